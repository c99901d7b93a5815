// q8_ffn.cu -- the elementwise steps of the routed expert FFN around the
// routed matmul (ds4 GPU code walkthrough, trace 5, ds4_gpu_routed_moe_one_tensor:
// gate and up projections of the selected experts, SwiGLU, down projection,
// weighted sum).  Both kernels are HBM-bound streams:
//
//   k_swiglu   mid = silu(min(gate, L)) * clamp(up, -L, L)  (MoE study page,
//              SwiGLU activation section; L = 0: no clamp), silu(g) = g / (1 + e^-g)
//              in fp32 with CUDA's expf and IEEE division.  12 bytes per value.
//   k_combine  out[t][o] = sum_j w[t*k+j] * y[t*k+j][o], slot order j = 0..k-1,
//              each product and sum rounded separately (no contraction), so the
//              result is the same on every run.  4(k+1) bytes per output value.
#include <cstdint>

#include "q8_common.cuh"
#include "q8_kernels.h"

namespace q8 {
namespace {

constexpr int FFN_THREADS = 256;

// n values; with ids, the values form rows of row_len (a multiple of 4) and a row
// whose pair has an expert id outside [0, n_expert) is written as zeros.
__global__ void __launch_bounds__(FFN_THREADS) k_swiglu(float *__restrict__ mid, const float *__restrict__ gate,
                                                       const float *__restrict__ up, uint64_t n, float limit,
                                                       const int32_t *__restrict__ ids, uint32_t n_expert,
                                                       uint64_t row_len) {
    const uint64_t n4 = n / 4;
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    const uint64_t tid = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (uint64_t i = tid; i < n4; i += stride) {
        const float4 g = reinterpret_cast<const float4 *>(gate)[i];
        const float4 u = reinterpret_cast<const float4 *>(up)[i];
        float4 m;
        m.x = swiglu1(g.x, u.x, limit);
        m.y = swiglu1(g.y, u.y, limit);
        m.z = swiglu1(g.z, u.z, limit);
        m.w = swiglu1(g.w, u.w, limit);
        if (ids) {
            const int32_t e = ids[(i * 4) / row_len];
            if (e < 0 || (uint32_t)e >= n_expert) m = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        }
        reinterpret_cast<float4 *>(mid)[i] = m;
    }
    // the last n % 4 values (only without ids: rows are multiples of 4 long)
    if (tid < n - n4 * 4) {
        const uint64_t i = n4 * 4 + tid;
        mid[i] = swiglu1(gate[i], up[i], limit);
    }
}

// Up to COMBINE_UNROLL experts per token: the rows' loads are all in flight at once
// (the loop's load-then-add took one memory round trip per expert: 6.0 us cold for
// 64 tokens x 6 experts x 4096).
constexpr int COMBINE_UNROLL = 8;

template <int V>
__global__ void __launch_bounds__(FFN_THREADS) k_combine(float *__restrict__ out, const float *__restrict__ y,
                                                        const float *__restrict__ w, uint64_t n_tok, uint32_t k,
                                                        uint64_t dim) {
    const uint64_t per_tok = dim / V;
    const uint64_t total = n_tok * per_tok;
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
        const uint64_t t = i / per_tok;
        const uint64_t o = (i - t * per_tok) * V;
        float acc[V];
#pragma unroll
        for (int v = 0; v < V; ++v) acc[v] = 0.0f;
        if (V == 4 && k <= COMBINE_UNROLL) {
            // every row load issued before the first use (one memory round trip, not k);
            // the products and sums in the same slot order
            float4 r[COMBINE_UNROLL];
            float wv[COMBINE_UNROLL];
#pragma unroll
            for (int j = 0; j < COMBINE_UNROLL; ++j)
                if ((uint32_t)j < k) {
                    const uint64_t p = t * k + (uint64_t)j;
                    wv[j] = w[p];
                    r[j] = *reinterpret_cast<const float4 *>(y + p * dim + o);
                }
#pragma unroll
            for (int j = 0; j < COMBINE_UNROLL; ++j)
                if ((uint32_t)j < k) {
                    acc[0] = __fadd_rn(acc[0], __fmul_rn(wv[j], r[j].x));
                    acc[1] = __fadd_rn(acc[1], __fmul_rn(wv[j], r[j].y));
                    acc[2] = __fadd_rn(acc[2], __fmul_rn(wv[j], r[j].z));
                    acc[3] = __fadd_rn(acc[3], __fmul_rn(wv[j], r[j].w));
                }
            *reinterpret_cast<float4 *>(out + t * dim + o) = make_float4(acc[0], acc[1], acc[2], acc[3]);
            continue;
        }
        for (uint32_t j = 0; j < k; ++j) {
            const uint64_t p = t * k + j;
            const float wj = w[p];
            const float *row = y + p * dim + o;
            if constexpr (V == 4) {
                const float4 r = *reinterpret_cast<const float4 *>(row);
                acc[0] = __fadd_rn(acc[0], __fmul_rn(wj, r.x));
                acc[1] = __fadd_rn(acc[1], __fmul_rn(wj, r.y));
                acc[2] = __fadd_rn(acc[2], __fmul_rn(wj, r.z));
                acc[3] = __fadd_rn(acc[3], __fmul_rn(wj, r.w));
            } else {
                acc[0] = __fadd_rn(acc[0], __fmul_rn(wj, row[0]));
            }
        }
        if constexpr (V == 4)
            *reinterpret_cast<float4 *>(out + t * dim + o) = make_float4(acc[0], acc[1], acc[2], acc[3]);
        else
            out[t * dim + o] = acc[0];
    }
}

int ffn_grid(uint64_t work, int num_sms) {
    const uint64_t blocks = (work + FFN_THREADS - 1) / FFN_THREADS;
    const uint64_t cap = (uint64_t)num_sms * 8;   // 8 resident 256-thread blocks per SM
    return (int)(blocks < 1 ? 1 : (blocks > cap ? cap : blocks));
}

}  // namespace

cudaError_t launch_swiglu(float *mid, const float *gate, const float *up, uint64_t n, float limit,
                          const int32_t *ids, uint32_t n_expert, uint64_t row_len, int num_sms, cudaStream_t st) {
    if (n == 0) return cudaSuccess;
    const uint64_t work = n / 4 > n % 4 ? n / 4 : n % 4;
    k_swiglu<<<ffn_grid(work, num_sms), FFN_THREADS, 0, st>>>(mid, gate, up, n, limit, ids, n_expert, row_len);
    return cudaGetLastError();
}

cudaError_t launch_combine(float *out, const float *y, const float *w, uint64_t n_tok, uint32_t k, uint64_t dim,
                           int num_sms, cudaStream_t st) {
    if (n_tok == 0 || dim == 0) return cudaSuccess;
    if (dim % 4 == 0)
        k_combine<4><<<ffn_grid(n_tok * dim / 4, num_sms), FFN_THREADS, 0, st>>>(out, y, w, n_tok, k, dim);
    else
        k_combine<1><<<ffn_grid(n_tok * dim, num_sms), FFN_THREADS, 0, st>>>(out, y, w, n_tok, k, dim);
    return cudaGetLastError();
}

}  // namespace q8
