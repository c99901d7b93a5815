// q8_quantize.cu -- activation quantiser kernels.
//
// The per-block arithmetic (quantize8) is in q8_quant.cuh.
//
// Thread mapping: four consecutive lanes own one block (eight values each,
// two 16-byte loads), the block maximum is two xor-shuffles away.  Work is
// memory bound (4 bytes read per value); grids are sized as a multiple of
// the SM count and loop over blocks.
#include <cuda.h>

#include "q8_common.cuh"
#include "q8_kernels.h"

#include "q8_quant.cuh"

namespace q8 {

// Canonical 34-byte blocks: xq[blk] for blk in [0, nblk), x read flat.
__global__ void __launch_bounds__(256) k_quantize_blocks(uint8_t *__restrict__ xq, const float *__restrict__ x,
                                                         uint64_t nblk) {
    const uint64_t lane_q = threadIdx.x & 3u;
    const uint64_t groups_per_cta = blockDim.x / 4;
    // Whole warps iterate together (the shuffles need all lanes): loop bound is per warp.
    for (uint64_t base = (uint64_t)blockIdx.x * groups_per_cta; base < nblk; base += (uint64_t)gridDim.x * groups_per_cta) {
        const uint64_t blk = base + threadIdx.x / 4;
        const bool live = blk < nblk;
        float x8[8];
        if (live) load8(x8, x + blk * QK + lane_q * 8);
        else {
#pragma unroll
            for (int i = 0; i < 8; ++i) x8[i] = 0.0f;
        }
        const QuantBlock r = quantize8(x8);
        if (live) {
            uint8_t *o = xq + blk * QB;
            if (lane_q == 0) *reinterpret_cast<uint16_t *>(o) = r.dh;
            uint16_t *qo = reinterpret_cast<uint16_t *>(o + 2 + lane_q * 8);
            qo[0] = (uint16_t)r.lo;
            qo[1] = (uint16_t)(r.lo >> 16);
            qo[2] = (uint16_t)r.hi;
            qo[3] = (uint16_t)(r.hi >> 16);
        }
    }
}

// Split planes for the matmul kernels: qplane [n_rows][in_dim] int8 and
// dplane [n_rows][nb] fp32 (the stored binary16 scale as fp32).  Output row r
// is quantised from x row src_row[r] when src_row is given (a negative entry
// gives a zero row), else from x row r when r < n_src, else it is zero.
// Four packed int8 -> two fp16x2 holding the same integers exactly (bytes 0, 1
// -> lo; 2, 3 -> hi): each byte biased to unsigned sits under the fp16 exponent
// of 1024 (1024 + q + 128), then 1152 is subtracted (exact; q = 0 gives +0, as
// the integer conversion does).
__device__ __forceinline__ void s8x4_to_f16x4(uint32_t w, uint32_t &lo, uint32_t &hi) {
    const uint32_t u = w ^ 0x80808080u;
    const uint32_t a = __byte_perm(u, 0x64646464u, 0x4140);
    const uint32_t b = __byte_perm(u, 0x64646464u, 0x4342);
    const uint32_t bias = 0x64806480u;   // fp16 (1152, 1152)
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(a), "r"(bias));
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(b), "r"(bias));
}

__device__ __forceinline__ void store_f16_quants(__half *dst, const QuantBlock &qb) {
    uint32_t h[4];
    s8x4_to_f16x4(qb.lo, h[0], h[1]);
    s8x4_to_f16x4(qb.hi, h[2], h[3]);
    *reinterpret_cast<uint4 *>(dst) = make_uint4(h[0], h[1], h[2], h[3]);
}

__global__ void __launch_bounds__(256, 8) k_quantize_planes(int8_t *__restrict__ qplane, float *__restrict__ dplane,
                                                         const float *__restrict__ x, uint64_t in_dim,
                                                         uint64_t n_rows, const int32_t *__restrict__ src_row,
                                                         uint64_t n_src) {
    // The matmul that follows only prefetches weights before it waits for this
    // grid to finish, so it may be scheduled now.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // when launched with programmatic serialisation: nothing is read or written
    // before the previous grid is done (it may still read the planes this kernel
    // rewrites); after a plain launch this returns at once
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const uint64_t nb = in_dim / QK;
    const uint64_t nblk = n_rows * nb;
    const uint64_t lane_q = threadIdx.x & 3u;
    const uint64_t groups_per_cta = blockDim.x / 4;
    for (uint64_t base = (uint64_t)blockIdx.x * groups_per_cta; base < nblk; base += (uint64_t)gridDim.x * groups_per_cta) {
        const uint64_t blk = base + threadIdx.x / 4;
        const bool live = blk < nblk;
        const uint64_t r = live ? blk / nb : 0;
        const uint64_t b = live ? blk - r * nb : 0;
        int64_t s = -1;
        if (live) s = src_row ? (int64_t)src_row[r] : (r < n_src ? (int64_t)r : -1);
        float x8[8];
        if (s >= 0) load8(x8, x + (uint64_t)s * in_dim + b * QK + lane_q * 8);
        else {
#pragma unroll
            for (int i = 0; i < 8; ++i) x8[i] = 0.0f;
        }
        const QuantBlock qb = quantize8(x8);
        if (live) {
            const uint32_t lo = qb.lo, hi = qb.hi;
            *reinterpret_cast<uint2 *>(qplane + r * in_dim + b * QK + lane_q * 8) = make_uint2(lo, hi);
            if (lane_q == 0) dplane[r * nb + b] = qb.d_stored;
        }
    }
}

// Routed pairs -> plane rows (see launch_quantize_pairs).  Same arithmetic and
// thread mapping as k_quantize_planes, over the pairs instead of the plane rows.
template <bool TC>
__global__ void __launch_bounds__(256) k_quantize_pairs(int8_t *__restrict__ qplane, float *__restrict__ dplane,
                                                        const float *__restrict__ x, uint64_t in_dim,
                                                        uint64_t n_pairs, uint32_t k, int x_per_pair,
                                                        const int32_t *__restrict__ dst_row,
                                                        __half *__restrict__ q16, float *__restrict__ dxT,
                                                        uint64_t n_ld, const PlanHeader *tc_plan) {
    // launched with programmatic serialisation: nothing is read before the previous grid is done
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // Only then may the matmul behind be scheduled: it reads the weights before its
    // own griddepcontrol.wait, and a kernel before this one may have written them.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const uint64_t tc_rows = TC ? (uint64_t)tc_plan->row_end : 0;
    const uint64_t nb = in_dim / QK;
    const uint64_t nblk = n_pairs * nb;
    const uint64_t lane_q = threadIdx.x & 3u;
    const uint64_t groups_per_cta = blockDim.x / 4;
    for (uint64_t base = (uint64_t)blockIdx.x * groups_per_cta; base < nblk; base += (uint64_t)gridDim.x * groups_per_cta) {
        const uint64_t blk = base + threadIdx.x / 4;
        const bool live = blk < nblk;
        const uint64_t pr = live ? blk / nb : 0;
        const uint64_t b = live ? blk - pr * nb : 0;
        const int64_t r = live ? (int64_t)dst_row[pr] : -1;
        float x8[8];
        if (r >= 0) load8(x8, x + (x_per_pair ? pr : pr / k) * in_dim + b * QK + lane_q * 8);
        else {
#pragma unroll
            for (int i = 0; i < 8; ++i) x8[i] = 0.0f;
        }
        const QuantBlock qb = quantize8(x8);
        if (r < 0) continue;   // bad id: no row (all lanes of the block agree)
        const uint64_t ru = (uint64_t)r;
        if (TC && ru < tc_rows) {
            store_f16_quants(q16 + ru * in_dim + b * QK + lane_q * 8, qb);
            if (lane_q == 0) dxT[b * n_ld + ru] = qb.d_stored;
        } else {
            const uint32_t lo = qb.lo, hi = qb.hi;
            *reinterpret_cast<uint2 *>(qplane + ru * in_dim + b * QK + lane_q * 8) = make_uint2(lo, hi);
            if (lane_q == 0) dplane[ru * nb + b] = qb.d_stored;
        }
    }
}

// Canonical blocks -> split planes (for pre-quantised activations).  One
// thread per (row, block); rows >= n_src are zero.
__global__ void __launch_bounds__(256) k_unpack_blocks(int8_t *__restrict__ qplane, float *__restrict__ dplane,
                                                       const uint8_t *__restrict__ xq, uint64_t in_dim,
                                                       uint64_t n_rows, uint64_t n_src) {
    const uint64_t nb = in_dim / QK;
    const uint64_t nblk = n_rows * nb;
    for (uint64_t blk = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; blk < nblk;
         blk += (uint64_t)gridDim.x * blockDim.x) {
        const uint64_t r = blk / nb, b = blk - r * nb;
        uint32_t w[8];
        float d = 0.0f;
        if (r < n_src) {
            const uint8_t *p = xq + blk * QB;   // same (row, block) index: xq is [n_src][nb]
            const uint16_t *p16 = reinterpret_cast<const uint16_t *>(p);
            d = half_bits_to_float(p16[0]);
#pragma unroll
            for (int i = 0; i < 8; ++i) w[i] = (uint32_t)p16[1 + 2 * i] | ((uint32_t)p16[2 + 2 * i] << 16);
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) w[i] = 0;
        }
        uint4 *o = reinterpret_cast<uint4 *>(qplane + r * in_dim + b * QK);
        o[0] = make_uint4(w[0], w[1], w[2], w[3]);
        o[1] = make_uint4(w[4], w[5], w[6], w[7]);
        dplane[blk] = d;
    }
}

// Prefill operand: fp16 quant plane q16 [n_ld][in_dim] (exact integers) and
// block-major scales dxT [nb][n_ld]; rows n_tok..n_ld-1 are zero.  Same
// arithmetic as the other quantiser kernels.
__global__ void __launch_bounds__(256) k_quantize_f16t(__half *__restrict__ q16, float *__restrict__ dxT,
                                                       const float *__restrict__ x, uint64_t in_dim, uint64_t n_tok,
                                                       uint64_t n_ld) {
    // launched with programmatic serialisation: nothing is read before the previous grid is done
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // Only then may the GEMM behind be scheduled: it reads these planes after its
    // griddepcontrol.wait, but the weights before it, and a kernel before this one
    // may have written them.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const uint64_t nb = in_dim / QK;
    const uint64_t nblk = n_ld * nb;
    const uint64_t lane_q = threadIdx.x & 3u;
    const uint64_t groups_per_cta = blockDim.x / 4;
    for (uint64_t base = (uint64_t)blockIdx.x * groups_per_cta; base < nblk; base += (uint64_t)gridDim.x * groups_per_cta) {
        const uint64_t blk = base + threadIdx.x / 4;
        const bool live = blk < nblk;
        const uint64_t r = live ? blk / nb : 0;
        const uint64_t b = live ? blk - r * nb : 0;
        float x8[8];
        if (live && r < n_tok) load8(x8, x + r * in_dim + b * QK + lane_q * 8);
        else {
#pragma unroll
            for (int i = 0; i < 8; ++i) x8[i] = 0.0f;
        }
        const QuantBlock qb = quantize8(x8);
        if (live) {
            store_f16_quants(q16 + r * in_dim + b * QK + lane_q * 8, qb);
            if (lane_q == 0) dxT[b * n_ld + r] = qb.d_stored;
        }
    }
}

// Canonical blocks [n_tok][nb] -> the prefill operand (as k_quantize_f16t).
__global__ void __launch_bounds__(256) k_unpack_f16t(__half *__restrict__ q16, float *__restrict__ dxT,
                                                     const uint8_t *__restrict__ xq, uint64_t in_dim, uint64_t n_tok,
                                                     uint64_t n_ld) {
    // launched with programmatic serialisation: nothing is read before the previous grid is done
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // Only then may the GEMM behind be scheduled: it reads these planes after its
    // griddepcontrol.wait, but the weights before it, and a kernel before this one
    // may have written them.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const uint64_t nb = in_dim / QK;
    const uint64_t nblk = n_ld * nb;
    for (uint64_t blk = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; blk < nblk;
         blk += (uint64_t)gridDim.x * blockDim.x) {
        const uint64_t r = blk / nb, b = blk - r * nb;
        uint4 *dst = reinterpret_cast<uint4 *>(q16 + r * in_dim + b * QK);
        if (r < n_tok) {
            const uint16_t *p16 = reinterpret_cast<const uint16_t *>(xq + blk * QB);
            dxT[b * n_ld + r] = half_bits_to_float(p16[0]);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t o[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const uint16_t two = p16[1 + c * 4 + e];
                    o[e] = (uint32_t)__half_as_ushort(__int2half_rn((int)(int8_t)(two & 0xff))) |
                           ((uint32_t)__half_as_ushort(__int2half_rn((int)(int8_t)(two >> 8))) << 16);
                }
                dst[c] = make_uint4(o[0], o[1], o[2], o[3]);
            }
        } else {
            dxT[b * n_ld + r] = 0.0f;
#pragma unroll
            for (int c = 0; c < 4; ++c) dst[c] = make_uint4(0, 0, 0, 0);
        }
    }
}

// RMSNorm feeding the quantiser: one CTA per token row (grid-stride over rows).
//   r = 1 / sqrt(mean_i x_i^2 + eps),  y_i = (x_i * r) * gamma_i,  xq = quantiser(y)
// The usual RMSNorm (the model's attn_norm / ffn_norm scales); the pages name the
// norm but print no formula.  The sum of squares runs in a fixed order -- each
// thread adds its own values in sequence (8 consecutive values per 2048-value
// stride), then a 5-level warp tree, then the 8 warps' sums in sequence -- so the
// result is the same on every run, and its relative error is at most
// (8 ceil(dim/2048) + 14) 2^-24.  Thread t's 8 values of a stride are lane
// (t & 3)'s part of block t/4, the quantiser's lane layout, so quantize8 applies
// unchanged: the quantised rows are the activation quantiser of the fp32 y.
constexpr int RMS_THREADS = 256;

__global__ void __launch_bounds__(RMS_THREADS) k_rmsnorm_quantize(uint8_t *__restrict__ xq, float *__restrict__ y,
                                                                 const float *__restrict__ x,
                                                                 const float *__restrict__ gamma, uint64_t dim,
                                                                 uint64_t n_tok, float eps) {
    __shared__ float part[RMS_THREADS / 32];
    __shared__ float r_sh;
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const uint64_t nb = dim / QK;
    const uint64_t lane_q = (uint64_t)(t & 3);
    for (uint64_t row = blockIdx.x; row < n_tok; row += gridDim.x) {
        const float *xr = x + row * dim;
        float s = 0.0f;
        for (uint64_t e = (uint64_t)t * 8; e < dim; e += RMS_THREADS * 8) {
            float x8[8];
            load8(x8, xr + e);
#pragma unroll
            for (int i = 0; i < 8; ++i) s = __fadd_rn(s, __fmul_rn(x8[i], x8[i]));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s = __fadd_rn(s, __shfl_xor_sync(0xffffffffu, s, o));
        if (lane == 0) part[warp] = s;
        __syncthreads();
        if (t == 0) {
            float tot = 0.0f;
            for (int w = 0; w < RMS_THREADS / 32; ++w) tot = __fadd_rn(tot, part[w]);
            r_sh = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(tot, (float)dim), eps)));
        }
        __syncthreads();
        const float r = r_sh;
        // whole CTA iterates together: the quantiser's shuffles need every lane
        for (uint64_t base = 0; base < dim; base += RMS_THREADS * 8) {
            const uint64_t e = base + (uint64_t)t * 8;
            const bool live = e < dim;
            float y8[8];
            if (live) {
                float x8[8], g8[8];
                load8(x8, xr + e);
                if (gamma) {
                    load8(g8, gamma + e);
                } else {
#pragma unroll
                    for (int i = 0; i < 8; ++i) g8[i] = 1.0f;
                }
#pragma unroll
                for (int i = 0; i < 8; ++i) y8[i] = __fmul_rn(__fmul_rn(x8[i], r), g8[i]);
                if (y) {
                    float4 *yo = reinterpret_cast<float4 *>(y + row * dim + e);
                    yo[0] = make_float4(y8[0], y8[1], y8[2], y8[3]);
                    yo[1] = make_float4(y8[4], y8[5], y8[6], y8[7]);
                }
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) y8[i] = 0.0f;
            }
            const QuantBlock qb = quantize8(y8);
            if (live) {
                uint8_t *o = xq + (row * nb + e / QK) * QB;
                if (lane_q == 0) *reinterpret_cast<uint16_t *>(o) = qb.dh;
                uint16_t *qo = reinterpret_cast<uint16_t *>(o + 2 + lane_q * 8);
                qo[0] = (uint16_t)qb.lo;
                qo[1] = (uint16_t)(qb.lo >> 16);
                qo[2] = (uint16_t)qb.hi;
                qo[3] = (uint16_t)(qb.hi >> 16);
            }
        }
        __syncthreads();   // part and r_sh are rewritten for the next row
    }
}

// The same operation, with the same arithmetic in the same order (bitwise the
// same results), for rows of at most NS * 2048 values: thread t keeps its values
// of the row (8 per 2048-value stride) and of gamma in registers, so x is read
// once, gamma once per CTA, and the next row's loads are issued before this row's
// reduction, keeping two rows in flight per CTA.
// MINB: CTAs per SM the register budget must allow (the kernel is bound by
// instruction issue and latency; 4 CTAs of 256 threads at 64 registers measured
// 25.2 us against 29.9 us at 3 CTAs for 4096 rows of 4096).
template <int NS, int MINB>
__global__ void __launch_bounds__(RMS_THREADS, MINB) k_rmsnorm_quantize_reg(uint8_t *__restrict__ xq, float *__restrict__ y,
                                                                     const float *__restrict__ x,
                                                                     const float *__restrict__ gamma, uint64_t dim,
                                                                     uint64_t n_tok, float eps) {
    __shared__ float part[RMS_THREADS / 32];
    __shared__ float r_sh;
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const uint64_t nb = dim / QK;
    const uint64_t lane_q = (uint64_t)(t & 3);
    float g[NS][8], xa[NS][8];
#pragma unroll
    for (int s = 0; s < NS; ++s) {
        const uint64_t e = (uint64_t)s * (RMS_THREADS * 8) + (uint64_t)t * 8;
        if (gamma && e < dim) {
            load8(g[s], gamma + e);
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) g[s][i] = 1.0f;
        }
    }
    // programmatic serialisation, as in the TMA-fed kernel: gamma before the wait,
    // dependents triggered when the CTA starts its last row
    asm volatile("griddepcontrol.wait;" ::: "memory");
    auto load_row = [&](float (&v)[NS][8], uint64_t row) {
#pragma unroll
        for (int s = 0; s < NS; ++s) {
            const uint64_t e = (uint64_t)s * (RMS_THREADS * 8) + (uint64_t)t * 8;
            if (row < n_tok && e < dim) {
                load8(v[s], x + row * dim + e);
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) v[s][i] = 0.0f;
            }
        }
    };
    load_row(xa, blockIdx.x);
    for (uint64_t row = blockIdx.x; row < n_tok; row += gridDim.x) {
        if (row + gridDim.x >= n_tok) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
        float xb[NS][8];
        load_row(xb, row + gridDim.x);   // the next row of this CTA, in flight meanwhile
        float sq = 0.0f;
#pragma unroll
        for (int s = 0; s < NS; ++s)
            if ((uint64_t)s * (RMS_THREADS * 8) + (uint64_t)t * 8 < dim) {
#pragma unroll
                for (int i = 0; i < 8; ++i) sq = __fadd_rn(sq, __fmul_rn(xa[s][i], xa[s][i]));
            }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sq = __fadd_rn(sq, __shfl_xor_sync(0xffffffffu, sq, o));
        if (lane == 0) part[warp] = sq;
        __syncthreads();
        if (t == 0) {
            float tot = 0.0f;
            for (int w = 0; w < RMS_THREADS / 32; ++w) tot = __fadd_rn(tot, part[w]);
            r_sh = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(tot, (float)dim), eps)));
        }
        __syncthreads();
        const float r = r_sh;
#pragma unroll
        for (int s = 0; s < NS; ++s) {
            const uint64_t e = (uint64_t)s * (RMS_THREADS * 8) + (uint64_t)t * 8;
            const bool live = e < dim;
            float y8[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) y8[i] = live ? __fmul_rn(__fmul_rn(xa[s][i], r), g[s][i]) : 0.0f;
            if (live && y) {
                float4 *yo = reinterpret_cast<float4 *>(y + row * dim + e);
                yo[0] = make_float4(y8[0], y8[1], y8[2], y8[3]);
                yo[1] = make_float4(y8[4], y8[5], y8[6], y8[7]);
            }
            const QuantBlock qb = quantize8(y8);   // every lane takes part: the block maximum is shuffled
            if (live) {
                uint8_t *o = xq + (row * nb + e / QK) * QB;
                if (lane_q == 0) *reinterpret_cast<uint16_t *>(o) = qb.dh;
                uint16_t *qo = reinterpret_cast<uint16_t *>(o + 2 + lane_q * 8);
                qo[0] = (uint16_t)qb.lo;
                qo[1] = (uint16_t)(qb.lo >> 16);
                qo[2] = (uint16_t)qb.hi;
                qo[3] = (uint16_t)(qb.hi >> 16);
            }
        }
#pragma unroll
        for (int s = 0; s < NS; ++s)
#pragma unroll
            for (int i = 0; i < 8; ++i) xa[s][i] = xb[s][i];
        __syncthreads();   // part and r_sh are rewritten for the next row
    }
}

// ------------------------------------------------------------------ RMSNorm, TMA-fed
// The same operation for rows of at most 4096 values, one lane per Q8_0 block.
// A CTA of T = 32 * ceil(nb / 32) threads takes one token row at a time (rows
// blockIdx.x, + gridDim.x, ...); thread t owns block t (the kernel is written for
// BPT blocks per thread, t, t + T, ...; two per thread for rows of 8192 held 2 CTAs
// of 205 registers per SM and ran 1.5x slower than the register kernel).  One TMA box brings a whole row into a ring of RMS_STAGES
// stages, so the CTA's next rows are in flight without holding registers.  The
// tensor map's 128-byte swizzle puts chunk j of block b at chunk j ^ (b & 7), so
// eight consecutive lanes reading chunk j of their own blocks hit eight different
// bank groups.  With a whole block in one lane, the block maximum needs no
// shuffles and the scale one division per block; one CTA barrier per row joins
// the warps' sums of squares.
// Sum of squares, in a fixed order: per thread, four accumulators over values
// 8c..8c+7 of each of its blocks in turn (fused multiply-adds), combined as
// (a0 + a1) + (a2 + a3); a 5-level warp tree; the warps' sums in sequence.  An x^2
// term meets at most 8 BPT + 2 + 5 + 3 = 18 roundings, inside the 8 ceil(dim/2048) + 14
// (at least 22) of the other kernels.
// y and the quantiser's decisions are computed exactly as there (the same
// products, quantize_block32 = quantize8's arithmetic), so the blocks are the
// activation quantiser of the kernel's own y.
constexpr int RMS_STAGES = 2;
constexpr int RMS_TMA_THREADS = 128;
constexpr uint32_t RMS_TMA_MAX_DIM = RMS_TMA_THREADS * QK;   // 4096: one block per lane

__device__ __forceinline__ void tma_load_blocks(void *dst, const CUtensorMap *map, int y, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
            "r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(y), "r"(smem_addr(bar))
        : "memory");
}

// The activation quantiser for one block held whole by one lane (v: its 32
// values in order): amax = max |v_i|, d = amax / 127 (IEEE), q_i = roundf(v_i / d)
// by quantize8's division-free test with the IEEE division where the test fails
// (so the same bytes as quantize8 and q8_quantize_act).  Returns the binary16
// scale; w: the quants packed, byte i of w[k] = q[4k + i].
// The test's threshold: qa = fl(v fl(1/d)) and fl(v / d) differ by at most
// (3u + u^2) 128 < 2.29e-5 (u = 2^-24, |v / d| <= 128), so |qa - k| < 0.5 - 3e-5
// keeps both in k's rounding interval.  A whole warp takes the slow branch when
// one of its lanes needs it, 32 blocks at a time: the tighter margin than
// quantize8's 1e-4 cuts that from about one warp-block in five to one in sixteen.
constexpr float RMS_TIE_TEST = 0.49997f;
__device__ __forceinline__ uint16_t quantize_block32(const float (&v)[32], uint32_t (&w)[8]) {
    float m[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int i = 0; i < 32; ++i) m[i & 3] = fmaxf(m[i & 3], fabsf(v[i]));
    const float amax = fmaxf(fmaxf(m[0], m[1]), fmaxf(m[2], m[3]));
    const float d = __fdiv_rn(amax, 127.0f);
    if (d == 0.0f) {
#pragma unroll
        for (int k = 0; k < 8; ++k) w[k] = 0u;
        return 0;
    }
    const float rd = __frcp_rn(d);   // inf for a subnormal d: every value then fails the test
    bool bad = false;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        uint32_t t[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float qa = __fmul_rn(v[4 * k + j], rd);
            const float sm = __fadd_rn(qa, ROUND_MAGIC);
            t[j] = __float_as_uint(sm);
            bad |= !(fabsf(__fsub_rn(qa, __fsub_rn(sm, ROUND_MAGIC))) < RMS_TIE_TEST);
        }
        w[k] = __byte_perm(__byte_perm(t[0], t[1], 0x0040), __byte_perm(t[2], t[3], 0x0040), 0x5410);
    }
    if (bad) {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const float qa = __fmul_rn(v[i], rd);
            const float sm = __fadd_rn(qa, ROUND_MAGIC);
            if (!(fabsf(__fsub_rn(qa, __fsub_rn(sm, ROUND_MAGIC))) < RMS_TIE_TEST)) {
                const uint32_t q = (uint32_t)(uint8_t)(int8_t)(int)roundf(__fdiv_rn(v[i], d));
                const int sh = 8 * (i & 3);
                w[i >> 2] = (w[i >> 2] & ~(0xffu << sh)) | (q << sh);
            }
        }
    }
    return __half_as_ushort(__float2half_rn(d));
}

// A quantised row staged in shared memory goes out in 16-byte stores when its
// global start is 16-byte aligned, else in 2-byte stores (coalesced either way:
// one lane per block wrote 34-byte strides, two bytes at a time).
__device__ __forceinline__ void store_row_out(uint8_t *dst, const uint8_t *src, uint32_t bytes, uint32_t t,
                                              uint32_t T) {
    if ((reinterpret_cast<uintptr_t>(dst) & 15u) == 0 && (bytes & 15u) == 0) {
        for (uint32_t c = t; c < bytes / 16; c += T)
            reinterpret_cast<uint4 *>(dst)[c] = reinterpret_cast<const uint4 *>(src)[c];
    } else {
        for (uint32_t c = t; c < bytes / 2; c += T)
            reinterpret_cast<uint16_t *>(dst)[c] = reinterpret_cast<const uint16_t *>(src)[c];
    }
}

template <int BPT, int MINB>
__global__ void __launch_bounds__(RMS_TMA_THREADS, MINB)
    k_rmsnorm_quantize_tma(const __grid_constant__ CUtensorMap xmap, uint8_t *__restrict__ xq, float *__restrict__ y,
                           const float *__restrict__ gamma, uint32_t dim, uint64_t n_tok, float eps, int *err,
                           uint64_t wait_ns, int withhold) {
    extern __shared__ uint8_t rms_dyn[];
    __shared__ uint64_t full[RMS_STAGES];
    __shared__ float part[2][RMS_TMA_THREADS / 32];
    __shared__ int abort_flag;
    const uint32_t T = blockDim.x, t = threadIdx.x, lane = t & 31u, warp = t >> 5, W = T >> 5;
    const uint32_t nb = dim / QK;
    const uint32_t stage_bytes = (nb * 128u + 1023u) & ~1023u;
    uint8_t *ring = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(rms_dyn) + 1023) & ~(uintptr_t)1023);
    const uint32_t row_out = nb * QB;                       // bytes of a quantised row
    const uint32_t out_stride = (row_out + 15u) & ~15u;
    uint8_t *outs = ring + RMS_STAGES * stage_bytes;       // two staged output rows
    const uint64_t G = gridDim.x;
    uint32_t issued = 0, par = 0;   // thread 0: stages with a copy not yet consumed, and its phase parity
    const uint64_t lim = wait_limit(wait_ns);
    if (t == 0) {
        for (int s = 0; s < RMS_STAGES; ++s) mbar_init(&full[s], 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    float g[BPT][32];
#pragma unroll
    for (int bl = 0; bl < BPT; ++bl) {
        const uint32_t bi = t + (uint32_t)bl * T;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            float4 q4 = make_float4(1.0f, 1.0f, 1.0f, 1.0f);
            if (gamma && bi < nb) q4 = __ldg(reinterpret_cast<const float4 *>(gamma + (size_t)bi * QK) + c);
            g[bl][4 * c] = q4.x; g[bl][4 * c + 1] = q4.y; g[bl][4 * c + 2] = q4.z; g[bl][4 * c + 3] = q4.w;
        }
    }
    // Launched with programmatic serialisation: the barrier set-up and gamma (which no
    // kernel that triggers early writes) overlap the preceding kernel's end; x is read
    // and xq written only after it is complete.  A CTA triggers its dependents once it
    // has issued its last row copy (4096 x 4096: 20.5 -> 19.8 us in graphs of calls).
    asm volatile("griddepcontrol.wait;" ::: "memory");
    bool trig = false;
    if (t == 0) {
        for (uint32_t s = 0; s < (uint32_t)RMS_STAGES && !withhold; ++s) {
            const uint64_t row = blockIdx.x + s * G;
            if (row < n_tok) {
                mbar_arrive_expect_tx(&full[s], nb * 128u);
                tma_load_blocks(ring + s * stage_bytes, &xmap, (int)(row * nb), &full[s]);
                issued |= 1u << s;
            }
        }
        if (blockIdx.x + (uint64_t)RMS_STAGES * G >= n_tok) {
            asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
            trig = true;
        }
    }
    __syncthreads();
    uint32_t i = 0;
    for (uint64_t row = blockIdx.x; row < n_tok; row += G, ++i) {
        const uint32_t s = i % RMS_STAGES, ph = (i / RMS_STAGES) & 1u;
        const bool ok = mbar_wait(&full[s], ph, err, &abort_flag, lim);
        const uint8_t *st = ring + s * stage_bytes;
        float v[BPT][32];
        float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int bl = 0; bl < BPT; ++bl) {
            const uint32_t bi = t + (uint32_t)bl * T;
            const bool live = ok && bi < nb;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                float4 c4 = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                if (live) c4 = *reinterpret_cast<const float4 *>(st + bi * 128u + (((uint32_t)j ^ (bi & 7u)) << 4));
                v[bl][4 * j] = c4.x; v[bl][4 * j + 1] = c4.y; v[bl][4 * j + 2] = c4.z; v[bl][4 * j + 3] = c4.w;
            }
#pragma unroll
            for (int c = 0; c < 4; ++c)
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    acc[c] = __fmaf_rn(v[bl][8 * c + e], v[bl][8 * c + e], acc[c]);
        }
        float sq = __fadd_rn(__fadd_rn(acc[0], acc[1]), __fadd_rn(acc[2], acc[3]));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sq = __fadd_rn(sq, __shfl_xor_sync(0xffffffffu, sq, o));
        if (lane == 0) part[i & 1u][warp] = sq;
        // every thread has read stage s and written its warp's sum (part is double-buffered
        // by row parity: the next row's writes cannot meet this row's reads)
        if (__syncthreads_or(!ok)) break;
        if (t == 0) {
            issued &= ~(1u << s);
            const uint64_t nrow = row + (uint64_t)RMS_STAGES * G;
            if (nrow < n_tok) {
                mbar_arrive_expect_tx(&full[s], nb * 128u);
                tma_load_blocks(ring + s * stage_bytes, &xmap, (int)(nrow * nb), &full[s]);
                issued |= 1u << s;
                par = (par & ~(1u << s)) | ((((i + RMS_STAGES) / RMS_STAGES) & 1u) << s);
            } else if (!trig) {
                asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
                trig = true;
            }
        }
        if (i > 0) store_row_out(xq + (row - G) * row_out, outs + ((i - 1) & 1u) * out_stride, row_out, t, T);
        float tot = 0.0f;
        for (uint32_t w = 0; w < W; ++w) tot = __fadd_rn(tot, part[i & 1u][w]);
        const float r = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(tot, (float)dim), eps)));
#pragma unroll
        for (int bl = 0; bl < BPT; ++bl) {
            const uint32_t bi = t + (uint32_t)bl * T;
            if (bi < nb) {
                float yv[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) yv[e] = __fmul_rn(__fmul_rn(v[bl][e], r), g[bl][e]);
                if (y) {
                    float4 *yo = reinterpret_cast<float4 *>(y + row * dim + (size_t)bi * QK);
#pragma unroll
                    for (int c = 0; c < 8; ++c) yo[c] = make_float4(yv[4 * c], yv[4 * c + 1], yv[4 * c + 2], yv[4 * c + 3]);
                }
                uint32_t w8[8];
                const uint16_t dh = quantize_block32(yv, w8);
                uint16_t *o = reinterpret_cast<uint16_t *>(outs + (i & 1u) * out_stride + bi * QB);
                o[0] = dh;
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    o[1 + 2 * k] = (uint16_t)w8[k];
                    o[2 + 2 * k] = (uint16_t)(w8[k] >> 16);
                }
            }
        }
    }
    // The CTA's last row (the loop ran to its end: i rows, none aborted).
    __syncthreads();
    if (i > 0 && !abort_flag) {
        const uint64_t last = blockIdx.x + (uint64_t)(i - 1) * G;
        if (last < n_tok) store_row_out(xq + last * row_out, outs + ((i - 1) & 1u) * out_stride, row_out, t, T);
    }
    // After an expired wait: let the copies still in flight land before the CTA's
    // shared memory goes away (each stage has at most one, the last issued on it).
    if (t == 0 && issued) {
        const uint64_t t_end = global_timer_ns() + WAIT_LIMIT_NS;
        for (uint32_t s = 0; s < (uint32_t)RMS_STAGES; ++s)
            if (issued & (1u << s)) mbar_drain(&full[s], (par >> s) & 1u, t_end);
    }
}

// ------------------------------------------------------------------ launchers
// Launch behind the previous kernel with programmatic serialisation: the
// launch overlaps that kernel's drain; the kernel waits for it in
// griddepcontrol.wait before reading anything.
template <class K, class... Args>
static cudaError_t launch_pdl(K kernel, int grid, int block, cudaStream_t st, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3((unsigned)block);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, args...);
    return e != cudaSuccess ? e : cudaGetLastError();
}

template <class K, class... Args>
static cudaError_t launch_pdl_smem(K kernel, int grid, int block, size_t smem, cudaStream_t st, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3((unsigned)block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, args...);
    return e != cudaSuccess ? e : cudaGetLastError();
}

static int grid_for(uint64_t work_items, int per_cta, int num_sms) {
    uint64_t need = (work_items + per_cta - 1) / per_cta;
    uint64_t cap = (uint64_t)num_sms * 8;
    if (need > cap) need = cap;
    return need ? (int)need : 1;
}

cudaError_t launch_quantize_blocks(uint8_t *xq, const float *x, uint64_t nblk, int num_sms, cudaStream_t st) {
    if (nblk == 0) return cudaSuccess;
    k_quantize_blocks<<<grid_for(nblk, 64, num_sms), 256, 0, st>>>(xq, x, nblk);
    return cudaGetLastError();
}

cudaError_t launch_quantize_planes(int8_t *qplane, float *dplane, const float *x, uint64_t in_dim, uint64_t n_rows,
                                   const int32_t *src_row, uint64_t n_src, int num_sms, cudaStream_t st,
                                   bool programmatic) {
    const uint64_t nblk = n_rows * (in_dim / QK);
    if (nblk == 0) return cudaSuccess;
    // Small inputs (the GEMV's 9-16 tokens) in CTAs of 128 threads at <= 32
    // registers (4096 registers): one fits on an SM beside a GEMV CTA (61,440
    // registers, 218 KB of shared memory).
    const int threads = nblk <= (uint64_t)num_sms * 32 ? 128 : 256;
    const int grid = grid_for(nblk, threads / 4, num_sms);
    // Behind a GEMV whose results cross the host link, a programmatic launch lets
    // this kernel sit beside that GEMV's CTAs while its writes drain, and the next
    // GEMV start its weight stream meanwhile (host-buffer calls at out 32768: 4
    // tokens 16.4 -> 13.9 us, 16 tokens 24.5 -> 21.7 us).  Between device-buffer
    // calls the plain launch measured faster (16-token calls back to back in a
    // graph 13.4 against 14.7 us).
    if (programmatic)
        return launch_pdl(k_quantize_planes, grid, threads, st, qplane, dplane, x, in_dim, n_rows, src_row, n_src);
    k_quantize_planes<<<grid, threads, 0, st>>>(qplane, dplane, x, in_dim, n_rows, src_row, n_src);
    return cudaGetLastError();
}

cudaError_t launch_quantize_f16t(__half *q16, float *dxT, const float *x, uint64_t in_dim, uint64_t n_tok,
                                 uint64_t n_ld, int num_sms, cudaStream_t st) {
    const uint64_t nblk = n_ld * (in_dim / QK);
    if (nblk == 0) return cudaSuccess;
    return launch_pdl(k_quantize_f16t, grid_for(nblk, 64, num_sms), 256, st, q16, dxT, x, in_dim, n_tok, n_ld);
}

cudaError_t launch_unpack_f16t(__half *q16, float *dxT, const uint8_t *xq, uint64_t in_dim, uint64_t n_tok,
                               uint64_t n_ld, int num_sms, cudaStream_t st) {
    const uint64_t nblk = n_ld * (in_dim / QK);
    if (nblk == 0) return cudaSuccess;
    return launch_pdl(k_unpack_f16t, grid_for(nblk, 256, num_sms), 256, st, q16, dxT, xq, in_dim, n_tok, n_ld);
}

cudaError_t launch_unpack_blocks(int8_t *qplane, float *dplane, const uint8_t *xq, uint64_t in_dim, uint64_t n_rows,
                                 uint64_t n_src, int num_sms, cudaStream_t st) {
    const uint64_t nblk = n_rows * (in_dim / QK);
    if (nblk == 0) return cudaSuccess;
    k_unpack_blocks<<<grid_for(nblk, 256, num_sms), 256, 0, st>>>(qplane, dplane, xq, in_dim, n_rows, n_src);
    return cudaGetLastError();
}

cudaError_t launch_quantize_pairs(int8_t *qplane, float *dplane, __half *q16, float *dxT, uint64_t n_ld,
                                  const PlanHeader *tc_plan, const float *x, uint64_t in_dim, uint64_t n_pairs,
                                  uint32_t k, int x_per_pair, const int32_t *dst_row, int num_sms, cudaStream_t st) {
    const uint64_t nblk = n_pairs * (in_dim / QK);
    if (nblk == 0) return cudaSuccess;
    const int grid = grid_for(nblk, 64, num_sms);
    if (tc_plan)
        return launch_pdl(k_quantize_pairs<true>, grid, 256, st, qplane, dplane, x, in_dim, n_pairs, k, x_per_pair,
                          dst_row, q16, dxT, n_ld, tc_plan);
    return launch_pdl(k_quantize_pairs<false>, grid, 256, st, qplane, dplane, x, in_dim, n_pairs, k, x_per_pair,
                      dst_row, (__half *)nullptr, (float *)nullptr, (uint64_t)0, (const PlanHeader *)nullptr);
}

template <int NS, int MINB>
static cudaError_t launch_rms_reg(uint8_t *xq, float *y, const float *x, const float *gamma, uint64_t dim,
                                  uint64_t n_tok, float eps, int num_sms, cudaStream_t st) {
    int per_sm = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_rmsnorm_quantize_reg<NS, MINB>,
                                                                  RMS_THREADS, 0);
    if (e != cudaSuccess) return e;
    const uint64_t cap = (uint64_t)num_sms * (uint64_t)(per_sm > 0 ? per_sm : 1);
    const int grid = (int)(n_tok < cap ? n_tok : cap);
    return launch_pdl(k_rmsnorm_quantize_reg<NS, MINB>, grid, RMS_THREADS, st, xq, y, x, gamma, dim, n_tok, eps);
}

bool encode_blocks_tmap(CUtensorMap *map, const float *x, uint64_t n_blocks, uint32_t box_blocks);

template <int BPT, int MINB>
static cudaError_t launch_rms_tma(const CUtensorMap &map, uint8_t *xq, float *y, const float *gamma, uint32_t dim,
                                  uint64_t n_tok, float eps, int *err, uint64_t wait_ns, int withhold, int num_sms,
                                  cudaStream_t st) {
    const uint32_t nb = dim / QK;
    const uint32_t warps = (nb + 31) / 32 < 4 ? (nb + 31) / 32 : 4;
    const int threads = (int)(32 * warps);
    const size_t smem = 1024 + (size_t)RMS_STAGES * ((nb * 128u + 1023u) & ~1023u) + 2 * ((nb * QB + 15u) & ~15u);
    auto k = k_rmsnorm_quantize_tma<BPT, MINB>;
    // the attribute once, at the largest size a call can ask for (rows of RMS_TMA_MAX_DIM);
    // the library's entry points run under one lock
    static bool attr_done = false;
    cudaError_t e;
    if (!attr_done) {
        const size_t smax = 1024 + (size_t)RMS_STAGES * (RMS_TMA_MAX_DIM / QK) * 128u +
                            2 * (((RMS_TMA_MAX_DIM / QK) * QB + 15u) & ~15u);
        e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smax);
        if (e != cudaSuccess) return e;
        attr_done = true;
    }
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, threads, smem);
    if (e != cudaSuccess) return e;
    const uint64_t cap = (uint64_t)num_sms * (uint64_t)(per_sm > 0 ? per_sm : 1);
    const int grid = (int)(n_tok < cap ? n_tok : cap);
    return launch_pdl_smem(k, grid, threads, smem, st, map, xq, y, gamma, dim, n_tok, eps, err, wait_ns, withhold);
}

bool rmsnorm_uses_tma(uint64_t dim, uint64_t n_tok, int num_sms) {
    return dim <= RMS_TMA_MAX_DIM && n_tok >= 12 * (uint64_t)num_sms && n_tok * (dim / QK) < (1ull << 31);
}

cudaError_t launch_rmsnorm_quantize(uint8_t *xq, float *y, const float *x, const float *gamma, uint64_t dim,
                                    uint64_t n_tok, float eps, int *err, uint64_t wait_ns, int withhold, int num_sms,
                                    cudaStream_t st) {
    if (n_tok == 0) return cudaSuccess;
    // Rows of up to 4096 values, at least three per CTA (four CTAs per SM): the
    // TMA-fed kernel, one lane per block.  It streams faster (4096 rows of 4096:
    // 20.3 against 21.5 us; of 1024: 8.6 against 9.9 us), but its chain per row is
    // longer, and with fewer rows the register kernel finishes first (1216 rows of
    // 4096: 8.7 against 9.8 us; 64 rows: 3.4 against 4.1 us).
    const uint64_t nb = dim / QK;
    CUtensorMap map;
    if (rmsnorm_uses_tma(dim, n_tok, num_sms) && encode_blocks_tmap(&map, x, n_tok * nb, (uint32_t)nb))
        return launch_rms_tma<1, 4>(map, xq, y, gamma, (uint32_t)dim, n_tok, eps, err, wait_ns, withhold, num_sms,
                                    st);
    // rows of up to 8192 values stay in registers; longer rows are read twice
    if (dim <= RMS_THREADS * 8) return launch_rms_reg<1, 4>(xq, y, x, gamma, dim, n_tok, eps, num_sms, st);
    if (dim <= 2 * RMS_THREADS * 8) return launch_rms_reg<2, 4>(xq, y, x, gamma, dim, n_tok, eps, num_sms, st);
    if (dim <= 4 * RMS_THREADS * 8) return launch_rms_reg<4, 2>(xq, y, x, gamma, dim, n_tok, eps, num_sms, st);
    const uint64_t cap = (uint64_t)num_sms * 8;
    const int grid = (int)(n_tok < cap ? n_tok : cap);
    k_rmsnorm_quantize<<<grid, RMS_THREADS, 0, st>>>(xq, y, x, gamma, dim, n_tok, eps);
    return cudaGetLastError();
}

}  // namespace q8
