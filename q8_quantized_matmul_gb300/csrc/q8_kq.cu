// q8_kq.cu -- the second weight format: Q2_K / Q4_K rows against Q8_K activations.
//
// Blocks of 256 weights (ds4 pages: model-architecture page, quantisation
// section 3, "Block layout"; the routed experts of the GPU code walkthrough,
// trace 5, and the MoE page's Q4_K expert path use them), packed as GGML's
// k-quants:
//   Q2_K (84 bytes): scales[16] (scale low nibble, min high nibble, one per
//     16-weight sub-block), qs[64], d, dmin (binary16).  Weight
//     128h + 32j + 16s + l is 2-bit field j of qs[32h + 16s + l], sub-block
//     8h + 2j + s.
//   Q4_K (144 bytes): d, dmin, scales[12] (6-bit scale and min of eight
//     32-weight sub-blocks), qs[128].  Weight 64c + l is the low nibble of
//     qs[32c + l] (sub-block 2c), weight 64c + 32 + l its high nibble.
//   value = d * sc * q - dmin * m.
// Activations are Q8_K (the quantiser the pages print: fp32 d = amax / 127,
// q = roundf(x / d) per 256 values), kept as planes: quants [rows][in_dim],
// scales [rows][in_dim / 256] and the sums of each 16 quants [rows][in_dim / 16]
// (the min term needs them).
//
// The product (same page, section 4, fixed-point dot): per sub-block the exact
// integers isum = sum q_w q_x (dp4a) and xsum = sum q_x, then in fp32
// d_x * (d * (sc * isum) - dmin * (m * xsum)), summed over sub-blocks and blocks.
// One lane takes one sub-block: Q4_K 8 lanes per block (4 blocks a warp pass),
// Q2_K 16 lanes (2 blocks).  A warp owns a weight row, reads each block once for
// all tokens of its group, and reduces its lanes' sums at the row's end.
#include "q8_common.cuh"
#include "q8_kernels.h"

namespace q8 {

namespace kq {
constexpr int THREADS = 256;
constexpr int WARPS = THREADS / 32;
constexpr int QKK = 256;
}  // namespace kq

// ---------------------------------------------------------------- Q8_K quantiser
// One warp per 256-value block, lane l holding values 8l .. 8l + 7.  Writes the
// planes (qx, dx, xs) and/or the canonical 292-byte blocks (fp32 d, int8 qs[256],
// int16 sums of each 16 quants).
__global__ void __launch_bounds__(256) k_quantize_q8k(int8_t *__restrict__ qx, float *__restrict__ dx,
                                                      int16_t *__restrict__ xs, uint8_t *__restrict__ blocks,
                                                      const float *__restrict__ x, uint64_t in_dim, uint64_t n_rows) {
    const uint64_t nsb = in_dim / kq::QKK;
    const uint64_t n_blk = n_rows * nsb;
    const int lane = threadIdx.x & 31;
    const uint64_t warp0 = ((uint64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const uint64_t nwarps = ((uint64_t)gridDim.x * blockDim.x) >> 5;
    for (uint64_t blk = warp0; blk < n_blk; blk += nwarps) {
        const uint64_t row = blk / nsb, b = blk - row * nsb;
        const float4 *src = reinterpret_cast<const float4 *>(x + row * in_dim + b * kq::QKK + 8 * lane);
        const float4 a0 = src[0], a1 = src[1];
        const float v[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
        const float d = __fdiv_rn(amax, 127.0f);
        uint32_t w[2] = {0u, 0u};
        int s = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int q = d != 0.0f ? (int)roundf(__fdiv_rn(v[i], d)) : 0;
            s += q;
            w[i >> 2] |= (uint32_t)(q & 0xff) << (8 * (i & 3));
        }
        s += __shfl_xor_sync(0xffffffffu, s, 1);   // lanes 2g, 2g + 1: the sum of quants 16g .. 16g + 15
        if (qx) {
            *reinterpret_cast<uint2 *>(qx + row * in_dim + b * kq::QKK + 8 * lane) = make_uint2(w[0], w[1]);
            if (lane == 0) dx[blk] = d;
            if ((lane & 1) == 0) xs[row * (in_dim / 16) + b * 16 + (lane >> 1)] = (int16_t)s;
        }
        if (blocks) {
            uint8_t *o = blocks + blk * 292;
            if (lane == 0) *reinterpret_cast<float *>(o) = d;
            reinterpret_cast<uint32_t *>(o + 4)[2 * lane] = w[0];
            reinterpret_cast<uint32_t *>(o + 4)[2 * lane + 1] = w[1];
            if ((lane & 1) == 0) reinterpret_cast<int16_t *>(o + 260)[lane >> 1] = (int16_t)s;
        }
    }
}

cudaError_t launch_quantize_q8k(int8_t *qx, float *dx, int16_t *xs, uint8_t *blocks, const float *x, uint64_t in_dim,
                                uint64_t n_rows, int num_sms, cudaStream_t st) {
    const uint64_t n_blk = n_rows * (in_dim / kq::QKK);
    if (n_blk == 0) return cudaSuccess;
    uint64_t grid = (n_blk + kq::WARPS - 1) / kq::WARPS;
    const uint64_t cap = (uint64_t)num_sms * 8;
    if (grid > cap) grid = cap;
    k_quantize_q8k<<<(unsigned)grid, kq::THREADS, 0, st>>>(qx, dx, xs, blocks, x, in_dim, n_rows);
    return cudaGetLastError();
}

// ---------------------------------------------------------------- GEMV
struct KqItem {
    int expert;
    int ntok;
    int xrow0;       // routed: first plane row of the token group; dense: first token
    uint32_t r0, nrows;
};

template <int TOKG>
__device__ __forceinline__ bool kq_item(const KqParams &p, int i, KqItem &it) {
    const int n_rb = (int)((p.out_dim + p.rows_per_item - 1) / p.rows_per_item);
    if (!p.plan) {
        const int n_tg = (int)((p.n_tok + TOKG - 1) / TOKG);
        if (i >= n_rb * n_tg) return false;
        const int tg = i / n_rb, rb = i - tg * n_rb;
        it.expert = 0;
        it.xrow0 = tg * TOKG;
        it.ntok = min(TOKG, (int)p.n_tok - it.xrow0);
        it.r0 = (uint32_t)rb * p.rows_per_item;
        it.nrows = min(p.rows_per_item, p.out_dim - it.r0);
        return true;
    }
    if (i >= p.plan->n_items) return false;
    const Segment *segs = reinterpret_cast<const Segment *>(p.plan + 1);
    int lo = 0, hi = p.plan->n_segments - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (segs[mid].item_start <= i) lo = mid;
        else hi = mid - 1;
    }
    const Segment s = segs[lo];
    const int local = i - s.item_start;
    const int tg = local / n_rb, rb = local - tg * n_rb;
    it.expert = s.expert;
    it.ntok = min(TOKG, s.count - tg * TOKG);
    it.xrow0 = s.row0 + tg * TOKG;
    it.r0 = (uint32_t)rb * p.rows_per_item;
    it.nrows = min(p.rows_per_item, p.out_dim - it.r0);
    return true;
}

__device__ __forceinline__ float f16_bits(uint32_t h) { return __half2float(__ushort_as_half((unsigned short)(h & 0xffffu))); }

__device__ __forceinline__ uint32_t byte_of(uint32_t w0, uint32_t w1, uint32_t w2, int k) {
    const uint32_t w = k < 4 ? w0 : (k < 8 ? w1 : w2);
    return (w >> (8 * (k & 3))) & 0xffu;
}

// This lane's sub-block of one block: 8 (Q4_K) or 4 (Q2_K) words of quants,
// each byte one weight of the 4 activations in the matching word of x, with
// the sub-block's scale, min and the block's d and dmin.
template <int FMT> struct SubBlock {
    static constexpr int WORDS = FMT == KQ_Q4 ? 8 : 4;
    uint32_t q[WORDS];
    int sc, m;
    float d, dmin;
    uint32_t xoff;   // offset of the sub-block's first value within the block
    uint32_t grp;    // first 16-value group of the sub-block within the block
};

template <int FMT>
__device__ __forceinline__ void load_sub(SubBlock<FMT> &u, const uint8_t *blk, int sub) {
    if constexpr (FMT == KQ_Q4) {
        const uint4 h = __ldg(reinterpret_cast<const uint4 *>(blk));
        u.d = f16_bits(h.x);
        u.dmin = f16_bits(h.x >> 16);
        const int j = sub;
        if (j < 4) {
            u.sc = (int)(byte_of(h.y, h.z, h.w, j) & 63u);
            u.m = (int)(byte_of(h.y, h.z, h.w, j + 4) & 63u);
        } else {
            u.sc = (int)((byte_of(h.y, h.z, h.w, j + 4) & 15u) | ((byte_of(h.y, h.z, h.w, j - 4) >> 6) << 4));
            u.m = (int)((byte_of(h.y, h.z, h.w, j + 4) >> 4) | ((byte_of(h.y, h.z, h.w, j) >> 6) << 4));
        }
        const int c = j >> 1, hi = j & 1;
        const uint4 *qs = reinterpret_cast<const uint4 *>(blk + 16 + 32 * c);
        const uint4 a = __ldg(qs), b = __ldg(qs + 1);
        const uint32_t raw[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
        for (int k = 0; k < 8; ++k) u.q[k] = (raw[k] >> (4 * hi)) & 0x0f0f0f0fu;
        u.xoff = 64u * c + 32u * hi;
        u.grp = 4u * c + 2u * hi;
    } else {
        const int sb = sub, h = sb >> 3, j = (sb >> 1) & 3, s = sb & 1;
        const uint32_t sw = __ldg(reinterpret_cast<const uint32_t *>(blk) + (sb >> 2));
        const uint32_t sbyte = (sw >> (8 * (sb & 3))) & 0xffu;
        u.sc = (int)(sbyte & 15u);
        u.m = (int)(sbyte >> 4);
        const uint32_t dd = __ldg(reinterpret_cast<const uint32_t *>(blk + 80));
        u.d = f16_bits(dd);
        u.dmin = f16_bits(dd >> 16);
        const uint32_t *qs = reinterpret_cast<const uint32_t *>(blk + 16 + 32 * h + 16 * s);
#pragma unroll
        for (int k = 0; k < 4; ++k) u.q[k] = (__ldg(qs + k) >> (2 * j)) & 0x03030303u;
        u.xoff = 128u * h + 32u * j + 16u * s;
        u.grp = (uint32_t)sb;
    }
}

template <int FMT, int TOKG>
__global__ void __launch_bounds__(kq::THREADS) k_kq_gemv(const KqParams p) {
    constexpr int LPB = FMT == KQ_Q4 ? 8 : 16;   // lanes per block, one sub-block each
    constexpr int BPP = 32 / LPB;                 // blocks per warp pass
    constexpr int BB = FMT == KQ_Q4 ? 144 : 84;   // bytes per block
    using SB = SubBlock<FMT>;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int sub = lane % LPB, bsel = lane / LPB;
    const uint32_t nsb = p.nsb;
    const uint64_t row_bytes = (uint64_t)nsb * BB;
    const uint64_t in_dim = p.in_dim;
    KqItem it;
    for (int i = blockIdx.x; kq_item<TOKG>(p, i, it); i += gridDim.x) {
        int arow[TOKG], orow[TOKG];
#pragma unroll
        for (int t = 0; t < TOKG; ++t) {
            const bool on = t < it.ntok;
            arow[t] = !on ? 0 : (p.plan ? p.src_row[it.xrow0 + t] : it.xrow0 + t);
            orow[t] = !on ? -1 : (p.plan ? p.row_to_out[it.xrow0 + t] : it.xrow0 + t);
        }
        const uint8_t *wmat = p.W + (uint64_t)it.expert * p.expert_stride;
        for (uint32_t r = it.r0 + warp; r < it.r0 + it.nrows; r += kq::WARPS) {
            const uint8_t *wrow = wmat + (uint64_t)r * row_bytes;
            float acc[TOKG];
#pragma unroll
            for (int t = 0; t < TOKG; ++t) acc[t] = 0.0f;
            for (uint32_t b0 = 0; b0 < nsb; b0 += BPP) {
                const uint32_t b = b0 + bsel;
                if (b >= nsb) continue;
                SB u;
                load_sub<FMT>(u, wrow + (uint64_t)b * BB, sub);
#pragma unroll
                for (int t = 0; t < TOKG; ++t) {
                    if (t >= it.ntok) break;
                    const uint64_t xr = (uint64_t)arow[t];
                    const int8_t *xq = p.qx + xr * in_dim + (uint64_t)b * kq::QKK + u.xoff;
                    int isum = 0, xsum;
                    if constexpr (FMT == KQ_Q4) {
                        const uint4 xa = __ldg(reinterpret_cast<const uint4 *>(xq));
                        const uint4 xb = __ldg(reinterpret_cast<const uint4 *>(xq) + 1);
                        isum = __dp4a((int)u.q[0], (int)xa.x, isum);
                        isum = __dp4a((int)u.q[1], (int)xa.y, isum);
                        isum = __dp4a((int)u.q[2], (int)xa.z, isum);
                        isum = __dp4a((int)u.q[3], (int)xa.w, isum);
                        isum = __dp4a((int)u.q[4], (int)xb.x, isum);
                        isum = __dp4a((int)u.q[5], (int)xb.y, isum);
                        isum = __dp4a((int)u.q[6], (int)xb.z, isum);
                        isum = __dp4a((int)u.q[7], (int)xb.w, isum);
                        const uint32_t s2 = __ldg(reinterpret_cast<const uint32_t *>(
                            p.xs + xr * (in_dim / 16) + (uint64_t)b * 16 + u.grp));
                        xsum = (int)(int16_t)(s2 & 0xffffu) + (int)(int16_t)(s2 >> 16);
                    } else {
                        const uint4 xa = __ldg(reinterpret_cast<const uint4 *>(xq));
                        isum = __dp4a((int)u.q[0], (int)xa.x, isum);
                        isum = __dp4a((int)u.q[1], (int)xa.y, isum);
                        isum = __dp4a((int)u.q[2], (int)xa.z, isum);
                        isum = __dp4a((int)u.q[3], (int)xa.w, isum);
                        xsum = (int)__ldg(p.xs + xr * (in_dim / 16) + (uint64_t)b * 16 + u.grp);
                    }
                    const float dxv = __ldg(p.dx + xr * nsb + b);
                    acc[t] += dxv * (u.d * (float)(u.sc * isum) - u.dmin * (float)(u.m * xsum));
                }
            }
            float mine = 0.0f;
#pragma unroll
            for (int t = 0; t < TOKG; ++t) {
                if (t >= it.ntok) break;
                float v = acc[t];
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
                if (lane == t) mine = v;
            }
            if (lane < it.ntok) {
                int o = -1;
#pragma unroll
                for (int t = 0; t < TOKG; ++t)
                    if (t == lane) o = orow[t];
                if (o >= 0) p.out[(uint64_t)o * p.out_dim + r] = mine;
            }
        }
    }
}

cudaError_t launch_kq_gemv(const KqParams &p, int tokg, int num_sms, cudaStream_t st) {
    const int grid = num_sms * 2;   // two resident CTAs per SM (128 registers a thread)
    if (p.fmt == KQ_Q4) {
        if (tokg == 8) k_kq_gemv<KQ_Q4, 8><<<grid, kq::THREADS, 0, st>>>(p);
        else if (tokg == 16) k_kq_gemv<KQ_Q4, 16><<<grid, kq::THREADS, 0, st>>>(p);
        else return cudaErrorInvalidValue;
    } else if (p.fmt == KQ_Q2) {
        if (tokg == 8) k_kq_gemv<KQ_Q2, 8><<<grid, kq::THREADS, 0, st>>>(p);
        else if (tokg == 16) k_kq_gemv<KQ_Q2, 16><<<grid, kq::THREADS, 0, st>>>(p);
        else return cudaErrorInvalidValue;
    } else {
        return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace q8
