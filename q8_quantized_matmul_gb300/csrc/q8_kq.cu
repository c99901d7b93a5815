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
// d_x * ((d * sc) * isum - (dmin * m) * xsum) (d * sc and dmin * m are exact in
// fp32), summed over sub-blocks and blocks.
// One lane takes two sub-blocks of a block, whose scaled integer sums it adds
// exactly before the fp32 step: Q4_K 4 lanes per block (8 blocks a warp pass),
// Q2_K 8 lanes (4 blocks).  A warp reads each block once for all tokens of its
// group and reduces its lanes' sums at the row's end.  In the streaming kernel a
// warp owns two weight rows of an item, so each activation load from shared
// memory (the limit there) serves two rows; in the direct kernel, one row.
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

// Work items are dealt to the CTAs in turn (item i to CTA i mod grid): routed
// items are ordered by the experts' pair counts, so contiguous ranges would give
// the first CTAs all the widest token groups.  The routing plan's segment table
// is searched per item; CTAs copy it to shared memory when it fits.
constexpr int KQ_SEG_CACHE = 1024;

struct KqSegs {
    const Segment *segs;   // shared-memory copy, or the plan's own table
    int nseg, n_items;
};

template <int TOKG>
__device__ __forceinline__ bool kq_item_at(const KqParams &p, const KqSegs &sg, int i, KqItem &it) {
    const int n_rb = (int)((p.out_dim + p.rows_per_item - 1) / p.rows_per_item);
    if (!p.plan) {
        if (i >= n_rb * (int)((p.n_tok + TOKG - 1) / TOKG)) return false;
        const int tg = i / n_rb, rb = i - tg * n_rb;
        it.expert = 0;
        it.xrow0 = tg * TOKG;
        it.ntok = min(TOKG, (int)p.n_tok - it.xrow0);
        it.r0 = (uint32_t)rb * p.rows_per_item;
        it.nrows = min(p.rows_per_item, p.out_dim - it.r0);
        return true;
    }
    if (i >= sg.n_items) return false;
    int lo = 0, hi = sg.nseg - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (sg.segs[mid].item_start <= i) lo = mid;
        else hi = mid - 1;
    }
    const Segment s = sg.segs[lo];
    const int local = i - s.item_start;
    const int tg = local / n_rb, rb = local - tg * n_rb;
    it.expert = s.expert;
    it.ntok = min(TOKG, s.count - tg * TOKG);
    it.xrow0 = s.row0 + tg * TOKG;
    it.r0 = (uint32_t)rb * p.rows_per_item;
    it.nrows = min(p.rows_per_item, p.out_dim - it.r0);
    return true;
}

// The segment table for kq_item_at: copied into cache (KQ_SEG_CACHE entries of
// shared memory) by threads [0, nthreads) when it fits; the caller synchronises
// those threads before the first lookup.
__device__ __forceinline__ KqSegs kq_segs(const KqParams &p, Segment *cache, int tid, int nthreads) {
    KqSegs sg{nullptr, 0, 0};
    if (!p.plan) return sg;
    const Segment *g = reinterpret_cast<const Segment *>(p.plan + 1);
    sg.nseg = p.plan->n_segments;
    sg.n_items = p.plan->n_items;
    if (sg.nseg <= KQ_SEG_CACHE) {
        for (int e = tid; e < sg.nseg; e += nthreads) cache[e] = g[e];
        sg.segs = cache;
    } else {
        sg.segs = g;
    }
    return sg;
}

__device__ __forceinline__ float f16_bits(uint32_t h) { return __half2float(__ushort_as_half((unsigned short)(h & 0xffffu))); }

// This lane's unit of one block: two sub-blocks.  Q4_K: chunk c (4 units a
// block), the low and high nibbles of qs[32c .. 32c + 31], sub-blocks 2c and
// 2c + 1, weights 64c .. 64c + 63.  Q2_K: unit 4h + j (8 units a block), field j
// of qs[32h .. 32h + 31], sub-blocks 8h + 2j and 8h + 2j + 1, weights
// 128h + 32j .. + 31.  q holds the weights one per byte (each word meets the
// matching word of the activations), the first sub-block's words first.  The
// two sub-blocks' scaled integer sums are combined exactly before the fp32 step.
template <int FMT> struct Unit {
    static constexpr int NW = FMT == KQ_Q4 ? 16 : 8;
    uint32_t q[NW];
    int sc0, sc1, m0, m1;
    float d, dmin;
};

// The words of a block this lane's unit needs, as loaded (all loads of a row's
// passes are issued before any is decoded).
template <int FMT> struct RawUnit {
    static constexpr int N = FMT == KQ_Q4 ? 12 : 10;
    uint32_t w[N];
};

template <int FMT> __host__ __device__ constexpr int units_per_block() { return FMT == KQ_Q4 ? 4 : 8; }

// Offsets of a unit within its block: its first activation value and first
// 16-value group of activation sums.
template <int FMT> __device__ __forceinline__ uint32_t unit_xoff(int u) {
    return FMT == KQ_Q4 ? 64u * (uint32_t)u : 128u * (uint32_t)(u >> 2) + 32u * (uint32_t)(u & 3);
}
template <int FMT> __device__ __forceinline__ uint32_t unit_grp(int u) {
    return FMT == KQ_Q4 ? 4u * (uint32_t)u : 8u * (uint32_t)(u >> 2) + 2u * (uint32_t)(u & 3);
}

// SMEM: the block lies in shared memory (plain loads; the read-only global
// path must not be used on shared addresses).
template <int FMT, bool SMEM>
__device__ __forceinline__ void load_raw(RawUnit<FMT> &r, const uint8_t *blk, int u) {
    auto ld4 = [](const uint32_t *p) { return SMEM ? *p : __ldg(p); };
    auto ld16 = [](const uint4 *p) { return SMEM ? *p : __ldg(p); };
    if constexpr (FMT == KQ_Q4) {
        const uint4 h = ld16(reinterpret_cast<const uint4 *>(blk));        // d, dmin, scales[12]
        const uint4 *qs = reinterpret_cast<const uint4 *>(blk + 16 + 32 * u);
        const uint4 a = ld16(qs), b = ld16(qs + 1);
        r.w[0] = h.x; r.w[1] = h.y; r.w[2] = h.z; r.w[3] = h.w;
        r.w[4] = a.x; r.w[5] = a.y; r.w[6] = a.z; r.w[7] = a.w;
        r.w[8] = b.x; r.w[9] = b.y; r.w[10] = b.z; r.w[11] = b.w;
    } else {   // Q2_K blocks are 4-byte aligned only
        const int h = u >> 2, j = u & 3;
        const uint32_t *qs = reinterpret_cast<const uint32_t *>(blk + 16 + 32 * h);
#pragma unroll
        for (int k = 0; k < 8; ++k) r.w[k] = ld4(qs + k);
        r.w[8] = ld4(reinterpret_cast<const uint32_t *>(blk) + 2 * h + (j >> 1));   // scales of 8h+2j, +1
        r.w[9] = ld4(reinterpret_cast<const uint32_t *>(blk + 80));                  // d, dmin
    }
}

template <int FMT>
__device__ __forceinline__ void decode_unit(Unit<FMT> &v, const RawUnit<FMT> &r, int u) {
    if constexpr (FMT == KQ_Q4) {
        v.d = f16_bits(r.w[0]);
        v.dmin = f16_bits(r.w[0] >> 16);
        // scales[0..3] in w[1], [4..7] in w[2], [8..11] in w[3]; sub-blocks 2u, 2u + 1
        const uint32_t sh0 = 8u * (uint32_t)((2 * u) & 3), sh1 = sh0 + 8u;
        if (u < 2) {
            v.sc0 = (int)((r.w[1] >> sh0) & 63u);
            v.sc1 = (int)((r.w[1] >> sh1) & 63u);
            v.m0 = (int)((r.w[2] >> sh0) & 63u);
            v.m1 = (int)((r.w[2] >> sh1) & 63u);
        } else {
            v.sc0 = (int)(((r.w[3] >> sh0) & 15u) | (((r.w[1] >> (sh0 + 6)) & 3u) << 4));
            v.sc1 = (int)(((r.w[3] >> sh1) & 15u) | (((r.w[1] >> (sh1 + 6)) & 3u) << 4));
            v.m0 = (int)(((r.w[3] >> (sh0 + 4)) & 15u) | (((r.w[2] >> (sh0 + 6)) & 3u) << 4));
            v.m1 = (int)(((r.w[3] >> (sh1 + 4)) & 15u) | (((r.w[2] >> (sh1 + 6)) & 3u) << 4));
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            v.q[k] = r.w[4 + k] & 0x0f0f0f0fu;
            v.q[8 + k] = (r.w[4 + k] >> 4) & 0x0f0f0f0fu;
        }
    } else {
        const int j = u & 3;
        const uint32_t s0 = 16u * (uint32_t)(j & 1), s1 = s0 + 8u;   // bytes of sub-blocks 8h+2j, +1 in w[8]
        v.sc0 = (int)((r.w[8] >> s0) & 15u);
        v.m0 = (int)((r.w[8] >> (s0 + 4)) & 15u);
        v.sc1 = (int)((r.w[8] >> s1) & 15u);
        v.m1 = (int)((r.w[8] >> (s1 + 4)) & 15u);
        v.d = f16_bits(r.w[9]);
        v.dmin = f16_bits(r.w[9] >> 16);
#pragma unroll
        for (int k = 0; k < 8; ++k) v.q[k] = (r.w[k] >> (2 * j)) & 0x03030303u;
    }
}

// Staged activation quants in shared memory: 16-byte unit u of a token row is
// stored at u ^ (block & 7) (16 units a 256-value block), so that the lanes of a
// warp pass, which read the same offsets of different blocks, spread over all
// eight 16-byte bank groups.
__device__ __forceinline__ uint32_t act_swz(uint32_t u) { return u ^ ((u >> 4) & 7u); }

// One token's activations for a unit: its quants (Q4_K 64, Q2_K 32) and its two
// sub-blocks' 16-value sums (packed int16 pairs).
template <int FMT> struct XUnit {
    static constexpr int NX = FMT == KQ_Q4 ? 4 : 2;
    uint4 x[NX];
    uint32_t g[FMT == KQ_Q4 ? 2 : 1];
};

// xrow: the token's quants (SMEM: the swizzled staged row), u0 the 16-byte unit
// of the unit's first value; xs: its 16-value sums from the unit's first group.
template <int FMT, bool SMEM>
__device__ __forceinline__ void load_x(XUnit<FMT> &a, const int8_t *xrow, uint32_t u0, const int16_t *xs) {
    const uint4 *x4 = reinterpret_cast<const uint4 *>(xrow);
#pragma unroll
    for (int k = 0; k < XUnit<FMT>::NX; ++k) a.x[k] = SMEM ? x4[act_swz(u0 + (uint32_t)k)] : __ldg(x4 + u0 + k);
    const uint32_t *g = reinterpret_cast<const uint32_t *>(xs);
#pragma unroll
    for (int k = 0; k < (FMT == KQ_Q4 ? 2 : 1); ++k) a.g[k] = SMEM ? g[k] : __ldg(g + k);
}

// The unit's term for one token, before the activation scale:
// d * (sc0 isum0 + sc1 isum1) - dmin * (m0 xsum0 + m1 xsum1), the integer sums
// exact.
template <int FMT>
__device__ __forceinline__ float term_x(const Unit<FMT> &v, const XUnit<FMT> &a) {
    int i0 = 0, i1 = 0, xs0, xs1;
    constexpr int H = Unit<FMT>::NW / 2;   // words of the first sub-block
#pragma unroll
    for (int k = 0; k < H; ++k) {
        const uint4 &xa = a.x[k >> 2];
        const uint32_t xw = (k & 3) == 0 ? xa.x : ((k & 3) == 1 ? xa.y : ((k & 3) == 2 ? xa.z : xa.w));
        i0 = __dp4a((int)v.q[k], (int)xw, i0);
    }
#pragma unroll
    for (int k = 0; k < H; ++k) {
        const uint4 &xa = a.x[(H + k) >> 2];
        const uint32_t xw = (k & 3) == 0 ? xa.x : ((k & 3) == 1 ? xa.y : ((k & 3) == 2 ? xa.z : xa.w));
        i1 = __dp4a((int)v.q[H + k], (int)xw, i1);
    }
    if constexpr (FMT == KQ_Q4) {
        xs0 = (int)(int16_t)(a.g[0] & 0xffffu) + (int)(int16_t)(a.g[0] >> 16);
        xs1 = (int)(int16_t)(a.g[1] & 0xffffu) + (int)(int16_t)(a.g[1] >> 16);
    } else {
        xs0 = (int)(int16_t)(a.g[0] & 0xffffu);
        xs1 = (int)(int16_t)(a.g[0] >> 16);
    }
    const int S = v.sc0 * i0 + v.sc1 * i1, M = v.m0 * xs0 + v.m1 * xs1;
    return fmaf(-v.dmin, (float)M, v.d * (float)S);
}

template <int FMT, bool SMEM>
__device__ __forceinline__ float unit_term(const Unit<FMT> &v, const int8_t *xrow, uint32_t u0, const int16_t *xs) {
    XUnit<FMT> a;
    load_x<FMT, SMEM>(a, xrow, u0, xs);
    return term_x<FMT>(v, a);
}

template <int FMT, int TOKG>
__global__ void __launch_bounds__(kq::THREADS, 2) k_kq_gemv(const KqParams p) {
    constexpr int LPB = units_per_block<FMT>();   // lanes per block, one unit (two sub-blocks) each
    constexpr int BPP = 32 / LPB;                 // blocks per warp pass
    constexpr int BB = FMT == KQ_Q4 ? 144 : 84;   // bytes per block
    constexpr int U = FMT == KQ_Q4 ? 2 : 4;       // warp passes whose loads are issued together
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int unit = lane % LPB, bsel = lane / LPB;
    const uint32_t xoff = unit_xoff<FMT>(unit), grp = unit_grp<FMT>(unit);
    const uint32_t nsb = p.nsb;
    const uint64_t row_bytes = (uint64_t)nsb * BB;
    const uint64_t in_dim = p.in_dim;
    __shared__ int arow[TOKG], orow[TOKG];   // the item's activation and output rows
    __shared__ Segment seg_cache[KQ_SEG_CACHE];
    const KqSegs sg = kq_segs(p, seg_cache, threadIdx.x, kq::THREADS);
    __syncthreads();
    KqItem it;
    for (int i = blockIdx.x; kq_item_at<TOKG>(p, sg, i, it); i += gridDim.x) {
        __syncthreads();   // every warp is done with the previous item's rows
        if (threadIdx.x < TOKG) {
            const int t = threadIdx.x;
            const bool on = t < it.ntok;
            arow[t] = !on ? 0 : (p.plan ? p.src_row[it.xrow0 + t] : it.xrow0 + t);
            orow[t] = !on ? -1 : (p.plan ? p.row_to_out[it.xrow0 + t] : it.xrow0 + t);
        }
        __syncthreads();
        const uint8_t *wmat = p.W + (uint64_t)it.expert * p.expert_stride;
        for (uint32_t r = it.r0 + warp; r < it.r0 + it.nrows; r += kq::WARPS) {
            const uint8_t *wrow = wmat + (uint64_t)r * row_bytes;
            float acc[TOKG];
#pragma unroll
            for (int t = 0; t < TOKG; ++t) acc[t] = 0.0f;
            for (uint32_t b0 = 0; b0 < nsb; b0 += BPP * U) {
                RawUnit<FMT> raw[U];
#pragma unroll
                for (int v = 0; v < U; ++v) {
                    const uint32_t b = b0 + (uint32_t)(v * BPP + bsel);
                    if (b < nsb) load_raw<FMT, false>(raw[v], wrow + (uint64_t)b * BB, unit);
                }
#pragma unroll
                for (int v = 0; v < U; ++v) {
                    const uint32_t b = b0 + (uint32_t)(v * BPP + bsel);
                    if (b >= nsb) continue;
                    Unit<FMT> un;
                    decode_unit<FMT>(un, raw[v], unit);
#pragma unroll
                    for (int t = 0; t < TOKG; ++t) {
                        if (t >= it.ntok) break;
                        const uint64_t xr = (uint64_t)arow[t];
                        const float term = unit_term<FMT, false>(
                            un, p.qx + xr * in_dim, (uint32_t)((b * kq::QKK + xoff) / 16u),
                            p.xs + xr * (in_dim / 16) + (uint64_t)b * 16 + grp);
                        acc[t] = fmaf(__ldg(p.dx + xr * nsb + b), term, acc[t]);
                    }
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
                const int o = orow[lane];
                if (o >= 0) p.out[(uint64_t)o * p.out_dim + r] = mine;
            }
        }
    }
}

// ---------------------------------------------------------------- staged GEMV
// The same product with the weights streamed through shared memory: a
// producer warp copies each work item's rows (contiguous in the matrix) into
// a ring of slots with bulk asynchronous copies (one per item for routed calls,
// one per row for dense ones), and the consumer warps take two rows of the slot
// each.  Needs 16-byte aligned rows (row bytes, the matrix and the expert
// stride multiples of 16) of at most SLOT_BYTES.
namespace kqs {
constexpr int NCONS = 14;                        // consumer warps (15 warps: 128 registers a thread)
constexpr int NGRP = 2;                          // groups of consumer warps, alternate fills
constexpr int WPG = NCONS / NGRP;                // warps of a group: two weight rows each per item
constexpr int THREADS = (NCONS + 1) * 32;
constexpr uint32_t SLOT_BYTES = 40 * 1024;       // a work item's rows (a multiple of 14 when they fit)
constexpr int CHUNK = 16;                        // consecutive items a CTA takes in turn
// Shared-memory layout per token group size: ring slots, then the token
// group's Q8_K planes (4864 bytes a token: in_dim up to 4096), then barriers.
template <int TOKG> struct Layout {
    static constexpr int NSLOT = TOKG == 8 ? 4 : 3;
    static constexpr uint32_t ACT_BYTES = TOKG * 4864;
    static constexpr size_t META_OFF = (size_t)NSLOT * SLOT_BYTES + ACT_BYTES;
    static constexpr size_t SEG_OFF = META_OFF + 2 * NSLOT * 8 + 16 + NSLOT * 36 * 4 + 8;   // ... + act_bar
    static constexpr size_t SMEM = SEG_OFF + KQ_SEG_CACHE * sizeof(Segment);
    static_assert(SMEM <= 227 * 1024, "shared memory");
};
// Bytes of one token's staged activations: quants, fp32 scales, int16 sums of 16.
__host__ __device__ constexpr uint64_t act_row_bytes(uint64_t in_dim) { return in_dim + in_dim / 64 + in_dim / 8; }
}  // namespace kqs

// Per-slot description of its work item, written by the producer before the
// slot's copy is armed (ntok < 0: no more items).  group identifies the token
// group (its first plane row): consecutive items of one group share staged
// activations.
struct KqSlotMeta {
    int ntok, group;
    uint32_t r0, nrows;
    int arow[16], orow[16];
};

template <int FMT, int TOKG>
__global__ void __launch_bounds__(kqs::THREADS, 1) k_kq_stream(const KqParams p) {
    using namespace kqs;
    constexpr int NSLOT = Layout<TOKG>::NSLOT;
    constexpr size_t META_OFF = Layout<TOKG>::META_OFF;
    constexpr int LPB = units_per_block<FMT>();   // lanes per block, one unit (two sub-blocks) each
    constexpr int BPP = 32 / LPB;
    constexpr int BB = FMT == KQ_Q4 ? 144 : 84;
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t *slots = smem;
    uint8_t *act = smem + (size_t)NSLOT * SLOT_BYTES;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + META_OFF);
    uint64_t *empty = full + NSLOT;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(empty + NSLOT);
    KqSlotMeta *meta = reinterpret_cast<KqSlotMeta *>(smem + META_OFF + 2 * NSLOT * 8 + 16);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < NSLOT; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], WPG);   // one group's warps consume a fill
        }
        mbar_init(reinterpret_cast<uint64_t *>(meta + NSLOT), NCONS);   // act_bar
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    const uint32_t nsb = p.nsb;
    const uint64_t row_bytes = (uint64_t)nsb * BB;
    if (warp == NCONS) {
        // ---------------- producer warp: item order, slot metadata, one bulk copy per item
        // Fills alternate between the two consumer groups (even fills: group 0).  A
        // token group may begin only at an even fill, so that both groups meet every
        // change of staged activations at the same pair of fills: an odd fill that
        // would start a new group carries a no-op item (no rows, same group) instead.
        // Two end markers, at an even fill and the next, close both groups.
        KqItem it;
        Segment *seg_cache = reinterpret_cast<Segment *>(smem + Layout<TOKG>::SEG_OFF);
        const KqSegs sg = kq_segs(p, seg_cache, lane, 32);
        __syncwarp();
        int group = -1, group_ntok = 0, my_arow = 0, my_orow = -1;
        // chunks of consecutive items (one token group, mostly) dealt in turn: the
        // staged activations change once per chunk; up to CHUNK items a chunk while
        // every CTA still gets about four chunks
        const int n_items = p.plan ? sg.n_items
                                   : (int)((p.out_dim + p.rows_per_item - 1) / p.rows_per_item) *
                                         (int)((p.n_tok + TOKG - 1) / TOKG);
        const int chunk = max(1, min(CHUNK, n_items / (4 * (int)gridDim.x)));
        uint32_t fills[NSLOT];
        for (int s2 = 0; s2 < NSLOT; ++s2) fills[s2] = 0;
        bool have = false, done = false;
        int ends = 0;
        for (uint32_t kf = 0, q = 0; ends < NGRP; ++kf) {
            if (!have && !done) {
                const int i = (((int)q / chunk) * (int)gridDim.x + (int)blockIdx.x) * chunk + (int)q % chunk;
                if (kq_item_at<TOKG>(p, sg, i, it)) {
                    have = true;
                    ++q;
                } else {
                    done = true;
                }
            }
            const bool odd = (kf & 1u) != 0u;
            // 0: end marker, 1: no-op, 2: the item
            const int kind = have ? ((odd && it.xrow0 != group) ? 1 : 2) : ((odd && ends == 0) ? 1 : 0);
            const uint32_t slot = kf % NSLOT, phase = (kf / NSLOT) & 1u;
            // after an abort nothing more is issued; consumers release only the
            // slots they saw land, so each slot has at most its last fill in flight
            bool ok = false;
            if (lane == 0) ok = mbar_wait(&empty[slot], phase ^ 1u, p.err, abort_flag) && !*abort_flag;
            ok = __shfl_sync(0xffffffffu, (int)ok, 0) != 0;
            if (!ok) break;
            KqSlotMeta &m = meta[slot];
            if (kind == 2 && it.xrow0 != group) {   // a new token group: its rows (lane t: token t)
                group = it.xrow0;
                group_ntok = it.ntok;
                const bool on = lane < it.ntok;
                my_arow = !on ? 0 : (p.plan ? p.src_row[it.xrow0 + lane] : it.xrow0 + lane);
                my_orow = !on ? -1 : (p.plan ? p.row_to_out[it.xrow0 + lane] : it.xrow0 + lane);
            }
            if (lane < TOKG) {
                m.arow[lane] = my_arow;
                m.orow[lane] = kind == 2 ? my_orow : -1;
            }
            if (lane == 0) {
                // a no-op keeps its group's tokens: a warp may stage the group from it
                m.ntok = kind == 2 ? it.ntok : (kind == 1 ? group_ntok : -1);
                m.group = kind == 0 ? -1 : group;
                m.r0 = kind == 2 ? it.r0 : 0u;
                m.nrows = kind == 2 ? it.nrows : 0u;
            }
            __syncwarp();
            // The item's bytes are armed first.  Routed calls (many items per CTA) copy an
            // item's rows, contiguous in the matrix and in the slot, with one bulk copy:
            // against one copy per row, Q4_K gate/up calls at the decode size took 331
            // instead of 376 us and down calls 363 instead of 457.  Dense calls (an item or
            // two per CTA) keep one copy per row, issued by one lane each so that the rows
            // stream in parallel: there the first rows land sooner (4-token calls 2-5 %).
            if (lane == 0) mbar_arrive_expect_tx(&full[slot], kind == 2 ? it.nrows * (uint32_t)row_bytes : 0u);
            __syncwarp();
            if (kind == 2 && p.plan) {
                if (lane == 0)
                    bulk_g2s(slots + (size_t)slot * SLOT_BYTES,
                             p.W + (uint64_t)it.expert * p.expert_stride + (uint64_t)it.r0 * row_bytes,
                             it.nrows * (uint32_t)row_bytes, &full[slot]);
            } else if (kind == 2) {
                for (uint32_t rr = (uint32_t)lane; rr < it.nrows; rr += 32)
                    bulk_g2s(slots + (size_t)slot * SLOT_BYTES + (size_t)rr * row_bytes,
                             p.W + (uint64_t)it.expert * p.expert_stride + (uint64_t)(it.r0 + rr) * row_bytes,
                             (uint32_t)row_bytes, &full[slot]);
            }
            ++fills[slot];
            if (kind == 2) have = false;
            if (kind == 0) ++ends;
        }
        if (lane == 0)
            for (int s2 = 0; s2 < NSLOT; ++s2)   // every copy lands before the CTA exits
                if (fills[s2]) mbar_wait(&full[s2], (fills[s2] - 1u) & 1u, p.err, nullptr);
        return;
    }
    // ---------------- consumers: two groups of WPG warps take alternate fills; warp
    // w of a group takes rows 2w + 14j and 2w + 14j + 1 of its items (items hold a
    // multiple of 14 rows when short rows allow), so each staged activation load
    // serves two weight rows.
    // The token group's activations are staged in shared memory once per group:
    // a bounded barrier (act_bar, two phases) first lets every warp finish the
    // previous group, then every warp copies its share and arrives again.
    const int unit = lane % LPB, bsel = lane / LPB;
    const uint32_t xoff = unit_xoff<FMT>(unit), grp = unit_grp<FMT>(unit);
    const uint64_t in_dim = p.in_dim;
    const uint32_t nxs = (uint32_t)(in_dim / 16);
    int8_t *qx_s = reinterpret_cast<int8_t *>(act);
    float *dx_s = reinterpret_cast<float *>(act + (size_t)TOKG * in_dim);
    int16_t *xs_s = reinterpret_cast<int16_t *>(act + (size_t)TOKG * in_dim + (size_t)TOKG * nsb * 4);
    uint64_t *act_bar = reinterpret_cast<uint64_t *>(meta + NSLOT);
    const int ctid = warp * 32 + lane;
    constexpr int CT = NCONS * 32;
    const int wg = warp / WPG, wr = warp % WPG;
    int group = -1;
    for (uint32_t kf = (uint32_t)wg;; kf += NGRP) {
        const uint32_t slot = kf % NSLOT, phase = (kf / NSLOT) & 1u;
        // a consumer whose wait failed leaves (an abort); it hands no slot back
        if (!mbar_wait(&full[slot], phase, p.err, abort_flag)) break;
        const KqSlotMeta &m = meta[slot];
        const int ntok = m.ntok;
        if (ntok < 0) break;   // the end marker: its slot needs no release
        if (m.group != group) {
            group = m.group;
            __syncwarp();
            if (lane == 0) mbar_arrive(act_bar);   // done with the previous group
            if (!mbar_wait(act_bar, 0u, p.err, abort_flag)) break;
            for (uint32_t e = (uint32_t)ctid; e < (uint32_t)ntok * nxs; e += CT) {
                const uint32_t t = e / nxs, c = e - t * nxs;
                reinterpret_cast<uint4 *>(qx_s + (size_t)t * in_dim)[act_swz(c)] =
                    __ldg(reinterpret_cast<const uint4 *>(p.qx + (uint64_t)m.arow[t] * in_dim) + c);
            }
            for (uint32_t e = (uint32_t)ctid; e < (uint32_t)ntok * nsb; e += CT) {
                const uint32_t t = e / nsb, c = e - t * nsb;
                dx_s[t * nsb + c] = __ldg(p.dx + (uint64_t)m.arow[t] * nsb + c);
            }
            for (uint32_t e = (uint32_t)ctid; e < (uint32_t)ntok * (nxs / 2); e += CT) {
                const uint32_t t = e / (nxs / 2), c = e - t * (nxs / 2);
                reinterpret_cast<uint32_t *>(xs_s + (size_t)t * nxs)[c] =
                    __ldg(reinterpret_cast<const uint32_t *>(p.xs + (uint64_t)m.arow[t] * nxs) + c);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(act_bar);   // this warp's share is staged
            if (!mbar_wait(act_bar, 1u, p.err, abort_flag)) break;
        }
        for (uint32_t ra = 2u * (uint32_t)wr; ra < m.nrows; ra += 2u * WPG) {
            const bool two = ra + 1u < m.nrows;
            const uint8_t *wa = slots + (size_t)slot * SLOT_BYTES + (size_t)ra * row_bytes;
            const uint8_t *wb = wa + (two ? row_bytes : 0);
            float acc[2][TOKG];
#pragma unroll
            for (int t = 0; t < TOKG; ++t) acc[0][t] = acc[1][t] = 0.0f;
            for (uint32_t b0 = 0; b0 < nsb; b0 += BPP) {
                const uint32_t b = b0 + (uint32_t)bsel;
                if (b >= nsb) continue;
                RawUnit<FMT> raw0, raw1;
                load_raw<FMT, true>(raw0, wa + (size_t)b * BB, unit);
                load_raw<FMT, true>(raw1, wb + (size_t)b * BB, unit);
                Unit<FMT> u0, u1;
                decode_unit<FMT>(u0, raw0, unit);
                decode_unit<FMT>(u1, raw1, unit);
#pragma unroll
                for (int t = 0; t < TOKG; ++t) {
                    if (t >= ntok) break;
                    XUnit<FMT> xa;
                    load_x<FMT, true>(xa, qx_s + (size_t)t * in_dim, (b * kq::QKK + xoff) / 16u,
                                      xs_s + (size_t)t * nxs + b * 16 + grp);
                    const float dxt = dx_s[t * nsb + b];
                    acc[0][t] = fmaf(dxt, term_x<FMT>(u0, xa), acc[0][t]);
                    acc[1][t] = fmaf(dxt, term_x<FMT>(u1, xa), acc[1][t]);
                }
            }
            float mine[2] = {0.0f, 0.0f};
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int t = 0; t < TOKG; ++t) {
                    if (t >= ntok) break;
                    float v = acc[h][t];
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
                    if (lane == t) mine[h] = v;
                }
            if (lane < ntok) {
                const int o = m.orow[lane];
                if (o >= 0) {
                    p.out[(uint64_t)o * p.out_dim + m.r0 + ra] = mine[0];
                    if (two) p.out[(uint64_t)o * p.out_dim + m.r0 + ra + 1u] = mine[1];
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
    }
}

uint32_t kq_stream_rows(uint64_t row_bytes, uint64_t in_dim, int tokg) {
    if (row_bytes == 0 || row_bytes % 16 || row_bytes > kqs::SLOT_BYTES) return 0;
    if (in_dim % 256 || kqs::act_row_bytes(in_dim) > 4864) return 0;
    // whole multiples of the consumers' 14 rows (every warp takes the same number
    // of row pairs) when a slot holds that many, at most 42: items of 56 short rows
    // (Q2_K, in_dim 2048) made the routed down call slower (368.5 us at 42 against
    // 387.9 us at 56; 381.8 us at 28)
    const uint64_t r = kqs::SLOT_BYTES / row_bytes;
    const uint64_t rows = r < (uint64_t)kqs::NCONS ? r : r / kqs::NCONS * kqs::NCONS;
    return (uint32_t)(rows > 3 * kqs::NCONS ? 3 * kqs::NCONS : rows);
}

template <int FMT, int TOKG> static cudaError_t launch_stream(const KqParams &p, int num_sms, cudaStream_t st) {
    static bool attr_done = false;
    if (!attr_done) {
        cudaError_t e = cudaFuncSetAttribute(k_kq_stream<FMT, TOKG>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)kqs::Layout<TOKG>::SMEM);
        if (e != cudaSuccess) return e;
        attr_done = true;
    }
    k_kq_stream<FMT, TOKG><<<num_sms, kqs::THREADS, kqs::Layout<TOKG>::SMEM, st>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_kq_stream(const KqParams &p, int tokg, int num_sms, cudaStream_t st) {
    const uint64_t row_bytes = (uint64_t)p.nsb * (p.fmt == KQ_Q4 ? 144 : 84);
    if (p.rows_per_item == 0 || p.rows_per_item > kq_stream_rows(row_bytes, p.in_dim, tokg))
        return cudaErrorInvalidValue;
    if (p.fmt == KQ_Q4) return tokg == 8 ? launch_stream<KQ_Q4, 8>(p, num_sms, st) : launch_stream<KQ_Q4, 16>(p, num_sms, st);
    if (p.fmt == KQ_Q2) return tokg == 8 ? launch_stream<KQ_Q2, 8>(p, num_sms, st) : launch_stream<KQ_Q2, 16>(p, num_sms, st);
    return cudaErrorInvalidValue;
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
