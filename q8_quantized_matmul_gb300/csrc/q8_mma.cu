// q8_mma.cu -- Q8_0 x Q8_0 matmul over raw 34-byte-block weight rows.
//
// Computes out[t][o] = sum_b d_w[o][b] d_x[t][b] isum_b[t][o] with isum_b the
// exact int32 dot of the two blocks' quants (ds4 pages: the Q8_0 matmul of the
// GPU code walkthrough, trace 3, and the fixed-point block dot of the
// model-architecture page, quantisation section 4).
//
// Structure (one persistent CTA per SM, warp-specialised):
//   * warp 8, one lane: producer.  Streams weight rows with 1-D bulk
//     asynchronous copies (TMA) into an NSTAGE-deep shared-memory ring, one
//     copy per row of a 16-row x KC-block chunk, completion counted on a full
//     mbarrier.  Rows land at a padded stride (an odd multiple of 16 bytes)
//     so the consumers' fragment loads are bank-conflict free.
//   * warps 0-7: consumers.  Warp w owns blocks j = w, w+8, ... of each chunk
//     for both 8-row groups.  Per block it issues one mma.sync m16n8k32 s8
//     (16 tokens x 8 rows x one 32-value block) giving the exact int32 block
//     dots, and folds them into fp32 accumulators with the two scales.  The
//     34-byte blocks start at 2 mod 4 for even j: those quants are rebuilt
//     from the two aligned words around them with one byte permute.
//   * at the end of a work item the eight warps' partial sums are added in a
//     fixed order through shared memory (deterministic, no atomics).
// A work item is (segment, 16-row block, group of up to 64 tokens); the
// weight chunk in shared memory is reused for every 16-token tile of the
// group.  Dense calls have one segment; routed-expert calls take the segment
// table written on the device by the routing kernels.
#include "q8_common.cuh"
#include "q8_kernels.h"

namespace q8 {

namespace mma_cfg {
constexpr int NCW = 8;                     // consumer warps
constexpr int NTHREADS = (NCW + 1) * 32;   // + one producer warp
constexpr int RBR = 16;                    // weight rows per work item
constexpr int KCMAX = 32;                  // blocks per chunk
constexpr int TGMAX = 4;                   // 16-token tiles per work item
constexpr int TOK_PER_ITEM = TGMAX * 16;
constexpr int NSTAGE = 8;
constexpr int RED_FLOATS = NCW * TOK_PER_ITEM * RBR;
}  // namespace mma_cfg

__device__ __forceinline__ bool get_item(const MmaParams &p, int i, int n_rb, Segment &seg, int &rb, int &tg) {
    using namespace mma_cfg;
    if (p.plan == nullptr) {
        const int tgn = ((int)p.n_tok + TOK_PER_ITEM - 1) / TOK_PER_ITEM;
        if (i >= n_rb * tgn) return false;
        rb = i / tgn;
        tg = i - rb * tgn;
        seg.expert = 0;
        seg.row0 = 0;
        seg.count = (int)p.n_tok;
        seg.item_start = 0;
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
    seg = segs[lo];
    const int tgn = (seg.count + TOK_PER_ITEM - 1) / TOK_PER_ITEM;
    const int local = i - seg.item_start;
    rb = local / tgn;
    tg = local - rb * tgn;
    return true;
}

__device__ __forceinline__ uint32_t lds32(const uint8_t *p) { return *reinterpret_cast<const uint32_t *>(p); }
__device__ __forceinline__ uint16_t lds16(const uint8_t *p) { return *reinterpret_cast<const uint16_t *>(p); }

__global__ void __launch_bounds__(mma_cfg::NTHREADS, 1)
    k_mma(const MmaParams p, uint32_t kc, uint32_t srow, uint32_t stage_bytes) {
    using namespace mma_cfg;
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t *stages = smem;
    float *red = reinterpret_cast<float *>(smem + (size_t)NSTAGE * stage_bytes);
    uint64_t *full = reinterpret_cast<uint64_t *>(red + RED_FLOATS);
    uint64_t *empty = full + NSTAGE;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(empty + NSTAGE);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < NSTAGE; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], NCW);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    const uint32_t nb = p.nb;
    const uint32_t nchunks = (nb + kc - 1) / kc;
    const int n_rb = (int)((p.out_dim + RBR - 1) / RBR);
    const uint64_t row_bytes = (uint64_t)nb * QB;

    if (warp == NCW) {
        // ---------------- producer
        if (lane == 0) {
            uint32_t stage = 0, phase = 0;
            uint32_t fills[NSTAGE];
            for (int s = 0; s < NSTAGE; ++s) fills[s] = 0;
            Segment seg;
            int rb, tg;
            for (int i = blockIdx.x; get_item(p, i, n_rb, seg, rb, tg); i += gridDim.x) {
                const uint32_t r0 = (uint32_t)rb * RBR;
                const uint32_t nr = min((uint32_t)RBR, p.out_dim - r0);
                const uint8_t *wb = p.W + (uint64_t)seg.expert * p.expert_stride + (uint64_t)r0 * row_bytes;
                for (uint32_t kk = 0; kk < nchunks; ++kk) {
                    const uint32_t kcur = min(kc, nb - kk * kc);
                    const uint32_t cbytes = kcur * QB;
                    // after an abort nothing more is issued (consumers release only
                    // stages they saw land, so each stage has at most one fill in flight)
                    const bool ok = mbar_wait(&empty[stage], phase ^ 1u, p.err, abort_flag) && !*abort_flag;
                    if (ok) {
                        mbar_arrive_expect_tx(&full[stage], nr * cbytes);
                        uint8_t *dst = stages + (size_t)stage * stage_bytes;
                        const uint8_t *src = wb + (uint64_t)kk * kc * QB;
                        for (uint32_t r = 0; r < nr; ++r) bulk_g2s(dst + r * srow, src + r * row_bytes, cbytes, &full[stage]);
                        ++fills[stage];
                    }
                    if (++stage == NSTAGE) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // Drain: every copy issued must have landed before the CTA exits.
            for (int s = 0; s < NSTAGE; ++s)
                if (fills[s]) mbar_wait(&full[s], (fills[s] - 1u) & 1u, p.err, nullptr);
        }
        return;
    }

    // ---------------- consumers
    const int g = lane >> 2, c = lane & 3;
    const uint64_t in_dim = p.in_dim;
    uint32_t stage = 0, phase = 0;
    Segment seg;
    int rb, tg;
    for (int i = blockIdx.x; get_item(p, i, n_rb, seg, rb, tg); i += gridDim.x) {
        const uint32_t r0 = (uint32_t)rb * RBR;
        const int tok0 = tg * TOK_PER_ITEM;
        const int ntok = min(TOK_PER_ITEM, seg.count - tok0);
        const int tiles = (ntok + 15) >> 4;
        const uint64_t xrow0 = (uint64_t)seg.row0 + tok0;

        float acc[TGMAX][2][4];
#pragma unroll
        for (int t = 0; t < TGMAX; ++t)
#pragma unroll
            for (int rg = 0; rg < 2; ++rg)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[t][rg][e] = 0.0f;

        for (uint32_t kk = 0; kk < nchunks; ++kk) {
            const uint32_t kcur = min(kc, nb - kk * kc);
            const bool staged = mbar_wait(&full[stage], phase, p.err, abort_flag);
            const uint8_t *st = stages + (size_t)stage * stage_bytes;
            const int nbw = (int)(kcur >> 3);   // this warp's blocks in the chunk

            // Weight fragments (B operand) and weight scales for this warp's blocks.
            uint32_t bq[KCMAX / 8][2][2];
            float bd[KCMAX / 8][2][2];
#pragma unroll
            for (int jj = 0; jj < KCMAX / 8; ++jj) {
                if (jj < nbw) {
                    const uint32_t j = (uint32_t)warp + 8u * jj;
#pragma unroll
                    for (int rg = 0; rg < 2; ++rg) {
                        const uint8_t *rowp = st + (uint32_t)(rg * 8 + g) * srow + j * QB;
                        if (warp & 1) {   // odd block: quants 4-byte aligned
                            bq[jj][rg][0] = lds32(rowp + 2 + 4 * c);
                            bq[jj][rg][1] = lds32(rowp + 18 + 4 * c);
                        } else {          // even block: quants at 2 mod 4
                            bq[jj][rg][0] = funnel16(lds32(rowp + 4 * c), lds32(rowp + 4 + 4 * c));
                            bq[jj][rg][1] = funnel16(lds32(rowp + 16 + 4 * c), lds32(rowp + 20 + 4 * c));
                        }
                        const uint8_t *drow = st + (uint32_t)(rg * 8 + 2 * c) * srow + j * QB;
                        bd[jj][rg][0] = half_bits_to_float(lds16(drow));
                        bd[jj][rg][1] = half_bits_to_float(lds16(drow + srow));
                    }
                }
            }

#pragma unroll
            for (int t = 0; t < TGMAX; ++t) {
                if (t < tiles) {
                    const uint64_t xr = xrow0 + (uint64_t)t * 16 + g;
#pragma unroll
                    for (int jj = 0; jj < KCMAX / 8; ++jj) {
                        if (jj < nbw) {
                            const uint32_t jb = kk * kc + (uint32_t)warp + 8u * jj;
                            const int8_t *xa = p.qx + xr * in_dim + (uint64_t)jb * QK + 4 * c;
                            uint32_t a[4];
                            a[0] = __ldg(reinterpret_cast<const uint32_t *>(xa));
                            a[1] = __ldg(reinterpret_cast<const uint32_t *>(xa + 8 * in_dim));
                            a[2] = __ldg(reinterpret_cast<const uint32_t *>(xa + 16));
                            a[3] = __ldg(reinterpret_cast<const uint32_t *>(xa + 8 * in_dim + 16));
                            const float dx0 = __ldg(p.dx + xr * nb + jb);
                            const float dx1 = __ldg(p.dx + (xr + 8) * nb + jb);
#pragma unroll
                            for (int rg = 0; rg < 2; ++rg) {
                                int d[4] = {0, 0, 0, 0};
                                mma_s8_16832(d, a, bq[jj][rg][0], bq[jj][rg][1]);
                                acc[t][rg][0] = fmaf((float)d[0], bd[jj][rg][0] * dx0, acc[t][rg][0]);
                                acc[t][rg][1] = fmaf((float)d[1], bd[jj][rg][1] * dx0, acc[t][rg][1]);
                                acc[t][rg][2] = fmaf((float)d[2], bd[jj][rg][0] * dx1, acc[t][rg][2]);
                                acc[t][rg][3] = fmaf((float)d[3], bd[jj][rg][1] * dx1, acc[t][rg][3]);
                            }
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0 && staged) mbar_arrive(&empty[stage]);   // a timed-out stage is never handed back
            if (++stage == NSTAGE) {
                stage = 0;
                phase ^= 1u;
            }
        }

        // Cross-warp reduction in a fixed order.
        float *rw = red + warp * (TOK_PER_ITEM * RBR);
#pragma unroll
        for (int t = 0; t < TGMAX; ++t) {
            if (t < tiles) {
#pragma unroll
                for (int rg = 0; rg < 2; ++rg) {
                    const int tok = t * 16 + g, row = rg * 8 + 2 * c;
                    rw[tok * RBR + row] = acc[t][rg][0];
                    rw[tok * RBR + row + 1] = acc[t][rg][1];
                    rw[(tok + 8) * RBR + row] = acc[t][rg][2];
                    rw[(tok + 8) * RBR + row + 1] = acc[t][rg][3];
                }
            }
        }
        named_bar_sync(1, NCW * 32);
        const int nout = tiles * 16 * RBR;
        for (int o = threadIdx.x; o < nout; o += NCW * 32) {
            float s = 0.0f;
#pragma unroll
            for (int w = 0; w < NCW; ++w) s += red[w * (TOK_PER_ITEM * RBR) + o];
            const int tok = o / RBR, row = o - tok * RBR;
            const int tl = tok0 + tok;
            if (tl < seg.count && r0 + (uint32_t)row < p.out_dim) {
                const int64_t orow = p.plan ? (int64_t)p.row_to_out[seg.row0 + tl] : (int64_t)tl;
                if (orow >= 0) p.out[(uint64_t)orow * p.out_dim + r0 + row] = s;
            }
        }
        named_bar_sync(1, NCW * 32);
    }
}

// Slow path for in_dim % 256 != 0 (rows not 16-byte aligned): one thread per
// output, blocks read in place.  Same arithmetic, sequential block order.
__global__ void __launch_bounds__(256) k_generic(const MmaParams p) {
    const uint32_t nb = p.nb;
    const uint64_t total_rows = p.plan ? (uint64_t)p.plan->n_rows : (uint64_t)p.n_tok;
    const uint64_t n = total_rows * p.out_dim;
    const Segment *segs = p.plan ? reinterpret_cast<const Segment *>(p.plan + 1) : nullptr;
    for (uint64_t idx = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < n; idx += (uint64_t)gridDim.x * blockDim.x) {
        const uint64_t r = idx / p.out_dim, o = idx - r * p.out_dim;
        int64_t orow = (int64_t)r;
        int expert = 0;
        if (p.plan) {
            orow = p.row_to_out[r];
            if (orow < 0) continue;
            int lo = 0, hi = p.plan->n_segments - 1;
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if ((uint64_t)segs[mid].row0 <= r) lo = mid;
                else hi = mid - 1;
            }
            if (p.plan->n_segments == 0 || r < (uint64_t)segs[lo].row0 ||
                r >= (uint64_t)segs[lo].row0 + (uint64_t)segs[lo].count)
                continue;   // row of another plan's segment
            expert = segs[lo].expert;
        }
        const uint8_t *w = p.W + (uint64_t)expert * p.expert_stride + o * (uint64_t)nb * QB;
        const int8_t *xq = p.qx + r * p.in_dim;
        float acc = 0.0f;
        for (uint32_t b = 0; b < nb; ++b) {
            const uint8_t *wb = w + (uint64_t)b * QB;
            const float dw = half_bits_to_float(*reinterpret_cast<const uint16_t *>(wb));
            int isum = 0;
#pragma unroll 8
            for (int i = 0; i < QK; ++i) isum += (int)(int8_t)wb[2 + i] * (int)xq[b * QK + i];
            acc = fmaf((float)isum, dw * p.dx[r * nb + b], acc);
        }
        p.out[(uint64_t)orow * p.out_dim + o] = acc;
    }
}

// ------------------------------------------------------------------ launchers
static size_t mma_smem_bytes(uint32_t stage_bytes) {
    using namespace mma_cfg;
    return (size_t)NSTAGE * stage_bytes + RED_FLOATS * sizeof(float) + 2 * NSTAGE * sizeof(uint64_t) + 16;
}

cudaError_t launch_mma(const MmaParams &p, int grid, cudaStream_t st) {
    using namespace mma_cfg;
    const uint32_t kc = p.nb < (uint32_t)KCMAX ? p.nb : (uint32_t)KCMAX;   // multiple of 8
    uint32_t srow = kc * QB;
    if (((srow / 16) & 1u) == 0) srow += 16;   // odd multiple of 16 bytes: conflict-free rows
    const uint32_t stage_bytes = (RBR * srow + 127u) & ~127u;
    const size_t smem = mma_smem_bytes(stage_bytes);
    static bool attr_done = false;   // per process; the limit is the same on every device
    if (!attr_done) {
        cudaError_t e = cudaFuncSetAttribute(k_mma, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)mma_smem_bytes(((RBR * (KCMAX * QB + 16)) + 127u) & ~127u));
        if (e != cudaSuccess) return e;
        attr_done = true;
    }
    k_mma<<<grid, NTHREADS, smem, st>>>(p, kc, srow, stage_bytes);
    return cudaGetLastError();
}

cudaError_t launch_generic(const MmaParams &p, int max_items_hint, int num_sms, cudaStream_t st) {
    int grid = (max_items_hint + 255) / 256;
    if (grid > num_sms * 8) grid = num_sms * 8;
    if (grid < 1) grid = 1;
    k_generic<<<grid, 256, 0, st>>>(p);
    return cudaGetLastError();
}

}  // namespace q8
