// q8_gemv.cu -- weight-streaming Q8_0 x Q8_0 matmul for up to 16 tokens (decode, and
// the small groups of routed experts).
//
// out[t][o] = sum_b d_w[o][b] d_x[t][b] isum_b, isum_b the exact int32 dot of one
// weight block and one activation block (ds4 pages: the Q8_0 matmul of the GPU
// code walkthrough, trace 3; the fixed-point block dot of the model-architecture
// page, quantisation section 4).  With a handful of tokens each weight byte is
// used a handful of times, so the kernel is bound by HBM: its job is to keep
// enough weight bytes in flight and to spend few instructions per byte.
//
// Layout of the work
//   * A CTA item is (segment, token group, row range).  A token group is up to
//     NT*8 tokens (NT = 1 or 2 N tiles of the MMA); its activation fragments are
//     staged once into shared memory in MMA-fragment order (converted to fp16,
//     exact for int8), so a warp reads one block's fragment with one 16-byte
//     load per lane and N tile.
//   * The row range is cut into 16-row sub-items (the MMA M dimension).  Each of
//     the 16 warps owns whole sub-items and streams their weight rows through its
//     own two-slot ring: one tiled TMA copy (cp.async.bulk.tensor) per slot of
//     16 rows x 8 blocks, over a tensor map that views the raw rows as 32-bit
//     words with a 76-word box, so rows land 304 bytes apart (an odd multiple of
//     16 bytes: the fragment loads are bank-conflict free).  The box's last 32
//     bytes per row belong to the next slot and are not used; words past the end
//     of a row and rows past out_dim are filled with zeros by the TMA.  When the
//     rows are too few for the warps, WPI warps split a sub-item's blocks and add
//     their partial sums through shared memory in a fixed order.
//   * Per block: the weight fragment (rows g and g+8, two 4-byte groups of
//     quants per lane) comes from 32-bit shared loads.  The sum over a block's 32
//     products does not depend on their order, so each lane may take any fixed
//     set of quant positions as long as the activation fragment uses the same
//     one: odd blocks (quants 4-byte aligned) use the natural MMA order; even
//     blocks (quants at 2 mod 4) give lanes 0-2 two aligned words each and lane
//     3 one aligned word plus the four edge bytes joined by one byte permute,
//     and the staged activations are permuted to match.  The quants are converted
//     to fp16 (exact: |q| <= 127), and two mma.sync m16n8k16 f16 per N tile give
//     the block dot (16 rows x 8 tokens x 32 values) in fp32, exact because
//     every product is an integer below 2^14 and every block sum below 2^24.
//     It is then scaled by d_w*d_x and added in fp32 with packed f32x2
//     instructions.  fp16 rather than int8 MMA: on GB300 mma.sync runs int8 at
//     251 and fp16 at 942 MAC per SM per clock (measured); the 8-token N tile
//     costs 8 or 16 MACs per weight, which int8 cannot deliver at the HBM rate.
//   * Memory-level parallelism: the ring is small, so at the start of an item
//     each warp also issues TMA L2 prefetches for all of its remaining slots;
//     HBM then sees the item's whole request at once and the ring refills from
//     L2 at low latency.
//   * Launched with programmatic stream serialisation: the weight prefetch starts
//     before the preceding quantiser kernel has finished; activations are read
//     only after griddepcontrol.wait.
#include <cuda.h>

#include "q8_common.cuh"
#include "q8_kernels.h"

namespace q8 {

namespace gv {
constexpr int NW = 16;                   // warps per CTA
constexpr int NTHREADS = NW * 32;
constexpr int ROWS = 16;                 // rows per sub-item
constexpr int KC = 8;                    // blocks per weight slot
constexpr int BOX_WORDS = (KC * QB + 32) / 4;   // 76 words per row of a slot
constexpr int SROW = BOX_WORDS * 4;      // 304 bytes: 19 x 16, an odd multiple of 16
constexpr int SLOT = ROWS * SROW;        // 4864 bytes
constexpr int NSLOT = 2;                 // ring depth per warp
constexpr int SUBMAX = 2;                // sub-items per warp per CTA item
constexpr int ACT_BYTES = 48 * 1024;     // activation fragments per chunk
constexpr int KA_MAX = ACT_BYTES / (32 * 16);  // blocks per chunk with one N tile (96)
constexpr int DX_FLOATS = KA_MAX * 16;   // scales of a chunk: [block][16 tokens]
constexpr int RING_BYTES = NW * NSLOT * SLOT;
constexpr size_t SMEM = RING_BYTES + ACT_BYTES + DX_FLOATS * 4 + NW * NSLOT * 8 + 64;
static_assert(SMEM <= 227 * 1024, "shared memory");
static_assert(SUBMAX * NW * ROWS >= GEMV_MAX_ROWS_PER_ITEM, "rows per item");
}  // namespace gv

__device__ __forceinline__ uint32_t lds32g(const uint8_t *p) { return *reinterpret_cast<const uint32_t *>(p); }

// Quant positions of an even block (block start 0 mod 4, quants at byte 2):
// lane c reads the aligned word 1+c of the block and, for c < 3, word 5+c;
// lane 3 instead joins the high half of word 0 with the low half of word 8
// ([q0, q1, q30, q31]) with one byte permute.  At a row pitch of 76 words the
// 32 lanes' addresses fall in 32 different banks.
//   logical 4c..4c+3    <- quants 4c+2..4c+5      (c < 3),  14..17 (c = 3)
//   logical 16+4c..+3   <- quants 4c+18..4c+21    (c < 3),  0, 1, 30, 31 (c = 3)
__device__ __forceinline__ int even_off_a(int c) { return 4 + 4 * c; }
__device__ __forceinline__ int even_off_b(int c) { return c < 3 ? 20 + 4 * c : 0; }

// (a0, a1) += (v0, v1) * (dx0, dx1) * dw with the accumulator pair in one
// 64-bit register: packed multiply by the token scales, packed FMA by {dw, dw}.
__device__ __forceinline__ void scale_acc64(uint64_t &acc, float v0, float v1, uint64_t dx01, uint64_t dwdw) {
    asm("{\n\t.reg .b64 v, u;\n\tmov.b64 v, {%1, %2};\n\t"
        "mul.rn.f32x2 u, v, %3;\n\t"
        "fma.rn.f32x2 %0, u, %4, %0;\n\t}"
        : "+l"(acc)
        : "f"(v0), "f"(v1), "l"(dx01), "l"(dwdw));
}

__device__ __forceinline__ uint64_t pack_same(float v) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %1};" : "=l"(r) : "f"(v));
    return r;
}

__device__ __forceinline__ float lo_of(uint64_t v) { return __uint_as_float((uint32_t)v); }
__device__ __forceinline__ float hi_of(uint64_t v) { return __uint_as_float((uint32_t)(v >> 32)); }

// D(16x8, f32) += A(16x16, f16, row) * B(16x8, f16, col).
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Four int8 -> two fp16x2 holding the same integers exactly (bytes 0,1 -> lo,
// bytes 2,3 -> hi): bias each byte to unsigned, place it under the fp16 exponent
// of 1024, then subtract 1024 + 128.
__device__ __forceinline__ void s8x4_to_h2x2(uint32_t w, uint32_t &lo, uint32_t &hi) {
    const uint32_t u = w ^ 0x80808080u;
    const uint32_t a = __byte_perm(u, 0x64646464u, 0x4140);
    const uint32_t b = __byte_perm(u, 0x64646464u, 0x4342);
    const uint32_t bias = 0x64806480u;   // fp16 (1152, 1152)
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(a), "r"(bias));
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(b), "r"(bias));
}

__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, int x, int y, int z, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar))
        : "memory");
}

// Bring a box of the tensor into L2 without a shared-memory destination.
__device__ __forceinline__ void tma_prefetch_l2_3d(const CUtensorMap *map, int x, int y, int z) {
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y), "r"(z)
                 : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Item decoding.  Returns false past the last item.
struct GItem {
    int expert;
    int xrow0;      // first activation-plane row of the token group
    int ntok;       // tokens in the group (<= NT*8)
    int tok0;       // index of the first token within its segment
    uint32_t r0;    // first weight row
    uint32_t nrows;
};

template <int NT>
__device__ __forceinline__ bool gemv_item(const GemvParams &p, int i, GItem &it) {
    constexpr int TOKG = NT * 8;
    if (!p.plan) {
        const uint32_t n_items = (p.out_dim + p.rows_per_item - 1) / p.rows_per_item;
        if ((uint32_t)i >= n_items) return false;
        it.expert = 0;
        it.xrow0 = 0;
        it.ntok = (int)p.n_tok;
        it.tok0 = 0;
        it.r0 = (uint32_t)i * p.rows_per_item;
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
    const int n_rb = (int)((p.out_dim + p.rows_per_item - 1) / p.rows_per_item);
    const int local = i - s.item_start;
    const int tg = local / n_rb, rb = local - tg * n_rb;
    it.expert = s.expert;
    it.tok0 = tg * TOKG;
    it.ntok = min(TOKG, s.count - it.tok0);
    it.xrow0 = s.row0 + it.tok0;
    it.r0 = (uint32_t)rb * p.rows_per_item;
    it.nrows = min(p.rows_per_item, p.out_dim - it.r0);
    return true;
}

template <int NT>
__global__ void __launch_bounds__(gv::NTHREADS, 1) k_gemv(const GemvParams p, const __grid_constant__ CUtensorMap tmap) {
    using namespace gv;
    constexpr int AFR = NT * 16;                    // activation fragment bytes per lane per block (fp16)
    constexpr int KA = (ACT_BYTES / (32 * AFR)) / KC * KC;   // blocks per activation chunk (96 or 48)

    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t *ring = smem;
    uint8_t *act = smem + RING_BYTES;
    float *dxs = reinterpret_cast<float *>(act + ACT_BYTES);
    uint64_t *bars = reinterpret_cast<uint64_t *>(dxs + DX_FLOATS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(bars + NW * NSLOT);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
    if (threadIdx.x == 0) {
        *abort_flag = 0;
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap)) : "memory");
    }
    if (lane == 0)
        for (int s = 0; s < NSLOT; ++s) mbar_init(&bars[warp * NSLOT + s], 1);
    fence_mbar_init();
    __syncthreads();

    const uint32_t nb = p.nb;
    const uint32_t nslots_row = (nb + KC - 1) / KC;          // weight slots per row
    const int kachunks = (int)((nb + KA - 1) / KA);
    uint8_t *myring = ring + (size_t)warp * NSLOT * SLOT;
    uint64_t *mybar = bars + warp * NSLOT;
    bool waited_dep = false;
    uint32_t qbase = 0;      // this warp's slots issued over all items (ring position and phase)

    for (int item_i = blockIdx.x;; item_i += gridDim.x) {
        GItem it;
        if (!gemv_item<NT>(p, item_i, it)) break;
        const int nsub = (int)((it.nrows + ROWS - 1) / ROWS);
        int wpi = (int)p.wpi;
        while (wpi > 1 && nsub * wpi > NW) wpi >>= 1;
        const int slice = warp % wpi;                        // this warp's K slice
        const int lane_group = warp / wpi;                   // which sub-item stream
        const int ngroups = NW / wpi;
        int my_nsub = 0;
        for (int s = lane_group; s < nsub; s += ngroups) ++my_nsub;
        if (my_nsub > SUBMAX) my_nsub = SUBMAX;              // the host keeps nsub <= ngroups*SUBMAX

        // This warp streams, for k = slice, slice+wpi, ... (its K slice) and for
        // each of its sub-items, one 16-row x KC-block slot.  Slot sequence
        // number q (k-major, sub-items inner); the ring position and mbarrier
        // phase come from the warp's running count gq = qbase + q.
        const uint32_t my_k = (nslots_row > (uint32_t)slice) ? (nslots_row - slice + wpi - 1) / wpi : 0;
        const uint32_t total = (uint32_t)my_nsub * my_k;
        auto issue = [&](uint32_t q) {
            if (lane == 0) {
                const uint32_t kk = q / (uint32_t)my_nsub;
                const int sub = (int)(q - kk * (uint32_t)my_nsub);
                const uint32_t kslot = (uint32_t)slice + kk * (uint32_t)wpi;
                const uint32_t gq = qbase + q;
                const int slot = (int)(gq % NSLOT);
                const uint32_t rs = it.r0 + (uint32_t)(lane_group + sub * ngroups) * ROWS;
                mbar_arrive_expect_tx(&mybar[slot], SLOT);
                tma_load_3d(myring + slot * SLOT, &tmap, (int)(kslot * (KC * QB / 4)), (int)rs, it.expert,
                            &mybar[slot]);
            }
        };

        uint64_t acc[SUBMAX][NT][2];   // packed fp32 pairs: [row g | row g+8] x tokens (2c, 2c+1)
#pragma unroll
        for (int s = 0; s < SUBMAX; ++s)
#pragma unroll
            for (int t = 0; t < NT; ++t) acc[s][t][0] = acc[s][t][1] = 0ull;

        for (uint32_t q0 = 0; q0 < total && q0 < NSLOT; ++q0) issue(q0);
        // The shared-memory ring holds only NSLOT slots per warp; ask L2 for all
        // of this warp's remaining slots now, so that HBM sees the whole item's
        // bytes at once and the ring refills from L2.
        if (lane == 0) {
            for (uint32_t q = NSLOT; q < total; ++q) {
                const uint32_t kq = q / (uint32_t)my_nsub;
                const int sub = (int)(q - kq * (uint32_t)my_nsub);
                const uint32_t kslot = (uint32_t)slice + kq * (uint32_t)wpi;
                const uint32_t rs = it.r0 + (uint32_t)(lane_group + sub * ngroups) * ROWS;
                tma_prefetch_l2_3d(&tmap, (int)(kslot * (KC * QB / 4)), (int)rs, it.expert);
            }
        }
        if (!waited_dep) {
            grid_dep_wait();      // activations are written by the preceding kernel
            waited_dep = true;
        }

        uint32_t kk = 0;
        for (int ch = 0; ch < kachunks; ++ch) {
            const uint32_t kb0 = (uint32_t)ch * KA;
            const uint32_t ka = min((uint32_t)KA, nb - kb0);
            // ---- stage this chunk's activation fragments (all warps), then sync
            __syncthreads();
            for (uint32_t e = threadIdx.x; e < ka * 32; e += NTHREADS) {
                const uint32_t b = e >> 5, l = e & 31;
                const uint32_t lg = l >> 2, lc = l & 3;
                const bool even = ((kb0 + b) & 1u) == 0;
                const int8_t *xr = p.qx + (uint64_t)(it.xrow0 + lg) * p.in_dim + (uint64_t)(kb0 + b) * QK;
                uint4 *dst = reinterpret_cast<uint4 *>(act + ((size_t)b * 32 + l) * AFR);
                // words of the activation block this lane's fragment is built from
                //   odd block: words c, 4+c;  even block: x[4c+2..4c+5] from words c, c+1 and
                //   x[4c+18..4c+21] from words c+4, c+5 (c < 3); lane 3: x[14..17] from words 3, 4
                //   and [x0, x1, x30, x31] from words 0, 7.
                const uint32_t i0 = even ? lc : lc;
                const uint32_t i1 = even ? lc + 1 : 4 + lc;
                const uint32_t i2 = lc < 3 ? lc + 4 : 0u;
                const uint32_t i3 = lc < 3 ? lc + 5 : 7u;
#pragma unroll
                for (int t = 0; t < NT; ++t) {
                    const uint32_t *xt = reinterpret_cast<const uint32_t *>(xr + (uint64_t)t * 8 * p.in_dim);
                    const uint32_t w0 = __ldg(xt + i0), w1 = __ldg(xt + i1);
                    uint32_t f0, f1;
                    if (!even) {
                        f0 = w0;
                        f1 = w1;
                    } else {
                        const uint32_t w2 = __ldg(xt + i2), w3 = __ldg(xt + i3);
                        f0 = funnel16(w0, w1);
                        f1 = lc < 3 ? funnel16(w2, w3) : __byte_perm(w2, w3, 0x7610);
                    }
                    uint4 h;
                    s8x4_to_h2x2(f0, h.x, h.y);   // MMA over the first quant group: b0, b1
                    s8x4_to_h2x2(f1, h.z, h.w);   // MMA over the second quant group
                    dst[t] = h;
                }
            }
            for (uint32_t e = threadIdx.x; e < ka * 16; e += NTHREADS) {
                const uint32_t b = e >> 4, t = e & 15;
                dxs[e] = (t < (uint32_t)(NT * 8)) ? __ldg(p.dx + (uint64_t)(it.xrow0 + t) * nb + kb0 + b) : 0.0f;
            }
            __syncthreads();
            // ---- consume this warp's slots whose K lies in the chunk
            for (; kk < my_k; ++kk) {
                const uint32_t kb = ((uint32_t)slice + kk * (uint32_t)wpi) * KC;
                if (kb >= kb0 + ka) break;                        // belongs to the next chunk
#pragma unroll
                for (int s = 0; s < SUBMAX; ++s) {
                    if (s < my_nsub) {
                        const uint32_t q = kk * (uint32_t)my_nsub + s;
                        const uint32_t gq = qbase + q;
                        const int slot = (int)(gq % NSLOT);
                        mbar_wait(&mybar[slot], (gq / NSLOT) & 1u, p.err, abort_flag);
                        const uint8_t *r0base = myring + slot * SLOT + g * SROW;
                        const uint32_t bl0 = kb - kb0;                    // first block of the slot in the chunk
                        const uint8_t *abase = act + ((size_t)bl0 * 32 + lane) * AFR;
                        const float *dbase = dxs + bl0 * 16 + 2 * c;
                        // Every slot holds KC = 8 blocks (nb % 8 == 0): 4 pairs.
#pragma unroll
                        for (uint32_t jp = 0; jp < KC / 2; ++jp) {
                            const uint8_t *e0 = r0base + jp * (2 * QB);   // even block, row g
                            const uint8_t *e8 = e0 + 8 * SROW;            // even block, row g+8
                            uint32_t w[2][4];   // [block][row g lo, row g+8 lo, row g hi, row g+8 hi]
                            {
                                const uint32_t sel = c < 3 ? 0x3210u : 0x5432u;
                                w[0][0] = lds32g(e0 + even_off_a(c));
                                w[0][1] = lds32g(e8 + even_off_a(c));
                                w[0][2] = __byte_perm(lds32g(e0 + even_off_b(c)), lds32g(e0 + 32), sel);
                                w[0][3] = __byte_perm(lds32g(e8 + even_off_b(c)), lds32g(e8 + 32), sel);
                            }
                            w[1][0] = lds32g(e0 + QB + 2 + 4 * c);
                            w[1][1] = lds32g(e8 + QB + 2 + 4 * c);
                            w[1][2] = lds32g(e0 + QB + 18 + 4 * c);
                            w[1][3] = lds32g(e8 + QB + 18 + 4 * c);
                            uint64_t dw0[2], dw8[2];
                            dw0[0] = pack_same(half_bits_to_float(*reinterpret_cast<const uint16_t *>(e0)));
                            dw8[0] = pack_same(half_bits_to_float(*reinterpret_cast<const uint16_t *>(e8)));
                            dw0[1] = pack_same(half_bits_to_float(*reinterpret_cast<const uint16_t *>(e0 + QB)));
                            dw8[1] = pack_same(half_bits_to_float(*reinterpret_cast<const uint16_t *>(e8 + QB)));
#pragma unroll
                            for (int h = 0; h < 2; ++h) {
                                const uint32_t bo = 2 * jp + h;                // block within the slot
                                uint32_t h0l, h0h, h1l, h1h, h2l, h2h, h3l, h3h;
                                s8x4_to_h2x2(w[h][0], h0l, h0h);     // row g,   first group
                                s8x4_to_h2x2(w[h][1], h1l, h1h);     // row g+8, first group
                                s8x4_to_h2x2(w[h][2], h2l, h2h);     // row g,   second group
                                s8x4_to_h2x2(w[h][3], h3l, h3h);     // row g+8, second group
                                const uint4 *af = reinterpret_cast<const uint4 *>(abase + (size_t)bo * 32 * AFR);
#pragma unroll
                                for (int t = 0; t < NT; ++t) {
                                    const uint64_t dx01 = *reinterpret_cast<const uint64_t *>(dbase + bo * 16 + t * 8);
                                    const uint4 b4 = af[t];
                                    float d[4] = {0.f, 0.f, 0.f, 0.f};
                                    mma_f16_16816(d, h0l, h1l, h0h, h1h, b4.x, b4.y);
                                    mma_f16_16816(d, h2l, h3l, h2h, h3h, b4.z, b4.w);
                                    scale_acc64(acc[s][t][0], d[0], d[1], dx01, dw0[h]);
                                    scale_acc64(acc[s][t][1], d[2], d[3], dx01, dw8[h]);
                                }
                            }
                        }
                        // slot consumed: refill it with the slot NSLOT ahead
                        __syncwarp();
                        fence_proxy_async_smem();
                        if (q + NSLOT < total) issue(q + NSLOT);
                    }
                }
            }
        }
        qbase += total;

        // ---- split-K partials (wpi > 1): add in slice order through shared memory
        float accf[SUBMAX][NT][4];
#pragma unroll
        for (int s = 0; s < SUBMAX; ++s)
#pragma unroll
            for (int t = 0; t < NT; ++t) {
                accf[s][t][0] = lo_of(acc[s][t][0]);
                accf[s][t][1] = hi_of(acc[s][t][0]);
                accf[s][t][2] = lo_of(acc[s][t][1]);
                accf[s][t][3] = hi_of(acc[s][t][1]);
            }
        if (wpi > 1) {
            __syncthreads();   // activation buffer reused for the partials
            float *red = reinterpret_cast<float *>(act);
            if (slice > 0) {
#pragma unroll
                for (int s = 0; s < SUBMAX; ++s)
#pragma unroll
                    for (int t = 0; t < NT; ++t)
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            red[(((warp * SUBMAX + s) * NT + t) * 4 + e) * 32 + lane] = accf[s][t][e];
            }
            __syncthreads();
            if (slice == 0) {
                for (int k = 1; k < wpi; ++k) {
                    const int w2 = warp + k;
#pragma unroll
                    for (int s = 0; s < SUBMAX; ++s)
#pragma unroll
                        for (int t = 0; t < NT; ++t)
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                accf[s][t][e] += red[(((w2 * SUBMAX + s) * NT + t) * 4 + e) * 32 + lane];
                }
            }
        }
        // ---- outputs
        if (slice == 0) {
#pragma unroll
            for (int s = 0; s < SUBMAX; ++s) {
                if (s < my_nsub) {
                    const uint32_t rs = it.r0 + (uint32_t)(lane_group + s * ngroups) * ROWS;
#pragma unroll
                    for (int t = 0; t < NT; ++t) {
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int tok = t * 8 + 2 * c + (e & 1);
                            const uint32_t row = rs + g + ((e & 2) ? 8 : 0);
                            if (tok < it.ntok && row < it.r0 + it.nrows) {
                                const int64_t orow = p.plan ? (int64_t)p.row_to_out[it.xrow0 + tok]
                                                            : (int64_t)(it.tok0 + tok);
                                if (orow >= 0) p.out[(uint64_t)orow * p.out_dim + row] = accf[s][t][e];
                            }
                        }
                    }
                }
            }
        }
        __syncthreads();   // item boundary: activation buffer reuse
    }
    if (!waited_dep) grid_dep_wait();
}

bool encode_rows_tmap(CUtensorMap *map, const void *W, uint64_t row_bytes, uint64_t rows, uint64_t n_mat,
                      uint64_t mat_stride, uint32_t box_words, uint32_t box_rows);

cudaError_t launch_gemv(const GemvParams &p, bool two_tiles, int grid, cudaStream_t st) {
    static bool attr_done[2] = {false, false};
    const void *fn = two_tiles ? (const void *)k_gemv<2> : (const void *)k_gemv<1>;
    if (!attr_done[two_tiles]) {
        cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)gv::SMEM);
        if (e != cudaSuccess) return e;
        attr_done[two_tiles] = true;
    }
    alignas(64) CUtensorMap tmap;
    const uint64_t row_bytes = (uint64_t)p.nb * QB;
    const uint64_t mats = p.plan ? p.n_expert : 1;
    if (!encode_rows_tmap(&tmap, p.W, row_bytes, p.out_dim, mats, p.plan ? p.expert_stride : (uint64_t)p.out_dim * row_bytes,
                          gv::BOX_WORDS, gv::ROWS))
        return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(gv::NTHREADS);
    cfg.dynamicSmemBytes = gv::SMEM;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    GemvParams pp = p;
    void *args[] = {&pp, &tmap};
    return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace q8
