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
//   * A CTA item is (segment, token group, row range).  The row range is cut into
//     16-row sub-items; the weights of an item stream through shared memory as
//     slots of 16 rows x 8 blocks, one tiled TMA copy (cp.async.bulk.tensor) per
//     slot over a tensor map that views the raw rows as 32-bit words with a
//     76-word box, so rows land 304 bytes apart (an odd multiple of 16 bytes:
//     the fragment loads below are bank-conflict free).  The box's last 32 bytes
//     per row belong to the next slot and are not used; words past the end of a
//     row and rows past out_dim are filled with zeros by the TMA.
//   * Warp specialisation.  One producer warp walks the CTA's slot sequence
//     (items in order; within an item, K-slot major and sub-items inner) and
//     issues every copy into a CTA-wide ring of 32 slots (152 KB in flight),
//     reusing a slot once its consumer has released it.  TMA issue stalls while
//     the SM's copy queue drains at the HBM rate, so only this warp ever waits
//     there.  Fourteen consumer warps own the sub-items (G = 14 / wpi groups,
//     sub-item s in group s mod G) and, when an item has fewer than 14
//     sub-items, wpi warps (2, 7 or 14) split its K slots and add their
//     partial sums through shared memory in a fixed order.  Consecutive slots of the
//     sequence belong to different warps, so the ring drains in arrival order.
//   * The token group's activations are staged once per K chunk by the consumer
//     warps, in the order the mode's inner loop reads them.
//   * Modes.  Mode 0 (at most 2 tokens): dp4a.  A lane owns one block column j
//     of the slot and four of its rows; it reads the block's 9 words, aligns the
//     quants with one byte permute per word and forms the int32 block dot with
//     8 dp4a per token; the 8 block columns of a row are added by shuffles at
//     the end.  Modes 1 and 2 (8 or 16 tokens): mma.sync m16n8k16 in fp16 on the
//     exact int8 values, one or two 8-token N tiles.  The weight fragment (rows
//     g and g+8, two 4-byte groups of quants per lane) comes from 32-bit shared
//     loads.  The sum over a block's 32 products does not depend on their order,
//     so each lane may take any fixed set of quant positions as long as the
//     activation fragment uses the same one: odd blocks (quants 4-byte aligned)
//     use the natural MMA order; even blocks (quants at 2 mod 4) give lanes 0-2
//     two aligned words each and lane 3 one aligned word plus the four edge
//     bytes joined by one byte permute, and the staged activations are permuted
//     to match.  fp32 accumulation of each block dot is exact (products below
//     2^14, block sums below 2^24); it is then scaled by d_w*d_x and added in
//     fp32 with packed f32x2 instructions.  fp16 rather than int8 MMA: on GB300
//     mma.sync runs int8 at 251 and fp16 at 942 MAC per SM per clock (measured).
//   * Gate/up pair (the routed FFN's first step, ds4 GPU code walkthrough, trace 5):
//     an item streams the gate's sub-items and then the up's, same rows, against
//     one staging of its activations; their results are staged side by side and
//     the epilogue writes swiglu1(gate, up) instead of either product.
//   * Small activations (at most 8 tokens, 1024 token-block pairs per CTA) are
//     quantised by the consumer warps themselves from the fp32 rows, with the
//     quantiser kernels' arithmetic: one kernel per call.  Otherwise the
//     quantiser kernel writes activation planes first.
//   * Launched with programmatic stream serialisation, so the launch and the
//     barrier set-up overlap the end of the preceding kernel.  Nothing written
//     by an earlier kernel is read before griddepcontrol.wait, except the
//     weights (which no kernel that triggers its dependents early writes),
//     behind this library's quantiser and in fused calls of 1-2 tokens: then
//     the first eight weight copies per SM go out before the wait (dense calls;
//     grouped calls stream on), the rest once it returns.  This kernel does not trigger early: measured
//     on GB300, an early trigger sped up runs of equal calls but slowed a
//     mixed decode step (a fused call followed by quantiser + GEMV) by 10 %.
#include <cuda.h>

#include "q8_common.cuh"
#include "q8_kernels.h"
#include "q8_quant.cuh"

namespace q8 {

namespace gv {
constexpr int NCW = 14;                          // consumer warps (15 warps: 128 registers each)
constexpr int PRODUCER = NCW;                    // warp index of the TMA producer
constexpr int NTHREADS = (NCW + 1) * 32;
constexpr int CONSUMER_THREADS = NCW * 32;
constexpr int ROWS = 16;                         // rows per sub-item
constexpr int KC = 8;                            // blocks per weight slot
constexpr int BOX_WORDS = (KC * QB + 32) / 4;    // 76 words per row of a slot
constexpr int SROW = BOX_WORDS * 4;              // 304 bytes: 19 x 16, an odd multiple of 16
constexpr int SLOT = ROWS * SROW;                // 4864 bytes
constexpr int NSLOT = 32;                        // CTA ring depth
constexpr uint32_t EARLY_SLOTS = 8;              // dense copies issued ahead of the grid dependency
constexpr int SUBMAX = (512 + NCW * 16 - 1) / (NCW * 16);   // sub-items per warp per CTA item
constexpr int ACT_BYTES = 40 * 1024;             // staged activations per chunk
constexpr int DX_FLOATS = 1280;                  // staged activation scales per chunk
constexpr int RING_BYTES = NSLOT * SLOT;
constexpr int QT_BYTES = 20736;                  // qtmp: natural-order quants of a chunk (fused quantiser, planes staging)
constexpr size_t SMEM = RING_BYTES + ACT_BYTES + DX_FLOATS * 4 + QT_BYTES + 2 * NSLOT * 8 + NSLOT * 4 + 16;
constexpr int BAR_CONSUMERS = 1;                 // named barrier of the consumer warps
constexpr int OUT_STRIDE = GEMV_MAX_ROWS_PER_ITEM;   // output staging: floats per token
static_assert(16 * OUT_STRIDE * 4 <= ACT_BYTES, "output staging fits the activation buffer");
static_assert(SMEM <= 227 * 1024, "shared memory");
static_assert(NSLOT >= 32, "one producer lane per slot of a batch");
static_assert(SUBMAX * NCW * ROWS >= GEMV_MAX_ROWS_PER_ITEM, "rows per item");
// Modes: 0 = dp4a, up to 2 tokens; 1 = fp16 MMA, one 8-token N tile; 2 = two N tiles.
template <int MODE> struct Mode {
    static constexpr int TOKG = MODE == 0 ? 2 : MODE * 8;          // tokens per group
    static constexpr int NT = MODE == 0 ? 1 : MODE;                // MMA N tiles
    static constexpr int ACT_BLOCK = MODE == 0 ? 80 : MODE * 512;   // staged activation bytes per block
    static constexpr int DXW = MODE == 0 ? 2 : 16;                  // staged scales per block
    static constexpr int KA = (ACT_BYTES / ACT_BLOCK) / KC * KC;    // blocks per chunk (512, 80, 40)
    static constexpr int NACC = MODE == 0 ? 8 : NT * 4;             // fp32 results per lane and sub-item
    static_assert(KA * DXW <= DX_FLOATS, "scale buffer");
    static_assert(NCW * NACC * 32 * 4 <= ACT_BYTES, "split-K buffer");
    static constexpr int QT_STRIDE = KA * QK + 16;                  // qtmp: bytes per token row of a chunk
    static_assert(MODE == 0 || TOKG * QT_STRIDE <= QT_BYTES, "fused quantiser buffer");
};
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

__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }


// dp4a mode: the four rows of a sub-item that lane group rb (lanes 8rb..8rb+7,
// one weight block each) reads in step i.  The sets {0,3,4,7} and {1,2,5,6} (and
// the same plus 8) put the 32 lanes' word addresses, block starts 34j bytes
// apart at a row pitch of 76 words, in 32 different banks.
__device__ __forceinline__ int dp4a_row(int rb, int i) {
    return (i >> 1) * 8 + (rb >> 1) * 4 + ((i & 1) ? 1 + (rb & 1) : 3 * (rb & 1));
}

// Item decoding.  Returns false past the last item.
struct GItem {
    int expert;
    int xrow0;      // first activation-plane row of the token group
    int ntok;       // tokens in the group
    int tok0;       // index of the first token within its segment
    uint32_t r0;    // first weight row
    uint32_t nrows;
};

// Kernel kinds: the dense product, a grouped (routed) one, a grouped gate/up pair.
constexpr int KIND_DENSE = 0, KIND_GROUPED = 1, KIND_PAIR = 2;

// GROUPED: p.plan is set (the variants are separate so that the dense kernel
// carries none of the plan decoding).
// Work enumeration (the producer and the consumers walk the same sequence).
// Dense: n_items contiguous ranges of whole sub-items, sizes differing by at most
// one (the split is computed on the host: a 64-bit division here would delay the
// first weight copy), dealt in turn.  Grouped: the class's work is the sequence
// of its token groups (plan order) times the output's units of U sixteen-row
// sub-items (U = 2 when a gate/up pair writes Q8_0 planes: whole 32-row blocks);
// CTA c takes units [c S / G, (c + 1) S / G) of the S units, so every SM streams
// the same amount, cut into items at token-group ends and after rows_per_item
// rows.  (Items of whole row blocks dealt in turn left the CTAs 6 or 7 items of
// up to 28 sub-items: 7 % of the stream idle at the decode size.)
struct ItemCursor {
    int i;                 // dense: the next item index
    uint64_t pos, end;     // grouped: the next unit and the end of this CTA's range
};

template <bool GROUPED>
__device__ __forceinline__ uint32_t group_units(const GemvParams &p) {
    const uint32_t u = (GROUPED && p.W2 && p.q_out) ? 2u : 1u;
    return ((p.out_dim + 15) / 16 + u - 1) / u;
}

template <bool GROUPED>
__device__ __forceinline__ void cursor_init(const GemvParams &p, ItemCursor &c) {
    c.i = (int)blockIdx.x;
    c.pos = c.end = 0;
    if constexpr (GROUPED) {
        const int n_rb = (int)((p.out_dim + p.rows_per_item - 1) / p.rows_per_item);
        const int prb = p.plan_rb ? (int)p.plan_rb : n_rb;
        // a GEMV class's item count is a multiple of the plan's row blocks per group
        const uint64_t total = (uint64_t)(p.plan->n_items / prb) * group_units<GROUPED>(p);
        c.pos = total * blockIdx.x / gridDim.x;
        c.end = total * (blockIdx.x + 1) / gridDim.x;
    }
}

// Returns false past the CTA's last item.
template <int TOKG, bool GROUPED>
__device__ __forceinline__ bool next_item(const GemvParams &p, ItemCursor &c, GItem &it) {
    if constexpr (!GROUPED) {
        const int i = c.i;
        c.i += (int)gridDim.x;
        if ((uint32_t)i >= p.n_items) return false;
        const uint32_t ui = (uint32_t)i;
        const uint32_t s0 = ui * p.sub_base + min(ui, p.sub_rem);
        const uint32_t s1 = s0 + p.sub_base + (ui < p.sub_rem ? 1u : 0u);
        it.expert = 0;
        it.xrow0 = 0;
        it.ntok = (int)p.n_tok;
        it.tok0 = 0;
        it.r0 = s0 * gv::ROWS;
        it.nrows = min((s1 - s0) * gv::ROWS, p.out_dim - it.r0);
        return true;
    } else {
        if (c.pos >= c.end) return false;
        const uint32_t usub = (p.W2 && p.q_out) ? 2u : 1u;   // sub-items a unit
        const uint64_t nu = group_units<GROUPED>(p);
        const uint64_t g = c.pos / nu;                        // token group within the class
        const uint32_t u0 = (uint32_t)(c.pos - g * nu);
        const int n_rb = (int)((p.out_dim + p.rows_per_item - 1) / p.rows_per_item);
        const int prb = p.plan_rb ? (int)p.plan_rb : n_rb;
        // the segment holding group g: its item_start / prb groups come before it
        const int gstart = (int)g * prb;
        const Segment *segs = reinterpret_cast<const Segment *>(p.plan + 1);
        int lo = 0, hi = p.plan->n_segments - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (segs[mid].item_start <= gstart) lo = mid;
            else hi = mid - 1;
        }
        const Segment s = segs[lo];
        const int tg = (int)g - s.item_start / prb;
        const uint64_t maxu = p.rows_per_item / (gv::ROWS * usub);
        uint64_t cnt = c.end - c.pos;
        if (cnt > nu - u0) cnt = nu - u0;
        if (cnt > maxu) cnt = maxu;
        it.expert = s.expert;
        it.tok0 = tg * TOKG;
        it.ntok = min(TOKG, s.count - it.tok0);
        it.xrow0 = s.row0 + it.tok0;
        it.r0 = u0 * usub * gv::ROWS;
        it.nrows = min((uint32_t)cnt * usub * gv::ROWS, p.out_dim - it.r0);
        c.pos += cnt;
        return true;
    }
}

// Bounded wait until the producer has armed round r of a slot.
__device__ __forceinline__ bool wait_armed(volatile uint32_t *armed, uint32_t r, int *err, volatile int *abort,
                                           uint64_t limit_ns) {
    if (*armed == r) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (*armed == r) return true;
        if ((it & 63u) == 0u) {
            if (*abort) return false;
            if (global_timer_ns() - t0 > limit_ns) {
                raise_error(err, DEV_ETIMEOUT);
                *abort = 1;
                return false;
            }
        }
    }
}

// Warps per sub-item for an item of nsub sub-items and nk K slots: the largest
// divisor of the consumer count (1, 2, 7, 14) that keeps every sub-item on its
// own group of wpi warps, with a K slot for each warp (so with wpi > 1 each warp
// holds one sub-item).  A single 16-row sub-item is split over all 14 warps.
__device__ __forceinline__ uint32_t item_wpi(uint32_t nsub, uint32_t nk) {
    uint32_t wpi = 1;
    for (uint32_t d = 2; d <= (uint32_t)gv::NCW; ++d)
        if (gv::NCW % d == 0 && nsub * d <= (uint32_t)gv::NCW && d <= nk) wpi = d;
    return wpi;
}

// The producer warp: every slot of every item of this CTA, in order, 32 at a
// time (lane l issues slot base + l).  One thread issuing alone is limited to
// about one tiled copy per 170 ns, well below the HBM rate; 32 lanes are not.
// After arming a slot's full barrier for round r (its use number) the lane
// publishes r in armed[slot].  Consumers of different warps take different
// slots and copies land out of order, so a warp may come to round r + 1 of a
// slot while round r has not landed; its parity wait would then see the
// previous phase as complete.  Waiting for armed[slot] == r first rules that
// out.  After an abort (a timed-out wait anywhere in the CTA) no further copy
// is issued, and consumers release only slots whose copy they saw land, so a
// slot never has two copies in flight: the drain at the end waits for each
// slot's last armed round only.  Returns the number of slots planned.
template <int TOKG, int KIND>
__device__ __forceinline__ uint32_t produce(const GemvParams &p, const CUtensorMap *tmap, const CUtensorMap *tmap2,
                                            uint8_t *ring, uint64_t *full, uint64_t *empty, volatile uint32_t *armed,
                                            volatile int *abort_flag, int lane, uint64_t lim) {
    using namespace gv;
    const uint32_t nk = (p.nb + KC - 1) / KC;
    uint32_t seqbase = 0;
    GItem it;
    constexpr bool PAIR = KIND == KIND_PAIR;
    ItemCursor cur;
    cursor_init<KIND != KIND_DENSE>(p, cur);
    while (next_item<TOKG, KIND != KIND_DENSE>(p, cur, it)) {
        const uint32_t nh = (it.nrows + ROWS - 1) / ROWS;   // sub-items of one matrix
        const uint32_t nsub = PAIR ? 2 * nh : nh;           // a pair: the gate's, then the up's
        const uint32_t total = nk * nsub;
        for (uint32_t base = 0; base < total; base += 32) {
            const uint32_t idx = base + (uint32_t)lane;
            // A dense call streaming ahead of griddepcontrol.wait (behind this
            // library's quantiser, or a fused 1-2-token call) issues only its first
            // EARLY_SLOTS copies before the wait, so that the consumers' activation
            // loads, issued once the wait returns, queue behind 39 KB of weights per SM
            // instead of 152 KB (decode step 31.3 -> 31.0 us; fused 1-token calls 7.5
            // us against 8.6 with every copy early; the grouped calls measured 1 %
            // slower with it).
            const bool hold = KIND == KIND_DENSE && p.weights_early && seqbase == 0 && base == 0;
            for (int pass = 0; pass < (hold ? 2 : 1); ++pass) {
                if (pass == 1) {
                    __syncwarp();
                    grid_dep_wait();
                }
                const bool mine = !hold || (pass == 0 ? idx < EARLY_SLOTS : idx >= EARLY_SLOTS);
                if (mine && idx < total) {
                    const uint32_t seq = seqbase + idx, slot = seq % NSLOT;
                    const uint32_t kk = idx / nsub, sub = idx - kk * nsub;
                    const bool second = PAIR && sub >= nh;
                    if (!p.withhold && mbar_wait(&empty[slot], ((seq / NSLOT) & 1u) ^ 1u, p.err, abort_flag, lim) &&
                        !*abort_flag) {
                        mbar_arrive_expect_tx(&full[slot], SLOT);
                        tma_load_3d(ring + (size_t)slot * SLOT, second ? tmap2 : tmap, (int)(kk * (KC * QB / 4)),
                                    (int)(it.r0 + (second ? sub - nh : sub) * ROWS), it.expert, &full[slot]);
                        __threadfence_block();
                        armed[slot] = seq / NSLOT;
                    }
                }
            }
            __syncwarp();
        }
        seqbase += total;
    }
    return seqbase;
}

// Stage one K chunk [kb0, kb0 + ka) of the token group's activations from the
// Q8_0 planes (consumer threads only; qtmp is the MMA modes' shared-memory
// copy of the rows).  All global loads of a thread are issued before any is used:
// under a saturated HBM stream each round trip costs a microsecond or more.
template <int MODE, bool TWO_PHASE>
__device__ __forceinline__ void stage_chunk(const GemvParams &p, const GItem &it, uint32_t kb0, uint32_t ka,
                                            uint8_t *act, float *dxs, uint8_t *qtmp) {
    using namespace gv;
    using M = Mode<MODE>;
    constexpr int NT = M::NT;
    const uint32_t nb = p.nb;
    if (MODE == 0) {
        // [block][token][8 words], 80 bytes per block.  The words are arranged to
        // meet the weight words of the block where they lie in the row:
        //   odd block (quants word-aligned, q0..q31 in words 1..8 of the read):
        //     A[0] = X[7], A[k] = X[k-1]
        //   even block (quants at 2 mod 4, words 1..7 hold q2..q29, the edge word
        //   holds q0, q1, q30, q31):  A[0] = [x0, x1, x30, x31], A[k] = x[4k-2 .. 4k+1]
        for (uint32_t e = threadIdx.x; e < ka * 2; e += CONSUMER_THREADS) {
            const uint32_t b = e >> 1, t = e & 1;
            uint32_t X[8] = {0, 0, 0, 0, 0, 0, 0, 0};
            float d = 0.0f;
            if (t < (uint32_t)it.ntok) {
                const uint4 *src = reinterpret_cast<const uint4 *>(p.qx + (uint64_t)(it.xrow0 + t) * p.in_dim +
                                                                   (uint64_t)(kb0 + b) * QK);
                const uint4 v0 = __ldg(src), v1 = __ldg(src + 1);
                d = __ldg(p.dx + (uint64_t)(it.xrow0 + t) * nb + kb0 + b);
                X[0] = v0.x; X[1] = v0.y; X[2] = v0.z; X[3] = v0.w;
                X[4] = v1.x; X[5] = v1.y; X[6] = v1.z; X[7] = v1.w;
            }
            uint32_t A[8];
            if ((kb0 + b) & 1u) {
                A[0] = X[7];
#pragma unroll
                for (int k = 1; k < 8; ++k) A[k] = X[k - 1];
            } else {
                A[0] = __byte_perm(X[0], X[7], 0x7610);
#pragma unroll
                for (int k = 1; k < 8; ++k) A[k] = funnel16(X[k - 1], X[k]);
            }
            uint4 *dst = reinterpret_cast<uint4 *>(act + (size_t)b * M::ACT_BLOCK + t * 32);
            dst[0] = make_uint4(A[0], A[1], A[2], A[3]);
            dst[1] = make_uint4(A[4], A[5], A[6], A[7]);
            dxs[e] = d;
        }
    } else {
        // MMA B fragments, fp16: [block][N tile][lane][16 bytes].  Rows past the
        // group's ntok are not read (routed planes leave their padding rows
        // unwritten): their fragments and scales are zero.
        // TWO_PHASE (dense calls): the group's token rows of the chunk go to qtmp
        // whole, in 16-byte loads (three per thread, all issued before the first
        // store), with the scales; after a consumer barrier the fragments are
        // built from qtmp.  Otherwise (routed items) each lane gathers its four
        // fragment words per N tile straight from global memory.  A dense call
        // stages once, at its start, where the load latency is exposed: there the
        // two phases are 9% faster at 16 tokens.  Routed items stage while the
        // weight stream runs, and the extra barrier cost them 0.3%.
        // Words of the activation block a lane's fragment is built from:
        //   odd block: words c, 4+c;  even block: x[4c+2..4c+5] from words c, c+1 and
        //   x[4c+18..4c+21] from words c+4, c+5 (c < 3); lane 3: x[14..17] from words 3, 4
        //   and [x0, x1, x30, x31] from words 0, 7.
        if (TWO_PHASE) {
            const uint32_t c16 = ka * (QK / 16);   // 16-byte pieces of a token row in the chunk
            constexpr int RC = (M::TOKG * M::KA * (QK / 16) + CONSUMER_THREADS - 1) / CONSUMER_THREADS;
            constexpr int RD = (M::KA * 16 + CONSUMER_THREADS - 1) / CONSUMER_THREADS;
            uint4 cv[RC];
            float dv[RD];
#pragma unroll
            for (int r = 0; r < RC; ++r) {
                const uint32_t e = threadIdx.x + (uint32_t)r * CONSUMER_THREADS;
                const uint32_t t = e / c16, c = e - t * c16;
                if (t < (uint32_t)it.ntok)
                    cv[r] = __ldg(reinterpret_cast<const uint4 *>(p.qx + (uint64_t)(it.xrow0 + t) * p.in_dim +
                                                                  (uint64_t)kb0 * QK) + c);
            }
#pragma unroll
            for (int r = 0; r < RD; ++r) {
                const uint32_t e = threadIdx.x + (uint32_t)r * CONSUMER_THREADS;
                const uint32_t b = e >> 4, t = e & 15;
                dv[r] = (e < ka * 16 && t < (uint32_t)(NT * 8) && t < (uint32_t)it.ntok)
                            ? __ldg(p.dx + (uint64_t)(it.xrow0 + t) * nb + kb0 + b)
                            : 0.0f;
            }
#pragma unroll
            for (int r = 0; r < RC; ++r) {
                const uint32_t e = threadIdx.x + (uint32_t)r * CONSUMER_THREADS;
                const uint32_t t = e / c16, c = e - t * c16;
                if (t < (uint32_t)it.ntok) *reinterpret_cast<uint4 *>(qtmp + (size_t)t * M::QT_STRIDE + (size_t)c * 16) = cv[r];
            }
#pragma unroll
            for (int r = 0; r < RD; ++r) {
                const uint32_t e = threadIdx.x + (uint32_t)r * CONSUMER_THREADS;
                if (e < ka * 16) dxs[e] = dv[r];
            }
            named_bar_sync(BAR_CONSUMERS, CONSUMER_THREADS);
            for (uint32_t e = threadIdx.x; e < ka * 32; e += CONSUMER_THREADS) {
                const uint32_t b = e >> 5, l = e & 31, lg = l >> 2, lc = l & 3;
                const bool even = ((kb0 + b) & 1u) == 0;
                const uint32_t i1 = even ? lc + 1 : 4 + lc;
                const uint32_t i2 = lc < 3 ? lc + 4 : 0u;
                const uint32_t i3 = lc < 3 ? lc + 5 : 7u;
#pragma unroll
                for (int t = 0; t < NT; ++t) {
                    const uint32_t *xt = reinterpret_cast<const uint32_t *>(qtmp + (size_t)(lg + 8 * t) * M::QT_STRIDE +
                                                                            (size_t)b * QK);
                    uint32_t f0, f1;
                    if (lg + 8 * t >= (uint32_t)it.ntok) {
                        f0 = 0;
                        f1 = 0;
                    } else if (!even) {
                        f0 = xt[lc];
                        f1 = xt[i1];
                    } else {
                        f0 = funnel16(xt[lc], xt[i1]);
                        f1 = lc < 3 ? funnel16(xt[i2], xt[i3]) : __byte_perm(xt[i2], xt[i3], 0x7610);
                    }
                    uint4 h;
                    s8x4_to_h2x2(f0, h.x, h.y);   // MMA over the first 16 quants: b0, b1
                    s8x4_to_h2x2(f1, h.z, h.w);   // MMA over the second 16 quants
                    *reinterpret_cast<uint4 *>(act + (size_t)b * M::ACT_BLOCK + (size_t)t * 512 + (size_t)l * 16) = h;
                }
            }
        } else {
            constexpr int R = (M::KA * 32 + CONSUMER_THREADS - 1) / CONSUMER_THREADS;
            uint32_t wv[R][NT][4];
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const uint32_t e = threadIdx.x + (uint32_t)r * CONSUMER_THREADS;
                if (e < ka * 32) {
                    const uint32_t b = e >> 5, l = e & 31, lg = l >> 2, lc = l & 3;
                    const bool even = ((kb0 + b) & 1u) == 0;
                    const uint32_t i1 = even ? lc + 1 : 4 + lc;
                    const uint32_t i2 = lc < 3 ? lc + 4 : 0u;
                    const uint32_t i3 = lc < 3 ? lc + 5 : 7u;
                    const int8_t *xr = p.qx + (uint64_t)(it.xrow0 + lg) * p.in_dim + (uint64_t)(kb0 + b) * QK;
#pragma unroll
                    for (int t = 0; t < NT; ++t) {
                        if (lg + 8u * (uint32_t)t < (uint32_t)it.ntok) {
                            const uint32_t *xt = reinterpret_cast<const uint32_t *>(xr + (uint64_t)t * 8 * p.in_dim);
                            wv[r][t][0] = __ldg(xt + lc);
                            wv[r][t][1] = __ldg(xt + i1);
                            wv[r][t][2] = __ldg(xt + i2);
                            wv[r][t][3] = __ldg(xt + i3);
                        } else {
                            wv[r][t][0] = wv[r][t][1] = wv[r][t][2] = wv[r][t][3] = 0u;
                        }
                    }
                }
            }
            constexpr int RD = (M::KA * 16 + CONSUMER_THREADS - 1) / CONSUMER_THREADS;
            float dv[RD];
#pragma unroll
            for (int r = 0; r < RD; ++r) {
                const uint32_t e = threadIdx.x + (uint32_t)r * CONSUMER_THREADS;
                const uint32_t b = e >> 4, t = e & 15;
                dv[r] = (e < ka * 16 && t < (uint32_t)(NT * 8) && t < (uint32_t)it.ntok)
                            ? __ldg(p.dx + (uint64_t)(it.xrow0 + t) * nb + kb0 + b)
                            : 0.0f;
            }
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const uint32_t e = threadIdx.x + (uint32_t)r * CONSUMER_THREADS;
                if (e < ka * 32) {
                    const uint32_t b = e >> 5, l = e & 31, lc = l & 3;
                    const bool even = ((kb0 + b) & 1u) == 0;
#pragma unroll
                    for (int t = 0; t < NT; ++t) {
                        uint32_t f0, f1;
                        if (!even) {
                            f0 = wv[r][t][0];
                            f1 = wv[r][t][1];
                        } else {
                            f0 = funnel16(wv[r][t][0], wv[r][t][1]);
                            f1 = lc < 3 ? funnel16(wv[r][t][2], wv[r][t][3]) : __byte_perm(wv[r][t][2], wv[r][t][3], 0x7610);
                        }
                        uint4 h;
                        s8x4_to_h2x2(f0, h.x, h.y);   // MMA over the first 16 quants: b0, b1
                        s8x4_to_h2x2(f1, h.z, h.w);   // MMA over the second 16 quants
                        *reinterpret_cast<uint4 *>(act + (size_t)b * M::ACT_BLOCK + (size_t)t * 512 + (size_t)l * 16) = h;
                    }
                }
            }
#pragma unroll
            for (int r = 0; r < RD; ++r) {
                const uint32_t e = threadIdx.x + (uint32_t)r * CONSUMER_THREADS;
                if (e < ka * 16) dxs[e] = dv[r];
            }
        }
    }
}

// Fused quantiser (dense path, x given): the CTA quantises tokens 0..TOKG-1 of
// chunk [kb0, kb0 + ka) from the fp32 rows itself, with the arithmetic of the
// quantiser kernels (four lanes per block), and writes the mode's layout.
// Only the group's real tokens are quantised; padding tokens get zero
// fragments and scales.  Loads are issued three rounds at a time before use.
template <int MODE>
__device__ __forceinline__ void stage_chunk_fused(const GemvParams &p, const GItem &it, uint32_t kb0, uint32_t ka,
                                                  uint8_t *act, float *dxs, uint8_t *qtmp) {
    using namespace gv;
    using M = Mode<MODE>;
    constexpr uint32_t GROUPS = CONSUMER_THREADS / 4;
    const uint32_t lane_q = threadIdx.x & 3u;
    const uint32_t ntok = (uint32_t)it.ntok;              // <= M::TOKG
    const uint32_t npair = ka * ntok;                     // (token, block) pairs, token-major
    const uint32_t rounds = (npair + GROUPS - 1) / GROUPS;
    constexpr int RB = 3;                                 // rounds whose loads are in flight together
    if (MODE != 0)   // padding tokens: zero scales (their fragments are zero, see below)
        for (uint32_t e = threadIdx.x; e < ka * 16; e += CONSUMER_THREADS)
            if ((e & 15u) >= ntok) dxs[e] = 0.0f;
    for (uint32_t r0 = 0; r0 < rounds; r0 += RB) {
        float xv[RB][8];
#pragma unroll
        for (int h = 0; h < RB; ++h) {
            const uint32_t pr = threadIdx.x / 4 + (r0 + h) * GROUPS;
            const uint32_t t = pr / ka, b = pr - t * ka;
            if (pr < npair)
                load8(xv[h], p.x + (uint64_t)t * p.in_dim + (uint64_t)(kb0 + b) * QK + lane_q * 8);
            else {
#pragma unroll
                for (int i = 0; i < 8; ++i) xv[h][i] = 0.0f;
            }
        }
#pragma unroll
        for (int h = 0; h < RB; ++h) {
            const uint32_t pr = threadIdx.x / 4 + (r0 + h) * GROUPS;
            const uint32_t t = pr / ka, b = pr - t * ka;
            const QuantBlock qb = quantize8_div(xv[h]);   // all lanes: the block maximum is shuffled
            const uint32_t lo = qb.lo, hi = qb.hi;
            if (MODE == 0) {
                // lane q holds words X[2q] = lo, X[2q+1] = hi; arrange as in stage_chunk
                const uint32_t nbw = __shfl_sync(0xffffffffu, lo, (threadIdx.x & ~3u) | ((lane_q + 1) & 3u));
                if (pr < npair && r0 + h < rounds) {
                    uint32_t *dst = reinterpret_cast<uint32_t *>(act + (size_t)b * M::ACT_BLOCK + t * 32);
                    if ((kb0 + b) & 1u) {
                        dst[2 * lane_q + 1] = lo;
                        dst[(2 * lane_q + 2) & 7u] = hi;
                    } else {
                        dst[2 * lane_q + 1] = funnel16(lo, hi);
                        if (lane_q < 3) dst[2 * lane_q + 2] = funnel16(hi, nbw);
                        else dst[0] = __byte_perm(nbw, hi, 0x7610);
                    }
                    if (lane_q == 0) dxs[b * 2 + t] = qb.d_stored;
                }
            } else {
                if (pr < npair && r0 + h < rounds) {
                    *reinterpret_cast<uint2 *>(qtmp + (size_t)t * M::QT_STRIDE + (size_t)b * QK + lane_q * 8) =
                        make_uint2(lo, hi);
                    if (lane_q == 0) dxs[b * 16 + t] = qb.d_stored;
                }
            }
        }
    }
    if (MODE == 0) return;
    named_bar_sync(BAR_CONSUMERS, CONSUMER_THREADS);
    // natural-order quants -> MMA B fragments, as stage_chunk does from the planes
    constexpr int NT = M::NT;
    for (uint32_t e = threadIdx.x; e < ka * 32; e += CONSUMER_THREADS) {
        const uint32_t b = e >> 5, l = e & 31, lg = l >> 2, lc = l & 3;
        const bool even = ((kb0 + b) & 1u) == 0;
        const uint32_t i1 = even ? lc + 1 : 4 + lc;
        const uint32_t i2 = lc < 3 ? lc + 4 : 0u;
        const uint32_t i3 = lc < 3 ? lc + 5 : 7u;
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            const uint32_t *xt = reinterpret_cast<const uint32_t *>(qtmp + (size_t)(lg + 8 * t) * M::QT_STRIDE +
                                                                    (size_t)b * QK);
            uint32_t f0, f1;
            if (lg + 8 * t >= ntok) {   // padding token: not quantised, zero fragment
                f0 = 0;
                f1 = 0;
            } else if (!even) {
                f0 = xt[lc];
                f1 = xt[i1];
            } else {
                f0 = funnel16(xt[lc], xt[i1]);
                f1 = lc < 3 ? funnel16(xt[i2], xt[i3]) : __byte_perm(xt[i2], xt[i3], 0x7610);
            }
            uint4 hh;
            s8x4_to_h2x2(f0, hh.x, hh.y);
            s8x4_to_h2x2(f1, hh.z, hh.w);
            *reinterpret_cast<uint4 *>(act + (size_t)b * M::ACT_BLOCK + (size_t)t * 512 + (size_t)l * 16) = hh;
        }
    }
}

// dp4a mode, one slot: lane = (row group rb, block column j).  Each row's
// block dot is 8 dp4a over the weight words as they lie in shared memory, the
// activation words having been arranged to match; one byte permute forms the
// edge word (odd block: word 8; even block: q0, q1, q30, q31).
__device__ __forceinline__ void slot_dp4a(const uint8_t *sbase, const uint8_t *act, const float *dxs, uint32_t bl0,
                                          int lane, float (&acc)[8], bool two_tokens) {
    using namespace gv;
    const int j = lane & 7, rb = lane >> 3;
    const uint32_t bl = bl0 + (uint32_t)j;
    const uint4 *xa = reinterpret_cast<const uint4 *>(act + (size_t)bl * Mode<0>::ACT_BLOCK);
    const uint4 x00 = xa[0], x01 = xa[1];
    const uint32_t A0[8] = {x00.x, x00.y, x00.z, x00.w, x01.x, x01.y, x01.z, x01.w};
    uint32_t A1[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    if (two_tokens) {
        const uint4 x10 = xa[2], x11 = xa[3];
        A1[0] = x10.x; A1[1] = x10.y; A1[2] = x10.z; A1[3] = x10.w;
        A1[4] = x11.x; A1[5] = x11.y; A1[6] = x11.z; A1[7] = x11.w;
    }
    const float dx0 = dxs[bl * 2], dx1 = dxs[bl * 2 + 1];
    // block j starts at byte 34j of the row: word-aligned when j is even, else at 2 mod 4
    const uint32_t sel = (j & 1) ? 0x7654u : 0x5432u;
    const int wbase = (34 * j) >> 2;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t *wr = reinterpret_cast<const uint32_t *>(sbase + dp4a_row(rb, i) * SROW) + wbase;
        uint32_t W[9];
#pragma unroll
        for (int k = 0; k < 9; ++k) W[k] = wr[k];
        const uint32_t dbits = (j & 1) ? (W[0] >> 16) : (W[0] & 0xffffu);
        const float dw = half_bits_to_float((uint16_t)dbits);
        const uint32_t edge = __byte_perm(W[0], W[8], sel);
        int s0 = __dp4a((int)edge, (int)A0[0], 0), s1 = 0;
        if (two_tokens) s1 = __dp4a((int)edge, (int)A1[0], 0);
#pragma unroll
        for (int k = 1; k < 8; ++k) {
            s0 = __dp4a((int)W[k], (int)A0[k], s0);
            if (two_tokens) s1 = __dp4a((int)W[k], (int)A1[k], s1);
        }
        acc[i] = fmaf((float)s0, dw * dx0, acc[i]);
        if (two_tokens) acc[4 + i] = fmaf((float)s1, dw * dx1, acc[4 + i]);
    }
}

// MMA modes, one slot: 16 rows x 8 blocks x NT*8 tokens.
template <int NT>
__device__ __forceinline__ void slot_mma(const uint8_t *sbase, const uint8_t *act, const float *dxs, uint32_t bl0,
                                         int lane, uint64_t (&acc)[NT][2]) {
    using namespace gv;
    constexpr int ACT_BLOCK = NT * 512;
    const int g = lane >> 2, c = lane & 3;
    const uint8_t *r0base = sbase + g * SROW;
    const uint8_t *abase = act + (size_t)bl0 * ACT_BLOCK + (size_t)lane * 16;
    const float *dbase = dxs + bl0 * 16 + 2 * c;
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
            s8x4_to_h2x2(w[h][0], h0l, h0h);     // row g,   first 16 quants
            s8x4_to_h2x2(w[h][1], h1l, h1h);     // row g+8, first 16 quants
            s8x4_to_h2x2(w[h][2], h2l, h2h);     // row g,   second 16 quants
            s8x4_to_h2x2(w[h][3], h3l, h3h);     // row g+8, second 16 quants
            const uint8_t *af = abase + (size_t)bo * ACT_BLOCK;   // + t * 512: N tile t
#pragma unroll
            for (int t = 0; t < NT; ++t) {
                const uint64_t dx01 = *reinterpret_cast<const uint64_t *>(dbase + bo * 16 + t * 8);
                const uint4 b4 = *reinterpret_cast<const uint4 *>(af + t * 512);
                float d[4] = {0.f, 0.f, 0.f, 0.f};
                mma_f16_16816(d, h0l, h1l, h0h, h1h, b4.x, b4.y);
                mma_f16_16816(d, h2l, h3l, h2h, h3h, b4.z, b4.w);
                scale_acc64(acc[t][0], d[0], d[1], dx01, dw0[h]);
                scale_acc64(acc[t][1], d[2], d[3], dx01, dw8[h]);
            }
        }
    }
}

// KIND: dense, grouped, or the grouped gate/up pair of GemvParams::W2.
// SUBM: sub-items a consumer warp holds in one item (items of at most 14 SUBM
// sub-items); the accumulators take SUBM x NT x 2 registers pairs, so the host
// picks the smallest that covers the call's items.
template <int MODE, int KIND, int SUBM>
__global__ void __launch_bounds__(gv::NTHREADS, 1) k_gemv(const GemvParams p, const __grid_constant__ CUtensorMap tmap,
                                                           const __grid_constant__ CUtensorMap tmap2) {
    using namespace gv;
    using M = Mode<MODE>;
    constexpr bool PAIR = KIND == KIND_PAIR;
    constexpr int NT = M::NT;
    constexpr int KA = M::KA;
    constexpr int NACC = M::NACC;

    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t *ring = smem;
    uint8_t *act = smem + RING_BYTES;
    float *dxs = reinterpret_cast<float *>(act + ACT_BYTES);
    uint8_t *qtmp = reinterpret_cast<uint8_t *>(dxs + DX_FLOATS);
    uint64_t *full = reinterpret_cast<uint64_t *>(qtmp + QT_BYTES);
    uint64_t *empty = full + NSLOT;
    volatile uint32_t *armed = reinterpret_cast<volatile uint32_t *>(empty + NSLOT);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(armed + NSLOT);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // one thread per ring slot initialises its barriers (one thread doing all 64
    // delays the first copy by about a microsecond)
    if (threadIdx.x < NSLOT) {
        const int s = threadIdx.x;
        if (s == 0) {
            *abort_flag = 0;
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap)) : "memory");
            if (PAIR) asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap2)) : "memory");
        }
        mbar_init(&full[s], 1);
        mbar_init(&empty[s], 1);
        armed[s] = 0xffffffffu;
        fence_mbar_init();
    }
    __syncthreads();

    const uint64_t lim = wait_limit(p.wait_ns);
    if (warp == PRODUCER) {
        if (!p.weights_early) grid_dep_wait();
        produce<M::TOKG, KIND>(p, &tmap, &tmap2, ring, full, empty, armed, abort_flag, lane, lim);
        // Every weight copy of this CTA is issued: a kernel launched behind this one
        // with programmatic serialisation may take the SMs freed from here on (its
        // reads of anything this grid writes wait in griddepcontrol.wait).
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
        // After a timed-out wait: let the copies still in flight land (with one
        // overall time limit) before the CTA's shared memory goes away.  Each slot
        // has at most one copy in flight, that of the last round armed on it.
        if (*abort_flag && lane == 0) {
            const uint64_t t_end = global_timer_ns() + WAIT_LIMIT_NS;
            for (int s = 0; s < NSLOT; ++s) {
                const uint32_t r = armed[s];
                if (r != 0xffffffffu) mbar_drain(&full[s], r & 1u, t_end);
            }
        }
        return;
    }

    const uint32_t nb = p.nb;
    const uint32_t nk = (nb + KC - 1) / KC;
    const int kachunks = (int)((nb + KA - 1) / KA);
    uint32_t seqbase = 0;
    bool waited_dep = false;

    ItemCursor cur;
    cursor_init<KIND != KIND_DENSE>(p, cur);
    for (;;) {
        GItem it;
        if (!next_item<M::TOKG, KIND != KIND_DENSE>(p, cur, it)) break;
        // sub-items: with a gate/up pair, nh of the gate and then nh of the up;
        // sub-item v's results are staged at local row 16v + r, so the up rows
        // follow the gate rows at 16 nh
        const uint32_t nh = (it.nrows + ROWS - 1) / ROWS;
        const uint32_t nsub = PAIR ? 2 * nh : nh;
        const uint32_t wpi = item_wpi(nsub, nk);
        const uint32_t ngroups = (uint32_t)NCW / wpi;
        const uint32_t slice = (uint32_t)warp % wpi, grp = (uint32_t)warp / wpi;
        if (!waited_dep) {
            grid_dep_wait();      // activations are written by the preceding kernel
            waited_dep = true;
        }

        float accf[SUBM][NACC];
        uint64_t acc[SUBM][NT][2];
#pragma unroll
        for (int s2 = 0; s2 < SUBM; ++s2) {
#pragma unroll
            for (int e = 0; e < NACC; ++e) accf[s2][e] = 0.0f;
#pragma unroll
            for (int t = 0; t < NT; ++t) acc[s2][t][0] = acc[s2][t][1] = 0ull;
        }

        uint32_t kk = slice;
        for (int ch = 0; ch < kachunks; ++ch) {
            const uint32_t kb0 = (uint32_t)ch * KA;
            const uint32_t ka = min((uint32_t)KA, nb - kb0);
            named_bar_sync(BAR_CONSUMERS, CONSUMER_THREADS);   // previous chunk or item done with act
            if (p.x) stage_chunk_fused<MODE>(p, it, kb0, ka, act, dxs, qtmp);
            else stage_chunk<MODE, KIND == KIND_DENSE>(p, it, kb0, ka, act, dxs, qtmp);
            named_bar_sync(BAR_CONSUMERS, CONSUMER_THREADS);
            for (; kk < nk; kk += wpi) {
                const uint32_t kb = kk * KC;
                if (kb >= kb0 + ka) break;                     // belongs to the next chunk
                const uint32_t bl0 = kb - kb0;
#pragma unroll
                for (int s2 = 0; s2 < SUBM; ++s2) {
                    const uint32_t sub = grp + (uint32_t)s2 * ngroups;
                    if (sub < nsub) {
                        const uint32_t seq = seqbase + kk * nsub + sub;
                        const uint32_t slot = seq % NSLOT;
                        bool ok = wait_armed(&armed[slot], seq / NSLOT, p.err, abort_flag, lim);
                        if (ok) ok = mbar_wait(&full[slot], (seq / NSLOT) & 1u, p.err, abort_flag, lim);
                        const uint8_t *sbase = ring + (size_t)slot * SLOT;
                        if (MODE == 0) {
                            float (&a8)[8] = *reinterpret_cast<float (*)[8]>(&accf[s2][0]);
                            slot_dp4a(sbase, act, dxs, bl0, lane, a8, it.ntok > 1);
                        } else {
                            slot_mma<NT>(sbase, act, dxs, bl0, lane, acc[s2]);
                        }
                        __syncwarp();
                        // a slot whose copy did not land (timed out) is never handed back
                        if (lane == 0 && ok) mbar_arrive(&empty[slot]);
                    }
                }
            }
        }
        seqbase += nk * nsub;
        const uint32_t nh_e = (it.nrows + ROWS - 1) / ROWS;   // recomputed: not kept live through the stream

        if (MODE != 0) {
#pragma unroll
            for (int s2 = 0; s2 < SUBM; ++s2)
#pragma unroll
                for (int t = 0; t < NT; ++t) {
                    accf[s2][t * 4 + 0] = lo_of(acc[s2][t][0]);
                    accf[s2][t * 4 + 1] = hi_of(acc[s2][t][0]);
                    accf[s2][t * 4 + 2] = lo_of(acc[s2][t][1]);
                    accf[s2][t * 4 + 3] = hi_of(acc[s2][t][1]);
                }
        }
        // ---- split-K partials (wpi > 1, one sub-item per warp): added in slice
        // order through shared memory
        if (wpi > 1) {
            named_bar_sync(BAR_CONSUMERS, CONSUMER_THREADS);   // act is reused for the partials
            float *red = reinterpret_cast<float *>(act);
            if (slice > 0) {
#pragma unroll
                for (int e = 0; e < NACC; ++e) red[(warp * NACC + e) * 32 + lane] = accf[0][e];
            }
            named_bar_sync(BAR_CONSUMERS, CONSUMER_THREADS);
            if (slice == 0) {
                for (uint32_t k = 1; k < wpi; ++k) {
                    const int w2 = warp + (int)k;
#pragma unroll
                    for (int e = 0; e < NACC; ++e) accf[0][e] += red[(w2 * NACC + e) * 32 + lane];
                }
            }
        }
        // ---- outputs: gathered per token in shared memory (the activation buffer,
        // free once every warp is past the compute and split-K steps), then
        // written as contiguous runs with 16-byte stores -- few, full transactions,
        // which matters most when the result lives in host memory
        named_bar_sync(BAR_CONSUMERS, CONSUMER_THREADS);
        float *obuf = reinterpret_cast<float *>(act);   // [token][row - r0], OUT_STRIDE floats a token
        if (MODE == 0) {
            // add the 8 block columns of each row (lanes differing in bits 0-2)
#pragma unroll
            for (int s2 = 0; s2 < SUBM; ++s2)
#pragma unroll
                for (int e = 0; e < NACC; ++e) {
                    float v = accf[s2][e];
                    v += __shfl_xor_sync(0xffffffffu, v, 1);
                    v += __shfl_xor_sync(0xffffffffu, v, 2);
                    v += __shfl_xor_sync(0xffffffffu, v, 4);
                    accf[s2][e] = v;
                }
            if (slice == 0 && (lane & 7) == 0) {
                const int rb = lane >> 3;
#pragma unroll
                for (int s2 = 0; s2 < SUBM; ++s2) {
                    const uint32_t sub = grp + (uint32_t)s2 * ngroups;
                    if (sub < nsub) {
#pragma unroll
                        for (int e = 0; e < NACC; ++e) {
                            const int tok = e >> 2;
                            const uint32_t rr = (uint32_t)dp4a_row(rb, e & 3);
                            const uint32_t hr = (PAIR && sub >= nh_e ? sub - nh_e : sub) * ROWS + rr;   // row in its matrix
                            if (tok < it.ntok && hr < it.nrows) obuf[tok * OUT_STRIDE + sub * ROWS + rr] = accf[s2][e];
                        }
                    }
                }
            }
        } else if (slice == 0) {
            const int g = lane >> 2, c = lane & 3;
#pragma unroll
            for (int s2 = 0; s2 < SUBM; ++s2) {
                const uint32_t sub = grp + (uint32_t)s2 * ngroups;
                if (sub < nsub) {
#pragma unroll
                    for (int t = 0; t < NT; ++t) {
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int tok = t * 8 + 2 * c + (e & 1);
                            const uint32_t rr = (uint32_t)g + ((e & 2) ? 8u : 0u);
                            const uint32_t hr = (PAIR && sub >= nh_e ? sub - nh_e : sub) * ROWS + rr;   // row in its matrix
                            if (tok < it.ntok && hr < it.nrows)
                                obuf[tok * OUT_STRIDE + sub * ROWS + rr] = accf[s2][t * 4 + e];
                        }
                    }
                }
            }
        }
        named_bar_sync(BAR_CONSUMERS, CONSUMER_THREADS);
        if (PAIR && p.q_out) {
            // mid = swiglu1(gate, up) as Q8_0 planes at the pair's activation-plane row:
            // four lanes a 32-value block (item rows and r0 are multiples of 32).  All
            // consumer threads run the same trips: the quantiser shuffles within a warp.
            const uint32_t nblk = it.nrows / QK, nbm = p.out_dim / QK;
            const uint32_t total = (uint32_t)it.ntok * nblk * 4;
            for (uint32_t base = 0; base < total; base += CONSUMER_THREADS) {
                const uint32_t e = base + threadIdx.x;
                const bool live = e < total;
                const uint32_t tok = live ? (e >> 2) / nblk : 0u, b = live ? (e >> 2) - tok * nblk : 0u;
                const uint32_t c0 = b * QK + (e & 3u) * 8;   // first of this lane's 8 values
                float v8[8];
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    v8[j] = live ? swiglu1(obuf[tok * OUT_STRIDE + c0 + j], obuf[tok * OUT_STRIDE + nh_e * ROWS + c0 + j],
                                           p.limit)
                                 : 0.0f;
                const QuantBlock qb = quantize8(v8);
                if (live) {
                    const uint64_t row = (uint64_t)(it.xrow0 + (int)tok);
                    *reinterpret_cast<uint2 *>(p.q_out + row * p.out_dim + it.r0 + c0) = make_uint2(qb.lo, qb.hi);
                    if ((e & 3u) == 0) p.d_out[row * nbm + it.r0 / QK + b] = qb.d_stored;
                }
            }
        } else if ((p.out_dim & 3u) == 0) {
            // every run starts 16-byte aligned (out is, r0 is a multiple of 16, out_dim of 4)
            // and is a whole number of float4 (nrows is a multiple of 4)
            const uint32_t nv = it.nrows >> 2;
            for (uint32_t e = threadIdx.x; e < (uint32_t)it.ntok * nv; e += CONSUMER_THREADS) {
                const uint32_t tok = e / nv, i = e - tok * nv;
                const int64_t orow = KIND != KIND_DENSE ? (int64_t)p.row_to_out[it.xrow0 + tok] : (int64_t)(it.tok0 + tok);
                if (orow >= 0) {
                    float4 v = *reinterpret_cast<const float4 *>(obuf + tok * OUT_STRIDE + 4 * i);
                    if (PAIR) {
                        const float4 u = *reinterpret_cast<const float4 *>(obuf + tok * OUT_STRIDE + nh_e * ROWS + 4 * i);
                        v = make_float4(swiglu1(v.x, u.x, p.limit), swiglu1(v.y, u.y, p.limit),
                                        swiglu1(v.z, u.z, p.limit), swiglu1(v.w, u.w, p.limit));
                    }
                    *reinterpret_cast<float4 *>(p.out + (uint64_t)orow * p.out_dim + it.r0 + 4 * i) = v;
                }
            }
        } else {
            for (uint32_t e = threadIdx.x; e < (uint32_t)it.ntok * it.nrows; e += CONSUMER_THREADS) {
                const uint32_t tok = e / it.nrows, i = e - tok * it.nrows;
                const int64_t orow = KIND != KIND_DENSE ? (int64_t)p.row_to_out[it.xrow0 + tok] : (int64_t)(it.tok0 + tok);
                if (orow >= 0) {
                    float v = obuf[tok * OUT_STRIDE + i];
                    if (PAIR) v = swiglu1(v, obuf[tok * OUT_STRIDE + nh_e * ROWS + i], p.limit);
                    p.out[(uint64_t)orow * p.out_dim + it.r0 + i] = v;
                }
            }
        }
    }
    if (!waited_dep) grid_dep_wait();
}

bool encode_rows_tmap(CUtensorMap *map, const void *W, uint64_t row_bytes, uint64_t rows, uint64_t n_mat,
                      uint64_t mat_stride, uint32_t box_words, uint32_t box_rows);

// The kernel variant of a call: kind, mode and sub-items per warp.
template <int KIND, int SUBM> static const void *gemv_fn(int mode) {
    if constexpr (KIND == KIND_DENSE) {
        return mode == 0 ? (const void *)k_gemv<0, KIND, SUBM>
                         : (mode == 1 ? (const void *)k_gemv<1, KIND, SUBM> : (const void *)k_gemv<2, KIND, SUBM>);
    } else {
        return mode == 1 ? (const void *)k_gemv<1, KIND, SUBM> : (const void *)k_gemv<2, KIND, SUBM>;
    }
}

cudaError_t launch_gemv(const GemvParams &p, int mode, int grid, cudaStream_t st) {
    if (mode < 0 || mode > 2 || (p.plan && mode == 0) || (p.W2 && !p.plan) || (p.q_out && !p.W2))
        return cudaErrorInvalidValue;
    const int kind = !p.plan ? KIND_DENSE : (p.W2 ? KIND_PAIR : KIND_GROUPED);
    // the most sub-items of one item (a pair's gate and up sub-items both count)
    uint32_t max_sub = !p.plan ? p.sub_base + (p.sub_rem ? 1u : 0u) : (p.rows_per_item + gv::ROWS - 1) / gv::ROWS;
    if (kind == KIND_PAIR) max_sub *= 2;
    const int subm = (int)((max_sub + gv::NCW - 1) / gv::NCW);
    if (subm < 1 || subm > (kind == KIND_DENSE ? 3 : 2)) return cudaErrorInvalidValue;
    static const void *const fns[3][3][3] = {
        {{gemv_fn<KIND_DENSE, 1>(0), gemv_fn<KIND_DENSE, 1>(1), gemv_fn<KIND_DENSE, 1>(2)},
         {gemv_fn<KIND_DENSE, 2>(0), gemv_fn<KIND_DENSE, 2>(1), gemv_fn<KIND_DENSE, 2>(2)},
         {gemv_fn<KIND_DENSE, 3>(0), gemv_fn<KIND_DENSE, 3>(1), gemv_fn<KIND_DENSE, 3>(2)}},
        {{nullptr, gemv_fn<KIND_GROUPED, 1>(1), gemv_fn<KIND_GROUPED, 1>(2)},
         {nullptr, gemv_fn<KIND_GROUPED, 2>(1), gemv_fn<KIND_GROUPED, 2>(2)},
         {nullptr, nullptr, nullptr}},
        {{nullptr, gemv_fn<KIND_PAIR, 1>(1), gemv_fn<KIND_PAIR, 1>(2)},
         {nullptr, gemv_fn<KIND_PAIR, 2>(1), gemv_fn<KIND_PAIR, 2>(2)},
         {nullptr, nullptr, nullptr}}};
    static bool attr_done[3][3][3] = {};
    const void *fn = fns[kind][subm - 1][mode];
    if (!fn) return cudaErrorInvalidValue;
    if (!attr_done[kind][subm - 1][mode]) {
        cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)gv::SMEM);
        if (e != cudaSuccess) return e;
        attr_done[kind][subm - 1][mode] = true;
    }
    alignas(64) CUtensorMap tmap, tmap2;
    const uint64_t row_bytes = (uint64_t)p.nb * QB;
    const uint64_t mats = p.plan ? p.n_expert : 1;
    const uint64_t mstride = p.plan ? p.expert_stride : (uint64_t)p.out_dim * row_bytes;
    if (!encode_rows_tmap(&tmap, p.W, row_bytes, p.out_dim, mats, mstride, gv::BOX_WORDS, gv::ROWS))
        return cudaErrorInvalidValue;
    if (p.W2) {
        // the pair's staged results take 2 x rows_per_item floats a token; Q8_0
        // output wants whole 32-value blocks in every item
        if (!p.plan || p.rows_per_item > gv::OUT_STRIDE / 2) return cudaErrorInvalidValue;
        if (p.q_out && (!p.d_out || p.rows_per_item % QK || p.out_dim % QK)) return cudaErrorInvalidValue;
        if (!encode_rows_tmap(&tmap2, p.W2, row_bytes, p.out_dim, mats, mstride, gv::BOX_WORDS, gv::ROWS))
            return cudaErrorInvalidValue;
    } else {
        tmap2 = tmap;
    }
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
    void *args[] = {&pp, &tmap, &tmap2};
    return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace q8
