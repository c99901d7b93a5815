// q8_tc.cu -- prefill GEMM on the 5th-generation tensor cores (tcgen05, TMEM).
//
// out[t][o] = sum_b d_w[o][b] d_x[t][b] isum_b[t][o] (ds4 pages: the Q8_0 matmul
// of the GPU code walkthrough, trace 3; fixed-point block dot of the
// model-architecture page, quantisation section 4; the pages route n_tok >= 2
// prefill to a tensor-core tier, concepts page section 4m).
//
// sm_103a has no int8 tcgen05.mma (ptxas rejects kind::i8 for it), so the int8
// arithmetic runs exactly on kind::f16: quants |q| <= 127 are exact in fp16,
// every product is an integer below 2^14 and a block's 32-product sum is below
// 2^24, exact in the fp32 accumulator.  The scales differ per 32-value block,
// so each block gets its own accumulator: two UMMAs (K = 16 each) write a fresh
// 128 x 128 fp32 tile into one of four TMEM slots, and the epilogue warps read
// it back (tcgen05.ld 16x256b: a thread holds four rows and a quarter of its
// warp's columns, so it loads a quarter of the activation scales a lane-per-row
// read would need) and fold it into fp32 registers as
// acc[o][t] += isum * d_x[t] * d_w[o] (packed f32x2 multiply and FMA).  That
// epilogue costs two fp32 operations per output per block, 1/16 of the MMA's
// multiply-adds, and the fp32 pipe, not the tensor pipe, sets the ceiling
// (about half the fp16 tensor rate).
//
// Warp roles (one persistent CTA per SM):
//   warp 0  TMA producer: per stage of K = 64 (two blocks) the fp16 activation
//           tile (128 x 64, 128-byte swizzle) and its two blocks' scales (1-D
//           bulk copies); with fp16 weights also the weight tile and scales
//           (six stages), with raw weights one copy of 8 raw Q8_0 blocks x 128
//           rows per four stages into a ring of two (four stages).
//   warp 1  allocates TMEM (512 columns) and issues the UMMAs from one thread;
//           tcgen05.commit signals "slot full" and, per stage, "stage consumed".
//   2..     epilogue, 8 warps (fp16 weights) or 16 (raw weights): warp w reads
//           TMEM lanes 32*(w%4).. and one column group (half or quarter of the
//           128); arrives "slot empty" after folding, "stage empty" after using
//           the stage's scales.
//   next    fp16 weights: the second MMA issuer.  Raw weights, two warps:
//           converters.  Each stage's weight tile is written
//           from the raw copy as exact fp16 in the layout the fp16 tensor map
//           gives, with the weight scales beside it, then handed to the tensor
//           core (proxy fence + the stage's "full" barrier).
// Dense work units are (128-row tile, 128-token tile, K split); with fewer tiles
// than SMs, K is split and the partial sums are added by a second kernel in a
// fixed order (deterministic).  Grouped units (routed experts) come from the
// routing plan: (expert group, 128-row tile, 128-token tile), output rows
// scattered through the plane-row -> output-row map.  Every wait is bounded.
#include <cuda.h>

#include "q8_common.cuh"
#include "q8_kernels.h"

namespace q8 {

namespace tc {
constexpr int BM = 128;                                // weight rows per tile (UMMA M)
constexpr int BN = 128;                                // tokens per tile (UMMA N)
constexpr int BK = 64;                                 // K elements per stage (two blocks)
constexpr int A_BYTES = BM * BK * 2;                   // 16384
constexpr int B_BYTES = BN * BK * 2;                   // 16384
constexpr int DX_BYTES = 2 * BN * 4;                   // 1024
constexpr int DW_BYTES = 2 * BM * 4;                   // 1024
constexpr int STAGE_BYTES = A_BYTES + B_BYTES + DX_BYTES + DW_BYTES;   // 34 KiB, 1 KiB aligned
constexpr int NSLOT_T = 4;                             // TMEM accumulator slots of BN columns
constexpr uint32_t TMEM_COLS = NSLOT_T * BN;           // 512
// Raw-weight variant: the A operand arrives as raw Q8_0 rows, 8 blocks (272
// bytes, 68 words) x 128 rows per copy, and converter warps write the fp16
// tile and the weight scales of each stage.
constexpr int RAW_KB = 8;                              // blocks per raw copy (K = 256)
constexpr int RAW_WORDS = RAW_KB * QB / 4;             // 68
constexpr int RAW_BYTES = BM * RAW_WORDS * 4;          // 34816 = 34 KiB
constexpr int NRAW = 2;                                // raw copies in flight
constexpr int NCONV = 2;                               // converter warps
static_assert(STAGE_BYTES % 1024 == 0 && RAW_BYTES % 1024 == 0, "stage alignment");

template <bool RAW> struct Cfg {
    static constexpr int NSTAGE = RAW ? 4 : 6;
    // Epilogue warps per TMEM lane quarter, each folding 128 / EPI_COLG columns.
    // With raw weights the converters share the schedulers and four warps per
    // quarter hide more latency; with fp16 weights two are faster (measured).
    static constexpr int EPI_COLG = RAW ? 4 : 2;
    static constexpr int NUM_EPI = 4 * EPI_COLG;
    // MMA issuers: the issuing thread shares its scheduler with two folding
    // epilogue warps and slows down while they fold; with fp16 weights a second
    // issuer on another scheduler takes every other stage.
    static constexpr int NMMA = RAW ? 1 : 2;
    static constexpr int NTHREADS = (2 + NUM_EPI + (RAW ? NCONV : 0) + (NMMA - 1)) * 32;
    static constexpr int W_EXTRA = 2 + NUM_EPI;   // second MMA issuer, or the first converter warp
    static constexpr int NRAWS = RAW ? NRAW : 0;
    // full, empty, tfull, tempty, done, raw full, raw empty
    static constexpr int NBAR = 2 * NSTAGE + 2 * NSLOT_T + 1 + 2 * NRAWS;
    static constexpr size_t SMEM =
        (size_t)NSTAGE * STAGE_BYTES + (size_t)NRAWS * RAW_BYTES + 1024 + NBAR * 8 + 16;
    static_assert(SMEM <= 227 * 1024, "shared memory");
};
}  // namespace tc

// ---------------------------------------------------------------- PTX wrappers
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, int x, int y, int z, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar))
        : "memory");
}

// Generic-proxy shared-memory writes -> visible to the tensor core (async proxy).
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tc_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
                 : "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, fp16 inputs, fp32 accumulate.
__device__ __forceinline__ void tc_mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// 16 lanes x 8 columns per repetition (NR repetitions, 8 columns apart): thread
// t gets, per repetition g, (lane t/4, columns 8g + 2(t%4) and + 1) in v[4g],
// v[4g+1] and the same columns of lane t/4 + 8 in v[4g+2], v[4g+3].
template <int NR>
__device__ __forceinline__ void tc_ld16x256(uint32_t taddr, uint32_t (&v)[4 * NR]) {
    if constexpr (NR == 8) {
        asm volatile(
            "tcgen05.ld.sync.aligned.16x256b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
            "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
            : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
              "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),
              "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]),
              "=r"(v[23]), "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]),
              "=r"(v[30]), "=r"(v[31])
            : "r"(taddr));
    } else if constexpr (NR == 4) {
        asm volatile(
            "tcgen05.ld.sync.aligned.16x256b.x4.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
            : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
              "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
            : "r"(taddr));
    } else if constexpr (NR == 2) {
        asm volatile("tcgen05.ld.sync.aligned.16x256b.x2.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                     : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7])
                     : "r"(taddr));
    } else {
        static_assert(NR == 1, "repetitions");
        asm volatile("tcgen05.ld.sync.aligned.16x256b.x1.b32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3])
                     : "r"(taddr));
    }
}

__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// No instruction: ties the registers of a finished tcgen05.ld to a point after
// tcgen05.wait::ld, so that no use of them is scheduled before the wait.
template <int N>
__device__ __forceinline__ void tc_regs_ready(uint32_t (&v)[N]) {
#pragma unroll
    for (int i = 0; i < N; i += 4) asm volatile("" : "+r"(v[i]), "+r"(v[i + 1]), "+r"(v[i + 2]), "+r"(v[i + 3]));
}

// Shared-memory matrix descriptor: K-major tile with 128-byte swizzle, rows 128
// bytes apart, 8-row groups 1024 bytes apart (the layout a 128-byte-swizzled
// TMA box of 64 fp16 per row produces).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);          // start address
    d |= (uint64_t)1 << 16;                            // leading byte offset (unused with swizzle)
    d |= (uint64_t)(1024u >> 4) << 32;                 // stride byte offset: 8-row group
    d |= (uint64_t)1 << 46;                            // descriptor version
    d |= (uint64_t)2 << 61;                            // 128-byte swizzle
    return d;
}

// Instruction descriptor: fp32 accumulate, fp16 A and B, both K-major, N x M.
__host__ __device__ constexpr uint32_t tc_idesc(int m, int n) {
    return (1u << 4) | (0u << 7) | (0u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

// (a0, a1) += (v0, v1) * (x0, x1) * (w, w), accumulator pair in one 64-bit register.
__device__ __forceinline__ void tc_fold(uint64_t &acc, uint32_t v0, uint32_t v1, float x0, float x1, uint64_t ww) {
    asm("{\n\t.reg .b64 v, x, t;\n\tmov.b64 v, {%1, %2};\n\tmov.b64 x, {%3, %4};\n\t"
        "mul.rn.f32x2 t, v, x;\n\t"
        "fma.rn.f32x2 %0, t, %5, %0;\n\t}"
        : "+l"(acc)
        : "r"(v0), "r"(v1), "f"(x0), "f"(x1), "l"(ww));
}

__device__ __forceinline__ uint64_t tc_pair(float w) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %1};" : "=l"(r) : "f"(w));
    return r;
}

// Four int8 -> two half2 (exact): bias each byte to unsigned, place it under the
// fp16 exponent of 1024, subtract 1024 + 128.
__device__ __forceinline__ void s8x4_to_half2x2(uint32_t w, uint32_t &lo, uint32_t &hi) {
    const uint32_t u = w ^ 0x80808080u;
    const uint32_t a = __byte_perm(u, 0x64646464u, 0x4140);
    const uint32_t b = __byte_perm(u, 0x64646464u, 0x4342);
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(a), "r"(0x64806480u));
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(b), "r"(0x64806480u));
}

// A predicate the whole warp agrees on (lane 0's value).
__device__ __forceinline__ bool warp_all(bool v) { return __shfl_sync(0xffffffffu, (int)v, 0) != 0; }

struct TcUnit {
    int mt, nt, kb0, kb1;
    int a_row, b_row;   // first weight row (in the expert) / b16 plane row of the tile,
                        // also the dwT / dxT column
    int n_valid;        // grouped: tokens of the tile that belong to the segment
    int expert;         // grouped: expert matrix of the tile
    int ncols;          // UMMA N of the tile: 128, or 64 / 32 for a group's short last tile
};

// Dense: units are (128-row tile, 128-token tile, K split).
__device__ __forceinline__ bool tc_unit_dense(const TcParams &p, int u, TcUnit &w) {
    const int m_tiles = (p.M + tc::BM - 1) / tc::BM;
    const int n_tiles = (p.N + tc::BN - 1) / tc::BN;
    const int units = m_tiles * n_tiles * p.ksplit;
    if (u >= units) return false;
    w.mt = u % m_tiles;                 // consecutive units share the activation tile
    const int r = u / m_tiles;
    w.nt = r % n_tiles;
    const int ks = r / n_tiles;
    w.kb0 = ks * p.kb_per;
    w.kb1 = min(p.nb, w.kb0 + p.kb_per);
    w.a_row = w.mt * tc::BM;
    w.b_row = w.nt * tc::BN;
    w.n_valid = tc::BN;
    w.expert = 0;
    w.ncols = tc::BN;
    return true;
}

// Grouped: the plan's segments in order, each m_tiles x ceil(count / 128)
// units from item_start on (weight tile fastest), on the segment's expert.
// Units only grow along a CTA's loop, so the segment cursor only moves forward.
__device__ __forceinline__ bool tc_unit_grouped(const TcParams &p, int u, TcUnit &w, int &seg) {
    const PlanHeader *h = p.plan;
    if (u >= h->n_items) return false;
    const Segment *sg = reinterpret_cast<const Segment *>(h + 1);
    const int nseg = h->n_segments;
    while (seg + 1 < nseg && sg[seg + 1].item_start <= u) ++seg;
    const int m_tiles = (p.M + tc::BM - 1) / tc::BM;
    const int v = u - sg[seg].item_start;
    w.mt = v % m_tiles;
    w.nt = v / m_tiles;
    w.kb0 = 0;
    w.kb1 = p.nb;
    w.a_row = w.mt * tc::BM;
    w.b_row = sg[seg].row0 + w.nt * tc::BN;
    w.n_valid = min(tc::BN, sg[seg].count - w.nt * tc::BN);
    w.expert = sg[seg].expert;
    w.ncols = w.n_valid > 64 ? 128 : (w.n_valid > 32 ? 64 : 32);
    return true;
}

template <bool G>
__device__ __forceinline__ bool tc_unit(const TcParams &p, int u, TcUnit &w, int &seg) {
    if constexpr (G) return tc_unit_grouped(p, u, w, seg);
    else return tc_unit_dense(p, u, w);
}

// One stage's share of a raw copy (blocks 2J, 2J + 1 of the copy's 8) for rows
// ct and ct + 64: fp16 quants into the stage's A tile in the 128-byte-swizzled
// K-major layout (row r at r * 128 bytes, 16-byte chunk c at c ^ (r % 8), the
// layout the fp16 tensor map writes), scales into dws[j][r].  The 68 bytes of a
// row's block pair start at word r * 68 + 17 J: five aligned 16-byte loads from
// word r * 68 + (17 J & ~3) cover them, and rows 8 apart fall in different
// bank groups.
template <int J>
__device__ __forceinline__ void tc_convert(const uint8_t *raw, uint8_t *a16, float *dws, int ct) {
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
        const int r = ct + rr * 64;
        const uint4 *src = reinterpret_cast<const uint4 *>(raw) + (r * tc::RAW_WORDS + ((17 * J) & ~3)) / 4;
        uint32_t w[20];
#pragma unroll
        for (int i = 0; i < 5; ++i) {
            const uint4 v = src[i];
            w[4 * i] = v.x;
            w[4 * i + 1] = v.y;
            w[4 * i + 2] = v.z;
            w[4 * i + 3] = v.w;
        }
        constexpr int o = (17 * J) & 3;   // word offset of the pair inside the loaded words
        uint8_t *row = a16 + r * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            uint32_t q0, q1;
            if (c < 4) {   // block 2J: quants at byte 2 of the pair
                q0 = funnel16(w[o + 2 * c], w[o + 2 * c + 1]);
                q1 = funnel16(w[o + 2 * c + 1], w[o + 2 * c + 2]);
            } else {       // block 2J + 1: quants at byte 36 (word 9)
                q0 = w[o + 9 + 2 * (c - 4)];
                q1 = w[o + 10 + 2 * (c - 4)];
            }
            uint32_t h0, h1, h2, h3;
            s8x4_to_half2x2(q0, h0, h1);
            s8x4_to_half2x2(q1, h2, h3);
            *reinterpret_cast<uint4 *>(row + ((c ^ (r & 7)) << 4)) = make_uint4(h0, h1, h2, h3);
        }
        dws[r] = half_bits_to_float((uint16_t)(w[o] & 0xffffu));
        dws[tc::BM + r] = half_bits_to_float((uint16_t)(w[o + 8] >> 16));
    }
}

// Epilogue warp state: stage ring and TMEM slot counters, carried across units.
struct TcEpi {
    uint8_t *smem;
    uint64_t *full, *empty, *tfull, *tempty;
    volatile int *abort_flag;
    uint64_t lim;         // wait limit (ns)
    uint32_t lane_addr;   // TMEM address of this warp's lane quarter
    int m, h, lane;       // tile row, column half, lane
    uint32_t stage, phase, blk;
};

// One unit of an epilogue warp: NCW = columns of this warp (half the unit's N).
// Per block, the warp's columns leave TMEM in one batch of x16 loads and are
// folded into acc as isum * d_x[t] * d_w[o]; then the unit's outputs are stored.
// One unit of an epilogue warp, NCW columns (its share of the unit's N), read
// from TMEM 16 lanes at a time (16x256b): each thread holds four rows (lanes
// t/4 + 0, 8, 16, 24 of its quarter) and 2 of every 8 columns, so per block it
// needs NCW/4 activation scales (NCW/8 shared-memory loads, each one wavefront)
// instead of all NCW.
template <int NCW, bool G, int NSTAGE>
__device__ __forceinline__ void tc_epilogue_unit(const TcParams &p, const TcUnit &w, TcEpi &e) {
    using namespace tc;
    constexpr int NG = NCW / 8;              // 8-column groups
    const int r4 = e.lane >> 2, c2 = 2 * (e.lane & 3);
    const int q32 = e.m - e.lane;            // first row of the warp's lane quarter
    uint64_t acc[2][2][NG];                  // [16-lane half][row + 0 / + 8][group]: fp32 pairs
#pragma unroll
    for (int a = 0; a < 2; ++a)
#pragma unroll
        for (int k = 0; k < 2; ++k)
#pragma unroll
            for (int g = 0; g < NG; ++g) acc[a][k][g] = 0ull;
    for (int kb = w.kb0; kb < w.kb1; kb += 2) {
        const uint8_t *st = e.smem + (size_t)e.stage * STAGE_BYTES;
        const bool staged = mbar_wait(&e.full[e.stage], e.phase, p.err, e.abort_flag, e.lim);
        const float *dxs = reinterpret_cast<const float *>(st + A_BYTES + B_BYTES);
        const float *dws = reinterpret_cast<const float *>(st + A_BYTES + B_BYTES + DX_BYTES);
        for (int j = 0; j < 2; ++j, ++e.blk) {
            const uint32_t slot = e.blk % NSLOT_T;
            mbar_wait(&e.tfull[slot], (e.blk / NSLOT_T) & 1u, p.err, e.abort_flag, e.lim);
            tc_fence_after();
            const uint32_t col0 = e.lane_addr + slot * BN + e.h * NCW;
            uint32_t v[2][4 * NG];
            tc_ld16x256<NG>(col0, v[0]);
            tc_ld16x256<NG>(col0 + (16u << 16), v[1]);
            uint64_t ww[2][2];
#pragma unroll
            for (int a = 0; a < 2; ++a)
#pragma unroll
                for (int k = 0; k < 2; ++k) ww[a][k] = tc_pair(dws[j * BM + q32 + 16 * a + 8 * k + r4]);
            const float *dxj = dxs + j * BN + e.h * NCW + c2;
            tc_wait_ld();
            tc_regs_ready(v[0]);
            tc_regs_ready(v[1]);
#pragma unroll
            for (int g = 0; g < NG; ++g) {
                const float2 x = *reinterpret_cast<const float2 *>(dxj + 8 * g);
#pragma unroll
                for (int a = 0; a < 2; ++a)
#pragma unroll
                    for (int k = 0; k < 2; ++k)
                        tc_fold(acc[a][k][g], v[a][4 * g + 2 * k], v[a][4 * g + 2 * k + 1], x.x, x.y, ww[a][k]);
            }
            // (handing the slot back before the fold, with the accumulator already in
            // registers, measured slower: the next block's MMAs then run against the fold)
            tc_fence_before();
            __syncwarp();
            if (e.lane == 0) mbar_arrive(&e.tempty[slot]);
        }
        __syncwarp();
        // a stage whose copies did not land (timed out) is never handed back
        if (e.lane == 0 && staged) mbar_arrive(&e.empty[e.stage]);
        if (++e.stage == NSTAGE) {
            e.stage = 0;
            e.phase ^= 1u;
        }
    }
    // ---- this unit's rows x this warp's tokens
    const int tok0 = e.h * NCW + c2;                  // within the tile
#pragma unroll
    for (int a = 0; a < 2; ++a)
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int row = w.mt * BM + q32 + 16 * a + 8 * k + r4;
            if (row >= p.M) continue;
#pragma unroll
            for (int g = 0; g < NG; ++g) {
                const int t = tok0 + 8 * g;
                const float lo = __uint_as_float((uint32_t)acc[a][k][g]);
                const float hi = __uint_as_float((uint32_t)(acc[a][k][g] >> 32));
                if constexpr (G) {
                    if (t < w.n_valid) p.out[(size_t)p.row_to_out[w.b_row + t] * p.M + row] = lo;
                    if (t + 1 < w.n_valid) p.out[(size_t)p.row_to_out[w.b_row + t + 1] * p.M + row] = hi;
                } else {
                    const int ks = w.kb0 / p.kb_per;
                    float *dst = p.partial ? p.partial + (size_t)ks * p.N * p.M : p.out;
                    const int tt = w.b_row + t;
                    if (tt < p.N) dst[(size_t)tt * p.M + row] = lo;
                    if (tt + 1 < p.N) dst[(size_t)(tt + 1) * p.M + row] = hi;
                }
            }
        }
}

template <bool G, bool RAW>
__global__ void __launch_bounds__(tc::Cfg<RAW>::NTHREADS, 1)
    k_tc_gemm(const TcParams p, const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB) {
    using namespace tc;
    constexpr int NSTAGE = Cfg<RAW>::NSTAGE;
    constexpr int NBAR = Cfg<RAW>::NBAR;
    constexpr int NUM_EPI = Cfg<RAW>::NUM_EPI, EPI_COLG = Cfg<RAW>::EPI_COLG, W_EXTRA = Cfg<RAW>::W_EXTRA;
    if constexpr (G) {
        // The GEMV launched behind this grid waits for it before it reads or
        // writes anything this grid touches; let it take the SMs this grid frees.
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
        if (p.plan->n_items == 0) return;
    }
    extern __shared__ uint8_t smem_raw[];
    const uint32_t base_s = smem_addr(smem_raw);
    uint8_t *smem = smem_raw + (((base_s + 1023u) & ~1023u) - base_s);      // 1 KiB aligned stages
    uint8_t *raw_s = smem + (size_t)NSTAGE * STAGE_BYTES;                     // raw copies (RAW only)
    uint64_t *bars = reinterpret_cast<uint64_t *>(raw_s + (size_t)Cfg<RAW>::NRAWS * RAW_BYTES);
    uint64_t *full = bars, *empty = bars + NSTAGE;
    uint64_t *tfull = bars + 2 * NSTAGE, *tempty = tfull + NSLOT_T, *done = tempty + NSLOT_T;
    uint64_t *raw_full = done + 1, *raw_empty = raw_full + Cfg<RAW>::NRAWS;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + NBAR);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < NSTAGE; ++s) {
            mbar_init(&full[s], RAW ? 1 + NCONV : 1);   // producer (+ every converter warp)
            mbar_init(&empty[s], 1 + NUM_EPI);           // MMA commit + every epilogue warp
        }
        for (int s = 0; s < NSLOT_T; ++s) {
            mbar_init(&tfull[s], 1);
            mbar_init(&tempty[s], NUM_EPI);
        }
        mbar_init(done, Cfg<RAW>::NMMA);
        for (int s = 0; s < Cfg<RAW>::NRAWS; ++s) {
            mbar_init(&raw_full[s], 1);
            mbar_init(&raw_empty[s], NCONV);
        }
        *abort_flag = 0;
        fence_mbar_init();
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmA)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmB)) : "memory");
    }
    if (warp == 1) {   // TMEM allocation (whole warp)
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const uint64_t lim = wait_limit(p.wait_ns);

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        // The whole warp walks the loop and waits (lane 0 issues): a warp with
        // one lane looping and 31 parked at the final barrier slows the other
        // warps of its scheduler.
        uint32_t stage = 0, phase = 0, rs = 0, rph = 0;
        uint32_t fills[NSTAGE] = {};
        uint32_t rfills[NRAW] = {};
        bool dep_waited = false;
        TcUnit w;
        int seg = 0;
        for (int u = blockIdx.x; tc_unit<G>(p, u, w, seg); u += gridDim.x) {
            const int m0 = w.a_row, n0 = w.b_row;
            for (int kb = w.kb0; kb < w.kb1; kb += 2) {
                if constexpr (RAW) {
                    if ((kb - w.kb0) % RAW_KB == 0) {   // next raw copy: 8 blocks x 128 rows
                        if (warp_all(!p.withhold && mbar_wait(&raw_empty[rs], rph ^ 1u, p.err, abort_flag, lim) &&
                                     !*abort_flag)) {
                            if (lane == 0) {
                                mbar_arrive_expect_tx(&raw_full[rs], RAW_BYTES);
                                tma_load_3d(raw_s + (size_t)rs * RAW_BYTES, &tmA, (kb / RAW_KB) * RAW_WORDS, m0,
                                            w.expert, &raw_full[rs]);
                            }
                            ++rfills[rs];
                        }
                        __syncwarp();
                        if (++rs == NRAW) {
                            rs = 0;
                            rph ^= 1u;
                        }
                    }
                }
                // After an abort nothing more is issued; consumers release only
                // stages and raw copies they saw land, so each has at most one copy
                // in flight (its last fill), which the drain below waits for.
                if (warp_all(!p.withhold && mbar_wait(&empty[stage], phase ^ 1u, p.err, abort_flag, lim) &&
                             !*abort_flag)) {
                    if (lane == 0) {
                        uint8_t *st = smem + (size_t)stage * STAGE_BYTES;
                        float *dxs = reinterpret_cast<float *>(st + A_BYTES + B_BYTES);
                        if constexpr (RAW) {
                            mbar_arrive_expect_tx(&full[stage], B_BYTES + DX_BYTES);
                        } else {
                            mbar_arrive_expect_tx(&full[stage], STAGE_BYTES);
                            tma_load_2d(st, &tmA, kb * QK, m0, &full[stage]);
                            float *dws = reinterpret_cast<float *>(st + A_BYTES + B_BYTES + DX_BYTES);
                            bulk_g2s(dws, p.dwT + (size_t)kb * p.m_ld + m0, BM * 4, &full[stage]);
                            bulk_g2s(dws + BM, p.dwT + (size_t)(kb + 1) * p.m_ld + m0, BM * 4, &full[stage]);
                        }
                        if (!dep_waited) {
                            // the activations come from the kernel just before this one (launched
                            // with programmatic serialisation); the weights and the plan are older
                            asm volatile("griddepcontrol.wait;" ::: "memory");
                            dep_waited = true;
                        }
                        tma_load_2d(st + A_BYTES, &tmB, kb * QK, n0, &full[stage]);
                        bulk_g2s(dxs, p.dxT + (size_t)kb * p.n_ld + n0, BN * 4, &full[stage]);
                        bulk_g2s(dxs + BN, p.dxT + (size_t)(kb + 1) * p.n_ld + n0, BN * 4, &full[stage]);
                    }
                    ++fills[stage];
                }
                __syncwarp();
                if (++stage == NSTAGE) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        if (*abort_flag && lane == 0) {
            // let every copy this warp issued land before the CTA exits
            const uint64_t t_end = global_timer_ns() + WAIT_LIMIT_NS;
            for (int s = 0; s < NSTAGE; ++s)
                if (fills[s]) mbar_drain(&full[s], (fills[s] - 1u) & 1u, t_end);
            for (int s = 0; s < NRAW; ++s)
                if (rfills[s]) mbar_drain(&raw_full[s], (rfills[s] - 1u) & 1u, t_end);
        }
        __syncwarp();
    } else if (warp == 1 || (Cfg<RAW>::NMMA > 1 && warp == W_EXTRA)) {
        // ------------------------------------------------ MMA issuers (stage s: issuer s % NMMA)
        // whole warp in the loop and the waits, lane 0 issues
        constexpr uint32_t NMMA = Cfg<RAW>::NMMA;
        const uint32_t which = warp == 1 ? 0u : 1u;
        uint32_t stage = 0, phase = 0, blk = 0, ks = 0;
        TcUnit w;
        int seg = 0;
        for (int u = blockIdx.x; tc_unit<G>(p, u, w, seg); u += gridDim.x) {
            const uint32_t idesc = tc_idesc(BM, w.ncols);
            for (int kb = w.kb0; kb < w.kb1; kb += 2, ++ks) {
                if (ks % NMMA != which) {   // the other issuer's stage
                    blk += 2;
                    if (++stage == NSTAGE) {
                        stage = 0;
                        phase ^= 1u;
                    }
                    continue;
                }
                const bool staged = mbar_wait(&full[stage], phase, p.err, abort_flag, lim);
                tc_fence_after();
                const uint32_t a_s = smem_addr(smem + (size_t)stage * STAGE_BYTES);
                const uint32_t b_s = a_s + A_BYTES;
                for (int j = 0; j < 2; ++j, ++blk) {
                    const uint32_t slot = blk % NSLOT_T;
                    const bool free_slot = mbar_wait(&tempty[slot], ((blk / NSLOT_T) & 1u) ^ 1u, p.err, abort_flag, lim);
                    tc_fence_after();
                    if (lane == 0 && staged && free_slot) {
                        const uint32_t d_tmem = tmem_base + slot * BN;
#pragma unroll
                        for (int k16 = 0; k16 < 2; ++k16) {
                            const uint32_t koff = (uint32_t)(2 * j + k16) * 32u;   // 16 fp16 = 32 bytes
                            tc_mma_f16(d_tmem, sw128_desc(a_s + koff), sw128_desc(b_s + koff), idesc, k16);
                        }
                    }
                    if (lane == 0) tc_commit(&tfull[slot]);
                    __syncwarp();
                }
                // the stage goes back to the producer once its MMAs are done, unless
                // its copies never landed (timed out)
                if (lane == 0 && staged) tc_commit(&empty[stage]);
                __syncwarp();
                if (++stage == NSTAGE) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        if (lane == 0) tc_commit(done);               // all MMAs issued by this thread
        __syncwarp();
        mbar_wait(done, 0, p.err, nullptr);           // the fixed 2 s limit: TMEM is freed after this
    } else if (warp < 2 + NUM_EPI) {
        // ------------------------------------------------ epilogue
        const int q = warp & 3;                       // TMEM lane quarter of this warp
        const int h = (warp - 2) >> 2;                // column group
        const int m = q * 32 + lane;                  // row within the tile
        const uint32_t lane_addr = tmem_base + ((uint32_t)(q * 32) << 16);
        TcEpi e{smem, full, empty, tfull, tempty, abort_flag, lim, lane_addr, m, h, lane, 0u, 0u, 0u};
        TcUnit w;
        int seg = 0;
        for (int u = blockIdx.x; tc_unit<G>(p, u, w, seg); u += gridDim.x) {
            if (w.ncols == 128) tc_epilogue_unit<128 / EPI_COLG, G, NSTAGE>(p, w, e);
            else if (w.ncols == 64) tc_epilogue_unit<64 / EPI_COLG, G, NSTAGE>(p, w, e);
            else tc_epilogue_unit<32 / EPI_COLG, G, NSTAGE>(p, w, e);
        }
    } else if constexpr (RAW) {
        // ------------------------------------------------ converters: raw copy -> fp16 A tile + scales
        const int ct = threadIdx.x - W_EXTRA * 32;   // 0 .. 63
        uint32_t stage = 0, phase = 0, rs = 0, rph = 0;
        TcUnit w;
        int seg = 0;
        for (int u = blockIdx.x; tc_unit<G>(p, u, w, seg); u += gridDim.x) {
            for (int kg = w.kb0; kg < w.kb1; kg += RAW_KB) {
                const bool raw_ok = mbar_wait(&raw_full[rs], rph, p.err, abort_flag, lim);
                const uint8_t *raw = raw_s + (size_t)rs * RAW_BYTES;
#pragma unroll
                for (int J = 0; J < RAW_KB / 2; ++J) {
                    const bool ok = mbar_wait(&empty[stage], phase ^ 1u, p.err, abort_flag, lim) && raw_ok;
                    if (ok) {
                        uint8_t *st = smem + (size_t)stage * STAGE_BYTES;
                        float *dws = reinterpret_cast<float *>(st + A_BYTES + B_BYTES + DX_BYTES);
                        if (J == 0) tc_convert<0>(raw, st, dws, ct);
                        else if (J == 1) tc_convert<1>(raw, st, dws, ct);
                        else if (J == 2) tc_convert<2>(raw, st, dws, ct);
                        else tc_convert<3>(raw, st, dws, ct);
                        fence_async_smem();
                    }
                    __syncwarp();
                    if (ok && lane == 0) mbar_arrive(&full[stage]);
                    if (++stage == NSTAGE) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                __syncwarp();
                if (raw_ok && lane == 0) mbar_arrive(&raw_empty[rs]);
                if (++rs == NRAW) {
                    rs = 0;
                    rph ^= 1u;
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS)
                     : "memory");
    }
}

// K-split partials -> out, adding the splits in order.
__global__ void __launch_bounds__(256) k_tc_reduce(float *__restrict__ out, const float *__restrict__ partial,
                                                   uint64_t n, int ksplit) {
    for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (uint64_t)gridDim.x * blockDim.x) {
        float s = partial[i];
        for (int k = 1; k < ksplit; ++k) s += partial[(uint64_t)k * n + i];
        out[i] = s;
    }
}

// Raw Q8_0 rows -> fp16 quant plane [rows][in_dim] (exact) and block-major
// scales dwT[b][m_ld] (fp32 of the stored binary16 scale).  A CTA converts tiles
// of 8 rows x 32 blocks: warp w takes row r0 + w and lane l block b0 + l, so a
// warp reads 32 consecutive 34-byte blocks (1088 contiguous bytes) and writes
// 32 consecutive 64-byte runs; the scales go through shared memory and leave
// as 32-byte runs of dwT.

__global__ void __launch_bounds__(256) k_tc_expand(__half *__restrict__ a16, float *__restrict__ dwT,
                                                   const uint8_t *__restrict__ W, uint32_t rows, uint32_t nb,
                                                   uint32_t m_ld) {
    __shared__ float ds[8][33];
    const uint32_t w = threadIdx.x >> 5, l = threadIdx.x & 31;
    const uint32_t tiles_r = (rows + 7) / 8, tiles_b = (nb + 31) / 32;
    const uint64_t tiles = (uint64_t)tiles_r * tiles_b;
    for (uint64_t tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
        const uint32_t tb = (uint32_t)(tile % tiles_b), tr = (uint32_t)(tile / tiles_b);
        const uint32_t r = tr * 8 + w, b = tb * 32 + l;
        if (r < rows && b < nb) {
            const uint16_t *src = reinterpret_cast<const uint16_t *>(W + ((uint64_t)r * nb + b) * QB);
            uint16_t h[17];
#pragma unroll
            for (int i = 0; i < 17; ++i) h[i] = __ldg(src + i);
            ds[w][l] = half_bits_to_float(h[0]);
            uint4 *dst = reinterpret_cast<uint4 *>(a16 + (uint64_t)r * nb * QK + (uint64_t)b * QK);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t o[4];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const uint32_t word = (uint32_t)h[1 + 4 * c + 2 * e] | ((uint32_t)h[2 + 4 * c + 2 * e] << 16);
                    s8x4_to_half2x2(word, o[2 * e], o[2 * e + 1]);
                }
                dst[c] = make_uint4(o[0], o[1], o[2], o[3]);
            }
        }
        __syncthreads();
        {
            const uint32_t bb = threadIdx.x >> 3, rr = threadIdx.x & 7;   // 32 blocks x 8 rows
            const uint32_t r2 = tr * 8 + rr, b2 = tb * 32 + bb;
            if (r2 < rows && b2 < nb) dwT[(uint64_t)b2 * m_ld + r2] = ds[rr][bb];
        }
        __syncthreads();
    }
}

bool encode_f16_tmap(CUtensorMap *map, const void *base, uint64_t cols, uint64_t rows, uint32_t box_cols,
                     uint32_t box_rows);
bool encode_rows_tmap(CUtensorMap *map, const void *W, uint64_t row_bytes, uint64_t rows, uint64_t n_mat,
                      uint64_t mat_stride, uint32_t box_words, uint32_t box_rows);

cudaError_t launch_tc_expand(__half *a16, float *dwT, const uint8_t *W, uint32_t rows, uint32_t nb, uint32_t m_ld,
                             int num_sms, cudaStream_t st) {
    const uint64_t tiles = (uint64_t)((rows + 7) / 8) * ((nb + 31) / 32);
    if (!tiles) return cudaSuccess;
    const uint64_t grid = tiles < (uint64_t)num_sms * 8 ? tiles : (uint64_t)num_sms * 8;
    k_tc_expand<<<(int)grid, 256, 0, st>>>(a16, dwT, W, rows, nb, m_ld);
    return cudaGetLastError();
}

template <bool G, bool RAW>
static cudaError_t launch_tc_variant(const TcParams &p, const CUtensorMap &tmA, const CUtensorMap &tmB, int grid,
                                     cudaStream_t st) {
    static bool attr_done = false;
    if (!attr_done) {
        cudaError_t e = cudaFuncSetAttribute(k_tc_gemm<G, RAW>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)tc::Cfg<RAW>::SMEM);
        if (e != cudaSuccess) return e;
        attr_done = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(tc::Cfg<RAW>::NTHREADS);
    cfg.dynamicSmemBytes = tc::Cfg<RAW>::SMEM;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, k_tc_gemm<G, RAW>, p, tmA, tmB);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess || G || p.ksplit == 1) return e;
    const uint64_t n = (uint64_t)p.N * p.M;
    uint64_t g = (n + 255) / 256;
    if (g > 4096) g = 4096;
    k_tc_reduce<<<(int)g, 256, 0, st>>>(p.out, p.partial, n, p.ksplit);
    return cudaGetLastError();
}

cudaError_t launch_tc_gemm(const TcParams &p, const __half *a16, const __half *b16, uint64_t n_rows_b, int grid,
                           cudaStream_t st) {
    if (p.plan) return cudaErrorInvalidValue;   // grouped units read raw weights
    alignas(64) CUtensorMap tmA, tmB;
    const uint64_t K = (uint64_t)p.nb * QK;
    if (!encode_f16_tmap(&tmA, a16, K, (uint64_t)p.M, tc::BK, tc::BM)) return cudaErrorInvalidValue;
    if (!encode_f16_tmap(&tmB, b16, K, n_rows_b, tc::BK, tc::BN)) return cudaErrorInvalidValue;
    return launch_tc_variant<false, false>(p, tmA, tmB, grid, st);
}

cudaError_t launch_tc_gemm_raw(const TcParams &p, const uint8_t *W, uint64_t n_mat, uint64_t mat_stride,
                               const __half *b16, uint64_t n_rows_b, int grid, cudaStream_t st) {
    if (p.nb % tc::RAW_KB || (!p.plan && p.kb_per % tc::RAW_KB)) return cudaErrorInvalidValue;
    alignas(64) CUtensorMap tmA, tmB;
    const uint64_t K = (uint64_t)p.nb * QK;
    if (!encode_rows_tmap(&tmA, W, (uint64_t)p.nb * QB, (uint64_t)p.M, n_mat, mat_stride, tc::RAW_WORDS, tc::BM))
        return cudaErrorInvalidValue;
    if (!encode_f16_tmap(&tmB, b16, K, n_rows_b, tc::BK, tc::BN)) return cudaErrorInvalidValue;
    return p.plan ? launch_tc_variant<true, true>(p, tmA, tmB, grid, st)
                  : launch_tc_variant<false, true>(p, tmA, tmB, grid, st);
}

}  // namespace q8
