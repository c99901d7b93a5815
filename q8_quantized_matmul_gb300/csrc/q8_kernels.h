// q8_kernels.h -- internal launch interface between the C ABI layer and the kernels.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace q8 {

// Segment table written by the routing kernels (grouped mode) or filled on
// the host (dense mode: one segment).  Segment s covers activation-plane rows
// [row0, row0 + count) (padded to a multiple of 16 rows with zero rows) and
// multiplies them by the weights of `expert`.
struct Segment {
    int32_t expert;
    int32_t row0;
    int32_t count;
    int32_t item_start;   // first work item of this segment
};

struct PlanHeader {      // device-side header before the segment array
    int32_t n_segments;
    int32_t n_items;
    int32_t n_rows;      // activation-plane rows used (multiple of 16)
    int32_t row_end;     // end of this class's rows (the tensor-core class holds rows [0, row_end))
};

struct MmaParams {
    const uint8_t *W;          // raw Q8_0 rows (dense) or the first expert's rows
    uint64_t expert_stride;    // bytes between experts
    uint64_t in_dim;
    uint32_t out_dim;
    uint32_t nb;               // in_dim / 32
    const int8_t *qx;          // activation quant plane [rows][in_dim]
    const float *dx;           // activation scale plane [rows][nb]
    float *out;                // [*][out_dim]
    int *err;                  // device error word
    // dense mode (plan == nullptr): one segment of n_tok rows, output row = plane row
    uint32_t n_tok;
    // grouped mode
    const PlanHeader *plan;    // header followed by Segment[n_segments]
    const int32_t *row_to_out; // plane row -> output row (-1: padding)
};

// Quantiser (q8_quantize.cu)
cudaError_t launch_quantize_blocks(uint8_t *xq, const float *x, uint64_t nblk, int num_sms, cudaStream_t st);
// programmatic: launch with programmatic stream serialisation (the kernel waits
// for the previous grid before it reads or writes anything).
cudaError_t launch_quantize_planes(int8_t *qplane, float *dplane, const float *x, uint64_t in_dim, uint64_t n_rows,
                                   const int32_t *src_row, uint64_t n_src, int num_sms, cudaStream_t st,
                                   bool programmatic = false);
// Routed pairs straight to their plane rows: pair p (activation row p, or p / k
// when x holds one row per token) goes to plane row dst_row[p]; padding rows are
// not written.  With tc_plan, rows [0, tc_plan->row_end) go to the tensor-core
// operand instead: fp16 quants q16[r][in_dim], scales dxT[b][n_ld].
cudaError_t launch_quantize_pairs(int8_t *qplane, float *dplane, __half *q16, float *dxT, uint64_t n_ld,
                                  const PlanHeader *tc_plan, const float *x, uint64_t in_dim, uint64_t n_pairs,
                                  uint32_t k, int x_per_pair, const int32_t *dst_row, int num_sms, cudaStream_t st);
cudaError_t launch_unpack_blocks(int8_t *qplane, float *dplane, const uint8_t *xq, uint64_t in_dim, uint64_t n_rows,
                                 uint64_t n_src, int num_sms, cudaStream_t st);

// Tensor-core (mma.sync int8) matmul over raw Q8_0 rows (q8_mma.cu).
// Requires nb % 8 == 0, W and expert_stride 16-byte aligned.
cudaError_t launch_mma(const MmaParams &p, int grid, cudaStream_t st);
// Any in_dim % 32 == 0 and 2-byte aligned W: one thread per output (slow path).
cudaError_t launch_generic(const MmaParams &p, int max_items_hint, int num_sms, cudaStream_t st);

// Routing (q8_moe.cu): buckets pairs by expert and writes three plans, one per
// size class of expert group: class 0 = groups of <= 8 rows (GEMV, one 8-token
// MMA tile), class 1 = more rows (GEMV, 16-token groups: a group of 60 rows is 4
// token groups, each streaming the expert's weights, which stay in L2 while the
// groups run side by side), class 2 = groups of more than MOE_TC_MIN_ROWS rows,
// at most tc_cap of them (the grouped tcgen05 GEMM on raw Q8_0 expert rows;
// items are 128-row x 128-token tiles).
// Experts are taken largest first, so the class-2 groups own plane rows
// [0, row_end).  Each plan is a PlanHeader followed by Segment[n_expert];
// GEMV items are rows_gemv rows x one token group.
//   row_to_out, src_row: int32[max_rows], max_rows = route_max_rows(n_pairs, n_expert)
//   dst_row (optional): int32[n_pairs], pair -> plane row (-1: bad id)
//   counts, row0_of: int32[n_expert] scratch
constexpr int ROUTE_CLASSES = 3;
constexpr int ROUTE_GEMV_CLASSES = 2;          // classes 0 and 1 run on the GEMV
constexpr int MOE_TC_MIN_ROWS = 16;            // class 2 takes groups of more rows than this
constexpr uint64_t MOE_TC_MIN_PAIRS = 1024;    // ... in batches of at least this many pairs
uint64_t route_max_rows(uint64_t n_pairs, uint64_t n_expert);
size_t route_plan_bytes(uint32_t n_expert);
cudaError_t launch_route(const int32_t *ids, uint64_t n_tok, uint32_t k, uint32_t n_expert, int x_per_pair,
                         uint32_t out_dim, uint32_t rows_gemv, uint32_t tc_cap, int32_t *counts, int32_t *row0_of,
                         uint8_t *plans, int32_t *row_to_out, int32_t *src_row, int32_t *dst_row, uint64_t max_rows,
                         float *out, int *err, int num_sms, cudaStream_t st);

// Weight-streaming GEMV (q8_gemv.cu).  Modes: 0 = dp4a, token groups of <= 2;
// 1 = fp16 MMA, one 8-token N tile; 2 = two N tiles (<= 16 tokens).
struct GemvParams {
    const uint8_t *W;
    uint64_t expert_stride;
    uint64_t in_dim;
    uint32_t out_dim;
    uint32_t nb;
    const int8_t *qx;          // activation quant plane [rows][in_dim] (groups padded to 16 rows)
    const float *dx;           // activation scale plane [rows][nb]
    const float *x;            // dense only: fp32 rows [n_tok][in_dim] quantised in the kernel (qx, dx unused)
    int weights_early;         // 1: the weight stream starts before griddepcontrol.wait (W is never
                               //    written by a kernel that triggers its dependents early)
    float *out;
    int *err;
    uint32_t n_tok;            // dense: the tokens (<= 8 or 16)
    uint32_t rows_per_item;    // grouped: rows per item, multiple of 16, <= 512
    uint32_t n_items;          // dense: items (contiguous runs of 16-row sub-items, <= 32 each)
    uint32_t sub_base;         // dense: every item has sub_base sub-items, the first sub_rem one more
    uint32_t sub_rem;
    const PlanHeader *plan;    // grouped: class plan; nullptr: dense
    const int32_t *row_to_out;
    uint32_t n_expert;         // grouped: number of expert matrices
    // Gate/up pair (grouped only; nullptr otherwise): W holds the gate and W2 the up
    // projections (same shape and expert stride).  An item streams both row ranges
    // against one staging of its activations, and out receives
    // swiglu1(gate, up, limit) instead of either product; rows_per_item <= 256.
    const uint8_t *W2;
    float limit;
    // With a pair: q_out / d_out non-null take mid as Q8_0 planes instead of fp32
    // rows in out (row = the activation-plane row of the pair, out_dim values a row;
    // the quantiser's arithmetic, so the bits of quantising the fp32 rows).
    int8_t *q_out;
    float *d_out;
    // Grouped: the plan's GEMV items were counted with plan_rb row blocks per token
    // group (0: this call's own ceil(out_dim / rows_per_item)), so one routing
    // serves products of different widths.
    uint32_t plan_rb;
    // Failure-detection test hook (zero in normal calls): wait_ns limits every wait
    // (0: the 2 s default); withhold != 0 makes the producer issue no copy, so the
    // consumers' waits run out, the kernel raises Q8_ETIMEOUT and returns.
    uint64_t wait_ns;
    int withhold;
};
constexpr uint32_t GEMV_MAX_ROWS_PER_ITEM = 512;
// Launched with programmatic stream serialisation; see GemvParams::weights_early.
cudaError_t launch_gemv(const GemvParams &p, int mode, int grid, cudaStream_t st);
inline int gemv_mode(uint64_t n_tok) { return n_tok <= 2 ? 0 : (n_tok <= 8 ? 1 : 2); }
// The dense GEMV quantises the activations itself when each CTA's share of that
// work stays small: at most 8 tokens and 1024 (token, block) pairs with the
// mode's token count.  (At 16 tokens the in-kernel quantiser delays the first
// MMA by more than the separate quantiser kernel costs.)
inline bool gemv_fuses_quantiser(uint64_t n_tok, uint64_t nb) {
    const uint64_t tok = n_tok <= 2 ? 2 : 8;
    return n_tok <= 8 && tok * nb <= 1024;
}
// Dense items: one per SM while there are enough 16-row sub-items, each at most
// GEMV_MAX_ROWS_PER_ITEM rows.
inline void gemv_dense_split(uint64_t out_dim, uint32_t n_items, uint32_t &base, uint32_t &rem) {
    const uint64_t nsub = (out_dim + 15) / 16;
    base = (uint32_t)(nsub / n_items);
    rem = (uint32_t)(nsub % n_items);
}
inline uint32_t gemv_dense_items(uint64_t out_dim, int num_sms) {
    const uint64_t nsub = (out_dim + 15) / 16;
    const uint64_t per = GEMV_MAX_ROWS_PER_ITEM / 16;
    uint64_t items = nsub < (uint64_t)num_sms ? nsub : (uint64_t)num_sms;
    if (items * per < nsub) items = (nsub + per - 1) / per;
    return (uint32_t)items;
}

// RMSNorm feeding the quantiser (q8_quantize.cu): per token row, y = x / sqrt(mean x^2 + eps)
// * gamma (gamma null: ones), xq = the activation quantiser of y ([n_tok][dim/32] blocks).
// x, gamma, y 16-byte aligned; y may be null; dim % 32 == 0.
// err: the device error word (an expired bounded wait of the TMA-fed kernel); wait_ns (0: the
// default limit) and withhold (issue no copy) are the failure-detection test hook, used only by
// the TMA-fed kernel, which rmsnorm_uses_tma() says the call will run.
bool rmsnorm_uses_tma(uint64_t dim, uint64_t n_tok, int num_sms);
cudaError_t launch_rmsnorm_quantize(uint8_t *xq, float *y, const float *x, const float *gamma, uint64_t dim,
                                    uint64_t n_tok, float eps, int *err, uint64_t wait_ns, int withhold, int num_sms,
                                    cudaStream_t st);

// Elementwise steps of the routed expert FFN (q8_ffn.cu).
//   launch_swiglu:  mid[i] = silu(min(gate[i], L)) * clamp(up[i], -L, L) (L = limit; 0: no
//                   clamp) for n values; gate, up, mid 16-byte aligned.  With ids, the values
//                   are rows of row_len (a multiple of 4) and the row of a pair whose id is
//                   outside [0, n_expert) is written as zeros.
//   launch_combine: out[t][o] = sum_j w[t*k+j] * y[t*k+j][o], j in order; out and y
//                   16-byte aligned.
cudaError_t launch_swiglu(float *mid, const float *gate, const float *up, uint64_t n, float limit,
                          const int32_t *ids, uint32_t n_expert, uint64_t row_len, int num_sms, cudaStream_t st);
cudaError_t launch_combine(float *out, const float *y, const float *w, uint64_t n_tok, uint32_t k, uint64_t dim,
                           int num_sms, cudaStream_t st);

// Prefill GEMM on tcgen05 (q8_tc.cu).  Weights as an fp16 plane [M][K] (from
// launch_tc_expand) with block-major scales dwT[nb][m_ld]; activations as an
// fp16 plane [n_ld rows][K] with block-major scales dxT[nb][n_ld]
// (launch_quantize_f16t / launch_unpack_f16t).  m_ld % 128 == 0, n_ld % 128 == 0,
// nb even.  With ksplit > 1, partial[ksplit][N][M] holds the K-split sums.
struct TcParams {
    int M;                 // weight rows (out_dim)
    int N;                 // tokens
    int nb;                // blocks per row
    int ksplit;            // K splits
    int kb_per;            // blocks per split (even)
    const float *dxT;
    const float *dwT;
    uint64_t n_ld, m_ld;
    float *out;            // [N][M]
    float *partial;        // [ksplit][N][M] or nullptr
    int *err;
    // grouped (routed experts, plan != nullptr; raw weights only): the units of
    // the class-2 plan.  Segment s multiplies its expert's rows by plane rows
    // [row0, row0 + count) and writes output row row_to_out[plane row].  N,
    // ksplit and kb_per are unused (no K split).
    const PlanHeader *plan;
    const int32_t *row_to_out;
    // Failure-detection test hook, as in GemvParams (zero in normal calls).
    uint64_t wait_ns;
    int withhold;
};
// Second weight format (q8_kq.cu): Q2_K / Q4_K rows against Q8_K activation
// planes (quants [rows][in_dim], fp32 scales [rows][in_dim/256], int16 sums of
// each 16 quants [rows][in_dim/16]).  Dense: tokens 0..n_tok-1, work items of
// rows_per_item rows x one token group.  Routed: the items of one GEMV-class
// routing plan (token groups of 8 for class 0, 16 for class 1); plane row i
// reads activation row src_row[i] and writes output row row_to_out[i].
constexpr int KQ_Q2 = 2, KQ_Q4 = 4;
struct KqParams {
    const uint8_t *W;
    uint64_t expert_stride;
    uint64_t in_dim;
    uint32_t out_dim;
    uint32_t nsb;              // blocks per row (in_dim / 256)
    int fmt;                   // KQ_Q2 or KQ_Q4
    const int8_t *qx;
    const float *dx;
    const int16_t *xs;
    float *out;                // [rows][out_dim]
    int *err;
    uint32_t n_tok;            // dense
    uint32_t rows_per_item;
    const PlanHeader *plan;    // routed: class plan; nullptr: dense
    const int32_t *src_row;
    const int32_t *row_to_out;
};
// x [n_rows][in_dim] -> the planes (qx, dx, xs; all or none) and/or canonical
// 292-byte Q8_K blocks (fp32 d, int8 qs[256], int16 sums of each 16 quants).
cudaError_t launch_quantize_q8k(int8_t *qx, float *dx, int16_t *xs, uint8_t *blocks, const float *x, uint64_t in_dim,
                                uint64_t n_rows, int num_sms, cudaStream_t st);
// tokg: 8 or 16 (the token group of the plan's class; dense: either).
cudaError_t launch_kq_gemv(const KqParams &p, int tokg, int num_sms, cudaStream_t st);
// The staged variant (weights through a shared-memory ring by bulk copies).
// kq_stream_rows: rows per work item it takes for rows of row_bytes and token
// groups of tokg (0: rows not 16-byte multiples, or the rows or the group's
// activations too long: use launch_kq_gemv).  W and the expert stride must be
// 16-byte aligned; rows_per_item <= kq_stream_rows(row bytes, in_dim, tokg).
uint32_t kq_stream_rows(uint64_t row_bytes, uint64_t in_dim, int tokg);
cudaError_t launch_kq_stream(const KqParams &p, int tokg, int num_sms, cudaStream_t st);

cudaError_t launch_tc_expand(__half *a16, float *dwT, const uint8_t *W, uint32_t rows, uint32_t nb, uint32_t m_ld,
                             int num_sms, cudaStream_t st);
// n_rows_b: rows of the b16 plane (the tensor map's extent).  Dense only.
cudaError_t launch_tc_gemm(const TcParams &p, const __half *a16, const __half *b16, uint64_t n_rows_b, int grid,
                           cudaStream_t st);
// The same GEMM with the weights read as raw Q8_0 rows (n_mat matrices of M rows,
// mat_stride bytes apart; grouped units take the segment's expert) and converted
// to fp16 in shared memory: no a16 / dwT planes.  nb % 8 == 0 and, dense,
// kb_per % 8 == 0; W and mat_stride 16-byte aligned.
cudaError_t launch_tc_gemm_raw(const TcParams &p, const uint8_t *W, uint64_t n_mat, uint64_t mat_stride,
                               const __half *b16, uint64_t n_rows_b, int grid, cudaStream_t st);
cudaError_t launch_quantize_f16t(__half *q16, float *dxT, const float *x, uint64_t in_dim, uint64_t n_tok,
                                 uint64_t n_ld, int num_sms, cudaStream_t st);
cudaError_t launch_unpack_f16t(__half *q16, float *dxT, const uint8_t *xq, uint64_t in_dim, uint64_t n_tok,
                               uint64_t n_ld, int num_sms, cudaStream_t st);

// Repack (q8_repack.cu)
cudaError_t launch_repack(uint8_t *Wp, const uint8_t *W, uint64_t in_dim, uint64_t rows, int num_sms,
                          cudaStream_t st);
cudaError_t launch_matmul_packed(float *out, const uint8_t *Wp, uint64_t in_dim, uint64_t out_dim,
                                 const int8_t *qx, const float *dx, uint64_t n_tok, int num_sms, cudaStream_t st);

}  // namespace q8
