/*
 * q8.h -- C ABI of the GB300 (sm_103a) Q8_0-weight x Q8_0-activation matmul library.
 *
 * The operation is the one the ds4 engine's "Q8_0 quantised matmul" entry
 * (GPU code walkthrough, trace 3, ds4_gpu_matmul_q8_0_tensor) performs:
 *
 *     out[t][o] = sum_b  d_w[o][b] * d_x[t][b] * sum_{i<32} q_w[o][b][i] * q_x[t][b][i]
 *
 * accumulated in fp32, where W holds out_dim rows of in_dim weights in Q8_0
 * blocks and the activations are quantised per 32-element block with the
 * formula printed for the Q8_K quantiser (model-architecture page,
 * quantisation section 1): d = max|x| / 127, q = roundf(x / d).
 *
 * Formats
 *   Q8_0 block: 34 bytes = fp16 scale d (IEEE binary16, little-endian) then
 *   int8 q[32].  A row of in_dim values is in_dim/32 consecutive blocks; a
 *   matrix is its rows back to back (row o = output o).  in_dim % 32 == 0
 *   (the pages' alignment requirement).
 *   Activations x: fp32, [n_tok][in_dim], row-major, token-major.
 *   Outputs out: fp32, [n_tok][out_dim], row-major.
 *
 * Conventions (all entry points)
 *   - Every pointer argument is a DEVICE pointer owned by the caller, unless
 *     an entry point says otherwise.  The library never frees caller memory.
 *   - Calls are asynchronous on `stream` (a cudaStream_t passed as void*;
 *     NULL = the legacy default stream) and return Q8_OK when the work was
 *     enqueued, or a negative Q8_E* code, in which case nothing was enqueued.
 *   - Arguments are validated on the host before any launch: null pointers,
 *     zero or misaligned dimensions and size overflow give Q8_EINVAL; W, x,
 *     out and xq must be 16-byte aligned, else Q8_EALIGN.  n_tok == 0 or
 *     out_dim == 0 is valid and does nothing.
 *   - Errors found on the device (an expert id out of range) never trap:
 *     the affected output rows are written as zeros and a device error word
 *     is raised; q8_last_error() reads and clears it.
 *   - Results are deterministic: the same inputs give the same bits on every
 *     run (fixed reduction order, no floating-point atomics).
 *   - The library keeps a per-device grow-only scratch buffer for quantised
 *     activations and routing tables (the pages' reused aligned Q8 scratch).
 *     Calls that use scratch must not run concurrently on different streams
 *     of the same device.  q8_release() frees it.
 *   - Kernels are launched with programmatic stream serialisation: a kernel
 *     may start while the one before it on the stream finishes, once that one
 *     has signalled its dependents.  Everything a kernel reads is read after
 *     it waits for its predecessor, except weights: the decode kernels may
 *     start streaming W, and q8_rmsnorm_quantize may load gamma, before that
 *     wait.  So W and gamma must not be written by a kernel that signals
 *     programmatic dependents before its writes (none of this library's
 *     kernels writes weights; a kernel that does not use programmatic
 *     launches is always waited for in full).
 */
#ifndef Q8_H
#define Q8_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define Q8_BLOCK 32        /* values per Q8_0 block */
#define Q8_BLOCK_BYTES 34  /* fp16 d + int8 q[32] */

enum q8_status {
    Q8_OK = 0,
    Q8_EINVAL = -1,      /* bad dimension, null pointer, in_dim % 32 != 0, overflow */
    Q8_EALIGN = -2,      /* a pointer is not 16-byte aligned */
    Q8_ERANGE = -3,      /* (device) an expert id was outside [0, n_expert) */
    Q8_ENOMEM = -4,      /* scratch allocation failed */
    Q8_ECUDA = -5,       /* a CUDA runtime call failed (no device, launch error, ...) */
    Q8_ETIMEOUT = -6,    /* (device) a kernel's bounded wait expired; outputs undefined */
    Q8_ESCRATCH = -7     /* the call needs more than the fixed scratch of q8_matmul_noalloc */
};

/* Library version (major*10000 + minor*100 + patch). */
int q8_version(void);

/* Human-readable name of a status code (static string). */
const char *q8_strerror(int status);

/*
 * Activation quantiser (model-architecture page, quantisation section 1,
 * applied to 32-element blocks with the scale stored as binary16).
 *   xq   out: n_tok * (in_dim/32) Q8_0 blocks, token-major ([n_tok][in_dim/32]).
 *   x    in:  fp32 [n_tok][in_dim].
 * Per block: amax = max|x_i| (fp32); d = amax / 127.0f (IEEE division);
 * if d == 0 every q_i = 0 and the stored d is +0; otherwise
 * q_i = (int8) roundf(x_i / d) (IEEE division by the fp32 d, halves away from
 * zero) and the stored d is d rounded to binary16 (nearest, ties to even,
 * subnormals kept).  Bit-exact: the same bytes as the CPU definition.
 * NaN/Inf inputs are outside the contract.
 */
int q8_quantize_act(void *xq, const float *x, uint64_t in_dim, uint64_t n_tok, void *stream);

/*
 * RMSNorm feeding the quantiser: the producer of a projection's input writes
 * the quantised activations directly, so the separate quantiser pass goes away
 * (the pages fold the HC RMS norm into the projection input: GPU concepts page,
 * §4m, and the fused RMS-norm producers of §4n).  Per token row t:
 *   r = 1 / sqrt(mean_i x[t][i]^2 + eps),  y[t][i] = (x[t][i] * r) * gamma[i]
 *   xq[t] = the q8_quantize_act quantiser of y[t]     (bit for bit)
 * The pages name the norm (attn_norm, ffn_norm) but print no formula; this is
 * the usual RMSNorm.  fp32 arithmetic: the sum of squares in a fixed order
 * (same bits on every run) with relative error at most (8 ceil(dim/2048) + 14)
 * 2^-24; sqrt and division are IEEE.
 *   xq     out: [n_tok][dim/32] Q8_0 blocks (input of q8_matmul_q).
 *   y      out: fp32 [n_tok][dim], the normalised rows, or NULL.
 *   x      in:  fp32 [n_tok][dim];  gamma in: fp32 [dim], or NULL for all ones.
 *   eps    > 0 and finite (else Q8_EINVAL); dim % 32 == 0.
 * xq, x, y and gamma 16-byte aligned (Q8_EALIGN).
 */
int q8_rmsnorm_quantize(void *xq, float *y, const float *x, const float *gamma, uint64_t dim,
                        uint64_t n_tok, float eps, void *stream);

/*
 * Q8_0 matmul from fp32 activations (GPU code walkthrough, trace 3:
 * ds4_gpu_matmul_q8_0_tensor(out, model_map, ..., weight_offset, in_dim,
 * out_dim, x, n_tok); here W is already a device pointer to the weight rows).
 *   out  out: fp32 [n_tok][out_dim].
 *   W    in:  out_dim rows of in_dim/32 Q8_0 blocks (34 bytes each).
 *   x    in:  fp32 [n_tok][in_dim]; quantised per block into library scratch
 *             with exactly the q8_quantize_act arithmetic.
 * n_tok <= 16 runs the weight-streaming decode kernel; larger n_tok the
 * prefill GEMM.  Both give out[t][o] = sum over blocks, in fp32, of
 * d_w*d_x*isum with isum the exact int32 block dot; the summation order
 * differs from a sequential loop only by fp32 rounding.
 */
int q8_matmul(float *out, const void *W, uint64_t in_dim, uint64_t out_dim,
              const float *x, uint64_t n_tok, void *stream);

/*
 * q8_matmul with the activations and the result in HOST memory, the way an
 * engine's decode step hands a token's activations to the GPU and reads the
 * result back; the weights stay resident on the device (the pages keep the
 * model mapped once and pass weight offsets into it).
 *   out_host  out: fp32 [n_tok][out_dim], host memory.
 *   W         in:  device pointer, as for q8_matmul (16-byte aligned).
 *   x_host    in:  fp32 [n_tok][in_dim], host memory.
 * When both buffers are page-locked (cudaHostAlloc, cudaMallocHost, or
 * cudaHostRegister with mapping; pinned torch tensors) and 16-byte aligned,
 * the q8_matmul kernels read x_host and write out_host directly through the
 * GPU's host link (NVLink-C2C on Grace systems): one call is just the kernels.
 * From 3 to 16 tokens x_host is then read once, by the quantiser kernel (not
 * by every CTA of the GEMV), and from 3 tokens and 12 x 152 16-row sub-items of
 * output up each CTA of the GEMV takes two items, so that the first one's
 * results cross the link while the second one's weights stream; those results
 * agree with q8_matmul's within the matmul's error bound (partial sums of two
 * warps are added in another order), all others bit for bit.
 * Otherwise, on `stream`, in order: x_host is copied into a library-owned
 * device staging buffer, the kernels run on it, and the result is copied to
 * out_host: the results of q8_matmul, bit for bit.
 * Host buffers need no alignment.  The work is asynchronous: x_host must stay
 * unchanged and out_host is valid only once `stream` has synchronised (with
 * pageable buffers the CUDA runtime stages the copies and the call may block
 * until they are done).  The staging buffer is grow-only, per device, counted
 * by q8_scratch_bytes and freed by q8_release; like the scratch, it must not
 * be used from two streams at once.
 */
int q8_matmul_host(float *out_host, const void *W, uint64_t in_dim, uint64_t out_dim,
                   const float *x_host, uint64_t n_tok, void *stream);

/*
 * Same product from activations already quantised by q8_quantize_act
 * (xq: [n_tok][in_dim/32] Q8_0 blocks, 16-byte aligned).
 */
int q8_matmul_q(float *out, const void *W, uint64_t in_dim, uint64_t out_dim,
                const void *xq, uint64_t n_tok, void *stream);

/*
 * Routed-expert matmul (GPU code walkthrough, trace 5: the per-expert
 * projections of ds4_gpu_routed_moe_one_tensor; MoE C notes, section 1: one
 * weight matrix per expert, only the selected ones are read).  Pairs are
 * p = t*k + j for token t and slot j; expert e = expert_ids[p].
 *   out               out: fp32 [n_tok*k][out_dim]; row p = W_e . x_row.
 *   W_experts         in:  n_expert matrices, expert e at byte offset
 *                          e*expert_stride_bytes, each out_dim rows of Q8_0 blocks.
 *   expert_stride_bytes    >= out_dim*(in_dim/32)*34, a multiple of 16.
 *   expert_ids        in:  int32 [n_tok][k] (device).
 *   x                 in:  fp32; x_per_pair == 0: [n_tok][in_dim], x_row = row t
 *                          (gate/up projections); x_per_pair != 0:
 *                          [n_tok*k][in_dim], x_row = row p (down projection).
 * Pairs are bucketed by expert on the device (stable in p), each expert's
 * weights are streamed once for all of its pairs.  An id outside
 * [0, n_expert) gives a zero row and raises Q8_ERANGE for q8_last_error().
 */
int q8_moe_matmul(float *out, const void *W_experts, uint32_t n_expert,
                  uint64_t expert_stride_bytes, const int32_t *expert_ids, uint32_t k,
                  uint64_t in_dim, uint64_t out_dim, const float *x, int x_per_pair,
                  uint64_t n_tok, void *stream);

/*
 * Second weight format: K-quant blocks against Q8_K activations (model-
 * architecture page, quantisation section 3, "Block layout": Q2_K and Q4_K
 * blocks of 256 weights; section 1: the 2-bit field order and the Q8_K
 * quantiser; section 4: the K-quant x Q8_K dot; the routed experts of the GPU
 * code walkthrough, trace 5, and the MoE page's Q4_K expert path use them).
 * The pages give the blocks' fields and sizes; the packing inside a block is
 * GGML's k-quant layout, the format the pages attribute these blocks to:
 *   Q2_K (fmt Q8_KQ_Q2_K, 84 bytes): scales[16], qs[64], d, dmin (binary16,
 *     little-endian).  Sub-block i (16 weights) has scale scales[i] & 15 and min
 *     scales[i] >> 4; weight 128h + 32j + 16s + l is 2-bit field j
 *     ((byte >> 2j) & 3) of qs[32h + 16s + l], in sub-block 8h + 2j + s.
 *   Q4_K (fmt Q8_KQ_Q4_K, 144 bytes): d, dmin, scales[12], qs[128].  Sub-block
 *     j (32 weights) has 6-bit scale and min: j < 4: s[j] & 63, s[j+4] & 63;
 *     j >= 4: (s[j+4] & 15) | (s[j-4] >> 6) << 4, (s[j+4] >> 4) | (s[j] >> 6) << 4.
 *     Weight 64c + l is the low nibble of qs[32c + l] (sub-block 2c), weight
 *     64c + 32 + l its high nibble (sub-block 2c + 1).
 *   Weight value: d * sc * q - dmin * m.
 * Rows are in_dim/256 consecutive blocks; in_dim % 256 == 0.
 *   Q8_K block (292 bytes): fp32 d = max|x| / 127, int8 qs[256] = roundf(x / d)
 *     (an all-zero block: d = 0, q = 0), then int16 sums of each 16 quants.
 *
 * q8_kq_row_bytes:  bytes of one row (0 for a bad fmt or in_dim).
 * q8_quantize_q8k:  xq (out, [n_tok][in_dim/256] Q8_K blocks, 4-byte aligned)
 *                   <- x (fp32 [n_tok][in_dim], 16-byte aligned); bit-exact to
 *                   the formula (IEEE fp32 division, roundf).
 * q8_kq_matmul:     out[t][o] = sum over blocks and sub-blocks of
 *                   d_x * (d * sc * sum q_w q_x - dmin * m * sum q_x), the
 *                   integer sums exact, the rest fp32; x is quantised to Q8_K in
 *                   the library scratch.  out fp32 [n_tok][out_dim]; W out_dim
 *                   rows (16-byte aligned for Q4_K, 4-byte for Q2_K).
 * q8_kq_moe_matmul: the routed product over K-quant experts, arguments as
 *                   q8_moe_matmul's (expert_stride_bytes >= one matrix, a
 *                   multiple of 16 for Q4_K and of 4 for Q2_K); an id outside
 *                   [0, n_expert) gives a zero row and raises Q8_ERANGE.
 * The matmuls run a weight-streaming kernel (dp4a on the integer quants, one
 * lane per two sub-blocks) over token groups of up to 16; more tokens re-read
 * the weights once per group.
 */
#define Q8_KQ_Q2_K 2
#define Q8_KQ_Q4_K 4
#define Q8_Q8K_BLOCK_BYTES 292
uint64_t q8_kq_row_bytes(uint64_t in_dim, int fmt);
int q8_quantize_q8k(void *xq, const float *x, uint64_t in_dim, uint64_t n_tok, void *stream);
int q8_kq_matmul(float *out, const void *W, int fmt, uint64_t in_dim, uint64_t out_dim,
                 const float *x, uint64_t n_tok, void *stream);
int q8_kq_moe_matmul(float *out, const void *W_experts, int fmt, uint32_t n_expert,
                     uint64_t expert_stride_bytes, const int32_t *expert_ids, uint32_t k,
                     uint64_t in_dim, uint64_t out_dim, const float *x, int x_per_pair,
                     uint64_t n_tok, void *stream);

/*
 * Routed expert FFN around the routed matmul (GPU code walkthrough, trace 5:
 * ds4_gpu_routed_moe_one_tensor runs, for the selected experts, the gate and up
 * projections, SwiGLU, the down projection and the weighted sum; the MoE study
 * page, SwiGLU activation section, gives mid = silu(gate) * up and the clamp).
 * Pairs p = t*k + j select expert e = expert_ids[p] with weight expert_weights[p]:
 *   gate[p] = W_gate[e] . x[t],  up[p] = W_up[e] . x[t]        (in_dim -> mid_dim)
 *   mid[p]  = silu(min(gate, limit)) * clamp(up, -limit, limit) (limit 0: no clamp)
 *   y[p]    = W_down[e] . mid[p]                               (mid_dim -> out_dim)
 *   out[t]  = sum_j expert_weights[t*k+j] * y[t*k+j]          (j in slot order)
 * x and mid are quantised per 32-block exactly as q8_quantize_act does, and
 * each projection is the q8_moe_matmul product (the gate and up projections
 * share one routing and one quantisation of x; below 1024 pairs one kernel
 * streams both against one staging of x and applies SwiGLU in its epilogue,
 * with the same bits as the separate steps).  silu(g) = g / (1 + e^-g) in
 * fp32 (CUDA expf, IEEE division).
 *   out               out: fp32 [n_tok][out_dim].
 *   W_gate, W_up      in:  n_expert matrices each, expert e at e*gate_up_stride_bytes,
 *                          each mid_dim rows of in_dim/32 Q8_0 blocks.
 *   W_down            in:  n_expert matrices, expert e at e*down_stride_bytes, each
 *                          out_dim rows of mid_dim/32 blocks.
 *   expert_ids        in:  int32 [n_tok][k];  expert_weights in: fp32 [n_tok][k].
 *   limit                  >= 0 (NaN or negative: Q8_EINVAL).
 *   x                 in:  fp32 [n_tok][in_dim].
 * in_dim and mid_dim are multiples of 32; strides are multiples of 16 and at
 * least one matrix long.  Intermediates (gate, up, mid, y) live in the
 * library scratch.  A pair with an id outside [0, n_expert) contributes zero
 * and raises Q8_ERANGE for q8_last_error().
 */
int q8_moe_ffn(float *out, const void *W_gate, const void *W_up, const void *W_down,
               uint32_t n_expert, uint64_t gate_up_stride_bytes, uint64_t down_stride_bytes,
               const int32_t *expert_ids, const float *expert_weights, uint32_t k,
               uint64_t in_dim, uint64_t mid_dim, uint64_t out_dim, float limit,
               const float *x, uint64_t n_tok, void *stream);

/*
 * The FFN's elementwise steps on their own.
 *   q8_swiglu:      mid[i] = silu(min(gate[i], limit)) * clamp(up[i], -limit, limit)
 *                   for i < n (limit 0: no clamp; NaN or negative: Q8_EINVAL);
 *                   mid, gate, up fp32, 16-byte aligned.
 *   q8_moe_combine: out[t][o] = sum_{j<k} weights[t*k+j] * y[t*k+j][o], j in
 *                   order, each product and sum rounded to fp32; out [n_tok][dim]
 *                   and y [n_tok*k][dim] 16-byte aligned, weights [n_tok*k]
 *                   4-byte aligned.
 */
int q8_swiglu(float *mid, const float *gate, const float *up, uint64_t n, float limit, void *stream);
int q8_moe_combine(float *out, const float *y, const float *weights, uint64_t n_tok, uint32_t k,
                   uint64_t dim, void *stream);

/*
 * Optional load-time repack of Q8_0 rows into a kernel-friendly layout (the
 * ROCm MXFP4 work on the pages found 16-byte aligned value slices with a
 * separate scale array fastest: GPU concepts page, §4c).  The repack copies or
 * widens bits exactly; the products over a packed buffer are the q8_matmul
 * products (same tolerance).
 *   Q8_LAYOUT_PLANES: int8 quant plane [rows][in_dim], then the fp16 scale plane
 *     [rows][in_dim/32]; the same 34 bytes per 32 weights.  Its matmul is a
 *     plain mma.sync kernel (reference speed: the library's fast kernels read raw
 *     Q8_0 rows in place, which TMA boxes make free of alignment costs).
 *   Q8_LAYOUT_TC: the tcgen05 GEMM's weight operand: fp16 quants [m_ld][in_dim]
 *     (exact integers), then fp32 scales block-major [in_dim/32][m_ld], m_ld =
 *     rows rounded up to 128, padding rows zero; 2 bytes per weight plus 4 per
 *     block.  Its matmul runs the tcgen05 GEMM on it directly for any n_tok,
 *     skipping the weight expansion q8_matmul performs per call above 2048
 *     tokens (or when in_dim/32 is not a multiple of 8).  in_dim must be a
 *     multiple of 64.
 *   q8_repack_bytes: size of the packed buffer (0 for a bad layout or in_dim).
 *   q8_repack:       Wp (out, device, q8_repack_bytes bytes, 16-byte aligned) <- W.
 *   q8_matmul_packed: as q8_matmul, weights from a q8_repack buffer of `layout`.
 * An unknown layout gives Q8_EINVAL.
 */
#define Q8_LAYOUT_PLANES 0
#define Q8_LAYOUT_TC 1
uint64_t q8_repack_bytes(uint64_t in_dim, uint64_t rows, int layout);
int q8_repack(void *Wp, const void *W, uint64_t in_dim, uint64_t rows, int layout, void *stream);
int q8_matmul_packed(float *out, const void *Wp, int layout, uint64_t in_dim, uint64_t out_dim,
                     const float *x, uint64_t n_tok, void *stream);

/*
 * q8_matmul without any device allocation.  This entry point has no
 * counterpart on the pages; it exists for callers that must not allocate
 * device memory from inside this library: for example an application whose
 * own pool allocator has reserved the device's memory up front (a cudaMalloc
 * here would fail or fragment its pool), or a latency-critical decode loop
 * that cannot afford the device-wide synchronisation and milliseconds that a
 * first-use cudaMalloc/cudaFree can cost.
 *
 * Same arguments, layouts and error codes as q8_matmul, and the same
 * quantised activations (bit for bit), but those live in one fixed array of
 * Q8_NOALLOC_SCRATCH_BYTES compiled into the library; every GPU that loads the
 * library holds that array until the process exits.  The kernels differ from
 * q8_matmul's: the quantiser always writes activation planes into the array;
 * up to 16 tokens on 16-byte-aligned rows (in_dim % 256 == 0) the
 * weight-streaming GEMV reads them; above 16 tokens an mma.sync int8 kernel
 * does (q8_matmul runs its tcgen05 GEMM there, whose fp16 operands would not
 * fit the array), so such calls are several times slower than q8_matmul's;
 * unaligned rows take the same plain kernel as q8_matmul.  The outputs
 * therefore agree with q8_matmul's within the matmul tolerance
 * (|diff| <= 1e-4 * sum_b |d_w d_x isum_b| + 1e-6 against the exact sum),
 * not bit for bit: the kernels add the blocks in different fp32 orders.
 * The call needs align256(n_pad*in_dim) + align256(n_pad*(in_dim/32)*4) bytes
 * of the array, with
 * n_pad = n_tok rounded up to a multiple of 16 (for example n_tok <= 16 with
 * in_dim <= 200000, or n_tok = 512 with in_dim <= 7168); larger calls return
 * Q8_ESCRATCH and enqueue nothing.  It never calls cudaMalloc, cudaFree or any
 * allocating routine.
 *
 * The first call on a device looks up the device address of that array
 * (cudaGetSymbolAddress) with the device current; make that first call
 * before any stream capture.  All calls share the one array and every call
 * rewrites the part it uses before reading it, so nothing needs clearing; but
 * calls whose work overlaps on the GPU (different streams without ordering)
 * race on it and must not be issued.
 */
#define Q8_NOALLOC_SCRATCH_BYTES (4u << 20)
int q8_matmul_noalloc(float *out, const void *W, uint64_t in_dim, uint64_t out_dim,
                      const float *x, uint64_t n_tok, void *stream);

/*
 * Synchronises `stream`, then returns and clears the device error word of
 * the current device: Q8_OK, Q8_ERANGE (an expert id was out of range) or
 * Q8_ETIMEOUT (a bounded wait inside a kernel expired), or Q8_ECUDA when the
 * synchronisation itself failed.
 */
int q8_last_error(void *stream);

/* Name of the last CUDA runtime error behind a Q8_ECUDA return ("cudaSuccess"
 * if none yet); for diagnostics. */
const char *q8_last_cuda_error(void);

/* Scratch bytes currently held on the current device, the staging buffer of
 * q8_matmul_host included (0 if none). */
uint64_t q8_scratch_bytes(void);

/* Frees the scratch and staging buffers of every device (synchronises each first). */
void q8_release(void);

/*
 * Kernel timing hook (for benchmarks).  q8_profile_arm(n) creates n pairs of
 * timing events on the current device (n = 0 destroys them and disarms).
 * While armed, every call that launches a matmul kernel (q8_matmul,
 * q8_matmul_q, q8_moe_matmul, q8_matmul_packed) records the next pair, in
 * round-robin order, on its own stream immediately before and after that
 * kernel -- also inside CUDA graph capture, where the records become graph
 * nodes.  q8_profile_used() is the number of pairs recorded since arming;
 * q8_profile_read(i, &ms) waits for pair i's end event and returns its
 * elapsed time in milliseconds.  Returns Q8_EINVAL for a pair never recorded.
 */
int q8_profile_arm(uint32_t n_pairs);
uint64_t q8_profile_used(void);
int q8_profile_read(uint32_t i, float *ms);

/*
 * Test hook: make the next `count` scratch allocations fail as if the device
 * were out of memory (they then return Q8_ENOMEM); 0 restores normal
 * behaviour.  Exists so that the allocation-failure path can be tested
 * without exhausting a shared GPU.
 */
void q8_debug_fail_next_alloc(int count);

/*
 * Test hook for the bounded waits inside the kernels (the pages give their
 * tensor-parallel poll gates a time budget and fail instead of hanging: GPU
 * concepts page, §4, distributed inference).  The next `count` dense matmul
 * kernels (the weight-streaming GEMV and the tcgen05 GEMM that q8_matmul,
 * q8_matmul_q and q8_matmul_host launch, and the TMA-fed kernel that
 * q8_rmsnorm_quantize runs for rows of at most 4096 values and at least 12
 * rows per SM) run with every wait limited to
 * limit_ns nanoseconds (0: the normal 2 s) and with their producer issuing no
 * copy at all, so the consumers wait on buffers that never fill.  Each such
 * kernel then raises Q8_ETIMEOUT for q8_last_error(), stops waiting, lets any
 * copy still in flight land and returns; its outputs are undefined.  Nothing
 * traps and the context stays usable.  count 0 disarms the hook.
 */
void q8_debug_expire_waits(int count, uint64_t limit_ns);

#ifdef __cplusplus
}
#endif

#endif /* Q8_H */
