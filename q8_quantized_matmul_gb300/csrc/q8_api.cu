// q8_api.cu -- the C ABI (include/q8.h): host-side validation, per-device
// scratch and error word, and dispatch to the kernels.
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/q8.h"
#include "q8_common.cuh"
#include "q8_kernels.h"

// Device error word (one per device context).  Kernels receive its address.
__device__ int g_q8_device_error = 0;

namespace {

constexpr int MAX_DEVICES = 64;
constexpr uint32_t MAX_EXPERTS = 16384;

struct DeviceState {
    bool ready = false;
    int num_sms = 0;
    int *err = nullptr;          // device address of g_q8_device_error
    void *scratch = nullptr;
    size_t scratch_bytes = 0;
    void *stage = nullptr;       // device copies of host activations and results (q8_matmul_host)
    size_t stage_bytes = 0;
};

std::mutex g_mutex;
DeviceState g_dev[MAX_DEVICES];
int g_fail_next_alloc = 0;
int g_expire_next = 0;            // q8_debug_expire_waits: dense kernels still to withhold their copies
uint64_t g_expire_limit_ns = 0;   // ... and their wait limit

// The failure-detection test hook, consumed by one dense GEMV or GEMM launch, or one
// launch of the TMA-fed RMSNorm kernel.
void take_expiry(uint64_t &wait_ns, int &withhold) {
    wait_ns = 0;
    withhold = 0;
    if (g_expire_next > 0) {
        --g_expire_next;
        wait_ns = g_expire_limit_ns;
        withhold = 1;
    }
}

// Kernel timing hook: event pairs recorded around the main matmul kernel.
struct Profile {
    int device = -1;
    uint32_t n = 0;
    uint64_t used = 0;
    cudaEvent_t *ev = nullptr;   // 2*n events
    uint8_t *recorded = nullptr; // per pair
} g_prof;

void profile_free() {
    if (g_prof.ev) {
        for (uint32_t i = 0; i < 2 * g_prof.n; ++i) cudaEventDestroy(g_prof.ev[i]);
        delete[] g_prof.ev;
        delete[] g_prof.recorded;
    }
    g_prof = Profile{};
}

// Launch `launch` between the next pair of timing events when armed.
template <class F> cudaError_t timed_launch(cudaStream_t st, F launch) {
    int dev = -1;
    cudaGetDevice(&dev);
    if (!g_prof.n || dev != g_prof.device) return launch();
    const uint32_t i = (uint32_t)(g_prof.used % g_prof.n);
    // Under stream capture a plain record only orders the capture; the
    // external flag makes it an event-record node of the graph.
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) {
        cudaGetLastError();
        cs = cudaStreamCaptureStatusNone;
    }
    const unsigned flags = cs == cudaStreamCaptureStatusActive ? cudaEventRecordExternal : cudaEventRecordDefault;
    cudaError_t e = cudaEventRecordWithFlags(g_prof.ev[2 * i], st, flags);
    if (e != cudaSuccess) return e;
    e = launch();
    if (e != cudaSuccess) return e;
    e = cudaEventRecordWithFlags(g_prof.ev[2 * i + 1], st, flags);
    g_prof.recorded[i] = 1;
    ++g_prof.used;
    return e;
}

cudaError_t g_last_cuda_error = cudaSuccess;   // for q8_last_cuda_error()

int status_of(cudaError_t e) {
    if (e == cudaSuccess) return Q8_OK;
    g_last_cuda_error = e;
    return Q8_ECUDA;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Current device's state, initialised on first use.
int get_device(DeviceState **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) {
        cudaGetLastError();
        return Q8_ECUDA;
    }
    DeviceState &s = g_dev[dev];
    if (!s.ready) {
        int sms = 0, major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
            cudaGetLastError();
            return Q8_ECUDA;
        }
        if (major * 10 + minor != 103) return Q8_ECUDA;   // built for sm_103a only
        void *err = nullptr;
        if (cudaGetSymbolAddress(&err, g_q8_device_error) != cudaSuccess) {
            cudaGetLastError();
            return Q8_ECUDA;
        }
        s.num_sms = sms;
        s.err = static_cast<int *>(err);
        s.ready = true;
    }
    *out = &s;
    return Q8_OK;
}

// Grow-only device buffer of at least `bytes`.  Growing synchronises the device
// (cudaFree does), so a call that grows it must not overlap work of another
// stream that still uses the old buffer -- scratch users are single-stream.
int reserve_buffer(void **buf, size_t *have, size_t bytes) {
    if (bytes <= *have) return Q8_OK;
    if (g_fail_next_alloc > 0) {
        --g_fail_next_alloc;
        return Q8_ENOMEM;
    }
    size_t want = bytes + bytes / 4;
    want = (want + ((size_t)1 << 20) - 1) & ~(((size_t)1 << 20) - 1);
    if (*buf) {
        cudaFree(*buf);
        *buf = nullptr;
        *have = 0;
    }
    void *p = nullptr;
    if (cudaMalloc(&p, want) != cudaSuccess) {
        cudaGetLastError();
        return Q8_ENOMEM;
    }
    *buf = p;
    *have = want;
    return Q8_OK;
}

int reserve_scratch(DeviceState *s, size_t bytes) { return reserve_buffer(&s->scratch, &s->scratch_bytes, bytes); }

size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

// Sub-allocations of the scratch buffer.
struct Carver {
    uint8_t *base;
    size_t off = 0;
    explicit Carver(void *b) : base(static_cast<uint8_t *>(b)) {}
    template <class T> T *take(size_t bytes) {
        T *p = reinterpret_cast<T *>(base + off);
        off = align256(off + bytes);
        return p;
    }
};

size_t planes_bytes(uint64_t rows, uint64_t in_dim) {
    return align256(rows * in_dim) + align256(rows * (in_dim / q8::QK) * sizeof(float));
}

int check_dims(uint64_t in_dim, uint64_t out_dim, uint64_t n_tok) {
    if (in_dim == 0 || in_dim % q8::QK) return Q8_EINVAL;
    if (in_dim > ((uint64_t)1 << 31) || out_dim > ((uint64_t)1 << 31) - 1 || n_tok > ((uint64_t)1 << 31) - 1)
        return Q8_EINVAL;
    const uint64_t nb = in_dim / q8::QK;
    if (out_dim && nb > (((uint64_t)1 << 62) / q8::QB) / out_dim) return Q8_EINVAL;
    if (n_tok && in_dim > ((uint64_t)1 << 40) / n_tok) return Q8_EINVAL;
    return Q8_OK;
}

// out = W x from activation planes already in scratch (n_pad rows), or, with
// x_fused given, from the fp32 rows quantised inside the GEMV.
// out_remote: the result lives in host memory (see q8_matmul_host).
int run_dense(DeviceState *s, float *out, const void *W, uint64_t in_dim, uint64_t out_dim, const int8_t *qx,
              const float *dx, const float *x_fused, uint64_t n_tok, cudaStream_t st, bool out_remote = false) {
    const uint32_t nb = (uint32_t)(in_dim / q8::QK);
    if (nb % 8 == 0 && n_tok <= 16) {
        q8::GemvParams g{};
        g.W = static_cast<const uint8_t *>(W);
        g.expert_stride = 0;
        g.in_dim = in_dim;
        g.out_dim = (uint32_t)out_dim;
        g.nb = nb;
        g.qx = qx;
        g.dx = dx;
        g.x = x_fused;
        g.out = out;
        g.err = s->err;
        g.n_tok = (uint32_t)n_tok;
        g.n_items = q8::gemv_dense_items(out_dim, s->num_sms);
        // A result in host memory crosses the host link at a fraction of the HBM
        // rate, and an item writes its results only once its last weights are in.
        // With 3 or more tokens (at least 384 KB of results for out 32768) each CTA
        // takes two items when each still keeps 12 of the 14 consumer warps busy (six
        // or more 16-row sub-items, two warps a sub-item): the first item's results
        // then cross the link while the second item's weights stream.
        const uint64_t nsub = (out_dim + 15) / 16;
        if (out_remote && n_tok >= 3 && nsub >= 12 * (uint64_t)g.n_items) g.n_items *= 2;
        q8::gemv_dense_split(out_dim, g.n_items, g.sub_base, g.sub_rem);
        g.plan = nullptr;
        g.row_to_out = nullptr;
        g.n_expert = 1;
        const int grid = (int)(g.n_items < (uint32_t)s->num_sms ? g.n_items : (uint32_t)s->num_sms);
        // Weights before the grid wait: behind the quantiser (planes), and for fused
        // calls of 1-2 tokens, whose 4-8 KB of fp32 rows barely queue behind the
        // early copies (1-token calls 8.17 -> 7.5 us, the mixed decode step 29.7 ->
        // 29.0 us; fused 3-8-token calls measured slower that way, 8.6 -> 9.2-9.9 us).
        g.weights_early = (!x_fused || n_tok <= 2) ? 1 : 0;
        take_expiry(g.wait_ns, g.withhold);
        return status_of(timed_launch(st, [&] { return q8::launch_gemv(g, q8::gemv_mode(n_tok), grid, st); }));
    }
    q8::MmaParams p{};
    p.W = static_cast<const uint8_t *>(W);
    p.expert_stride = 0;
    p.in_dim = in_dim;
    p.out_dim = (uint32_t)out_dim;
    p.nb = nb;
    p.qx = qx;
    p.dx = dx;
    p.out = out;
    p.err = s->err;
    p.n_tok = (uint32_t)n_tok;
    p.plan = nullptr;
    p.row_to_out = nullptr;
    if (p.nb % 8 == 0) {
        const uint64_t items = ((out_dim + 15) / 16) * ((n_tok + 63) / 64);
        const int grid = (int)(items < (uint64_t)s->num_sms ? items : (uint64_t)s->num_sms);
        return status_of(timed_launch(st, [&] { return q8::launch_mma(p, grid, st); }));
    }
    const int hint = (int)((n_tok * out_dim) > (1u << 30) ? (1u << 30) : n_tok * out_dim);
    return status_of(timed_launch(st, [&] { return q8::launch_generic(p, hint, s->num_sms, st); }));
}

// Prefill (n_tok > 16, even number of blocks per row): tcgen05 GEMM on fp16
// operands, activations quantised straight into the fp16 operand; K is split
// when the output tiles do not fill the GPU.  Up to TC_RAW_MAX_TOKENS tokens
// (and in_dim / 32 a multiple of 8) the GEMM reads the raw Q8_0 rows and
// converts them in shared memory; beyond that the weights are first expanded
// to an fp16 plane with block-major scales (measured: the raw-weight GEMM is
// faster than expansion plus GEMM up to 2048 tokens and about even at 4096).
constexpr uint64_t TC_RAW_MAX_TOKENS = 2048;
// a16_pre / dwT_pre: weights already in the GEMM's fp16 operand layout (a
// Q8_LAYOUT_TC buffer; m_ld = out_dim rounded up to 128), used as they are.
int run_tc(DeviceState *s, float *out, const void *W, uint64_t in_dim, uint64_t out_dim, const float *x,
           const void *xq, uint64_t n_tok, cudaStream_t st, const __half *a16_pre = nullptr,
           const float *dwT_pre = nullptr) {
    const uint64_t nb = in_dim / q8::QK;
    const bool packed = a16_pre != nullptr;
    const bool raw = !packed && nb % 8 == 0 && n_tok <= TC_RAW_MAX_TOKENS;   // raw Q8_0 rows, no fp16 plane
    const uint64_t kb_align = raw ? 8 : 2;
    const uint64_t m_ld = (out_dim + 127) & ~(uint64_t)127;
    const uint64_t n_ld = (n_tok + 127) & ~(uint64_t)127;
    const uint64_t tiles = (m_ld / 128) * (n_ld / 128);
    const uint64_t sms = (uint64_t)s->num_sms;
    uint64_t ksplit = 1;
    if (tiles < sms) {
        ksplit = sms / tiles;
        const uint64_t max_split = nb / 16 > 0 ? nb / 16 : 1;   // keep >= 16 blocks per split
        if (ksplit > max_split) ksplit = max_split;
        if (ksplit < 1) ksplit = 1;
        // With long K, more splits than fit one wave can fill the SMs better: 32 tiles
        // in 4 splits leave 24 of 152 SMs idle, 9 splits run 288 units in two full
        // waves of 114 blocks each (in 32768 -> out 1024 at 512 tokens: 114.3 ->
        // 111.5 us).  Only while a split keeps >= 96 blocks (short splits pay the
        // pipeline's fill: 7 splits of 18 blocks took 4096 -> 2048 from 35.6 to 42.9
        // us); 0.004 per split for the partial sums.
        double best = 1.0 / (double)ksplit + 0.004 * (double)ksplit;
        for (uint64_t k = ksplit + 1; k <= 64 && nb / k >= 96; ++k) {
            const uint64_t waves = (tiles * k + sms - 1) / sms;
            const double t = (double)waves / (double)k + 0.004 * (double)k;
            if (t < best - 1e-12) {
                best = t;
                ksplit = k;
            }
        }
    } else {
        // Tiles fill the SMs but may end in a thin last wave (256 tiles: 1.68 waves,
        // 0.84 of the SMs busy on average): split K when that fills the waves better,
        // keeping >= 64 blocks per split and charging 0.01 per extra split for the
        // partial sums' traffic.
        double best = 0.0;
        for (uint64_t k = 1; k <= 8 && nb / k >= 64; ++k) {
            const uint64_t units = tiles * k, waves = (units + sms - 1) / sms;
            const double score = (double)units / (double)(waves * sms) - 0.01 * (double)(k - 1);
            if (score > best + 1e-9) {
                best = score;
                ksplit = k;
            }
        }
    }
    uint64_t kb_per = (nb + ksplit - 1) / ksplit;
    kb_per = (kb_per + kb_align - 1) / kb_align * kb_align;
    ksplit = (nb + kb_per - 1) / kb_per;
    const bool expand = !raw && !packed;
    const size_t need = (expand ? align256(out_dim * in_dim * 2) + align256(nb * m_ld * 4) : 0) +
                        align256(n_ld * in_dim * 2) + align256(nb * n_ld * 4) +
                        (ksplit > 1 ? align256(ksplit * n_tok * out_dim * 4) : 0);
    int rc = reserve_scratch(s, need);
    if (rc) return rc;
    Carver cv(s->scratch);
    const __half *a16 = packed ? a16_pre : nullptr;
    const float *dwT = packed ? dwT_pre : nullptr;
    __half *a16_x = expand ? cv.take<__half>(out_dim * in_dim * 2) : nullptr;
    float *dwT_x = expand ? cv.take<float>(nb * m_ld * 4) : nullptr;
    __half *b16 = cv.take<__half>(n_ld * in_dim * 2);
    float *dxT = cv.take<float>(nb * n_ld * 4);
    float *partial = ksplit > 1 ? cv.take<float>(ksplit * n_tok * out_dim * 4) : nullptr;
    if (expand) {
        if ((rc = status_of(q8::launch_tc_expand(a16_x, dwT_x, static_cast<const uint8_t *>(W), (uint32_t)out_dim,
                                                 (uint32_t)nb, (uint32_t)m_ld, s->num_sms, st))))
            return rc;
        a16 = a16_x;
        dwT = dwT_x;
    }
    cudaError_t e = x ? q8::launch_quantize_f16t(b16, dxT, x, in_dim, n_tok, n_ld, s->num_sms, st)
                      : q8::launch_unpack_f16t(b16, dxT, static_cast<const uint8_t *>(xq), in_dim, n_tok, n_ld,
                                               s->num_sms, st);
    if ((rc = status_of(e))) return rc;
    q8::TcParams p{};
    p.M = (int)out_dim;
    p.N = (int)n_tok;
    p.nb = (int)nb;
    p.ksplit = (int)ksplit;
    p.kb_per = (int)kb_per;
    p.dxT = dxT;
    p.dwT = dwT;
    p.n_ld = n_ld;
    p.m_ld = m_ld;
    p.out = out;
    p.partial = partial;
    p.err = s->err;
    take_expiry(p.wait_ns, p.withhold);
    const uint64_t units = tiles * ksplit;
    const int grid = (int)(units < (uint64_t)s->num_sms ? units : (uint64_t)s->num_sms);
    if (raw)
        return status_of(timed_launch(st, [&] {
            return q8::launch_tc_gemm_raw(p, static_cast<const uint8_t *>(W), 1, 0, b16, n_ld, grid, st);
        }));
    return status_of(timed_launch(st, [&] { return q8::launch_tc_gemm(p, a16, b16, n_ld, grid, st); }));
}

// One routed-expert product, or two that share the routing and the quantised
// activations (the gate and up projections of an expert FFN): W[w] -> out[w].
struct MoeCall {
    const void *W[2] = {nullptr, nullptr};
    float *out[2] = {nullptr, nullptr};
    int n_w = 1;
    uint32_t n_expert = 0;
    uint64_t stride = 0;          // bytes between experts' matrices
    const int32_t *ids = nullptr;
    uint32_t k = 0;
    uint64_t in_dim = 0, out_dim = 0;
    const float *x = nullptr;
    int x_per_pair = 0;
    uint64_t n_tok = 0;
    // Gate/up pair: W[0] gate, W[1] up, and out[0] receives swiglu1(gate, up, limit)
    // from one GEMV pass per class (GEMV path without a tensor-core class only).
    bool pair = false;
    float limit = 0.0f;
};

// Scratch layout of a routed call.
struct MoeLayout {
    uint64_t nb = 0, n_pairs = 0, max_rows = 0, tc_cap = 0, tc_ld = 0;
    size_t plan_bytes = 0, need = 0;
    bool gemv_path = false;
};

MoeLayout moe_layout(const MoeCall &c) {
    MoeLayout L;
    L.nb = c.in_dim / q8::QK;
    L.n_pairs = c.n_tok * c.k;
    L.max_rows = q8::route_max_rows(L.n_pairs, c.n_expert);
    L.plan_bytes = q8::route_plan_bytes(c.n_expert);
    // Tensor-core class: experts of more than MOE_TC_MIN_ROWS rows, read as raw
    // Q8_0 rows by the grouped GEMM; their activation rows go to the fp16 operand.
    if (L.nb % 8 == 0 && L.n_pairs >= q8::MOE_TC_MIN_PAIRS) {
        L.tc_cap = L.n_pairs / (q8::MOE_TC_MIN_ROWS + 1);
        if (L.tc_cap > c.n_expert) L.tc_cap = c.n_expert;
    }
    const uint64_t tc_rows =
        L.max_rows < L.n_pairs + 15 * L.tc_cap + 16 ? L.max_rows : L.n_pairs + 15 * L.tc_cap + 16;
    L.tc_ld = ((tc_rows + 127) & ~(uint64_t)127) + 128;   // a tile may start at the last row
    const size_t tc_bytes = L.tc_cap ? align256(L.tc_ld * c.in_dim * 2) + align256(L.nb * L.tc_ld * 4) : 0;
    L.gemv_path = L.nb % 8 == 0;   // routed GEMV / tensor-core kernels (else the generic kernel)
    L.need = align256(c.n_expert * 4) * 2 + q8::ROUTE_CLASSES * L.plan_bytes + align256(L.max_rows * 4) * 2 +
             (L.gemv_path ? align256(L.n_pairs * 4) : 0) + planes_bytes(L.max_rows, c.in_dim) + tc_bytes;
    return L;
}

// Routing, one quantisation of the activations, then the kernels of each weight
// set; scratch at `base` holds L.need bytes.  Rows of pairs with an id out of
// range are zeroed in out[0] only.
int moe_run(DeviceState *s, const MoeCall &c, const MoeLayout &L, void *base, cudaStream_t st) {
    Carver cv(base);
    int32_t *counts = cv.take<int32_t>(c.n_expert * 4);
    int32_t *row0_of = cv.take<int32_t>(c.n_expert * 4);
    uint8_t *plans = cv.take<uint8_t>(q8::ROUTE_CLASSES * L.plan_bytes);
    int32_t *row_to_out = cv.take<int32_t>(L.max_rows * 4);
    int32_t *src_row = cv.take<int32_t>(L.max_rows * 4);
    int32_t *dst_row = L.gemv_path ? cv.take<int32_t>(L.n_pairs * 4) : nullptr;
    int8_t *qx = cv.take<int8_t>(L.max_rows * c.in_dim);
    float *dx = cv.take<float>(L.max_rows * L.nb * sizeof(float));
    __half *b16 = L.tc_cap ? cv.take<__half>(L.tc_ld * c.in_dim * 2) : nullptr;
    float *dxT = L.tc_cap ? cv.take<float>(L.nb * L.tc_ld * 4) : nullptr;
    // GEMV items of up to 448 rows: 28 sixteen-row sub-items, two for each of the 14
    // consumer warps.  (128-row items left 6 of the warps idle; at 64 tokens, top-6,
    // the calls took 395 / 430 us with 128-row items, 352 / 374 with 224, 336 / 345
    // with 448.)  A gate/up pair streams two matrices per item: 224 rows of each.
    if (c.pair && (!L.gemv_path || L.tc_cap)) return Q8_EINVAL;
    const uint32_t rows_cap = c.pair ? 224 : 448;
    uint32_t rows_gemv = (uint32_t)((c.out_dim + 15) & ~(uint64_t)15);
    if (rows_gemv > rows_cap) rows_gemv = rows_cap;
    cudaError_t e = q8::launch_route(c.ids, c.n_tok, c.k, c.n_expert, c.x_per_pair, (uint32_t)c.out_dim, rows_gemv,
                                     (uint32_t)L.tc_cap, counts, row0_of, plans, row_to_out, src_row, dst_row,
                                     L.max_rows, c.out[0], s->err, s->num_sms, st);
    if (e != cudaSuccess) return status_of(e);
    auto plan_of = [&](int cls) { return reinterpret_cast<const q8::PlanHeader *>(plans + cls * L.plan_bytes); };
    // The GEMV and tensor-core kernels read only the real rows: the quantiser walks
    // the pairs and leaves the padding rows unwritten.  The generic kernel gets
    // zero padding rows.
    if (L.gemv_path)
        e = q8::launch_quantize_pairs(qx, dx, b16, dxT, L.tc_ld, L.tc_cap ? plan_of(2) : nullptr, c.x, c.in_dim,
                                      L.n_pairs, c.k, c.x_per_pair, dst_row, s->num_sms, st);
    else
        e = q8::launch_quantize_planes(qx, dx, c.x, c.in_dim, L.max_rows, src_row, 0, s->num_sms, st);
    if (e != cudaSuccess) return status_of(e);
    for (int w = 0; w < (c.pair ? 1 : c.n_w); ++w) {
        const uint8_t *W = static_cast<const uint8_t *>(c.W[w]);
        float *out = c.out[w];
        q8::MmaParams p{};
        p.W = W;
        p.expert_stride = c.stride;
        p.in_dim = c.in_dim;
        p.out_dim = (uint32_t)c.out_dim;
        p.nb = (uint32_t)L.nb;
        p.qx = qx;
        p.dx = dx;
        p.out = out;
        p.err = s->err;
        p.n_tok = 0;
        p.row_to_out = row_to_out;
        if (!L.gemv_path) {   // no tensor-core class here (tc_cap == 0)
            const int hint = (int)(L.max_rows * c.out_dim > (1u << 30) ? (1u << 30) : L.max_rows * c.out_dim);
            e = timed_launch(st, [&] {
                for (int cls = 0; cls < q8::ROUTE_GEMV_CLASSES; ++cls) {
                    p.plan = plan_of(cls);
                    cudaError_t e2 = q8::launch_generic(p, hint, s->num_sms, st);
                    if (e2 != cudaSuccess) return e2;
                }
                return cudaSuccess;
            });
            if (e != cudaSuccess) return status_of(e);
            continue;
        }
        q8::GemvParams g{};
        g.W = W;
        g.expert_stride = c.stride;
        g.in_dim = c.in_dim;
        g.out_dim = (uint32_t)c.out_dim;
        g.nb = (uint32_t)L.nb;
        g.qx = qx;
        g.dx = dx;
        g.out = out;
        g.err = s->err;
        g.n_tok = 0;
        g.rows_per_item = rows_gemv;
        g.weights_early = 1;   // behind the quantiser, the grouped GEMM or another routed GEMV
        g.row_to_out = row_to_out;
        g.n_expert = c.n_expert;
        if (c.pair) {
            g.W2 = static_cast<const uint8_t *>(c.W[1]);
            g.limit = c.limit;
        }
        q8::TcParams tp{};
        tp.M = (int)c.out_dim;
        tp.N = 0;
        tp.nb = (int)L.nb;
        tp.ksplit = 1;
        tp.kb_per = (int)L.nb;
        tp.dxT = dxT;
        tp.dwT = nullptr;
        tp.n_ld = L.tc_ld;
        tp.m_ld = 0;
        tp.out = out;
        tp.partial = nullptr;
        tp.err = s->err;
        tp.plan = plan_of(2);
        tp.row_to_out = row_to_out;
        e = timed_launch(st, [&] {
            if (L.tc_cap) {
                cudaError_t e2 = q8::launch_tc_gemm_raw(tp, W, c.n_expert, c.stride, b16, L.tc_ld, s->num_sms, st);
                if (e2 != cudaSuccess) return e2;
            }
            g.plan = plan_of(0);
            cudaError_t e2 = q8::launch_gemv(g, 1, s->num_sms, st);
            if (e2 != cudaSuccess) return e2;
            g.plan = plan_of(1);
            return q8::launch_gemv(g, 2, s->num_sms, st);
        });
        if (e != cudaSuccess) return status_of(e);
    }
    return Q8_OK;
}

// Host checks of a routed product's arguments (dimensions, expert count, stride).
int check_moe(uint32_t n_expert, uint64_t stride, uint32_t k, uint64_t in_dim, uint64_t out_dim, uint64_t n_tok) {
    int rc = check_dims(in_dim, out_dim, n_tok);
    if (rc) return rc;
    if (n_expert == 0 || n_expert > MAX_EXPERTS || k == 0 || k > n_expert) return Q8_EINVAL;
    if (stride < out_dim * (in_dim / q8::QK) * q8::QB) return Q8_EINVAL;
    if (n_tok * k > ((uint64_t)1 << 31) - 1) return Q8_EINVAL;
    return Q8_OK;
}

}  // namespace

namespace q8 {
// Device address of the current device's error word (nullptr if the device is unusable).
int *device_error_word() {
    std::lock_guard<std::mutex> lk(g_mutex);
    DeviceState *s;
    return get_device(&s) ? nullptr : s->err;
}

// Status of a CUDA runtime result for entry points defined in other files: a
// failure is recorded for q8_last_cuda_error() and becomes Q8_ECUDA.
int record_cuda_status(cudaError_t e) {
    std::lock_guard<std::mutex> lk(g_mutex);
    return status_of(e);
}
}  // namespace q8

extern "C" {

int q8_version(void) { return 10100; }

const char *q8_strerror(int status) {
    switch (status) {
        case Q8_OK: return "ok";
        case Q8_EINVAL: return "invalid argument";
        case Q8_EALIGN: return "pointer not 16-byte aligned";
        case Q8_ERANGE: return "expert id out of range";
        case Q8_ENOMEM: return "scratch allocation failed";
        case Q8_ECUDA: return "CUDA runtime error";
        case Q8_ETIMEOUT: return "bounded wait expired inside a kernel";
        case Q8_ESCRATCH: return "call exceeds the fixed scratch of q8_matmul_noalloc";
        default: return "unknown status";
    }
}

int q8_quantize_act(void *xq, const float *x, uint64_t in_dim, uint64_t n_tok, void *stream) {
    int rc = check_dims(in_dim, 1, n_tok);
    if (rc) return rc;
    if (n_tok == 0) return Q8_OK;
    if (!xq || !x) return Q8_EINVAL;
    if (!aligned16(xq) || !aligned16(x)) return Q8_EALIGN;
    std::lock_guard<std::mutex> lk(g_mutex);
    DeviceState *s;
    if ((rc = get_device(&s))) return rc;
    return status_of(q8::launch_quantize_blocks(static_cast<uint8_t *>(xq), x, n_tok * (in_dim / q8::QK), s->num_sms,
                                                static_cast<cudaStream_t>(stream)));
}

// Device address of a page-locked host buffer (cudaHostAlloc, cudaMallocHost or
// cudaHostRegister with mapping), 16-byte aligned, that the current device can
// address; nullptr for pageable memory or anything else.
static void *mapped_host_pointer(const void *p) {
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    if (a.type != cudaMemoryTypeHost || !a.devicePointer || !aligned16(a.devicePointer)) return nullptr;
    return a.devicePointer;
}

// The dense product with arguments already validated, under g_mutex.
// host_io: x and out are host memory mapped into the device's address space.
static int dispatch_matmul(DeviceState *s, float *out, const void *W, uint64_t in_dim, uint64_t out_dim,
                           const float *x, const void *xq, uint64_t n_tok, cudaStream_t st, bool host_io = false) {
    int rc;
    const uint64_t nb = in_dim / q8::QK;
    if (n_tok > 16 && nb % 2 == 0) return run_tc(s, out, W, in_dim, out_dim, x, xq, n_tok, st);
    // small activations: one kernel, the GEMV quantises them itself.  For host
    // activations only up to 2 tokens: every CTA reads all of x over the host link
    // (measured per call at out 32768: 1 token 11.5 us fused against 14.4 us
    // through the quantiser; 4 tokens, 152 x 16 KB, 21 against 16 us), where the
    // quantiser reads each value once.
    if (x && (!host_io || n_tok <= 2) && nb % 8 == 0 && q8::gemv_fuses_quantiser(n_tok, nb))
        return run_dense(s, out, W, in_dim, out_dim, nullptr, nullptr, x, n_tok, st);
    const uint64_t n_pad = (n_tok + 15) & ~(uint64_t)15;
    if ((rc = reserve_scratch(s, planes_bytes(n_pad, in_dim)))) return rc;
    Carver cv(s->scratch);
    int8_t *qx = cv.take<int8_t>(n_pad * in_dim);
    float *dx = cv.take<float>(n_pad * nb * sizeof(float));
    cudaError_t e = x ? q8::launch_quantize_planes(qx, dx, x, in_dim, n_pad, nullptr, n_tok, s->num_sms, st, host_io)
                      : q8::launch_unpack_blocks(qx, dx, static_cast<const uint8_t *>(xq), in_dim, n_pad, n_tok,
                                                 s->num_sms, st);
    if (e != cudaSuccess) return status_of(e);
    return run_dense(s, out, W, in_dim, out_dim, qx, dx, nullptr, n_tok, st, host_io);
}

int q8_rmsnorm_quantize(void *xq, float *y, const float *x, const float *gamma, uint64_t dim, uint64_t n_tok,
                        float eps, void *stream) {
    int rc = check_dims(dim, 1, n_tok);
    if (rc) return rc;
    if (!(eps > 0.0f) || eps == __builtin_inff()) return Q8_EINVAL;   // NaN, zero, negative or infinite
    if (n_tok == 0) return Q8_OK;
    if (!xq || !x) return Q8_EINVAL;
    if (!aligned16(xq) || !aligned16(x) || (y && !aligned16(y)) || (gamma && !aligned16(gamma))) return Q8_EALIGN;
    std::lock_guard<std::mutex> lk(g_mutex);
    DeviceState *s;
    if ((rc = get_device(&s))) return rc;
    uint64_t wait_ns = 0;
    int withhold = 0;
    if (q8::rmsnorm_uses_tma(dim, n_tok, s->num_sms)) take_expiry(wait_ns, withhold);
    return status_of(q8::launch_rmsnorm_quantize(static_cast<uint8_t *>(xq), y, x, gamma, dim, n_tok, eps, s->err,
                                                 wait_ns, withhold, s->num_sms, static_cast<cudaStream_t>(stream)));
}

static int matmul_common(float *out, const void *W, uint64_t in_dim, uint64_t out_dim, const float *x,
                         const void *xq, uint64_t n_tok, void *stream) {
    int rc = check_dims(in_dim, out_dim, n_tok);
    if (rc) return rc;
    if (n_tok == 0 || out_dim == 0) return Q8_OK;
    if (!out || !W || (!x && !xq)) return Q8_EINVAL;
    if (!aligned16(out) || !aligned16(W) || (x && !aligned16(x)) || (xq && !aligned16(xq))) return Q8_EALIGN;
    std::lock_guard<std::mutex> lk(g_mutex);
    DeviceState *s;
    if ((rc = get_device(&s))) return rc;
    return dispatch_matmul(s, out, W, in_dim, out_dim, x, xq, n_tok, static_cast<cudaStream_t>(stream));
}

int q8_matmul(float *out, const void *W, uint64_t in_dim, uint64_t out_dim, const float *x, uint64_t n_tok,
              void *stream) {
    if (!x && n_tok) return Q8_EINVAL;
    return matmul_common(out, W, in_dim, out_dim, x, nullptr, n_tok, stream);
}

int q8_matmul_host(float *out_host, const void *W, uint64_t in_dim, uint64_t out_dim, const float *x_host,
                   uint64_t n_tok, void *stream) {
    int rc = check_dims(in_dim, out_dim, n_tok);
    if (rc) return rc;
    if (n_tok == 0 || out_dim == 0) return Q8_OK;
    if (!out_host || !W || !x_host) return Q8_EINVAL;
    if (!aligned16(W)) return Q8_EALIGN;
    if (out_dim > (((uint64_t)1 << 40) / n_tok)) return Q8_EINVAL;
    std::lock_guard<std::mutex> lk(g_mutex);
    DeviceState *s;
    if ((rc = get_device(&s))) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // Page-locked host buffers are mapped into the device's address space and the
    // GPU reaches them over its host link: the kernels then read x and write the
    // result there directly, with no staging copies.
    const float *xd_host = static_cast<const float *>(mapped_host_pointer(x_host));
    float *od_host = static_cast<float *>(mapped_host_pointer(out_host));
    if (xd_host && od_host) return dispatch_matmul(s, od_host, W, in_dim, out_dim, xd_host, nullptr, n_tok, st, true);
    const size_t x_bytes = n_tok * in_dim * sizeof(float), out_bytes = n_tok * out_dim * sizeof(float);
    if ((rc = reserve_buffer(&s->stage, &s->stage_bytes, align256(x_bytes) + align256(out_bytes)))) return rc;
    Carver cv(s->stage);
    float *xd = cv.take<float>(x_bytes);
    float *od = cv.take<float>(out_bytes);
    if ((rc = status_of(cudaMemcpyAsync(xd, x_host, x_bytes, cudaMemcpyHostToDevice, st)))) return rc;
    if ((rc = dispatch_matmul(s, od, W, in_dim, out_dim, xd, nullptr, n_tok, st))) return rc;
    return status_of(cudaMemcpyAsync(out_host, od, out_bytes, cudaMemcpyDeviceToHost, st));
}

int q8_matmul_q(float *out, const void *W, uint64_t in_dim, uint64_t out_dim, const void *xq, uint64_t n_tok,
                void *stream) {
    if (!xq && n_tok) return Q8_EINVAL;
    return matmul_common(out, W, in_dim, out_dim, nullptr, xq, n_tok, stream);
}

int q8_moe_matmul(float *out, const void *W_experts, uint32_t n_expert, uint64_t expert_stride_bytes,
                  const int32_t *expert_ids, uint32_t k, uint64_t in_dim, uint64_t out_dim, const float *x,
                  int x_per_pair, uint64_t n_tok, void *stream) {
    int rc = check_moe(n_expert, expert_stride_bytes, k, in_dim, out_dim, n_tok);
    if (rc) return rc;
    if (n_tok == 0 || out_dim == 0) return Q8_OK;
    if (!out || !W_experts || !expert_ids || !x) return Q8_EINVAL;
    if (!aligned16(out) || !aligned16(W_experts) || !aligned16(x) || (expert_stride_bytes & 15u) ||
        (reinterpret_cast<uintptr_t>(expert_ids) & 3u))
        return Q8_EALIGN;
    std::lock_guard<std::mutex> lk(g_mutex);
    DeviceState *s;
    if ((rc = get_device(&s))) return rc;
    MoeCall c;
    c.W[0] = W_experts;
    c.out[0] = out;
    c.n_expert = n_expert;
    c.stride = expert_stride_bytes;
    c.ids = expert_ids;
    c.k = k;
    c.in_dim = in_dim;
    c.out_dim = out_dim;
    c.x = x;
    c.x_per_pair = x_per_pair;
    c.n_tok = n_tok;
    const MoeLayout L = moe_layout(c);
    if ((rc = reserve_scratch(s, L.need))) return rc;
    return moe_run(s, c, L, s->scratch, static_cast<cudaStream_t>(stream));
}

int q8_swiglu(float *mid, const float *gate, const float *up, uint64_t n, float limit, void *stream) {
    if (!(limit >= 0.0f)) return Q8_EINVAL;   // negative or NaN
    if (n == 0) return Q8_OK;
    if (n > ((uint64_t)1 << 60)) return Q8_EINVAL;
    if (!mid || !gate || !up) return Q8_EINVAL;
    if (!aligned16(mid) || !aligned16(gate) || !aligned16(up)) return Q8_EALIGN;
    int rc;
    int sms;
    {
        std::lock_guard<std::mutex> lk(g_mutex);
        DeviceState *s;
        if ((rc = get_device(&s))) return rc;
        sms = s->num_sms;
    }
    return status_of(q8::launch_swiglu(mid, gate, up, n, limit, nullptr, 0, 0, sms, static_cast<cudaStream_t>(stream)));
}

int q8_moe_combine(float *out, const float *y, const float *weights, uint64_t n_tok, uint32_t k, uint64_t dim,
                   void *stream) {
    if (k == 0) return Q8_EINVAL;
    if (n_tok == 0 || dim == 0) return Q8_OK;
    if (n_tok > ((uint64_t)1 << 40) / k || dim > ((uint64_t)1 << 60) / (n_tok * k)) return Q8_EINVAL;
    if (!out || !y || !weights) return Q8_EINVAL;
    if (!aligned16(out) || !aligned16(y) || (reinterpret_cast<uintptr_t>(weights) & 3u)) return Q8_EALIGN;
    int rc;
    int sms;
    {
        std::lock_guard<std::mutex> lk(g_mutex);
        DeviceState *s;
        if ((rc = get_device(&s))) return rc;
        sms = s->num_sms;
    }
    return status_of(q8::launch_combine(out, y, weights, n_tok, k, dim, sms, static_cast<cudaStream_t>(stream)));
}

// The routed FFN when every expert group of both projections is on the GEMV (in_dim
// and mid_dim multiples of 256, fewer than 1024 pairs): one routing serves both.
// Plane rows depend only on the pairs, and a GEMV counts its items from its own
// width (GemvParams::plan_rb), so: routing -> gathering quantiser of x -> gate/up
// pair GEMVs writing mid as Q8_0 planes at the pairs' plane rows -> down GEMVs on
// those planes -> weighted sum.  The routing zeroes y's row of a pair with a bad id.
static int ffn_gemv_run(DeviceState *s, const MoeCall &gu, const MoeLayout &L, const void *W_down,
                        uint64_t down_stride, uint64_t out_dim, float limit, const float *expert_weights, float *out,
                        cudaStream_t st) {
    const uint64_t mid_dim = gu.out_dim;
    const uint64_t nbm = mid_dim / q8::QK;
    if ((L.nb % 8) || (nbm % 8) || L.tc_cap) return Q8_EINVAL;
    int rc;
    const size_t region = align256(L.need);
    if ((rc = reserve_scratch(s, region + planes_bytes(L.max_rows, mid_dim) + align256(L.n_pairs * out_dim * 4))))
        return rc;
    Carver cv(s->scratch);
    int32_t *counts = cv.take<int32_t>(gu.n_expert * 4);
    int32_t *row0_of = cv.take<int32_t>(gu.n_expert * 4);
    uint8_t *plans = cv.take<uint8_t>(q8::ROUTE_CLASSES * L.plan_bytes);
    int32_t *row_to_out = cv.take<int32_t>(L.max_rows * 4);
    int32_t *src_row = cv.take<int32_t>(L.max_rows * 4);
    int32_t *dst_row = cv.take<int32_t>(L.n_pairs * 4);
    int8_t *qx = cv.take<int8_t>(L.max_rows * gu.in_dim);
    float *dx = cv.take<float>(L.max_rows * L.nb * sizeof(float));
    Carver cv2(static_cast<uint8_t *>(s->scratch) + region);
    int8_t *qmid = cv2.take<int8_t>(L.max_rows * mid_dim);
    float *dmid = cv2.take<float>(L.max_rows * nbm * sizeof(float));
    float *y = cv2.take<float>(L.n_pairs * out_dim * 4);
    // pair items of 224 rows of each matrix (14 + 14 sub-items); the routing counts
    // its items for the down projection's width
    const uint32_t rows_pair = mid_dim < 224 ? (uint32_t)mid_dim : 224u;
    uint32_t rows_down = (uint32_t)((out_dim + 15) & ~(uint64_t)15);
    if (rows_down > 448) rows_down = 448;
    const uint32_t rows_route = 224;
    const uint32_t plan_rb = (uint32_t)((out_dim + rows_route - 1) / rows_route);
    cudaError_t e = q8::launch_route(gu.ids, gu.n_tok, gu.k, gu.n_expert, 0, (uint32_t)out_dim, rows_route, 0, counts,
                                     row0_of, plans, row_to_out, src_row, dst_row, L.max_rows, y, s->err, s->num_sms,
                                     st);
    if (e != cudaSuccess) return status_of(e);
    e = q8::launch_quantize_pairs(qx, dx, nullptr, nullptr, 0, nullptr, gu.x, gu.in_dim, L.n_pairs, gu.k, 0, dst_row,
                                  s->num_sms, st);
    if (e != cudaSuccess) return status_of(e);
    auto plan_of = [&](int cls) { return reinterpret_cast<const q8::PlanHeader *>(plans + cls * L.plan_bytes); };
    q8::GemvParams g{};
    g.W = static_cast<const uint8_t *>(gu.W[0]);
    g.W2 = static_cast<const uint8_t *>(gu.W[1]);
    g.expert_stride = gu.stride;
    g.in_dim = gu.in_dim;
    g.out_dim = (uint32_t)mid_dim;
    g.nb = (uint32_t)L.nb;
    g.qx = qx;
    g.dx = dx;
    g.err = s->err;
    g.rows_per_item = rows_pair;
    g.plan_rb = plan_rb;
    g.weights_early = 1;   // behind this library's quantiser
    g.row_to_out = row_to_out;
    g.n_expert = gu.n_expert;
    g.limit = limit;
    g.q_out = qmid;
    g.d_out = dmid;
    auto classes = [&](q8::GemvParams &gp) {
        return timed_launch(st, [&] {
            gp.plan = plan_of(0);
            cudaError_t e2 = q8::launch_gemv(gp, 1, s->num_sms, st);
            if (e2 != cudaSuccess) return e2;
            gp.plan = plan_of(1);
            return q8::launch_gemv(gp, 2, s->num_sms, st);
        });
    };
    if ((rc = status_of(classes(g)))) return rc;
    q8::GemvParams d{};
    d.W = static_cast<const uint8_t *>(W_down);
    d.expert_stride = down_stride;
    d.in_dim = mid_dim;
    d.out_dim = (uint32_t)out_dim;
    d.nb = (uint32_t)nbm;
    d.qx = qmid;
    d.dx = dmid;
    d.out = y;
    d.err = s->err;
    d.rows_per_item = rows_down;
    d.plan_rb = plan_rb;
    d.weights_early = 1;   // behind the pair GEMV, which writes no weights
    d.row_to_out = row_to_out;
    d.n_expert = gu.n_expert;
    if ((rc = status_of(classes(d)))) return rc;
    return status_of(q8::launch_combine(out, y, expert_weights, gu.n_tok, gu.k, out_dim, s->num_sms, st));
}

int q8_moe_ffn(float *out, const void *W_gate, const void *W_up, const void *W_down, uint32_t n_expert,
               uint64_t gate_up_stride_bytes, uint64_t down_stride_bytes, const int32_t *expert_ids,
               const float *expert_weights, uint32_t k, uint64_t in_dim, uint64_t mid_dim, uint64_t out_dim,
               float limit, const float *x, uint64_t n_tok, void *stream) {
    int rc = check_moe(n_expert, gate_up_stride_bytes, k, in_dim, mid_dim, n_tok);
    if (rc) return rc;
    if ((rc = check_moe(n_expert, down_stride_bytes, k, mid_dim, out_dim, n_tok))) return rc;
    if (mid_dim == 0 || !(limit >= 0.0f)) return Q8_EINVAL;
    if (n_tok == 0 || out_dim == 0) return Q8_OK;
    if (!out || !W_gate || !W_up || !W_down || !expert_ids || !expert_weights || !x) return Q8_EINVAL;
    if (!aligned16(out) || !aligned16(W_gate) || !aligned16(W_up) || !aligned16(W_down) || !aligned16(x) ||
        (gate_up_stride_bytes & 15u) || (down_stride_bytes & 15u) ||
        (reinterpret_cast<uintptr_t>(expert_ids) & 3u) || (reinterpret_cast<uintptr_t>(expert_weights) & 3u))
        return Q8_EALIGN;
    std::lock_guard<std::mutex> lk(g_mutex);
    DeviceState *s;
    if ((rc = get_device(&s))) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const uint64_t n_pairs = n_tok * k;
    MoeCall gu;   // gate and up: in_dim -> mid_dim on the token rows, one routing
    gu.W[0] = W_gate;
    gu.W[1] = W_up;
    gu.n_w = 2;
    gu.n_expert = n_expert;
    gu.stride = gate_up_stride_bytes;
    gu.ids = expert_ids;
    gu.k = k;
    gu.in_dim = in_dim;
    gu.out_dim = mid_dim;
    gu.x = x;
    gu.x_per_pair = 0;
    gu.n_tok = n_tok;
    MoeCall dn = gu;   // down: mid_dim -> out_dim on the pair rows of mid
    dn.W[0] = W_down;
    dn.W[1] = nullptr;
    dn.out[1] = nullptr;
    dn.n_w = 1;
    dn.stride = down_stride_bytes;
    dn.in_dim = mid_dim;
    dn.out_dim = out_dim;
    dn.x_per_pair = 1;
    const MoeLayout Lgu = moe_layout(gu), Ldn = moe_layout(dn);
    if (Lgu.gemv_path && Ldn.gemv_path && !Lgu.tc_cap && !Ldn.tc_cap)
        return ffn_gemv_run(s, gu, Lgu, W_down, down_stride_bytes, out_dim, limit, expert_weights, out, st);
    // scratch: the routed calls' region (reused by both), then gate, up, mid and y
    const size_t region = align256(Lgu.need > Ldn.need ? Lgu.need : Ldn.need);
    const size_t mid_bytes = align256(n_pairs * mid_dim * 4);
    if ((rc = reserve_scratch(s, region + 3 * mid_bytes + align256(n_pairs * out_dim * 4)))) return rc;
    Carver cv(static_cast<uint8_t *>(s->scratch) + region);
    float *gate = cv.take<float>(n_pairs * mid_dim * 4);
    float *up = cv.take<float>(n_pairs * mid_dim * 4);
    float *mid = cv.take<float>(n_pairs * mid_dim * 4);
    float *y = cv.take<float>(n_pairs * out_dim * 4);
    if (Lgu.gemv_path && !Lgu.tc_cap) {
        // Every gate/up group on the GEMV, the down projection not (mid_dim not a
        // multiple of 256): gate and up rows stream through one kernel per class
        // against one staging of the activations, and its epilogue writes
        // mid = swiglu1(gate, up) as fp32 rows.  The routing zeroes the mid row of
        // a pair with a bad id.
        gu.pair = true;
        gu.limit = limit;
        gu.out[0] = mid;
        if ((rc = moe_run(s, gu, Lgu, s->scratch, st))) return rc;
    } else {
        gu.out[0] = gate;
        gu.out[1] = up;
        if ((rc = moe_run(s, gu, Lgu, s->scratch, st))) return rc;
        // a pair with a bad id: its gate row is zero, its up row unwritten; mid is zeroed
        if ((rc = status_of(q8::launch_swiglu(mid, gate, up, n_pairs * mid_dim, limit, expert_ids, n_expert, mid_dim,
                                              s->num_sms, st))))
            return rc;
    }
    dn.x = mid;
    dn.out[0] = y;
    if ((rc = moe_run(s, dn, Ldn, s->scratch, st))) return rc;
    return status_of(q8::launch_combine(out, y, expert_weights, n_tok, k, out_dim, s->num_sms, st));
}

// ---- second weight format: K-quant blocks against Q8_K activations

static uint64_t kq_block_bytes(int fmt) {
    return fmt == Q8_KQ_Q2_K ? 84u : (fmt == Q8_KQ_Q4_K ? 144u : 0u);
}

uint64_t q8_kq_row_bytes(uint64_t in_dim, int fmt) {
    const uint64_t bb = kq_block_bytes(fmt);
    if (!bb || in_dim == 0 || in_dim % 256 || in_dim > ((uint64_t)1 << 40)) return 0;
    return in_dim / 256 * bb;
}

// Dimensions of a K-quant product with n_rows activation rows.
static int check_kq(int fmt, uint64_t in_dim, uint64_t out_dim, uint64_t n_rows) {
    if (!kq_block_bytes(fmt) || in_dim == 0 || in_dim % 256 || in_dim > ((uint64_t)1 << 40)) return Q8_EINVAL;
    if (out_dim > ((uint64_t)1 << 31) || (out_dim && in_dim / 256 > (((uint64_t)1 << 62) / 144) / out_dim))
        return Q8_EINVAL;
    if (n_rows && in_dim > ((uint64_t)1 << 40) / n_rows) return Q8_EINVAL;
    return Q8_OK;
}

static size_t q8k_planes_bytes(uint64_t rows, uint64_t in_dim) {
    return align256(rows * in_dim) + align256(rows * (in_dim / 256) * 4) + align256(rows * (in_dim / 16) * 2);
}

struct Q8kPlanes {
    int8_t *qx;
    float *dx;
    int16_t *xs;
};

static Q8kPlanes take_q8k_planes(Carver &cv, uint64_t rows, uint64_t in_dim) {
    Q8kPlanes q;
    q.qx = cv.take<int8_t>(rows * in_dim);
    q.dx = cv.take<float>(rows * (in_dim / 256) * 4);
    q.xs = cv.take<int16_t>(rows * (in_dim / 16) * 2);
    return q;
}

// Rows per GEMV work item: a multiple of the CTA's 8 warps, 8..64, about four
// items per CTA slot (4 CTAs per SM) when the rows allow.
static uint32_t kq_rows_per_item(uint64_t out_dim, uint64_t groups, int num_sms) {
    uint64_t want = (out_dim * groups + (uint64_t)num_sms * 16 - 1) / ((uint64_t)num_sms * 16);
    want = (want + 7) & ~(uint64_t)7;
    if (want < 8) want = 8;
    if (want > 64) want = 64;
    return (uint32_t)want;
}

int q8_quantize_q8k(void *xq, const float *x, uint64_t in_dim, uint64_t n_tok, void *stream) {
    int rc = check_kq(Q8_KQ_Q4_K, in_dim, 1, n_tok);
    if (rc) return rc;
    if (n_tok == 0) return Q8_OK;
    if (!xq || !x) return Q8_EINVAL;
    if (!aligned16(x) || (reinterpret_cast<uintptr_t>(xq) & 3u)) return Q8_EALIGN;
    std::lock_guard<std::mutex> lk(g_mutex);
    DeviceState *s;
    if ((rc = get_device(&s))) return rc;
    return status_of(q8::launch_quantize_q8k(nullptr, nullptr, nullptr, static_cast<uint8_t *>(xq), x, in_dim, n_tok,
                                             s->num_sms, static_cast<cudaStream_t>(stream)));
}

int q8_kq_matmul(float *out, const void *W, int fmt, uint64_t in_dim, uint64_t out_dim, const float *x,
                 uint64_t n_tok, void *stream) {
    int rc = check_kq(fmt, in_dim, out_dim, n_tok);
    if (rc) return rc;
    if (n_tok == 0 || out_dim == 0) return Q8_OK;
    if (!out || !W || !x) return Q8_EINVAL;
    if (!aligned16(out) || !aligned16(x) ||
        (reinterpret_cast<uintptr_t>(W) & (fmt == Q8_KQ_Q4_K ? 15u : 3u)))
        return Q8_EALIGN;
    if (n_tok > ((uint64_t)1 << 31) - 1) return Q8_EINVAL;
    std::lock_guard<std::mutex> lk(g_mutex);
    DeviceState *s;
    if ((rc = get_device(&s))) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if ((rc = reserve_scratch(s, q8k_planes_bytes(n_tok, in_dim)))) return rc;
    Carver cv(s->scratch);
    const Q8kPlanes q = take_q8k_planes(cv, n_tok, in_dim);
    cudaError_t e = q8::launch_quantize_q8k(q.qx, q.dx, q.xs, nullptr, x, in_dim, n_tok, s->num_sms, st);
    if (e != cudaSuccess) return status_of(e);
    const int tokg = n_tok <= 8 ? 8 : 16;
    const uint32_t stream_rows = aligned16(W) ? q8::kq_stream_rows(q8_kq_row_bytes(in_dim, fmt), in_dim, tokg) : 0;
    q8::KqParams p{};
    p.W = static_cast<const uint8_t *>(W);
    p.in_dim = in_dim;
    p.out_dim = (uint32_t)out_dim;
    p.nsb = (uint32_t)(in_dim / 256);
    p.fmt = fmt;
    p.qx = q.qx;
    p.dx = q.dx;
    p.xs = q.xs;
    p.out = out;
    p.err = s->err;
    p.n_tok = (uint32_t)n_tok;
    if (stream_rows) {   // weights staged through shared memory by bulk copies
        // a dense call has few items: fewer rows an item (in steps of the 14 the
        // consumers share) while that keeps fewer than two items per SM
        uint32_t rows = stream_rows;
        const uint64_t groups = (n_tok + tokg - 1) / tokg;
        while (rows > 14 && ((out_dim + rows - 1) / rows) * groups < 2 * (uint64_t)s->num_sms) rows -= 14;
        p.rows_per_item = rows;
        return status_of(timed_launch(st, [&] { return q8::launch_kq_stream(p, tokg, s->num_sms, st); }));
    }
    p.rows_per_item = kq_rows_per_item(out_dim, (n_tok + tokg - 1) / tokg, s->num_sms);
    return status_of(timed_launch(st, [&] { return q8::launch_kq_gemv(p, tokg, s->num_sms, st); }));
}

int q8_kq_moe_matmul(float *out, const void *W_experts, int fmt, uint32_t n_expert, uint64_t expert_stride_bytes,
                     const int32_t *expert_ids, uint32_t k, uint64_t in_dim, uint64_t out_dim, const float *x,
                     int x_per_pair, uint64_t n_tok, void *stream) {
    if (n_expert == 0 || n_expert > MAX_EXPERTS || k == 0 || k > n_expert) return Q8_EINVAL;
    if (n_tok > (((uint64_t)1 << 31) - 1) / k) return Q8_EINVAL;
    const uint64_t n_pairs = n_tok * k, x_rows = x_per_pair ? n_pairs : n_tok;
    int rc = check_kq(fmt, in_dim, out_dim, x_rows);
    if (rc) return rc;
    if (expert_stride_bytes < out_dim * q8_kq_row_bytes(in_dim, fmt)) return Q8_EINVAL;
    if (n_tok == 0 || out_dim == 0) return Q8_OK;
    if (!out || !W_experts || !expert_ids || !x) return Q8_EINVAL;
    const uintptr_t wmask = fmt == Q8_KQ_Q4_K ? 15u : 3u;
    if (!aligned16(out) || !aligned16(x) || (reinterpret_cast<uintptr_t>(W_experts) & wmask) ||
        (expert_stride_bytes & wmask) || (reinterpret_cast<uintptr_t>(expert_ids) & 3u))
        return Q8_EALIGN;
    std::lock_guard<std::mutex> lk(g_mutex);
    DeviceState *s;
    if ((rc = get_device(&s))) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const uint64_t max_rows = q8::route_max_rows(n_pairs, n_expert);
    const size_t plan_bytes = q8::route_plan_bytes(n_expert);
    const size_t need = align256(n_expert * 4) * 2 + q8::ROUTE_CLASSES * align256(plan_bytes) +
                        align256(max_rows * 4) * 2 + q8k_planes_bytes(x_rows, in_dim);
    if ((rc = reserve_scratch(s, need))) return rc;
    Carver cv(s->scratch);
    int32_t *counts = cv.take<int32_t>(n_expert * 4);
    int32_t *row0_of = cv.take<int32_t>(n_expert * 4);
    uint8_t *plans = cv.take<uint8_t>(q8::ROUTE_CLASSES * plan_bytes);
    int32_t *row_to_out = cv.take<int32_t>(max_rows * 4);
    int32_t *src_row = cv.take<int32_t>(max_rows * 4);
    const Q8kPlanes q = take_q8k_planes(cv, x_rows, in_dim);
    // staged kernel when rows, matrix and stride are 16-byte multiples: items of its
    // rows per slot; else the direct kernel, items of 32 rows
    const uint32_t stream_rows = aligned16(W_experts) && (expert_stride_bytes & 15u) == 0
                                     ? q8::kq_stream_rows(q8_kq_row_bytes(in_dim, fmt), in_dim, 16)
                                     : 0;
    const uint32_t rows_item = stream_rows ? stream_rows : 32;
    cudaError_t e = q8::launch_route(expert_ids, n_tok, k, n_expert, x_per_pair, (uint32_t)out_dim, rows_item, 0,
                                     counts, row0_of, plans, row_to_out, src_row, nullptr, max_rows, out, s->err,
                                     s->num_sms, st);
    if (e != cudaSuccess) return status_of(e);
    if ((e = q8::launch_quantize_q8k(q.qx, q.dx, q.xs, nullptr, x, in_dim, x_rows, s->num_sms, st)) != cudaSuccess)
        return status_of(e);
    q8::KqParams p{};
    p.W = static_cast<const uint8_t *>(W_experts);
    p.expert_stride = expert_stride_bytes;
    p.in_dim = in_dim;
    p.out_dim = (uint32_t)out_dim;
    p.nsb = (uint32_t)(in_dim / 256);
    p.fmt = fmt;
    p.qx = q.qx;
    p.dx = q.dx;
    p.xs = q.xs;
    p.out = out;
    p.err = s->err;
    p.rows_per_item = rows_item;
    p.src_row = src_row;
    p.row_to_out = row_to_out;
    return status_of(timed_launch(st, [&] {
        for (int cls = 0; cls < q8::ROUTE_GEMV_CLASSES; ++cls) {
            p.plan = reinterpret_cast<const q8::PlanHeader *>(plans + cls * plan_bytes);
            cudaError_t e2 = stream_rows ? q8::launch_kq_stream(p, cls == 0 ? 8 : 16, s->num_sms, st)
                                         : q8::launch_kq_gemv(p, cls == 0 ? 8 : 16, s->num_sms, st);
            if (e2 != cudaSuccess) return e2;
        }
        return cudaSuccess;
    }));
}

uint64_t q8_repack_bytes(uint64_t in_dim, uint64_t rows, int layout) {
    if (in_dim == 0 || in_dim % q8::QK || check_dims(in_dim, rows, 1)) return 0;
    const uint64_t nb = in_dim / q8::QK;
    if (layout == Q8_LAYOUT_PLANES) return rows * in_dim + rows * nb * 2;
    if (layout == Q8_LAYOUT_TC) {
        if (in_dim % 64) return 0;   // the GEMM takes K in stages of two blocks
        const uint64_t m_ld = (rows + 127) & ~(uint64_t)127;
        return m_ld * in_dim * 2 + nb * m_ld * 4;
    }
    return 0;
}

int q8_repack(void *Wp, const void *W, uint64_t in_dim, uint64_t rows, int layout, void *stream) {
    int rc = check_dims(in_dim, rows, 1);
    if (rc) return rc;
    if (layout != Q8_LAYOUT_PLANES && layout != Q8_LAYOUT_TC) return Q8_EINVAL;
    if (layout == Q8_LAYOUT_TC && in_dim % 64) return Q8_EINVAL;
    if (rows == 0) return Q8_OK;
    if (!Wp || !W) return Q8_EINVAL;
    if (!aligned16(Wp) || !aligned16(W)) return Q8_EALIGN;
    std::lock_guard<std::mutex> lk(g_mutex);
    DeviceState *s;
    if ((rc = get_device(&s))) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (layout == Q8_LAYOUT_PLANES)
        return status_of(q8::launch_repack(static_cast<uint8_t *>(Wp), static_cast<const uint8_t *>(W), in_dim, rows,
                                           s->num_sms, st));
    // the GEMM's operand: padding rows and their scales zero, then every real row widened
    const uint64_t nb = in_dim / q8::QK, m_ld = (rows + 127) & ~(uint64_t)127;
    if ((rc = status_of(cudaMemsetAsync(Wp, 0, q8_repack_bytes(in_dim, rows, layout), st)))) return rc;
    uint8_t *base = static_cast<uint8_t *>(Wp);
    return status_of(q8::launch_tc_expand(reinterpret_cast<__half *>(base), reinterpret_cast<float *>(base + m_ld * in_dim * 2),
                                          static_cast<const uint8_t *>(W), (uint32_t)rows, (uint32_t)nb, (uint32_t)m_ld,
                                          s->num_sms, st));
}

int q8_matmul_packed(float *out, const void *Wp, int layout, uint64_t in_dim, uint64_t out_dim, const float *x,
                     uint64_t n_tok, void *stream) {
    int rc = check_dims(in_dim, out_dim, n_tok);
    if (rc) return rc;
    if (layout != Q8_LAYOUT_PLANES && layout != Q8_LAYOUT_TC) return Q8_EINVAL;
    if (layout == Q8_LAYOUT_TC && in_dim % 64) return Q8_EINVAL;
    if (n_tok == 0 || out_dim == 0) return Q8_OK;
    if (!out || !Wp || !x) return Q8_EINVAL;
    if (!aligned16(out) || !aligned16(Wp) || !aligned16(x)) return Q8_EALIGN;
    std::lock_guard<std::mutex> lk(g_mutex);
    DeviceState *s;
    if ((rc = get_device(&s))) return rc;
    if (layout == Q8_LAYOUT_TC) {
        const uint64_t m_ld = (out_dim + 127) & ~(uint64_t)127;
        const uint8_t *base = static_cast<const uint8_t *>(Wp);
        return run_tc(s, out, nullptr, in_dim, out_dim, x, nullptr, n_tok, static_cast<cudaStream_t>(stream),
                      reinterpret_cast<const __half *>(base), reinterpret_cast<const float *>(base + m_ld * in_dim * 2));
    }
    const uint64_t n_pad = (n_tok + 15) & ~(uint64_t)15;
    if ((rc = reserve_scratch(s, planes_bytes(n_pad, in_dim)))) return rc;
    Carver cv(s->scratch);
    int8_t *qx = cv.take<int8_t>(n_pad * in_dim);
    float *dx = cv.take<float>(n_pad * (in_dim / q8::QK) * sizeof(float));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if ((rc = status_of(q8::launch_quantize_planes(qx, dx, x, in_dim, n_pad, nullptr, n_tok, s->num_sms, st))))
        return rc;
    return status_of(timed_launch(st, [&] {
        return q8::launch_matmul_packed(out, static_cast<const uint8_t *>(Wp), in_dim, out_dim, qx, dx, n_tok,
                                        s->num_sms, st);
    }));
}

int q8_last_error(void *stream) {
    std::lock_guard<std::mutex> lk(g_mutex);
    DeviceState *s;
    int rc = get_device(&s);
    if (rc) return rc;
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        cudaGetLastError();
        return status_of(e);
    }
    int v = 0, zero = 0;
    if ((e = cudaMemcpy(&v, s->err, sizeof(int), cudaMemcpyDeviceToHost)) != cudaSuccess ||
        (e = cudaMemcpy(s->err, &zero, sizeof(int), cudaMemcpyHostToDevice)) != cudaSuccess) {
        cudaGetLastError();
        return status_of(e);
    }
    return v;
}

uint64_t q8_scratch_bytes(void) {
    std::lock_guard<std::mutex> lk(g_mutex);
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) {
        cudaGetLastError();
        return 0;
    }
    return g_dev[dev].scratch_bytes + g_dev[dev].stage_bytes;
}

void q8_release(void) {
    std::lock_guard<std::mutex> lk(g_mutex);
    int cur = -1;
    if (cudaGetDevice(&cur) != cudaSuccess) {
        cudaGetLastError();
        return;
    }
    for (int d = 0; d < MAX_DEVICES; ++d) {
        if (!g_dev[d].scratch && !g_dev[d].stage) continue;
        cudaSetDevice(d);
        cudaDeviceSynchronize();
        cudaFree(g_dev[d].scratch);
        cudaFree(g_dev[d].stage);
        g_dev[d].scratch = g_dev[d].stage = nullptr;
        g_dev[d].scratch_bytes = g_dev[d].stage_bytes = 0;
    }
    cudaSetDevice(cur);
}

int q8_profile_arm(uint32_t n_pairs) {
    std::lock_guard<std::mutex> lk(g_mutex);
    profile_free();
    if (n_pairs == 0) return Q8_OK;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return Q8_ECUDA;
    }
    g_prof.ev = new cudaEvent_t[2 * n_pairs];
    g_prof.recorded = new uint8_t[n_pairs]();
    for (uint32_t i = 0; i < 2 * n_pairs; ++i) {
        if (cudaEventCreate(&g_prof.ev[i]) != cudaSuccess) {
            cudaGetLastError();
            for (uint32_t j = 0; j < i; ++j) cudaEventDestroy(g_prof.ev[j]);
            delete[] g_prof.ev;
            delete[] g_prof.recorded;
            g_prof = Profile{};
            return Q8_ECUDA;
        }
    }
    g_prof.n = n_pairs;
    g_prof.device = dev;
    return Q8_OK;
}

uint64_t q8_profile_used(void) {
    std::lock_guard<std::mutex> lk(g_mutex);
    return g_prof.used;
}

int q8_profile_read(uint32_t i, float *ms) {
    std::lock_guard<std::mutex> lk(g_mutex);
    if (!ms || i >= g_prof.n || !g_prof.recorded[i]) return Q8_EINVAL;
    if (cudaEventSynchronize(g_prof.ev[2 * i + 1]) != cudaSuccess ||
        cudaEventElapsedTime(ms, g_prof.ev[2 * i], g_prof.ev[2 * i + 1]) != cudaSuccess) {
        cudaGetLastError();
        return Q8_ECUDA;
    }
    return Q8_OK;
}

const char *q8_last_cuda_error(void) {
    std::lock_guard<std::mutex> lk(g_mutex);
    return cudaGetErrorName(g_last_cuda_error);
}

void q8_debug_fail_next_alloc(int count) {
    std::lock_guard<std::mutex> lk(g_mutex);
    g_fail_next_alloc = count > 0 ? count : 0;
}

void q8_debug_expire_waits(int count, uint64_t limit_ns) {
    std::lock_guard<std::mutex> lk(g_mutex);
    g_expire_next = count > 0 ? count : 0;
    g_expire_limit_ns = limit_ns;
}

}  // extern "C"
