// q8_noalloc.cu -- q8_matmul_noalloc: the matmul with its scratch in a fixed
// device array, for callers that must not allocate device memory through this
// library (an application whose own pool allocator owns the device's memory,
// or a decode loop that cannot take the synchronisation and latency of a
// first-use cudaMalloc).  The pages have no counterpart.  The quantiser
// always writes activation planes into the fixed array; up to 16 tokens the
// weight-streaming GEMV reads them (as q8_matmul does from 9 tokens on), above
// that the mma.sync kernel of the odd block counts does (q8_matmul runs its
// tcgen05 GEMM there, whose operands would not fit the array), and rows that
// are not 16-byte aligned take the plain slow kernel, as in q8_matmul.  The
// results agree with q8_matmul's within the matmul tolerance, not bit for bit:
// the kernels add the blocks in different fp32 orders.
#include <cstdint>
#include <mutex>

#include "../../include/q8.h"
#include "q8_common.cuh"
#include "q8_kernels.h"

namespace q8 {
int *device_error_word();                 // q8_api.cu
int record_cuda_status(cudaError_t e);    // q8_api.cu: Q8_OK, or Q8_ECUDA with the error recorded
}

namespace {

// The scratch: quantised activation planes of the current call (int8 plane,
// then fp32 scale plane).  Every GPU that loads the library holds it until the
// process exits.  The quantiser writes every byte a call reads (padding rows
// included) before the matmul reads it, so the array never needs clearing.
static __device__ __align__(256) uint8_t g_noalloc_scratch[Q8_NOALLOC_SCRATCH_BYTES];

constexpr int MAX_DEVICES = 64;

struct NoallocDevice {
    bool ready = false;
    uint8_t *scratch = nullptr;   // device address of g_noalloc_scratch on that device
    int num_sms = 0;
};

std::mutex g_na_mutex;
NoallocDevice g_na[MAX_DEVICES];

size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

// Once per device, with the device current: the array's device address.
int noalloc_device(NoallocDevice **out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) {
        cudaGetLastError();
        return q8::record_cuda_status(e != cudaSuccess ? e : cudaErrorInvalidDevice);
    }
    NoallocDevice &d = g_na[dev];
    if (!d.ready) {
        void *ptr = nullptr;
        if ((e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch)) != cudaSuccess || !ptr) {
            cudaGetLastError();
            return q8::record_cuda_status(e != cudaSuccess ? e : cudaErrorInvalidSymbol);
        }
        int sms = 0;
        if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) {
            cudaGetLastError();
            return q8::record_cuda_status(e);
        }
        d.scratch = static_cast<uint8_t *>(ptr);
        d.num_sms = sms;
        d.ready = true;
    }
    *out = &d;
    return Q8_OK;
}

}  // namespace

extern "C" int q8_matmul_noalloc(float *out, const void *W, uint64_t in_dim, uint64_t out_dim, const float *x,
                                 uint64_t n_tok, void *stream) {
    // Argument rules of q8_matmul.
    if (in_dim == 0 || in_dim % q8::QK) return Q8_EINVAL;
    if (in_dim > ((uint64_t)1 << 31) || out_dim > ((uint64_t)1 << 31) - 1 || n_tok > ((uint64_t)1 << 31) - 1)
        return Q8_EINVAL;
    const uint64_t nb = in_dim / q8::QK;
    if (out_dim && nb > (((uint64_t)1 << 62) / q8::QB) / out_dim) return Q8_EINVAL;
    if (n_tok && in_dim > ((uint64_t)1 << 40) / n_tok) return Q8_EINVAL;
    if (n_tok == 0 || out_dim == 0) return Q8_OK;
    if (!out || !W || !x) return Q8_EINVAL;
    const auto a16 = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    if (!a16(out) || !a16(W) || !a16(x)) return Q8_EALIGN;
    // The planes must fit the fixed array.
    const uint64_t n_pad = (n_tok + 15) & ~(uint64_t)15;
    const size_t q_bytes = align256(n_pad * in_dim);
    const size_t need = q_bytes + align256(n_pad * nb * sizeof(float));
    if (need > Q8_NOALLOC_SCRATCH_BYTES) return Q8_ESCRATCH;

    std::lock_guard<std::mutex> lk(g_na_mutex);
    NoallocDevice *d;
    int rc = noalloc_device(&d);
    if (rc) return rc;
    int *err = q8::device_error_word();
    if (!err) return Q8_ECUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int8_t *qx = reinterpret_cast<int8_t *>(d->scratch);
    float *dx = reinterpret_cast<float *>(d->scratch + q_bytes);
    if ((rc = q8::record_cuda_status(
             q8::launch_quantize_planes(qx, dx, x, in_dim, n_pad, nullptr, n_tok, d->num_sms, st))))
        return rc;

    // Up to 16 tokens on 16-byte-aligned rows: the weight-streaming GEMV from planes.
    if (nb % 8 == 0 && n_tok <= 16) {
        q8::GemvParams g{};
        g.W = static_cast<const uint8_t *>(W);
        g.in_dim = in_dim;
        g.out_dim = (uint32_t)out_dim;
        g.nb = (uint32_t)nb;
        g.qx = qx;
        g.dx = dx;
        g.out = out;
        g.err = err;
        g.n_tok = (uint32_t)n_tok;
        g.n_items = q8::gemv_dense_items(out_dim, d->num_sms);
        q8::gemv_dense_split(out_dim, g.n_items, g.sub_base, g.sub_rem);
        g.n_expert = 1;
        const int grid = (int)(g.n_items < (uint32_t)d->num_sms ? g.n_items : (uint32_t)d->num_sms);
        g.weights_early = 1;   // the preceding kernel is the quantiser
        return q8::record_cuda_status(q8::launch_gemv(g, q8::gemv_mode(n_tok), grid, st));
    }
    // More tokens: the mma.sync kernel on aligned rows, else the plain kernel.
    q8::MmaParams p{};
    p.W = static_cast<const uint8_t *>(W);
    p.in_dim = in_dim;
    p.out_dim = (uint32_t)out_dim;
    p.nb = (uint32_t)nb;
    p.qx = qx;
    p.dx = dx;
    p.out = out;
    p.err = err;
    p.n_tok = (uint32_t)n_tok;
    if (nb % 8 == 0) {
        const uint64_t items = ((out_dim + 15) / 16) * ((n_tok + 63) / 64);
        const int grid = (int)(items < (uint64_t)d->num_sms ? items : (uint64_t)d->num_sms);
        return q8::record_cuda_status(q8::launch_mma(p, grid, st));
    }
    const uint64_t hint = n_tok * out_dim > (1u << 30) ? (1u << 30) : n_tok * out_dim;
    return q8::record_cuda_status(q8::launch_generic(p, (int)hint, d->num_sms, st));
}
