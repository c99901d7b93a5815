// q8_common.cuh -- device helpers shared by the library's kernels (sm_103a only).
//
// Inline PTX for mbarriers, bulk asynchronous copies (TMA) and bounded waits.
// Every wait in this library is bounded: when a limit expires the kernel
// records Q8_DEV_ETIMEOUT in the device error word and stops waiting, so a
// bug can produce wrong numbers and an error code but never a hung GPU.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>

#if defined(__CUDA_ARCH__) && (__CUDA_ARCH__ != 1030)
#error "this library is built for sm_103a (GB300) only"
#endif

namespace q8 {

constexpr int QK = 32;          // values per Q8_0 block
constexpr int QB = 34;          // bytes per Q8_0 block

// Device error word values (mirrored by q8_status in q8.h).
constexpr int DEV_ERANGE = -3;
constexpr int DEV_ETIMEOUT = -6;

// ~2 s at 1 ns per %globaltimer tick: far beyond any legitimate wait.  Kernels
// take their limit as a parameter (0 = this default); the drains of copies in
// flight after an abort always use this default.
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;

__host__ __device__ __forceinline__ uint64_t wait_limit(uint64_t ns) { return ns ? ns : WAIT_LIMIT_NS; }

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void raise_error(int *err, int code) {
    if (err) atomicCAS(err, 0, code);
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for the phase with the given parity to complete.  Returns
// false (and raises Q8_ETIMEOUT) when limit_ns expires; once `*abort` is set
// (a CTA-wide flag in shared memory) it returns false within 256 retries.
// A caller whose wait failed must not release the buffer it guards: the copy
// may still be in flight, and only the producer's drain may wait for it.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, int *err, volatile int *abort,
                                          uint64_t limit_ns = WAIT_LIMIT_NS) {
    if (mbar_try_wait(bar, parity)) return true;
    uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 255u) == 0u) {
            if (abort && *abort) return false;
            if (global_timer_ns() - t0 > limit_ns) {
                raise_error(err, DEV_ETIMEOUT);
                if (abort) *abort = 1;
                return false;
            }
        }
    }
}

// After an abort: wait, until the global-timer deadline t_end at the latest, for
// a phase whose copies may still be in flight, so that no bulk copy lands after
// the CTA has exited.
__device__ __forceinline__ void mbar_drain(uint64_t *bar, uint32_t parity, uint64_t t_end) {
    while (!mbar_try_wait(bar, parity))
        if (global_timer_ns() > t_end) return;
}

// ---------------------------------------------------------------- bulk copy (TMA, 1-D)
// Global -> shared, completion counted on `bar` in bytes.  src and dst must be
// 16-byte aligned and bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// ---------------------------------------------------------------- named barriers
__device__ __forceinline__ void named_bar_sync(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// ---------------------------------------------------------------- small math
__device__ __forceinline__ float half_bits_to_float(uint16_t h) {
    return __half2float(__ushort_as_half(h));
}

// Four int8 at byte offset 2 mod 4: combine the two aligned words around them.
__device__ __forceinline__ uint32_t funnel16(uint32_t lo, uint32_t hi) {
    return __byte_perm(lo, hi, 0x5432);
}

// Integer MMA: D(16x8, s32) += A(16x32, s8, row) * B(32x8, s8, col).
__device__ __forceinline__ void mma_s8_16832(int (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+r"(d[0]), "+r"(d[1]), "+r"(d[2]), "+r"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// SwiGLU of one gate/up pair (MoE study page, SwiGLU activation section):
// silu(min(g, L)) * clamp(u, -L, L), L = limit (0: no clamp), silu(g) = g / (1 + e^-g)
// in fp32 with CUDA's expf and IEEE division.  The routed FFN's separate pass and
// the gate/up pair GEMV's epilogue both use it, so they give the same bits.
__device__ __forceinline__ float swiglu1(float g, float u, float limit) {
    if (limit > 0.0f) {
        g = fminf(g, limit);
        u = fminf(fmaxf(u, -limit), limit);
    }
    return g / (1.0f + expf(-g)) * u;
}

}  // namespace q8
