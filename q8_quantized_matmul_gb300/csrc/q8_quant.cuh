// q8_quant.cuh -- the per-block activation quantiser, shared by the quantiser
// kernels and the GEMV's fused staging.
//
// The arithmetic is the per-block quantiser of the ds4 pages (model-architecture
// page, quantisation section 1, printed for Q8_K) applied to 32-element blocks:
//   amax = max|x_i|,  d = amax / 127 (IEEE fp32 division),
//   q_i = (int8) roundf(x_i / d) (IEEE division by the fp32 d, halves away from zero),
//   stored d = binary16(d) (round to nearest even, subnormals kept);
//   d == 0 (all-zero block, or an fp32 underflow) stores d = +0 and q = 0.
// The library is built without fast-math, so '/' is the IEEE division and
// roundf / __float2half_rn are CUDA's correctly specified routines.
#pragma once

#include <cuda_fp16.h>

#include "q8_common.cuh"

namespace q8 {

struct QuantBlock {
    int8_t q[8];      // this lane's eight quants
    uint32_t lo, hi;  // the same packed: q[0..3], q[4..7] (byte i = q[i])
    uint16_t dh;      // stored binary16 scale (same on the four lanes)
    float d_stored;   // dh as fp32 (exact)
};

// 1.5 * 2^23: adding it to |v| < 2^22 rounds v to the nearest integer (ties to
// even) and leaves that integer, as two's complement, in the low bits of the sum.
constexpr float ROUND_MAGIC = 12582912.0f;

// x8: this lane's eight values of the block; lanes 4i..4i+3 hold one block.
//
// q_i = roundf(x_i / d), with x_i / d the IEEE fp32 quotient, without dividing in
// the common case.  With u = 2^-24 and rd = fl(1/d) = (1/d)(1 + e1), the product
// qa = fl(x rd) = (x/d)(1 + e1)(1 + e2) and the quotient fl(x/d) = (x/d)(1 + e3),
// |e_i| <= u, differ by at most (3u + u^2)|x/d| < 2.3e-5 while |x/d| <= 128.
// roundf changes value only at half-integers, so when qa is more than 1e-4 from
// every half-integer both lie on the same side of all of them and roundf(qa) =
// roundf(fl(x/d)); away from half-integers roundf and round-half-even agree, so
// the fast path rounds qa with one add of ROUND_MAGIC (the quant is the sum's
// low byte) and checks the distance |qa - k| < 0.4999 (exact: k and qa are
// within 1/2).  |qa| <= 127 (1 + 3u), so k never leaves [-127, 127].  A value
// that fails the check (about 2e-4 of evenly spread values, and every exact tie)
// takes the IEEE division; so does every value of a block whose d is subnormal
// enough for its reciprocal to overflow (qa is then infinite or NaN and fails).
// The warp takes the slow path only when one of its lanes needs it.
__device__ __forceinline__ QuantBlock quantize8(const float (&x8)[8]) {
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(x8[i]));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    const float d = __fdiv_rn(amax, 127.0f);
    QuantBlock r;
    uint32_t w[2] = {0u, 0u};   // packed quants, byte i of w[h] = q[4h + i]
    uint32_t bad = 0;
    if (d != 0.0f) {
        const float rd = __frcp_rn(d);   // inf for a subnormal d: every value then fails the check
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint32_t t[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int i = 4 * h + j;
                const float qa = __fmul_rn(x8[i], rd);
                const float sm = __fadd_rn(qa, ROUND_MAGIC);
                const float k = __fsub_rn(sm, ROUND_MAGIC);
                t[j] = __float_as_uint(sm);
                bad |= (fabsf(__fsub_rn(qa, k)) < 0.4999f ? 0u : 1u) << i;
            }
            w[h] = __byte_perm(__byte_perm(t[0], t[1], 0x0040), __byte_perm(t[2], t[3], 0x0040), 0x5410);
        }
        r.dh = __half_as_ushort(__float2half_rn(d));
    } else {
        r.dh = 0;
    }
    if (__any_sync(0xffffffffu, bad != 0u)) {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (bad & (1u << i)) {
                const uint32_t q = (uint32_t)(uint8_t)(int8_t)(int)roundf(__fdiv_rn(x8[i], d));
                const int sh = 8 * (i & 3);
                w[i >> 2] = (w[i >> 2] & ~(0xffu << sh)) | (q << sh);
            }
    }
    r.lo = w[0];
    r.hi = w[1];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        r.q[i] = (int8_t)(r.lo >> (8 * i));
        r.q[4 + i] = (int8_t)(r.hi >> (8 * i));
    }
    r.d_stored = half_bits_to_float(r.dh);
    return r;
}

// The same quantiser with an IEEE division per value (same results, bit for bit).
// The GEMV's in-kernel staging uses it: there it measured slightly faster (4-token
// decode calls 9.35 against 9.6 us), while the kernels that quantise whole
// activation matrices, bound by instruction issue, gain from quantize8.
__device__ __forceinline__ QuantBlock quantize8_div(const float (&x8)[8]) {
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(x8[i]));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    const float d = __fdiv_rn(amax, 127.0f);
    QuantBlock r;
    if (d != 0.0f) {
#pragma unroll
        for (int i = 0; i < 8; ++i) r.q[i] = static_cast<int8_t>(static_cast<int>(roundf(__fdiv_rn(x8[i], d))));
        r.dh = __half_as_ushort(__float2half_rn(d));
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) r.q[i] = 0;
        r.dh = 0;
    }
    r.lo = r.hi = 0u;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        r.lo |= (uint32_t)(uint8_t)r.q[i] << (8 * i);
        r.hi |= (uint32_t)(uint8_t)r.q[4 + i] << (8 * i);
    }
    r.d_stored = half_bits_to_float(r.dh);
    return r;
}

__device__ __forceinline__ void load8(float (&x8)[8], const float *p) {
    const float4 a = __ldg(reinterpret_cast<const float4 *>(p));
    const float4 b = __ldg(reinterpret_cast<const float4 *>(p) + 1);
    x8[0] = a.x; x8[1] = a.y; x8[2] = a.z; x8[3] = a.w;
    x8[4] = b.x; x8[5] = b.y; x8[6] = b.z; x8[7] = b.w;
}

}  // namespace q8
