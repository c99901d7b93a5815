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
    uint16_t dh;      // stored binary16 scale (same on the four lanes)
    float d_stored;   // dh as fp32 (exact)
};

// roundf(x / d), with x / d the IEEE fp32 quotient, without dividing in the
// common case.  With u = 2^-24 and rd = fl(1/d) = (1/d)(1 + e1), the product
// qa = fl(x rd) = (x/d)(1 + e1)(1 + e2) and the quotient fl(x/d) = (x/d)(1 + e3),
// |e_i| <= u, differ by at most (3u + u^2)|x/d| < 2.3e-5 while |x/d| <= 128.
// roundf changes value only at half-integers, so when qa is more than 1e-4 from
// every half-integer (and |qa| < 127.75) both lie on the same side of all of them
// and roundf(qa) = roundf(fl(x/d)).  Otherwise (about 2e-4 of evenly spread
// values, and every exact tie) the quotient is taken with the IEEE division; a
// subnormal d whose reciprocal overflows always takes the division.
// Away from half-integers roundf and round-half-even agree, so the fast path is
// one rint and the distance |qa - k| < 0.4999 (exact: k and qa are within 1/2).
__device__ __forceinline__ float round_quotient(float x, float d, float rd) {
    const float qa = __fmul_rn(x, rd);
    const float k = rintf(qa);
    if (fabsf(__fsub_rn(qa, k)) < 0.4999f && fabsf(qa) < 127.75f) return k;
    return roundf(__fdiv_rn(x, d));
}

// x8: this lane's eight values of the block; lanes 4i..4i+3 hold one block.
__device__ __forceinline__ QuantBlock quantize8(const float (&x8)[8]) {
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(x8[i]));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    const float d = __fdiv_rn(amax, 127.0f);
    QuantBlock r;
    if (d != 0.0f) {
        const float rd = __frcp_rn(d);   // inf for a subnormal d: every value then takes the division
#pragma unroll
        for (int i = 0; i < 8; ++i) r.q[i] = static_cast<int8_t>(static_cast<int>(round_quotient(x8[i], d, rd)));
        r.dh = __half_as_ushort(__float2half_rn(d));
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) r.q[i] = 0;
        r.dh = 0;
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
