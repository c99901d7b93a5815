// q8_repack.cu -- load-time repack of Q8_0 rows into split planes, and the
// matmul over that layout.
//
// Packed layout for `rows` rows of in_dim values (same 34 bytes per 32 weights):
//   [0, rows*in_dim)                 int8 quant plane, row-major (row o at o*in_dim)
//   [rows*in_dim, + rows*nb*2)       fp16 scale plane, row-major ([rows][nb])
// Rows of the quant plane are 32-byte aligned, so fragment loads need no byte
// permutes (the ds4 pages report the aligned-slice + separate-scale layout as
// the faster one for their ROCm MoE tiles).  The repack copies bits; it does
// no arithmetic.
#include "q8_common.cuh"
#include "q8_kernels.h"

namespace q8 {

// One thread per block: 34 bytes in, 32 + 2 bytes out.
__global__ void __launch_bounds__(256) k_repack(uint8_t *__restrict__ Wp, const uint8_t *__restrict__ W,
                                                uint64_t in_dim, uint64_t rows) {
    const uint64_t nb = in_dim / QK;
    const uint64_t nblk = rows * nb;
    uint16_t *dplane = reinterpret_cast<uint16_t *>(Wp + rows * in_dim);
    for (uint64_t blk = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; blk < nblk; blk += (uint64_t)gridDim.x * blockDim.x) {
        const uint16_t *src = reinterpret_cast<const uint16_t *>(W + blk * QB);
        uint32_t w[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) w[i] = (uint32_t)src[1 + 2 * i] | ((uint32_t)src[2 + 2 * i] << 16);
        uint4 *dst = reinterpret_cast<uint4 *>(Wp + blk * QK);   // row o, block b -> o*in_dim + b*32 = blk*32
        dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
        dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
        dplane[blk] = src[0];
    }
}

// One warp per (8-row group, 16-token tile); blocks in order; mma.sync s8.
__global__ void __launch_bounds__(256) k_matmul_packed(float *__restrict__ out, const uint8_t *__restrict__ Wp,
                                                       uint64_t in_dim, uint64_t out_dim,
                                                       const int8_t *__restrict__ qx, const float *__restrict__ dx,
                                                       uint64_t n_tok) {
    const uint64_t nb = in_dim / QK;
    const int lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
    const uint64_t n_rg = (out_dim + 7) / 8, n_tt = (n_tok + 15) / 16;
    const uint64_t items = n_rg * n_tt;
    const int8_t *qp = reinterpret_cast<const int8_t *>(Wp);
    const uint16_t *dp = reinterpret_cast<const uint16_t *>(Wp + out_dim * in_dim);
    const uint64_t warps = (uint64_t)gridDim.x * (blockDim.x >> 5);
    for (uint64_t it = (uint64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); it < items; it += warps) {
        const uint64_t rg = it / n_tt, tt = it - rg * n_tt;
        const uint64_t rowb = rg * 8 + g;             // B row (weight) of this lane
        const uint64_t rowc0 = rg * 8 + 2 * c;        // output rows of this lane's accumulators
        const bool vb = rowb < out_dim, v0 = rowc0 < out_dim, v1 = rowc0 + 1 < out_dim;
        const uint64_t xr = tt * 16 + g;              // padded plane: always in range
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        for (uint64_t b = 0; b < nb; ++b) {
            uint32_t b0 = 0, b1 = 0;
            if (vb) {
                const int8_t *wq = qp + rowb * in_dim + b * QK + 4 * c;
                b0 = __ldg(reinterpret_cast<const uint32_t *>(wq));
                b1 = __ldg(reinterpret_cast<const uint32_t *>(wq + 16));
            }
            const float dw0 = v0 ? half_bits_to_float(__ldg(dp + rowc0 * nb + b)) : 0.f;
            const float dw1 = v1 ? half_bits_to_float(__ldg(dp + (rowc0 + 1) * nb + b)) : 0.f;
            const int8_t *xa = qx + xr * in_dim + b * QK + 4 * c;
            uint32_t a[4];
            a[0] = __ldg(reinterpret_cast<const uint32_t *>(xa));
            a[1] = __ldg(reinterpret_cast<const uint32_t *>(xa + 8 * in_dim));
            a[2] = __ldg(reinterpret_cast<const uint32_t *>(xa + 16));
            a[3] = __ldg(reinterpret_cast<const uint32_t *>(xa + 8 * in_dim + 16));
            const float dx0 = __ldg(dx + xr * nb + b), dx1 = __ldg(dx + (xr + 8) * nb + b);
            int d[4] = {0, 0, 0, 0};
            mma_s8_16832(d, a, b0, b1);
            acc[0] = fmaf((float)d[0], dw0 * dx0, acc[0]);
            acc[1] = fmaf((float)d[1], dw1 * dx0, acc[1]);
            acc[2] = fmaf((float)d[2], dw0 * dx1, acc[2]);
            acc[3] = fmaf((float)d[3], dw1 * dx1, acc[3]);
        }
        const uint64_t t0 = tt * 16 + g, t1 = t0 + 8;
        if (t0 < n_tok) {
            if (v0) out[t0 * out_dim + rowc0] = acc[0];
            if (v1) out[t0 * out_dim + rowc0 + 1] = acc[1];
        }
        if (t1 < n_tok) {
            if (v0) out[t1 * out_dim + rowc0] = acc[2];
            if (v1) out[t1 * out_dim + rowc0 + 1] = acc[3];
        }
    }
}

cudaError_t launch_repack(uint8_t *Wp, const uint8_t *W, uint64_t in_dim, uint64_t rows, int num_sms,
                          cudaStream_t st) {
    const uint64_t nblk = rows * (in_dim / QK);
    if (!nblk) return cudaSuccess;
    uint64_t grid = (nblk + 255) / 256;
    if (grid > (uint64_t)num_sms * 16) grid = (uint64_t)num_sms * 16;
    k_repack<<<(int)grid, 256, 0, st>>>(Wp, W, in_dim, rows);
    return cudaGetLastError();
}

cudaError_t launch_matmul_packed(float *out, const uint8_t *Wp, uint64_t in_dim, uint64_t out_dim,
                                 const int8_t *qx, const float *dx, uint64_t n_tok, int num_sms, cudaStream_t st) {
    const uint64_t items = ((out_dim + 7) / 8) * ((n_tok + 15) / 16);
    if (!items) return cudaSuccess;
    uint64_t grid = (items + 7) / 8;
    if (grid > (uint64_t)num_sms * 16) grid = (uint64_t)num_sms * 16;
    k_matmul_packed<<<(int)grid, 256, 0, st>>>(out, Wp, in_dim, out_dim, qx, dx, n_tok);
    return cudaGetLastError();
}

}  // namespace q8
