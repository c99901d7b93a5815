// q8_tmap.cu -- host helper: tensor maps (TMA descriptors) over raw Q8_0 rows.
//
// The driver's cuTensorMapEncodeTiled is reached through the runtime's
// driver-entry-point query, so the library does not link libcuda directly.
#include <cuda.h>
#include <cuda_runtime.h>

#include "q8_kernels.h"

namespace q8 {

namespace {
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

bool load_encoder() {
    if (g_encode) return true;
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn) {
        cudaGetLastError();
        return false;
    }
    g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    return true;
}
}  // namespace

// Rows of raw Q8_0 blocks viewed as 32-bit words: dims {row_bytes/4, rows, n_mat},
// strides {row_bytes, mat_stride}; box {box_words, box_rows, 1}; no swizzle;
// out-of-bounds words read as zero.
bool encode_rows_tmap(CUtensorMap *map, const void *W, uint64_t row_bytes, uint64_t rows, uint64_t n_mat,
                      uint64_t mat_stride, uint32_t box_words, uint32_t box_rows) {
    if (!load_encoder()) return false;
    if (row_bytes % 16 || mat_stride % 16 || (reinterpret_cast<uintptr_t>(W) & 15u)) return false;
    cuuint64_t dims[3] = {row_bytes / 4, rows, n_mat};
    cuuint64_t strides[2] = {row_bytes, n_mat > 1 ? mat_stride : rows * row_bytes};
    cuuint32_t box[3] = {box_words, box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<void *>(W), dims, strides, box, estr,
                                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Row-major fp16 matrix [rows][cols] with a 128-byte-swizzled box of
// box_cols (64) x box_rows: the canonical K-major operand layout of tcgen05.
bool encode_f16_tmap(CUtensorMap *map, const void *base, uint64_t cols, uint64_t rows, uint32_t box_cols,
                     uint32_t box_rows) {
    if (!load_encoder()) return false;
    if ((cols * 2) % 16 || (reinterpret_cast<uintptr_t>(base) & 15u)) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(base), dims, strides, box,
                                estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// fp32 rows cut into Q8_0 blocks: a [n_blocks][32] view of x (one 128-byte row
// per block) with a box of box_blocks blocks and the 128-byte swizzle, so that in
// shared memory the 16-byte chunk j of block b lies at chunk j ^ (b & 7) of the
// block's 128 bytes (the box must land 1024-byte aligned).
bool encode_blocks_tmap(CUtensorMap *map, const float *x, uint64_t n_blocks, uint32_t box_blocks) {
    if (!load_encoder()) return false;
    if ((reinterpret_cast<uintptr_t>(x) & 15u) || n_blocks == 0 || n_blocks > (1ull << 32)) return false;
    cuuint64_t dims[2] = {32, n_blocks};
    cuuint64_t strides[1] = {128};
    cuuint32_t box[2] = {32, box_blocks};
    cuuint32_t estr[2] = {1, 1};
    const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(x), dims, strides, box,
                                estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace q8
