// TMA tensor-map construction shared by the GEMM translation units.
#pragma once
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

namespace moe {

inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return (PFN_cuTensorMapEncodeTiled_v12000) nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }();
  return fn;
}

// 2-D bf16 tensor [rows, cols] row-major, 128-byte swizzled boxes of
// box_cols x box_rows; out-of-bounds elements read as zero.
inline bool make_map(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows,
                     uint32_t box_cols, uint32_t box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D tensor [rows, cols] row-major of `dtype` (elem_bytes each), boxes of
// box_cols x box_rows, unswizzled unless `swizzle` says otherwise (128-byte
// swizzle: box rows of 128 bytes, 16-byte chunk q of row r at
// r*128 + ((q ^ (r % 8)) * 16)); out-of-bounds elements read as zero. The row
// pitch cols*elem_bytes must be a multiple of 16.
inline bool make_map_plain(CUtensorMap* m, CUtensorMapDataType dtype, uint32_t elem_bytes,
                           const void* base, uint64_t cols, uint64_t rows, uint32_t box_cols,
                           uint32_t box_rows,
                           CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_NONE) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn || (cols * elem_bytes) % 16 != 0) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * elem_bytes};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(m, dtype, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// MN-major operand tiles in one copy: a 3-D view of a bf16 [rows, cols]
// matrix as (64 columns, rows, cols/64 chunks), strides (row pitch, 128 B),
// box {64, box_rows, box_chunks}: shared memory receives [chunk][row][64],
// the 128-byte-swizzled MN-major layout with 64-element chunks.
inline bool make_map_mn3d(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows,
                          uint32_t box_rows, uint32_t box_chunks) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn || cols % 64 != 0) return false;
  cuuint64_t dims[3] = {64, rows, cols / 64};
  cuuint64_t strides[2] = {cols * 2, 128};
  cuuint32_t box[3] = {64, box_rows, box_chunks};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace moe
