// Host-side construction of TMA tensor maps (bf16, 2-D, 128-byte swizzle).
//
// The driver's cuTensorMapEncodeTiled is reached through the runtime's
// driver-entry-point query, so the library has no link-time dependency on
// libcuda and can be loaded (for argument validation and symbol checks) on a
// machine without a GPU driver.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

namespace h3 {

inline PFN_cuTensorMapEncodeTiled_v12000 tmap_encoder() {
  // looked up once per process (a function-local static: thread-safe initialisation)
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    return PFN_cuTensorMapEncodeTiled_v12000(nullptr);
  }();
  return fn;
}

// A row-major bf16 matrix [rows][cols] with a row pitch of `row_stride_elems`
// elements, read in boxes of box_rows x box_cols (box_cols * 2 must be 128 for
// the 128-byte swizzle).  Rows past `rows` read as zero.
inline bool make_tmap_bf16_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                              uint64_t row_stride_elems, uint32_t box_rows, uint32_t box_cols) {
  auto enc = tmap_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {row_stride_elems * 2};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// The same matrix in boxes of box_rows x 32 elements (64-byte rows, 64-byte
// swizzle), e.g. for bulk tensor stores from a staging tile.
inline bool make_tmap_bf16_2d_sw64(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                                   uint64_t row_stride_elems, uint32_t box_rows) {
  auto enc = tmap_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {row_stride_elems * 2};
  cuuint32_t box[2] = {32, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// A row-major byte matrix (fp8 values) [rows][cols] with a row pitch of
// `row_stride` bytes, read in boxes of box_rows x 128 bytes (128-byte swizzle).
inline bool make_tmap_u8_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                            uint64_t row_stride, uint32_t box_rows) {
  auto enc = tmap_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {row_stride};
  cuuint32_t box[2] = {128, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace h3
