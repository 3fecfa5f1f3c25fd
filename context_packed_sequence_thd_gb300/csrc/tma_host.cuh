// tma_host.cuh -- host-side TMA tensor maps for THD tensors (one per
// translation unit that launches TMA kernels).
#pragma once

#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"

namespace cpthd {
namespace tma {

inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// [rows, H, D] bf16 (or fp16) viewed as a 3-D tensor (D, H, rows): boxes of
// 64 (d) x 1 (head) x box_rows (rows), 128-byte swizzle, zero fill outside.
inline int make_thd_map(CUtensorMap* map, const void* base, int64_t rows, int H, int D,
                        int box_rows, bool f16 = false) {
  auto enc = encode_fn();
  if (!enc) return CP_ERR_CUDA;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)rows};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2};
  cuuint32_t box[3] = {64, 1, (cuuint32_t)box_rows};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                   const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? CP_OK : CP_ERR_CUDA;
}

// [rows, H, D] bf16 (or fp16) viewed as a 2-D tensor (H*D, rows) for row gathers:
// boxes of 64 columns x 1 row, 128-byte swizzle (tile::gather4 loads four
// arbitrary rows of one box column per instruction).
inline int make_row_gather_map(CUtensorMap* map, const void* base, int64_t rows, int H, int D,
                               bool f16 = false) {
  auto enc = encode_fn();
  if (!enc) return CP_ERR_CUDA;
  cuuint64_t dims[2] = {(cuuint64_t)H * D, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)H * D * 2};
  cuuint32_t box[2] = {64, 1};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                   const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? CP_OK : CP_ERR_CUDA;
}

// fp32 [rows, H, D] viewed as a 3-D tensor (D, H, rows): boxes of 32 (d) x
// 1 (head) x 32 (rows) = 32 rows of 128 bytes, 128-byte swizzle (the
// shared-memory layout of the dK/dV epilogue's staging buffers).
inline int make_f32_rows_map(CUtensorMap* map, const void* base, int64_t rows, int H, int D) {
  auto enc = encode_fn();
  if (!enc) return CP_ERR_CUDA;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)rows};
  cuuint64_t strides[2] = {(cuuint64_t)D * 4, (cuuint64_t)H * D * 4};
  cuuint32_t box[3] = {32, 1, 32};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? CP_OK : CP_ERR_CUDA;
}

}  // namespace tma
}  // namespace cpthd
