// Host-side TMA tensor-map encoding.  The driver entry point is fetched
// through the runtime once, so the library does not link libcuda directly.

#include <cudaTypedefs.h>

#include <mutex>

#include "tma_host.h"

namespace mla {

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
  });
  return fn;
}

bool make_tmap_bf16_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows,
                       uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_rows,
                       int swizzle_bytes) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {row_stride_bytes};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t es[2] = {1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                        strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        swizzle_bytes == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
                        : swizzle_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                              : CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

static bool encode_3d(CUtensorMap* map, CUtensorMapDataType type, const void* base,
                      uint64_t inner, uint64_t rows, uint64_t planes, uint64_t row_stride_bytes,
                      uint64_t plane_stride_bytes, uint32_t box_inner, uint32_t box_rows) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[3] = {inner, rows, planes};
  cuuint64_t strides[2] = {row_stride_bytes, plane_stride_bytes};
  cuuint32_t box[3] = {box_inner, box_rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  const CUresult r = fn(map, type, 3, const_cast<void*>(base), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_tmap_bf16_3d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows,
                       uint64_t planes, uint64_t row_stride_bytes, uint64_t plane_stride_bytes,
                       uint32_t box_inner, uint32_t box_rows) {
  return encode_3d(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, inner, rows, planes,
                   row_stride_bytes, plane_stride_bytes, box_inner, box_rows);
}

bool make_tmap_f32_3d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows,
                      uint64_t planes, uint64_t row_stride_bytes, uint64_t plane_stride_bytes,
                      uint32_t box_inner, uint32_t box_rows) {
  return encode_3d(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, base, inner, rows, planes,
                   row_stride_bytes, plane_stride_bytes, box_inner, box_rows);
}

}  // namespace mla
