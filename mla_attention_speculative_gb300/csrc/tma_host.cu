// Host-side TMA tensor-map encoding.  The driver entry point is fetched
// through the runtime once, so the library does not link libcuda directly.

#include <cudaTypedefs.h>

#include <cstring>
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

// Encoding a tensor map is a driver call made several times per verify call;
// the maps depend only on what is encoded (type, address, extents, strides,
// box, swizzle), so each thread keeps the recent ones.
namespace {
struct MapKey {
  int type, rank, swizzle;
  const void* base;
  uint64_t dims[4], strides[3];
  uint32_t box[4];
};
struct MapEntry {
  MapKey key;
  CUtensorMap map;
  bool valid;
};
constexpr int kMapCache = 256;
thread_local MapEntry t_maps[kMapCache];

uint64_t key_hash(const MapKey& k) {
  uint64_t h = 1469598103934665603ull;
  const unsigned char* p = reinterpret_cast<const unsigned char*>(&k);
  for (size_t i = 0; i < sizeof(MapKey); ++i) h = (h ^ p[i]) * 1099511628211ull;
  return h;
}

// Encodes through the cache; false if the driver rejects the parameters.
bool encode_cached(CUtensorMap* map, CUtensorMapDataType type, int rank, const void* base,
                   const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box,
                   CUtensorMapSwizzle swizzle) {
  MapKey k;
  std::memset(&k, 0, sizeof(k));  // padding included: the key is hashed and compared bytewise
  k.type = (int)type;
  k.rank = rank;
  k.swizzle = (int)swizzle;
  k.base = base;
  for (int i = 0; i < rank; ++i) {
    k.dims[i] = dims[i];
    k.box[i] = box[i];
  }
  for (int i = 0; i + 1 < rank; ++i) k.strides[i] = strides[i];
  MapEntry& e = t_maps[key_hash(k) % kMapCache];
  if (e.valid && std::memcmp(&e.key, &k, sizeof(k)) == 0) {
    *map = e.map;
    return true;
  }
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint32_t es[4] = {1, 1, 1, 1};
  const CUresult r = fn(map, type, (cuuint32_t)rank, const_cast<void*>(base), dims, strides, box,
                        es, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return false;
  e.key = k;
  e.map = *map;
  e.valid = true;
  return true;
}
}  // namespace

bool make_tmap_bf16_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows,
                       uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_rows,
                       int swizzle_bytes) {
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {row_stride_bytes};
  const cuuint32_t box[2] = {box_inner, box_rows};
  return encode_cached(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box,
                       swizzle_bytes == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
                       : swizzle_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                             : CU_TENSOR_MAP_SWIZZLE_NONE);
}

static bool encode_3d(CUtensorMap* map, CUtensorMapDataType type, const void* base,
                      uint64_t inner, uint64_t rows, uint64_t planes, uint64_t row_stride_bytes,
                      uint64_t plane_stride_bytes, uint32_t box_inner, uint32_t box_rows) {
  const cuuint64_t dims[3] = {inner, rows, planes};
  const cuuint64_t strides[2] = {row_stride_bytes, plane_stride_bytes};
  const cuuint32_t box[3] = {box_inner, box_rows, 1};
  return encode_cached(map, type, 3, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
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

bool make_tmap_bf16_4d(CUtensorMap* map, const void* base, const uint64_t dims[4],
                       const uint64_t strides_bytes[3], const uint32_t box[4]) {
  const cuuint64_t d[4] = {dims[0], dims[1], dims[2], dims[3]};
  const cuuint64_t st[3] = {strides_bytes[0], strides_bytes[1], strides_bytes[2]};
  const cuuint32_t b[4] = {box[0], box[1], box[2], box[3]};
  return encode_cached(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, base, d, st, b,
                       CU_TENSOR_MAP_SWIZZLE_128B);
}

}  // namespace mla
