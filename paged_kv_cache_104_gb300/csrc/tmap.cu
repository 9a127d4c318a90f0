// TMA tensor-map encoding through cudaGetDriverEntryPointByVersion, with a
// cache: a map depends only on its base address, its shape and its kind, so
// a launch over the same pool (or the same q buffer) reuses the map encoded
// by an earlier one instead of encoding it again.
#include <cuda_runtime.h>

#include <map>
#include <mutex>
#include <tuple>

#include "tmap.h"

namespace pkv {
namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static const EncodeTiledFn fn = [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<EncodeTiledFn>(ptr);
    return static_cast<EncodeTiledFn>(nullptr);
  }();
  return fn;
}

enum MapKind { kPoolBf16 = 0, kPoolU8 = 1, kRowsBf16 = 2, kPoolBlocksBf16 = 3, kRows32Bf16 = 4 };
using Key = std::tuple<int, const void*, int64_t, int>;

std::mutex g_map_mu;
std::map<Key, CUtensorMap> g_maps;

// Look the map up, or encode it with `enc` and remember it.
template <typename Enc>
bool cached(CUtensorMap* map, MapKind kind, const void* base, int64_t n, int m, Enc enc) {
  const Key key{kind, base, n, m};
  {
    std::lock_guard<std::mutex> lock(g_map_mu);
    auto it = g_maps.find(key);
    if (it != g_maps.end()) {
      *map = it->second;
      return true;
    }
  }
  if (!enc(map)) return false;
  std::lock_guard<std::mutex> lock(g_map_mu);
  if (g_maps.size() >= 4096) g_maps.clear();   // bounded: start over
  g_maps[key] = *map;
  return true;
}

}  // namespace

bool encode_pool_map_bf16(CUtensorMap* map, const void* base, int64_t rows) {
  EncodeTiledFn f = encode_fn();
  if (!f || rows <= 0 || rows >= (1ll << 31) - 1) return false;
  return cached(map, kPoolBf16, base, rows, 0, [&](CUtensorMap* m) {
    cuuint64_t dims[2] = {128, (cuuint64_t)rows};
    cuuint64_t strides[1] = {128 * 2};
    cuuint32_t box[2] = {64, 16};
    cuuint32_t estr[2] = {1, 1};
    return f(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  });
}

bool encode_pool_map_u8(CUtensorMap* map, const void* base, int64_t rows) {
  EncodeTiledFn f = encode_fn();
  if (!f || rows <= 0 || rows >= (1ll << 31) - 1) return false;
  return cached(map, kPoolU8, base, rows, 0, [&](CUtensorMap* m) {
    cuuint64_t dims[2] = {128, (cuuint64_t)rows};
    cuuint64_t strides[1] = {128};
    cuuint32_t box[2] = {128, 16};
    cuuint32_t estr[2] = {1, 1};
    return f(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  });
}

bool encode_rows_map_bf16(CUtensorMap* map, const void* base, int64_t n, int heads) {
  EncodeTiledFn f = encode_fn();
  if (!f || n <= 0 || heads <= 0) return false;
  return cached(map, kRowsBf16, base, n, heads, [&](CUtensorMap* m) {
    cuuint64_t dims[3] = {128, (cuuint64_t)heads, (cuuint64_t)n};
    cuuint64_t strides[2] = {128 * 2, (cuuint64_t)heads * 128 * 2};
    cuuint32_t box[3] = {64, 1, 128};
    cuuint32_t estr[3] = {1, 1, 1};
    return f(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  });
}

bool encode_latent_block_map(CUtensorMap* map, const void* base, int64_t num_blocks) {
  EncodeTiledFn f = encode_fn();
  if (!f || num_blocks <= 0 || 2 * num_blocks >= (1ll << 31) - 1) return false;
  return cached(map, kPoolBlocksBf16, base, num_blocks, 0, [&](CUtensorMap* m) {
    // element (x, y, z, w) = column x of half z of row y of 8-row group w
    cuuint64_t dims[4] = {64, 8, 2, (cuuint64_t)(2 * num_blocks)};
    cuuint64_t strides[3] = {256, 128, 2048};
    cuuint32_t box[4] = {64, 8, 2, 2};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    return f(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  });
}

bool encode_rows32_map_bf16(CUtensorMap* map, const void* base, int64_t rows) {
  EncodeTiledFn f = encode_fn();
  if (!f || rows <= 0 || rows >= (1ll << 31) - 1) return false;
  return cached(map, kRows32Bf16, base, rows, 0, [&](CUtensorMap* m) {
    cuuint64_t dims[2] = {128, (cuuint64_t)rows};
    cuuint64_t strides[1] = {128 * 2};
    cuuint32_t box[2] = {64, 32};
    cuuint32_t estr[2] = {1, 1};
    return f(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  });
}

}  // namespace pkv
