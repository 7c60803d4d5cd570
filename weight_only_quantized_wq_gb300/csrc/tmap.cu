// tmap.cu -- 2-D TMA tensor maps for the kernels, encoded through the
// runtime's driver entry point (no libcuda link) and cached by their values.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>
#include <unordered_map>

#include "kernels.h"

namespace wq {

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// Looked up once per process; a function-local static is initialised once
// even when several host threads make their first call together.
EncodeTiledFn encode_fn() {
  static const EncodeTiledFn fn = []() -> EncodeTiledFn {
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<EncodeTiledFn>(f);
    return nullptr;
  }();
  return fn;
}

struct Key {
  uintptr_t base;
  uint64_t cols, rows;
  uint32_t box_cols, box_rows;
  int elem_bytes, swizzle;
  bool operator==(const Key &o) const { return std::memcmp(this, &o, sizeof(Key)) == 0; }
};

struct KeyHash {
  size_t operator()(const Key &k) const {
    uint64_t h = k.base * 0x9E3779B97F4A7C15ull;
    h ^= (k.cols + 0x51ull) * 0xC2B2AE3D27D4EB4Full;
    h ^= (k.rows + 0x7Full) * 0x165667B19E3779F9ull;
    h ^= ((uint64_t)k.box_cols << 32 | k.box_rows) * 0x27D4EB2F165667C5ull;
    h ^= (uint64_t)(k.elem_bytes * 1024 + k.swizzle);
    return (size_t)(h ^ (h >> 29));
  }
};

}  // namespace

bool encode_2d(CUtensorMap *m, const void *base, int elem_bytes, uint64_t cols, uint64_t rows, uint32_t box_cols,
               uint32_t box_rows, int swizzle) {
  Key key;
  std::memset(&key, 0, sizeof(key));  // padding bytes take part in the comparison
  key.base = reinterpret_cast<uintptr_t>(base);
  key.cols = cols;
  key.rows = rows;
  key.box_cols = box_cols;
  key.box_rows = box_rows;
  key.elem_bytes = elem_bytes;
  key.swizzle = swizzle;
  static std::unordered_map<Key, CUtensorMap, KeyHash> cache;
  static std::mutex mu;
  {
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end()) {
      *m = it->second;
      return true;
    }
  }
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * (uint64_t)elem_bytes};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUtensorMapDataType dt = elem_bytes == 4   ? CU_TENSOR_MAP_DATA_TYPE_UINT32
                                 : elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16
                                                   : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const CUtensorMapSwizzle sw = swizzle == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
                                : swizzle == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                : swizzle == 32 ? CU_TENSOR_MAP_SWIZZLE_32B
                                                : CU_TENSOR_MAP_SWIZZLE_NONE;
  if (fn(m, dt, 2, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
         swizzle ? CU_TENSOR_MAP_L2_PROMOTION_L2_256B : CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  std::lock_guard<std::mutex> lock(mu);
  if (cache.size() > 4096) cache.clear();  // bounded
  cache.emplace(key, *m);
  return true;
}

}  // namespace wq
