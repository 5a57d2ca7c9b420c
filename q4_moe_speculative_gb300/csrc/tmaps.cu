// tmaps.cu — TMA tensor maps for the kernels: encoded through the runtime's driver entry
// point and kept in a small cache keyed by their parameters (a decode loop calls the same
// layer with the same tensors every step).
#include <cstring>
#include <mutex>

#include "kernels.h"

namespace dsmoe {
namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
  static const EncodeTiledFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &qr) != cudaSuccess ||
        qr != cudaDriverEntryPointSuccess)
      return static_cast<EncodeTiledFn>(nullptr);
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

struct MapKey {
  const void* base;
  uint64_t d0, d1, d2;
  uint32_t b0, b1, b2, kind;
};

bool same_key(const MapKey& a, const MapKey& b) {
  return a.base == b.base && a.d0 == b.d0 && a.d1 == b.d1 && a.d2 == b.d2 && a.b0 == b.b0 &&
         a.b1 == b.b1 && a.b2 == b.b2 && a.kind == b.kind;
}

cudaError_t cached_map(CUtensorMap* out, const MapKey& key) {
  constexpr int kSlots = 64;
  static std::mutex mu;
  static MapKey keys[kSlots];
  static CUtensorMap maps[kSlots];
  static int used = 0, next = 0;
  {
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < used; ++i)
      if (same_key(keys[i], key)) { *out = maps[i]; return cudaSuccess; }
  }
  const EncodeTiledFn f = encode_tiled();
  if (!f) return cudaErrorNotSupported;
  CUresult r;
  if (key.kind == 2) {
    // bf16 block keys [layer][block][128 values]: boxes of 64 values x b1 blocks x 1 layer,
    // 128-byte swizzle (the K-major operand layout of the tensor-core scorer)
    const cuuint64_t dims[3] = {128, key.d1, key.d2};
    const cuuint64_t strides[2] = {256, key.d0};
    const cuuint32_t box[3] = {64, key.b1, 1};
    const cuuint32_t es[3] = {1, 1, 1};
    r = f(out, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<void*>(key.base), dims, strides, box,
          es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  } else {
    return cudaErrorInvalidValue;
  }
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  std::lock_guard<std::mutex> lock(mu);
  keys[next] = key;
  maps[next] = *out;
  next = (next + 1) % kSlots;
  if (used < kSlots) ++used;
  return cudaSuccess;
}

}  // namespace

cudaError_t key_tile_map(CUtensorMap* out, const uint16_t* keys, int N, int L,
                         int64_t key_stride, int box_rows) {
  MapKey k{};
  k.base = keys; k.d0 = (uint64_t)key_stride * 2; k.d1 = (uint64_t)N; k.d2 = (uint64_t)L;
  k.b1 = (uint32_t)box_rows; k.kind = 2;
  return cached_map(out, k);
}

}  // namespace dsmoe
