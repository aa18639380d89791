// tmap.hpp -- host-side creation of TMA tensor maps (cuTensorMapEncodeTiled,
// reached through the runtime's driver entry point so the library needs no
// link-time dependency on libcuda).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

namespace nsa {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_tiled_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// bf16 tensor map with 128-byte swizzle.  dims/strides innermost first;
// strides are in bytes for dims 1..rank-1.  Returns false on failure.
inline bool make_tmap_bf16(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                           const uint64_t* strides_bytes, const uint32_t* box,
                           CUtensorMapL2promotion l2 = CU_TENSOR_MAP_L2_PROMOTION_L2_256B) {
  EncodeTiledFn fn = encode_tiled_fn();
  if (fn == nullptr) return false;
  cuuint64_t gd[5], gs[4];
  cuuint32_t bd[5], es[5];
  for (int i = 0; i < rank; ++i) {
    gd[i] = dims[i];
    bd[i] = box[i];
    es[i] = 1;
  }
  for (int i = 0; i < rank - 1; ++i) gs[i] = strides_bytes[i];
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void*>(base), gd, gs, bd, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, l2, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// K or V, token-major [B,T,G,d] or head-major [B,G,T,d], as a 4-D map with
// 64-column x ``tokens``-token boxes of one head.  Coordinates are
// (column, g, token, b) for token-major and (column, token, g, b) for
// head-major (dimensions always in increasing stride order).
inline bool make_kv_map(CUtensorMap* map, const void* base, int B, int T, int G, int d, int tokens,
                        bool head_major) {
  const uint64_t e = 2;
  if (!head_major) {
    const uint64_t dims[4] = {(uint64_t)d, (uint64_t)G, (uint64_t)T, (uint64_t)B};
    const uint64_t str[3] = {d * e, (uint64_t)G * d * e, (uint64_t)T * G * d * e};
    const uint32_t box[4] = {64, 1, (uint32_t)tokens, 1};
    return make_tmap_bf16(map, base, 4, dims, str, box);
  }
  const uint64_t dims[4] = {(uint64_t)d, (uint64_t)T, (uint64_t)G, (uint64_t)B};
  const uint64_t str[3] = {d * e, (uint64_t)T * d * e, (uint64_t)G * T * d * e};
  const uint32_t box[4] = {64, (uint32_t)tokens, 1, 1};
  return make_tmap_bf16(map, base, 4, dims, str, box);
}

}  // namespace nsa
