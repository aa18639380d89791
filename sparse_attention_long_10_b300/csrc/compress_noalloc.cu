// compress_noalloc.cu -- nsa_compress_kv_noalloc: the compression step with
// its scratch memory in a fixed, file-scope device array instead of a
// caller-provided workspace.
//
// Who needs it: callers that cannot allocate device memory at the point where
// they compress KV blocks -- for example a serving loop whose device memory is
// planned once up front and never grows, or an embedding C program that is
// only handed tensor pointers and owns no device allocator.  cudaMalloc can
// also synchronise the device, which such latency-bound callers avoid.  The
// caller still passes its inputs and outputs; only the scratch moves here.
//
// The scratch is the status word (256 B) followed by the two fp32 bias
// vectors flatten(PE) @ W (dk and dv floats, each 256-byte aligned).  Every
// GPU that loads libnsa.so holds this array until the process exits.
#include <cuda_runtime.h>

#include <mutex>

#include "common.cuh"
#include "kernels.hpp"
#include "nsa.h"

namespace {

// Fixed maximum: status word + bias_k + bias_v for dk, dv <= 256.
constexpr size_t kNoAllocScratchBytes = 256 + 1024 + 1024;
static_assert(kNoAllocScratchBytes >= 256 + 256 * sizeof(float) * 2, "scratch covers dk, dv <= 256");

static __device__ __align__(256) uint8_t g_compress_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices];   // device address of g_compress_scratch, per device

// Device address of the scratch array on the current device.  Resolved once
// per device, with that device current, and cached.
int scratch_for_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return NSA_ERR_NO_DEVICE;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_compress_scratch) != cudaSuccess || p == nullptr) return NSA_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return NSA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" int nsa_compress_kv_noalloc(const nsa_cfg* cfg, int layout, const void* k, const void* v, void* kc,
                                       void* vc, void* stream) {
  // the same argument rules, in the same order, as nsa_compress_kv
  int rc = nsa::check_nsa_cfg(cfg);
  if (rc != NSA_OK) return rc;
  const nsa_cfg& c = *cfg;
  if (layout != NSA_LAYOUT_BTGD && layout != NSA_LAYOUT_BGTD) return NSA_ERR_INVALID_ARG;
  if ((rc = nsa::check_nsa_phi(cfg)) != NSA_OK) return rc;
  for (const void* p : {k, v}) {
    if (p == nullptr) return NSA_ERR_INVALID_ARG;
    if (!aligned16(p)) return NSA_ERR_MISALIGNED;
  }
  const int Nc = nsa_num_compressed(cfg);
  if (Nc > 0) {
    for (const void* p : {static_cast<const void*>(kc), static_cast<const void*>(vc)}) {
      if (p == nullptr) return NSA_ERR_INVALID_ARG;
      if (!aligned16(p)) return NSA_ERR_MISALIGNED;
    }
  }
  // the fixed scratch must hold the status word and both bias vectors; the
  // cfg rules (dk, dv <= 256) keep this true today, the check keeps it true
  // if those rules are ever widened
  const size_t off_bk = 256;
  const size_t off_bv = nsa::align_up(off_bk + sizeof(float) * (size_t)c.dk, 256);
  const size_t need = nsa::align_up(off_bv + sizeof(float) * (size_t)c.dv, 256);
  if (need > kNoAllocScratchBytes) return NSA_ERR_WORKSPACE;
  int dev = -1, major = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess || major != 10)
    return NSA_ERR_NO_DEVICE;
  void* scratch = nullptr;
  rc = scratch_for_current_device(&scratch);
  if (rc != NSA_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the array keeps the previous call's contents: clear the status word
  if (cudaMemsetAsync(scratch, 0, 256, s) != cudaSuccess) return NSA_ERR_CUDA;
  if (Nc == 0) return NSA_OK;
  uint8_t* base = static_cast<uint8_t*>(scratch);
  nsa::DeviceStatus* st = reinterpret_cast<nsa::DeviceStatus*>(base);
  rc = nsa::launch_compress_one(c, layout, k, c.dk, c.pe_k, c.w_k, kc, reinterpret_cast<float*>(base + off_bk), st, s);
  if (rc != NSA_OK) return rc;
  return nsa::launch_compress_one(c, layout, v, c.dv, c.pe_v, c.w_v, vc, reinterpret_cast<float*>(base + off_bv), st,
                                  s);
}

extern "C" int nsa_compress_kv_noalloc_status(void* stream) {
  void* scratch = nullptr;
  int rc = scratch_for_current_device(&scratch);
  if (rc != NSA_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  nsa::DeviceStatus h;
  if (cudaMemcpyAsync(&h, scratch, sizeof(h), cudaMemcpyDeviceToHost, s) != cudaSuccess) return NSA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return NSA_ERR_CUDA;
  if (cudaMemsetAsync(scratch, 0, sizeof(h), s) != cudaSuccess) return NSA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return NSA_ERR_CUDA;
  return h.code != NSA_OK ? h.code : h.arg_code;
}
