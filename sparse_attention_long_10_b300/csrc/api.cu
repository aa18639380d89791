// api.cu -- the extern "C" surface of libnsa.so (declared in include/nsa.h):
// argument validation, workspace carving, launch sequencing.  No allocation,
// no synchronisation except in nsa_device_status().
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "kernels.hpp"
#include "nsa.h"

using namespace nsa;

namespace {

constexpr size_t kHeader = sizeof(DeviceStatus);

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool is_pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

// Device check, cached per device id: needs an sm_100-family GPU (tcgen05).
int check_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return NSA_ERR_NO_DEVICE;
  static int cached[64];  // 0 unknown, 1 ok, 2 bad
  if (dev < 0 || dev >= 64) return NSA_ERR_NO_DEVICE;
  if (cached[dev] == 0) {
    int major = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return NSA_ERR_NO_DEVICE;
    cached[dev] = (major == 10) ? 1 : 2;
  }
  return cached[dev] == 1 ? NSA_OK : NSA_ERR_NO_DEVICE;
}

int validate_cfg(const nsa_cfg* c) {
  if (c == nullptr) return NSA_ERR_INVALID_ARG;
  if (c->B < 1 || c->T < 1 || c->H < 1 || c->G < 1 || c->dk < 1 || c->dv < 1) return NSA_ERR_INVALID_ARG;
  if (c->l < 1 || c->d < 1 || c->lsel < 1 || c->n < 1 || c->w < 1) return NSA_ERR_INVALID_ARG;
  if (c->H % c->G != 0) return NSA_ERR_INVALID_ARG;
  const int hpg = c->H / c->G;
  if (!is_pow2(hpg) || hpg > 128) return NSA_ERR_UNSUPPORTED;
  if (c->l != 32 || c->d != 16 || c->lsel != 64) return NSA_ERR_UNSUPPORTED;
  if (c->n < 3 || c->n > 32) return NSA_ERR_UNSUPPORTED;
  if (c->dk % 64 != 0 || c->dv % 64 != 0 || c->dk > 256 || c->dv > 256) return NSA_ERR_UNSUPPORTED;
  if ((long long)c->T > (1ll << 24) || (long long)c->B * c->T > (1ll << 26)) return NSA_ERR_UNSUPPORTED;
  return NSA_OK;
}

int validate_phi(const nsa_cfg* c) {
  const void* p[4] = {c->pe_k, c->pe_v, c->w_k, c->w_v};
  for (const void* x : p) {
    if (x == nullptr) return NSA_ERR_INVALID_ARG;
    if (!aligned16(x)) return NSA_ERR_MISALIGNED;
  }
  return NSA_OK;
}

int check_ptrs(std::initializer_list<const void*> ps) {
  for (const void* x : ps) {
    if (x == nullptr) return NSA_ERR_INVALID_ARG;
    if (!aligned16(x)) return NSA_ERR_MISALIGNED;
  }
  return NSA_OK;
}

int num_compressed(const nsa_cfg& c) { return c.T < c.l ? 0 : (c.T - c.l) / c.d + 1; }

// ---- workspace layout -------------------------------------------------------
struct CompressWs {
  size_t bias_k, bias_v, end;
};
CompressWs compress_ws(const nsa_cfg& c) {
  CompressWs w;
  w.bias_k = kHeader;
  w.bias_v = align_up(w.bias_k + sizeof(float) * c.dk, 256);
  w.end = align_up(w.bias_v + sizeof(float) * c.dv, 256);
  return w;
}

struct PrefillWs {
  CompressWs cw;
  size_t part, idx, end;
};

// multi-token decode: status word, then the partial and kept blocks of R rows
struct MultiWs {
  size_t part, idx, end;
};
MultiWs multi_ws(const nsa_cfg& c, int R) {
  MultiWs w;
  w.part = kHeader;
  w.idx = align_up(w.part + sizeof(float) * (size_t)c.B * R * c.H * c.dv, 256);
  w.end = align_up(w.idx + sizeof(int32_t) * (size_t)c.B * R * c.G * c.n, 256);
  return w;
}
PrefillWs prefill_ws(const nsa_cfg& c) {
  PrefillWs w;
  w.cw = compress_ws(c);
  w.part = w.cw.end;
  w.idx = align_up(w.part + sizeof(float) * (size_t)c.B * c.T * c.H * c.dv, 256);
  w.end = align_up(w.idx + sizeof(int32_t) * (size_t)c.B * c.T * c.G * c.n, 256);
  return w;
}

// shapes the prefill kernels implement (beyond validate_cfg)
int prefill_supported(const nsa_cfg& c) {
  const int hpg = c.H / c.G;
  if (hpg > 16 || c.n > 16 || (c.dv != 64 && c.dv != 128) || c.T > 65536) return NSA_ERR_UNSUPPORTED;
  if (cmp_win_smem_bytes(c) > smem_max() || sel_smem_bytes(c) > smem_max()) return NSA_ERR_UNSUPPORTED;
  return NSA_OK;
}

// shapes the dense comparison implements (beyond validate_cfg)
int full_attn_supported(const nsa_cfg& c) {
  const int hpg = c.H / c.G;
  if (hpg > 16 || (c.dv != 64 && c.dv != 128)) return NSA_ERR_UNSUPPORTED;
  if (cmp_win_smem_bytes(c, true) > smem_max()) return NSA_ERR_UNSUPPORTED;
  return NSA_OK;
}

int check_ws(void* ws, size_t ws_bytes, size_t need) {
  if (ws == nullptr) return NSA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return NSA_ERR_MISALIGNED;
  if (ws_bytes < need) return NSA_ERR_WORKSPACE;
  return NSA_OK;
}

int run_compress(const nsa_cfg& c, int layout, const void* k, const void* v, void* kc, void* vc, uint8_t* ws,
                 cudaStream_t s) {
  const CompressWs w = compress_ws(c);
  DeviceStatus* st = reinterpret_cast<DeviceStatus*>(ws);
  int rc = launch_compress_one(c, layout, k, c.dk, c.pe_k, c.w_k, kc, reinterpret_cast<float*>(ws + w.bias_k), st, s);
  if (rc != NSA_OK) return rc;
  return launch_compress_one(c, layout, v, c.dv, c.pe_v, c.w_v, vc, reinterpret_cast<float*>(ws + w.bias_v), st, s);
}

}  // namespace

namespace nsa {

int check_nsa_cfg(const nsa_cfg* cfg) { return validate_cfg(cfg); }
int check_nsa_phi(const nsa_cfg* cfg) { return cfg == nullptr ? NSA_ERR_INVALID_ARG : validate_phi(cfg); }

int ensure_smem_attr(const void* func, size_t bytes) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return NSA_ERR_NO_DEVICE;
  struct Entry {
    const void* func;
    int dev;
    size_t bytes;
  };
  constexpr int kMax = 256;
  static Entry table[kMax];
  static int used = 0;
  static std::mutex mu;
  std::lock_guard<std::mutex> lk(mu);
  int slot = -1;
  for (int i = 0; i < used; ++i)
    if (table[i].func == func && table[i].dev == dev) {
      if (table[i].bytes >= bytes) return NSA_OK;
      slot = i;
      break;
    }
  if (cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) != cudaSuccess)
    return NSA_ERR_CUDA;
  if (slot < 0) {
    if (used == kMax) return NSA_OK;   // table full: the attribute is set, only not remembered
    slot = used++;
  }
  table[slot] = Entry{func, dev, bytes};
  return NSA_OK;
}

}  // namespace nsa

extern "C" {

const char* nsa_status_string(int status) {
  switch (status) {
    case NSA_OK: return "NSA_OK";
    case NSA_ERR_INVALID_ARG: return "NSA_ERR_INVALID_ARG";
    case NSA_ERR_UNSUPPORTED: return "NSA_ERR_UNSUPPORTED";
    case NSA_ERR_MISALIGNED: return "NSA_ERR_MISALIGNED";
    case NSA_ERR_WORKSPACE: return "NSA_ERR_WORKSPACE";
    case NSA_ERR_CUDA: return "NSA_ERR_CUDA";
    case NSA_ERR_DEVICE_TIMEOUT: return "NSA_ERR_DEVICE_TIMEOUT";
    case NSA_ERR_NO_DEVICE: return "NSA_ERR_NO_DEVICE";
    default: return "NSA_ERR_UNKNOWN";
  }
}

int nsa_version(void) { return 200; }

int nsa_num_compressed(const nsa_cfg* cfg) {
  if (validate_cfg(cfg) != NSA_OK) return -1;
  return num_compressed(*cfg);
}

size_t nsa_compress_workspace_size(const nsa_cfg* cfg) {
  if (validate_cfg(cfg) != NSA_OK) return 0;
  return compress_ws(*cfg).end;
}

int nsa_compress_kv(const nsa_cfg* cfg, int layout, const void* k, const void* v, void* kc, void* vc, void* ws,
                    size_t ws_bytes, void* stream) {
  int rc = validate_cfg(cfg);
  if (rc != NSA_OK) return rc;
  if (layout != NSA_LAYOUT_BTGD && layout != NSA_LAYOUT_BGTD) return NSA_ERR_INVALID_ARG;
  if ((rc = validate_phi(cfg)) != NSA_OK) return rc;
  if ((rc = check_ptrs({k, v})) != NSA_OK) return rc;
  if (num_compressed(*cfg) > 0 && (rc = check_ptrs({kc, vc})) != NSA_OK) return rc;
  if ((rc = check_ws(ws, ws_bytes, compress_ws(*cfg).end)) != NSA_OK) return rc;
  if ((rc = check_device()) != NSA_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(ws, 0, kHeader, s) != cudaSuccess) return NSA_ERR_CUDA;
  if (num_compressed(*cfg) == 0) return NSA_OK;
  return run_compress(*cfg, layout, k, v, kc, vc, static_cast<uint8_t*>(ws), s);
}

size_t nsa_prefill_workspace_size(const nsa_cfg* cfg) {
  if (validate_cfg(cfg) != NSA_OK) return 0;
  return prefill_ws(*cfg).end;
}

int nsa_prefill_fwd(const nsa_cfg* cfg, const void* q, const void* k, const void* v, const void* gates, void* kc,
                    void* vc, void* out, int32_t* idx_out, void* ws, size_t ws_bytes, void* stream) {
  int rc = validate_cfg(cfg);
  if (rc != NSA_OK) return rc;
  const nsa_cfg& c = *cfg;
  if ((rc = prefill_supported(c)) != NSA_OK) return rc;
  const bool given = (c.flags & NSA_FLAG_KC_GIVEN) != 0;
  const int Nc = num_compressed(c);
  if (!given && (rc = validate_phi(cfg)) != NSA_OK) return rc;
  if ((rc = check_ptrs({q, k, v, gates, out})) != NSA_OK) return rc;
  if (Nc > 0 && (rc = check_ptrs({kc, vc})) != NSA_OK) return rc;
  if (idx_out != nullptr && !aligned16(idx_out)) return NSA_ERR_MISALIGNED;
  const PrefillWs w = prefill_ws(c);
  if ((rc = check_ws(ws, ws_bytes, w.end)) != NSA_OK) return rc;
  if ((rc = check_device()) != NSA_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  DeviceStatus* st = reinterpret_cast<DeviceStatus*>(wsb);
  if (cudaMemsetAsync(ws, 0, kHeader, s) != cudaSuccess) return NSA_ERR_CUDA;
  if (!given && Nc > 0 && (rc = run_compress(c, NSA_LAYOUT_BTGD, k, v, kc, vc, wsb, s)) != NSA_OK) return rc;
  void* part = wsb + w.part;
  int32_t* idx = idx_out != nullptr ? idx_out : reinterpret_cast<int32_t*>(wsb + w.idx);
  if ((rc = launch_cmp_win(c, q, k, v, kc, vc, gates, part, idx, st, s)) != NSA_OK) return rc;
  return launch_sel(c, q, k, v, gates, idx, part, out, st, s);
}

size_t nsa_prefill_bwd_workspace_size(const nsa_cfg* cfg) {
  if (validate_cfg(cfg) != NSA_OK || bwd_supported(*cfg) != NSA_OK) return 0;
  return bwd_ws(*cfg, kHeader).end;
}

int nsa_prefill_bwd(const nsa_cfg* cfg, const void* q, const void* k, const void* v, const void* gates,
                    const void* kc, const void* vc, const int32_t* idx, const float* slc_lse, const float* slc_o,
                    const void* dout, float* dq, float* dk, float* dv, float* dgates, float* dw_k, float* dw_v,
                    float* dpe_k, float* dpe_v, void* ws, size_t ws_bytes, void* stream) {
  int rc = validate_cfg(cfg);
  if (rc != NSA_OK) return rc;
  const nsa_cfg& c = *cfg;
  if ((rc = bwd_supported(c)) != NSA_OK) return rc;
  if ((rc = validate_phi(cfg)) != NSA_OK) return rc;
  if ((rc = check_ptrs({q, k, v, gates, idx, dout, dq, dk, dv, dgates, dw_k, dw_v, dpe_k, dpe_v})) != NSA_OK)
    return rc;
  if (num_compressed(c) > 0 && (rc = check_ptrs({kc, vc})) != NSA_OK) return rc;
  if ((slc_lse == nullptr) != (slc_o == nullptr)) return NSA_ERR_INVALID_ARG;
  if (slc_lse != nullptr && (rc = check_ptrs({slc_lse, slc_o})) != NSA_OK) return rc;
  const BwdWs w = bwd_ws(c, kHeader);
  if ((rc = check_ws(ws, ws_bytes, w.end)) != NSA_OK) return rc;
  if ((rc = check_device()) != NSA_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(ws, 0, kHeader, s) != cudaSuccess) return NSA_ERR_CUDA;
  BwdPtrs p{q, k, v, gates, kc, vc, dout, idx, slc_lse, slc_o, dq, dk, dv, dgates, dw_k, dw_v, dpe_k, dpe_v};
  return launch_prefill_bwd(c, p, static_cast<uint8_t*>(ws), w, s);
}

int nsa_prefill_fwd_train(const nsa_cfg* cfg, const void* q, const void* k, const void* v, const void* gates,
                          void* kc, void* vc, void* out, int32_t* idx_out, float* slc_lse, float* slc_o, void* ws,
                          size_t ws_bytes, void* stream) {
  int rc = validate_cfg(cfg);
  if (rc != NSA_OK) return rc;
  const nsa_cfg& c = *cfg;
  if ((rc = prefill_supported(c)) != NSA_OK) return rc;
  const bool given = (c.flags & NSA_FLAG_KC_GIVEN) != 0;
  const int Nc = num_compressed(c);
  if (!given && (rc = validate_phi(cfg)) != NSA_OK) return rc;
  if ((rc = check_ptrs({q, k, v, gates, out, idx_out, slc_lse, slc_o})) != NSA_OK) return rc;
  if (Nc > 0 && (rc = check_ptrs({kc, vc})) != NSA_OK) return rc;
  const PrefillWs w = prefill_ws(c);
  if ((rc = check_ws(ws, ws_bytes, w.end)) != NSA_OK) return rc;
  if ((rc = check_device()) != NSA_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  DeviceStatus* st = reinterpret_cast<DeviceStatus*>(wsb);
  if (cudaMemsetAsync(ws, 0, kHeader, s) != cudaSuccess) return NSA_ERR_CUDA;
  if (!given && Nc > 0 && (rc = run_compress(c, NSA_LAYOUT_BTGD, k, v, kc, vc, wsb, s)) != NSA_OK) return rc;
  void* part = wsb + w.part;
  if ((rc = launch_cmp_win(c, q, k, v, kc, vc, gates, part, idx_out, st, s)) != NSA_OK) return rc;
  return launch_sel(c, q, k, v, gates, idx_out, part, out, st, s, QueryRows(), slc_lse, slc_o);
}

size_t nsa_full_attn_workspace_size(const nsa_cfg* cfg) {
  if (validate_cfg(cfg) != NSA_OK || full_attn_supported(*cfg) != NSA_OK) return 0;
  return kHeader;
}

int nsa_full_attn_fwd(const nsa_cfg* cfg, const void* q, const void* k, const void* v, void* out, void* ws,
                      size_t ws_bytes, void* stream) {
  int rc = validate_cfg(cfg);
  if (rc != NSA_OK) return rc;
  const nsa_cfg& c = *cfg;
  if ((rc = full_attn_supported(c)) != NSA_OK) return rc;
  if ((rc = check_ptrs({q, k, v, out})) != NSA_OK) return rc;
  if ((rc = check_ws(ws, ws_bytes, kHeader)) != NSA_OK) return rc;
  if ((rc = check_device()) != NSA_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(ws, 0, kHeader, s) != cudaSuccess) return NSA_ERR_CUDA;
  return launch_cmp_win(c, q, k, v, nullptr, nullptr, nullptr, out, nullptr, reinterpret_cast<DeviceStatus*>(ws), s,
                        true);
}

size_t nsa_decode_multi_workspace_size(const nsa_cfg* cfg, int m) {
  if (validate_cfg(cfg) != NSA_OK || prefill_supported(*cfg) != NSA_OK || m < 1 || m > cfg->T) return 0;
  return multi_ws(*cfg, m).end;
}

int nsa_decode_multi(const nsa_cfg* cfg, int m, const void* q, const void* kcache, const void* vcache,
                     const void* kc, const void* vc, const void* gates, void* out, int32_t* idx_out, void* ws,
                     size_t ws_bytes, void* stream) {
  int rc = validate_cfg(cfg);
  if (rc != NSA_OK) return rc;
  const nsa_cfg& c = *cfg;
  if (m < 1 || m > c.T) return NSA_ERR_INVALID_ARG;
  if ((rc = prefill_supported(c)) != NSA_OK) return rc;
  if ((rc = check_ptrs({q, kcache, vcache, gates, out})) != NSA_OK) return rc;
  if (num_compressed(c) > 0 && (rc = check_ptrs({kc, vc})) != NSA_OK) return rc;
  if (idx_out != nullptr && !aligned16(idx_out)) return NSA_ERR_MISALIGNED;
  const MultiWs w = multi_ws(c, m);
  if ((rc = check_ws(ws, ws_bytes, w.end)) != NSA_OK) return rc;
  if ((rc = check_device()) != NSA_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  DeviceStatus* st = reinterpret_cast<DeviceStatus*>(wsb);
  if (cudaMemsetAsync(ws, 0, kHeader, s) != cudaSuccess) return NSA_ERR_CUDA;
  QueryRows rows;
  rows.R = m;
  rows.qoff = c.T - m;
  rows.head_major = true;
  void* part = wsb + w.part;
  int32_t* idx = idx_out != nullptr ? idx_out : reinterpret_cast<int32_t*>(wsb + w.idx);
  if ((rc = launch_cmp_win(c, q, kcache, vcache, kc, vc, gates, part, idx, st, s, false, rows)) != NSA_OK) return rc;
  return launch_sel(c, q, kcache, vcache, gates, idx, part, out, st, s, rows);
}

size_t nsa_decode_workspace_size(const nsa_cfg* cfg) {
  if (validate_cfg(cfg) != NSA_OK || decode_supported(*cfg) != NSA_OK) return 0;
  return decode_ws_bytes(*cfg);
}

int nsa_decode_step(const nsa_cfg* cfg, const void* q, const void* kcache, const void* vcache, const void* kc,
                    const void* vc, const int32_t* seq_lens, const void* gates, void* out, int32_t* idx_out,
                    void* ws, size_t ws_bytes, void* stream) {
  int rc = validate_cfg(cfg);
  if (rc != NSA_OK) return rc;
  const nsa_cfg& c = *cfg;
  if ((rc = decode_supported(c)) != NSA_OK) return rc;
  if ((rc = check_ptrs({q, kcache, vcache, gates, out})) != NSA_OK) return rc;
  if (num_compressed(c) > 0 && (rc = check_ptrs({kc, vc})) != NSA_OK) return rc;
  if (idx_out != nullptr && !aligned16(idx_out)) return NSA_ERR_MISALIGNED;
  if (seq_lens != nullptr && (reinterpret_cast<uintptr_t>(seq_lens) & 3u) != 0) return NSA_ERR_MISALIGNED;
  if ((rc = check_ws(ws, ws_bytes, decode_ws_bytes(c))) != NSA_OK) return rc;
  if ((rc = check_device()) != NSA_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(ws, 0, decode_zero_bytes(c), s) != cudaSuccess) return NSA_ERR_CUDA;
  return launch_decode(c, q, kcache, vcache, kc, vc, seq_lens, gates, out, idx_out, static_cast<uint8_t*>(ws), s);
}

int validate_dsa(const dsa_cfg* c) {
  if (c == nullptr) return NSA_ERR_INVALID_ARG;
  if (c->B < 1 || c->T < 1 || c->HI < 1 || c->dI < 1 || c->H < 1 || c->dk < 1 || c->dv < 1 || c->topk < 1)
    return NSA_ERR_INVALID_ARG;
  return dsa_supported(*c);
}

size_t dsa_decode_workspace_size(const dsa_cfg* cfg) {
  if (validate_dsa(cfg) != NSA_OK) return 0;
  return dsa_ws_bytes(*cfg);
}

int dsa_decode_step(const dsa_cfg* cfg, const void* qI, const void* wI, const void* kI, const void* q,
                    const void* k, const void* v, const int32_t* seq_lens, void* out, int32_t* idx_out, void* ws,
                    size_t ws_bytes, void* stream) {
  int rc = validate_dsa(cfg);
  if (rc != NSA_OK) return rc;
  if ((rc = check_ptrs({qI, wI, kI, q, k, out})) != NSA_OK) return rc;
  // v == NULL: values are the first dv columns of the key rows (latent KV)
  if (v == nullptr ? cfg->dv > cfg->dk : !aligned16(v)) return v == nullptr ? NSA_ERR_INVALID_ARG : NSA_ERR_MISALIGNED;
  if (idx_out != nullptr && !aligned16(idx_out)) return NSA_ERR_MISALIGNED;
  if (seq_lens != nullptr && (reinterpret_cast<uintptr_t>(seq_lens) & 3u) != 0) return NSA_ERR_MISALIGNED;
  if ((rc = check_ws(ws, ws_bytes, dsa_ws_bytes(*cfg))) != NSA_OK) return rc;
  if ((rc = check_device()) != NSA_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(ws, 0, dsa_zero_bytes(*cfg), s) != cudaSuccess) return NSA_ERR_CUDA;
  return launch_dsa(*cfg, qI, wI, kI, q, k, v, seq_lens, out, idx_out, static_cast<uint8_t*>(ws), s);
}

// The prefill form runs the decode kernels over B*T query rows.
static bool prefill_rows_cfg(const dsa_cfg* cfg, dsa_cfg* rows) {
  if (cfg == nullptr || cfg->B < 1 || cfg->T < 1 || (long long)cfg->B * cfg->T > 65535) return false;
  *rows = *cfg;
  rows->B = cfg->B * cfg->T;
  return true;
}

size_t dsa_prefill_workspace_size(const dsa_cfg* cfg) {
  dsa_cfg rc;
  if (!prefill_rows_cfg(cfg, &rc) || validate_dsa(&rc) != NSA_OK) return 0;
  return dsa_ws_bytes(rc);
}

int dsa_prefill_fwd(const dsa_cfg* cfg, const void* qI, const void* wI, const void* kI, const void* q, const void* k,
                    const void* v, void* out, int32_t* idx_out, void* ws, size_t ws_bytes, void* stream) {
  int rc = validate_dsa(cfg);
  if (rc != NSA_OK) return rc;
  dsa_cfg rows;
  if (!prefill_rows_cfg(cfg, &rows)) return NSA_ERR_UNSUPPORTED;
  if ((rc = validate_dsa(&rows)) != NSA_OK) return rc;
  if ((rc = check_ptrs({qI, wI, kI, q, k, out})) != NSA_OK) return rc;
  // v == NULL: values are the first dv columns of the key rows (latent KV)
  if (v == nullptr ? cfg->dv > cfg->dk : !aligned16(v)) return v == nullptr ? NSA_ERR_INVALID_ARG : NSA_ERR_MISALIGNED;
  if (idx_out != nullptr && !aligned16(idx_out)) return NSA_ERR_MISALIGNED;
  if ((rc = check_ws(ws, ws_bytes, dsa_ws_bytes(rows))) != NSA_OK) return rc;
  if ((rc = check_device()) != NSA_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(ws, 0, dsa_zero_bytes(rows), s) != cudaSuccess) return NSA_ERR_CUDA;
  return launch_dsa(rows, qI, wI, kI, q, k, v, nullptr, out, idx_out, static_cast<uint8_t*>(ws), s, cfg->T);
}

int nsa_device_status(void* ws, void* stream) {
  if (ws == nullptr) return NSA_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  DeviceStatus h;
  if (cudaMemcpyAsync(&h, ws, sizeof(h), cudaMemcpyDeviceToHost, s) != cudaSuccess) return NSA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return NSA_ERR_CUDA;
  if (cudaMemsetAsync(ws, 0, sizeof(h), s) != cudaSuccess) return NSA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return NSA_ERR_CUDA;
  return h.code != NSA_OK ? h.code : h.arg_code;
}

}  // extern "C"
