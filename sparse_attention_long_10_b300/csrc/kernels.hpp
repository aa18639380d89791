// kernels.hpp -- host-side launchers of the NSA / DSA kernels (internal to
// libnsa.so; the public surface is include/nsa.h).
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "nsa.h"

namespace nsa {

struct DeviceStatus;

// Largest dynamic shared memory any kernel of the library asks for (bytes).
constexpr size_t smem_max() { return 232448; }  // 227 KB

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Raises ``func``'s dynamic shared-memory limit to at least ``bytes`` on the
// current device.  A function attribute belongs to one device context, so the
// setting is remembered per (function, device); thread-safe.  Returns a status.
int ensure_smem_attr(const void* func, size_t bytes);

// The argument rules every NSA entry point applies to ``cfg`` and to its phi
// parameters (api.cu); each returns NSA_OK or the status the call returns.
int check_nsa_cfg(const nsa_cfg* cfg);
int check_nsa_phi(const nsa_cfg* cfg);

// ---- compression (compress.cu)
size_t compress_smem_bytes(int N);
// One of K or V: X in ``layout``, dX = head dim = output dim.
int launch_compress_one(const nsa_cfg& c, int layout, const void* X, int dX, const void* pe, const void* W,
                        void* out, float* bias_ws, DeviceStatus* st, cudaStream_t stream);

// ---- prefill (prefill_cmp_win.cu, prefill_sel.cu)
// Query rows of a prefill-kernel launch.  Default: one row per position
// (R = T, qoff = 0, k/v token-major [B,T,G,d]).  A multi-token decode runs
// R rows at positions qoff .. qoff+R-1 against head-major caches [B,G,T,d];
// q, gates, out, the partial and idx are then addressed by row.
struct QueryRows {
  int R = 0;          // 0: T
  int qoff = 0;
  bool head_major = false;
};

size_t cmp_win_smem_bytes(const nsa_cfg& c, bool dense = false);
size_t sel_smem_bytes(const nsa_cfg& c);
// compressed attention + block scores + top-n + window; writes
// part = g_cmp*O_cmp + g_win*O_win (fp32 [B,T,H,dv]) and idx [B,T,G,n].
// dense: exact causal full attention of q over k/v written to ``part``
// (no compressed branch, no selection, gates unused).
int launch_cmp_win(const nsa_cfg& c, const void* q, const void* k, const void* v, const void* kc, const void* vc,
                   const void* gates, void* part, int32_t* idx, DeviceStatus* st, cudaStream_t s,
                   bool dense = false, const QueryRows& rows = QueryRows());
// selected attention; out = part + g_slc*O_slc.  slc_lse / slc_o (both or
// neither, token-major prefill only): also write the branch's log2-domain
// log-sum-exp [B,T,H] and O_slc [B,T,H,dv] (fp32) for the backward pass.
int launch_sel(const nsa_cfg& c, const void* q, const void* k, const void* v, const void* gates, const int32_t* idx,
               const void* part, void* out, DeviceStatus* st, cudaStream_t s,
               const QueryRows& rows = QueryRows(), float* slc_lse = nullptr, float* slc_o = nullptr);

// ---- decode (decode.cu)
int decode_supported(const nsa_cfg& c);
size_t decode_ws_bytes(const nsa_cfg& c);
// bytes at the start of the decode workspace (status word + counters) that
// must be zero when the step starts
size_t decode_zero_bytes(const nsa_cfg& c);
// lens: nullable device array [B] of sequence lengths (each in [1, c.T])
int launch_decode(const nsa_cfg& c, const void* q, const void* kcache, const void* vcache, const void* kc,
                  const void* vc, const int32_t* lens, const void* gates, void* out, int32_t* idx_out, uint8_t* ws,
                  cudaStream_t s);

// ---- DSA decode (dsa.cu)
int dsa_supported(const dsa_cfg& c);
size_t dsa_ws_bytes(const dsa_cfg& c);
size_t dsa_zero_bytes(const dsa_cfg& c);
// lens: nullable device array [B] of context lengths (each in [1, c.T])
// c.B is the number of query rows; rows_per_seq = 1 for the decode step (one
// row per sequence), T for the prefill (row r is position r mod T of sequence
// r / T).
int launch_dsa(const dsa_cfg& c, const void* qI, const void* wI, const void* kI, const void* q, const void* k,
               const void* v, const int32_t* lens, void* out, int32_t* idx_out, uint8_t* ws, cudaStream_t s,
               int rows_per_seq = 1);

// ---- prefill backward (backward.cu)
struct BwdPtrs {
  const void *q, *k, *v, *gates, *kc, *vc, *dout;
  const int32_t* idx;
  const float *slc_lse, *slc_o;   // nullable: the forward's saved selected-branch statistics
  float *dq, *dk, *dv, *dgates, *dw_k, *dw_v, *dpe_k, *dpe_v;
};
// byte offsets of the backward's scratch inside the workspace; [zero_begin,
// zero_end) and [dkc, zero_begin) are cleared by every call
struct BwdWs {
  size_t lse, dgw, dkc, dvc, zero_begin, cnt, fill, csum, zero_end, offs, nunits, inv, units[3], end;
  size_t cap[3];
};
int bwd_supported(const nsa_cfg& c);
BwdWs bwd_ws(const nsa_cfg& c, size_t header);
int launch_prefill_bwd(const nsa_cfg& c, const BwdPtrs& p, uint8_t* ws, const BwdWs& w, cudaStream_t s);

}  // namespace nsa
