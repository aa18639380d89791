/*
 * nsa.h -- C ABI of libnsa.so: the forward hot path of Native Sparse Attention
 * (NSA) and of a DSA-style indexed sparse decode on one NVIDIA B300 (sm_103a).
 *
 * Sources (cited by page title and section):
 *  [P2] "AI 모델의 '긴 문장 처리' 한계 돌파, 딥시크의 새 어텐션 기술 화제", section II:
 *       three parallel attention paths (compressed coarse tokens, selected fine
 *       tokens, sliding window); l=32, d=16, l'=64, n=16 (1 initial + 2 local
 *       blocks included), w=512.  Section III.3: a 64k decode step reads 5,632
 *       tokens instead of 65,536.
 *  [P3] deepdaiv newsletter no. 82, paragraphs on token compression, token
 *       selection (block importance from the compressed tokens, blockwise
 *       selection for contiguous memory access) and the sliding window.
 *  [P4] "딥시크 희소 어텐션 DSA 원리: 라이트닝 인덱서와 상위 2048 토큰 선택 구조 해설",
 *       "쉽게 이해하기": ReLU-weighted indexer with keys shared by its heads,
 *       top-2048 selection, softmax over the selected set only.
 *
 * Conventions for every call
 *  - All tensors are bf16, row-major, dense, in device memory of the current
 *    CUDA device; base pointers must be 16-byte aligned.  Index outputs are
 *    int32.  Query head h uses KV head floor(h / (H/G)).
 *  - The caller owns every buffer and the stream.  The library never
 *    allocates, frees or synchronises; scratch memory is the caller's
 *    workspace ``ws`` of at least the size the matching *_workspace_size()
 *    call returns (256-byte aligned).
 *  - Calls are asynchronous on ``stream`` (a cudaStream_t passed as void*;
 *    NULL = legacy default stream).  Host-side validation runs first: on any
 *    invalid argument the call returns an error and launches nothing.
 *  - Kernels never trap.  Every device-side wait is bounded; a wait that
 *    runs out records NSA_ERR_DEVICE_TIMEOUT in the workspace status word,
 *    which nsa_device_status() reads back.
 *  - No C++ exception crosses this boundary.
 */
#ifndef NSA_H_
#define NSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---------------------------------------------------------------- status */
enum nsa_status_code {
  NSA_OK = 0,
  NSA_ERR_INVALID_ARG = 1,     /* null pointer, non-positive size, bad enum  */
  NSA_ERR_UNSUPPORTED = 2,     /* shape outside what the kernels implement   */
  NSA_ERR_MISALIGNED = 3,      /* a pointer not 16-byte (ws: 256-byte) aligned */
  NSA_ERR_WORKSPACE = 4,       /* ws_bytes smaller than the required size    */
  NSA_ERR_CUDA = 5,            /* a CUDA runtime/driver call failed          */
  NSA_ERR_DEVICE_TIMEOUT = 6,  /* a bounded device-side wait ran out         */
  NSA_ERR_NO_DEVICE = 7        /* no usable sm_100-family device             */
};

/* Human-readable name of a status code (static string, never NULL). */
const char* nsa_status_string(int status);

/* ABI version of this header (major*100 + minor). */
int nsa_version(void);

/* ---------------------------------------------------------------- NSA config */
/* Flags for nsa_cfg.flags */
#define NSA_FLAG_KC_GIVEN 1u   /* nsa_prefill_fwd: kc/vc already hold the compressed
                                  cache; skip the compression step */
#define NSA_FLAG_TEST_STALL 0x80000000u
                               /* test hook of the failure path (no counterpart on the
                                  pages): in the compression step the first CTA's producer
                                  never signals one pipeline stage, so a bounded device
                                  wait runs out after 0.5 s.  The call then records
                                  NSA_ERR_DEVICE_TIMEOUT (nsa_device_status), its outputs
                                  are not valid, and the next call on the same workspace
                                  runs normally.  Never set in normal use. */

typedef struct nsa_cfg {
  int B;        /* sequences                                            */
  int T;        /* tokens per sequence (decode: cache length; query at T-1) */
  int H;        /* query heads                                          */
  int G;        /* KV heads (GQA groups); H % G == 0                    */
  int dk;       /* query/key head dim                                   */
  int dv;       /* value head dim                                       */
  int l;        /* compression block length        (pages: 32)          */
  int d;        /* compression stride              (pages: 16)          */
  int lsel;     /* selection block length l'       (pages: 64)          */
  int n;        /* selected blocks per query       (pages: 16)          */
  int w;        /* sliding-window length           (pages: 512)         */
  float scale;  /* softmax scale of all three branches; <= 0 -> 1/sqrt(dk) */
  unsigned flags;
  /* compression map phi [P2 II.1, P3]: block i of one KV head is
     flatten(X[d*i : d*i+l] + PE) @ W.  Device pointers, bf16:           */
  const void* pe_k;  /* [l, dk]                                          */
  const void* pe_v;  /* [l, dv]                                          */
  const void* w_k;   /* [l*dk, dk]                                       */
  const void* w_v;   /* [l*dv, dv]                                       */
} nsa_cfg;

/* Supported shapes: l=32, d=16, lsel=64, 3 <= n <= 32, 1 <= w,
   dk and dv multiples of 64 with dk <= 256 and dv <= 256, H/G a power of two
   between 1 and 128, T >= 1, B >= 1.  Anything else -> NSA_ERR_UNSUPPORTED. */

/* Layout of the K/V tensors handed to nsa_compress_kv */
#define NSA_LAYOUT_BTGD 0   /* [B, T, G, d]  (prefill inputs)        */
#define NSA_LAYOUT_BGTD 1   /* [B, G, T, d]  (head-major decode cache) */

/* Number of compressed blocks per KV head: floor((T-l)/d)+1, or 0 if T < l. */
int nsa_num_compressed(const nsa_cfg* cfg);

/* Workspace bytes needed by nsa_compress_kv / nsa_prefill_fwd /
   nsa_decode_step for this cfg (0 on an invalid cfg). */
size_t nsa_compress_workspace_size(const nsa_cfg* cfg);
size_t nsa_prefill_workspace_size(const nsa_cfg* cfg);
size_t nsa_decode_workspace_size(const nsa_cfg* cfg);

/*
 * nsa_compress_kv -- token compression [P2 II.1; P3, token compression]
 *   kc[b,g,i,:] = bf16( flatten(k[b, d*i : d*i+l, g, :] + pe_k) @ w_k )
 *   vc[b,g,i,:] = bf16( flatten(v[b, d*i : d*i+l, g, :] + pe_v) @ w_v )
 * for i < Nc = nsa_num_compressed(cfg).  Accumulation is fp32; each output
 * is rounded once to bf16.
 *   k, v    : layout NSA_LAYOUT_BTGD ([B,T,G,dk] / [B,T,G,dv]) or
 *             NSA_LAYOUT_BGTD ([B,G,T,dk] / [B,G,T,dv])
 *   kc, vc  : out, [B, G, Nc, dk] / [B, G, Nc, dv]
 *   phi parameters come from cfg (pe_k, pe_v, w_k, w_v).
 */
int nsa_compress_kv(const nsa_cfg* cfg, int layout, const void* k, const void* v,
                    void* kc, void* vc, void* ws, size_t ws_bytes, void* stream);

/*
 * nsa_compress_kv_noalloc -- the same computation as nsa_compress_kv, for
 * callers that cannot allocate device memory when they compress: a serving
 * loop whose device memory is planned once and never grows, or an embedding
 * program that is handed tensor pointers but owns no device allocator (and
 * avoids cudaMalloc, which can synchronise the device).  It takes no
 * workspace and allocates nothing: its scratch (status word + the two fp32
 * flatten(PE) @ W bias vectors, at most 2304 bytes) lives in a fixed static
 * device array of the library, held by every GPU that loads it until exit.
 * The pages have no counterpart of this entry point.
 *   - The first call on a device resolves that array's device address (with
 *     the device current) and caches it; make that first call before any
 *     stream capture.
 *   - Every call shares the one array: calls that can overlap on the GPU
 *     (different streams without ordering) race on it.  Each call clears the
 *     status word before it launches.
 *   - Arguments, outputs and argument errors as nsa_compress_kv; a cfg whose
 *     biases do not fit the array returns NSA_ERR_WORKSPACE (unreachable
 *     while dk, dv <= 256 is a cfg rule).
 *   - The status word is read back with nsa_compress_kv_noalloc_status().
 */
int nsa_compress_kv_noalloc(const nsa_cfg* cfg, int layout, const void* k, const void* v,
                            void* kc, void* vc, void* stream);

/*
 * nsa_compress_kv_noalloc_status -- the status word of the fixed array that
 * nsa_compress_kv_noalloc uses, on the current device: synchronises
 * ``stream``, returns the code the kernels of the last no-alloc call
 * recorded (NSA_OK if none, NSA_ERR_DEVICE_TIMEOUT if a bounded wait ran out
 * and the outputs were left unwritten) and clears it.  Like the call itself
 * it allocates nothing.  No counterpart on the pages.
 */
int nsa_compress_kv_noalloc_status(void* stream);

/*
 * nsa_prefill_fwd -- NSA forward over whole sequences [P2 II; P3].
 * For every sequence b, query position t and head h (group g):
 *   compressed : softmax over the complete compressed blocks i (d*i+l-1 <= t)
 *   scores     : S[t,g,j] = sum_{h in g} sum_i w(i,j) p_cmp[t,h,i], w = shared
 *                d-chunks of compressed block i and selection block j
 *   selection  : blocks 0, j_t, j_t-1 (j_t = t/lsel) plus the top n-3 other
 *                causal blocks by S, ties to the lower index (all blocks if
 *                j_t < n); attention over their tokens s <= t
 *   window     : attention over s in (t-w, t]
 *   out[b,t,h,:] = g_cmp*O_cmp + g_slc*O_slc + g_win*O_win
 *   q     : [B,T,H,dk]     k : [B,T,G,dk]     v : [B,T,G,dv]
 *   gates : [B,T,H,3] (cmp, slc, win)
 *   kc,vc : [B,G,Nc,dk] / [B,G,Nc,dv]; written by this call (compression
 *           step) unless cfg->flags has NSA_FLAG_KC_GIVEN, then read only
 *   out   : [B,T,H,dv]
 *   idx_out (nullable): [B,T,G,n] int32, the kept blocks ascending, -1 padded
 */
int nsa_prefill_fwd(const nsa_cfg* cfg, const void* q, const void* k, const void* v,
                    const void* gates, void* kc, void* vc, void* out, int32_t* idx_out,
                    void* ws, size_t ws_bytes, void* stream);

/*
 * nsa_prefill_fwd_train -- nsa_prefill_fwd that also saves what the backward
 * pass reads of the selected branch: its log-sum-exp and its output before
 * the gate.
 *   idx_out : [B,T,G,n] int32 (required here)
 *   slc_lse : out, fp32 [B,T,H]: the row's log-sum-exp in base 2 over its
 *             kept keys, m + log2(sum_j 2^(u_j - m)) with u_j = s_j * scale *
 *             log2(e) and m = max_j u_j
 *   slc_o   : out, fp32 [B,T,H,dv]: O_slc = sum_j P_j v_j
 * Everything else as nsa_prefill_fwd (same workspace size).
 */
int nsa_prefill_fwd_train(const nsa_cfg* cfg, const void* q, const void* k, const void* v,
                          const void* gates, void* kc, void* vc, void* out, int32_t* idx_out,
                          float* slc_lse, float* slc_o, void* ws, size_t ws_bytes, void* stream);

/*
 * nsa_prefill_bwd -- NSA backward pass over whole sequences: the gradients of
 * sum(dout * out) for out = nsa_prefill_fwd(...) [P2 II; the pages' training
 * figure, 6.0x faster than full attention at 64k, P2 III.3].  The pages give
 * no backward formula; these are the gradients of the forward under three
 * readings: the kept blocks idx are constants (top-n has no gradient), the
 * bf16 rounding of the compressed cache passes gradients unchanged, and the
 * gradients of pe_k / pe_v / w_k / w_v sum over every sequence and KV head.
 * Per branch (softmax attention, P = softmax(scale q K^T), dO_b = g_b dout):
 *   dV_j += P_j dO_b,  dS_j = P_j (dO_b . V_j - dO_b . O_b),
 *   dq += scale sum_j dS_j K_j,  dK_j += scale dS_j q,  dgates_b = dout . O_b,
 * and the compressed branch's dKc / dVc flow through the compression map
 * (dW += flatten(X_i + PE)^T dXc_i, dX[16 i + r] += (dXc_i W^T)[r], dPE).
 *   q, k, v, gates, kc, vc : the forward's inputs and its compressed cache
 *   idx   : [B,T,G,n] int32, the forward's kept blocks (its idx_out)
 *   slc_lse, slc_o (nullable, both or neither): the selected branch's
 *           statistics saved by nsa_prefill_fwd_train; given, the backward
 *           skips its own statistics pass over the kept blocks (dgates of
 *           that branch is then dout . slc_o, with the forward's bf16 P)
 *   dout  : [B,T,H,dv] bf16, the upstream gradient
 *   dq    : out, fp32 [B,T,H,dk]      dk, dv : out, fp32 [B,T,G,dk] / [B,T,G,dv]
 *   dgates: out, fp32 [B,T,H,3]       dw_k, dw_v : out, fp32 [l*dk,dk] / [l*dv,dv]
 *   dpe_k, dpe_v : out, fp32 [l,dk] / [l,dv]
 *   ws    : nsa_prefill_bwd_workspace_size(cfg) bytes
 * Every output is overwritten.  dk, dv, dw_* are sums of fp32 reductions in
 * an order that varies between runs (the last bits can differ).
 * Supported: H/G <= 16, n <= 16, dk 128 or 192, dv 64 or 128, T <= 65536,
 * 16*B*G <= 65535 (cfg rules as nsa_prefill_fwd).
 */
size_t nsa_prefill_bwd_workspace_size(const nsa_cfg* cfg);
int nsa_prefill_bwd(const nsa_cfg* cfg, const void* q, const void* k, const void* v,
                    const void* gates, const void* kc, const void* vc, const int32_t* idx,
                    const float* slc_lse, const float* slc_o,
                    const void* dout, float* dq, float* dk, float* dv, float* dgates,
                    float* dw_k, float* dw_v, float* dpe_k, float* dpe_v,
                    void* ws, size_t ws_bytes, void* stream);

/*
 * nsa_decode_step -- one new token per sequence [P2 II, III.3]: row t = len-1
 * of the prefill definition, read from the caches (the cache already holds
 * the new token).  Per KV head it reads the visible compressed entries, the
 * n selected blocks and the w-token window of its own sequence.
 *   q      : [B,H,dk]        gates : [B,H,3]
 *   kcache : [B,G,T,dk]      vcache : [B,G,T,dv]   (head-major; T = capacity)
 *   kc, vc : [B,G,Nc,dk] / [B,G,Nc,dv] compressed caches at capacity T
 *            (nsa_compress_kv with NSA_LAYOUT_BGTD; entry i only depends on
 *            tokens 16i .. 16i+31, so a shorter sequence uses a prefix)
 *   seq_lens (nullable): device int32 [B], sequence b's length len_b in
 *            [1, T]; NULL means every sequence has length T.  The values are
 *            read on the device: a length outside [1, T] is recorded as
 *            NSA_ERR_INVALID_ARG in the workspace status word
 *            (nsa_device_status) and that sequence is read as empty (its
 *            out is zero, its idx_out all -1); the others are unaffected.
 *   out    : [B,H,dv]
 *   idx_out (nullable): [B,G,n] int32
 */
int nsa_decode_step(const nsa_cfg* cfg, const void* q, const void* kcache, const void* vcache,
                    const void* kc, const void* vc, const int32_t* seq_lens, const void* gates,
                    void* out, int32_t* idx_out, void* ws, size_t ws_bytes, void* stream);

/*
 * nsa_full_attn_fwd -- exact causal full attention, the dense comparison the
 * pages measure NSA against (9.0x forward at 64k, [P2] section III.3):
 *   out[b,t,h,:] = softmax_{s <= t}(q[b,t,h,:] . k[b,s,g,:] * scale) @ v[b,:,g,:]
 * with g = floor(h / (H/G)) and scale from cfg.  It runs the window path of
 * the prefill kernel with a window covering the whole prefix, no compressed
 * branch and gate 1.  Only B, T, H, G, dk, dv and scale of cfg are used (the
 * rest must still pass the cfg rules); phi and gates are not read.
 *   q [B,T,H,dk]   k [B,T,G,dk]   v [B,T,G,dv]   out [B,T,H,dv]
 *   ws: nsa_full_attn_workspace_size(cfg) bytes (the status word).
 * Supported: H/G <= 16, dv 64 or 128.
 */
size_t nsa_full_attn_workspace_size(const nsa_cfg* cfg);
int nsa_full_attn_fwd(const nsa_cfg* cfg, const void* q, const void* k, const void* v, void* out,
                      void* ws, size_t ws_bytes, void* stream);

/*
 * nsa_decode_multi -- m new tokens per sequence at once (a chunk of tokens,
 * or draft tokens checked together): rows t = T-m .. T-1 of the prefill
 * definition [P2 II; P3], each query with its own compressed attention,
 * block scores, top-n selection and window, read from the caches that
 * already hold the m tokens.  The 128-row tiles of the compressed and window
 * branches cover 128/(H/G) of the m queries at once, so the chunk shares
 * every compressed and window K/V tile it reads.
 *   q      : [B,m,H,dk]      gates : [B,m,H,3]     out : [B,m,H,dv]
 *   kcache : [B,G,T,dk]      vcache : [B,G,T,dv]   (head-major, T = length)
 *   kc, vc : [B,G,Nc,dk] / [B,G,Nc,dv] compressed caches (nsa_compress_kv,
 *            NSA_LAYOUT_BGTD); read only
 *   idx_out (nullable): [B,m,G,n] int32
 *   ws     : nsa_decode_multi_workspace_size(cfg, m) bytes
 * 1 <= m <= T; shapes as nsa_prefill_fwd (H/G <= 16, n <= 16, dv 64 or 128,
 * T <= 65536).
 */
size_t nsa_decode_multi_workspace_size(const nsa_cfg* cfg, int m);
int nsa_decode_multi(const nsa_cfg* cfg, int m, const void* q, const void* kcache, const void* vcache,
                     const void* kc, const void* vc, const void* gates, void* out, int32_t* idx_out,
                     void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------- DSA */
typedef struct dsa_cfg {
  int B;       /* batch rows (one query token each, at position T-1)  */
  int T;       /* context length                                      */
  int HI;      /* indexer heads                                       */
  int dI;      /* indexer head dim                                    */
  int H;       /* attention query heads (one shared KV)               */
  int dk;      /* key dim                                             */
  int dv;      /* value dim                                           */
  int topk;    /* positions kept per query (pages: 2048)              */
  float scale; /* <= 0 -> 1/sqrt(dk)                                  */
} dsa_cfg;
/* Supported: 1 <= HI <= 8, dI in {64, 128, 256}, 1 <= H <= 16, dk a multiple
   of 64 up to 640, dv in {64, 128, 256, 512}, 1 <= topk, B <= 65535,
   T <= 2^28; every device pointer 16-byte aligned.  Anything else returns
   NSA_ERR_UNSUPPORTED (shape) or NSA_ERR_INVALID_ARG (pointer). */

size_t dsa_decode_workspace_size(const dsa_cfg* cfg);

/*
 * dsa_decode_step -- indexed sparse decode [P4, "쉽게 이해하기"]; row b's
 * context holds T_b tokens and its query sits at T_b - 1:
 *   I[b,s]   = sum_h wI[b,h] * max(0, qI[b,h,:] . kI[b,s,:])    for s < T_b
 *   keep     = the min(topk,T_b) positions of largest fp32 I, ties to the lower s
 *   out[b,h] = softmax_{s in keep}(q[b,h,:] . k[b,s,:] * scale) @ v[b,keep,:]
 *   qI [B,HI,dI]   wI [B,HI]   kI [B,T,dI]   q [B,H,dk]   k [B,T,dk]
 *   v [B,T,dv]     out [B,H,dv]      (T = capacity)
 *   seq_lens (nullable): device int32 [B], T_b in [1, T]; NULL means T for
 *            every row.  Read on the device: a length outside [1, T] is
 *            recorded as NSA_ERR_INVALID_ARG (nsa_device_status) and that row
 *            is read as empty (out zero, idx_out row -1); the others are
 *            unaffected.
 *   idx_out (nullable): [B, min(topk,T)] int32, ascending, -1 past min(topk,T_b)
 * v may be NULL when dv <= dk: value row s is then the first dv columns of
 * key row s -- the latent KV of multi-head latent attention, on which the
 * page builds DSA (one cached latent per token, positional part in the last
 * dk-dv columns) -- and only the key rows are fetched.  A NULL v with
 * dv > dk returns NSA_ERR_INVALID_ARG.
 */
int dsa_decode_step(const dsa_cfg* cfg, const void* qI, const void* wI, const void* kI,
                    const void* q, const void* k, const void* v, const int32_t* seq_lens,
                    void* out, int32_t* idx_out, void* ws, size_t ws_bytes, void* stream);

/*
 * dsa_prefill_fwd -- DSA over whole sequences [P4, "쉽게 이해하기": the
 * selection is made independently for every query token]: every position t of
 * sequence b is a query with its own indexer query and weights, scoring and
 * keeping among its causal prefix s <= t (itself included):
 *   I[b,t,s]   = sum_h wI[b,t,h] * max(0, qI[b,t,h,:] . kI[b,s,:])     s <= t
 *   keep(b,t)  = the min(topk, t+1) positions of largest fp32 I, ties to the lower s
 *   out[b,t,h] = softmax_{s in keep}(q[b,t,h,:] . k[b,s,:] * scale) @ v[b,keep,:]
 *   qI [B,T,HI,dI]   wI [B,T,HI]   kI [B,T,dI]   q [B,T,H,dk]   k [B,T,dk]
 *   v [B,T,dv] (or NULL: the first dv columns of k, as in dsa_decode_step)
 *   out [B,T,H,dv]
 *   idx_out (nullable): [B,T,min(topk,T)] int32, ascending, -1 past min(topk,t+1)
 *   ws     : dsa_prefill_workspace_size(cfg) bytes
 * The rows run through the decode step's kernels (row b*T + t reads the keys
 * of sequence b with context t+1), so B*T <= 65535 and the shapes of
 * dsa_decode_step apply; anything else returns NSA_ERR_UNSUPPORTED.
 */
size_t dsa_prefill_workspace_size(const dsa_cfg* cfg);
int dsa_prefill_fwd(const dsa_cfg* cfg, const void* qI, const void* wI, const void* kI,
                    const void* q, const void* k, const void* v, void* out, int32_t* idx_out,
                    void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------- profiling */
/* No counterpart on the pages: measurement support.  When enabled, every
   kernel launch of the library is bracketed by two CUDA events on its
   stream.  nsa_profile_read() synchronises them and, for up to max_kernels
   distinct kernel names (comma-joined into ``names``, at most name_cap
   bytes including the terminator), stores the launch count and the summed
   device time in ms, then forgets the records.  Returns the number of names
   (or a negative status on a CUDA error: -NSA_ERR_CUDA). */
int nsa_profile_enable(int on);
int nsa_profile_read(int max_kernels, char* names, size_t name_cap, int* launches, float* total_ms);

/* ---------------------------------------------------------------- status word */
/* Synchronises ``stream``, returns the status the kernels of the last call on
   ``ws`` recorded (NSA_OK if none) and clears it: a device-side failure (such
   as NSA_ERR_DEVICE_TIMEOUT, after which the call's outputs are not valid)
   first, else a bad argument that only the device could see (such as a
   sequence length out of range, whose sequence was skipped). */
int nsa_device_status(void* ws, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* NSA_H_ */
