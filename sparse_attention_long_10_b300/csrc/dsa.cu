// dsa.cu -- DSA-style indexed sparse decode [page "딥시크 희소 어텐션 DSA 원리:
// 라이트닝 인덱서와 상위 2048 토큰 선택 구조 해설", section "쉽게 이해하기": a
// lightning indexer scores every past token with a weighted sum of ReLU dot
// products over a few small heads whose keys are shared; the 2048 best tokens
// are kept, independently per query; attention runs over the kept tokens only,
// its softmax normalised over that set].
//
// One query token per batch row b at position T-1.  Five launches:
//   dsa_index   I[s] = sum_h w_h * max(0, qI_h . kI_s) for every s (warp MMA,
//               kI streamed by TMA); writes an order-preserving 32-bit key of
//               the fp32 score and a 4096-bin histogram of the key's top 12
//               bits per row.
//   dsa_thresh  exact radix select of the kk-th best (key, position) pair,
//               ties to the lower position: the first level comes from the
//               histogram, the boundary bin's candidates are collected and the
//               last CTA of the row resolves them (12 + 8 more key bits, then
//               the position); it also counts the kept positions per part.
//   dsa_compact ordered compaction of the kept positions (ascending).
//   dsa_attn    softmax(q K_sel^T * scale) V_sel over the kept positions:
//               rows gathered by untiled bulk copies, warp MMA, split over
//               CTAs of 64 kept positions, each leaving (max, sum, O);
//   dsa_merge   merges a row's splits, one CTA per (head, row).
// The last indexer CTA of a row finds the first radix cut from the row's
// histogram.
#include "common.cuh"
#include "kernels.hpp"
#include "profiler.hpp"
#include "tmap.hpp"
#include "warp_mma.cuh"

namespace nsa {

namespace {

constexpr int kIdxThreads = 160;    // 4 compute warps + 1 TMA producer warp
constexpr int kIdxTile = 128;       // keys per indexer tile
constexpr int kIdxStages = 4;
constexpr int kIdxPartMax = 4096;   // most positions per indexer CTA
constexpr int kBins = 4096;         // first radix level: top 12 bits
constexpr int kSelThreads = 256;
constexpr int kSelPart = 2048;      // positions per threshold / compaction CTA
constexpr int kCandCap = 8192;      // boundary-bin candidates kept per row
constexpr int kAttnThreads = 160;   // 4 compute warps + 1 gather warp
constexpr int kAttnTile = 32;       // kept tokens per attention tile
constexpr int kAttnTilesPerCta = 2;
constexpr int kAttnStages = 2;

struct DsaArgs {
  int B, T, HI, dI, H, dk, dv, kk;  // T: context capacity; kk = min(topk, T) (row stride of idx)
  int topk;
  const int32_t* lens;              // nullable [B]: context length of each row (query at len-1)
  int nparts;                       // threshold / compaction parts per row
  int idx_part;                     // positions per indexer CTA (a multiple of kIdxTile)
  int attn_ctas;                    // attention CTAs per row
  int all;                          // kk == T: every position is kept
  float sc2;                        // softmax scale * log2(e)
  const __nv_bfloat16* qI;          // [B,HI,dI]
  const __nv_bfloat16* wI;          // [B,HI]
  const __nv_bfloat16* q;           // [B,H,dk]
  const __nv_bfloat16* k;           // [B,T,dk]
  const __nv_bfloat16* v;           // [B,T,dv]; unused when v_from_k
  int v_from_k;                     // values are the first dv columns of k (latent KV)
  __nv_bfloat16* out;               // [B,H,dv]
  int32_t* idx_out;                 // nullable [B,kk]
  uint32_t* keys;                   // [B,T]
  uint32_t* hist;                   // [B,kBins]
  uint32_t* cand;                   // [B,kCandCap,2] (key, position)
  uint32_t* cand_n;                 // [B]
  uint32_t* gtcnt;                  // [B,nparts] keys above the boundary bin
  uint32_t* offs;                   // [B,nparts] output offset of each part
  uint32_t* thr;                    // [B,2] (K*, I*): the kk-th kept pair
  uint32_t* cut1;                   // [B,2] first-level cut: boundary bin B1, count above it
  int32_t* idx;                     // [B,kk] kept positions, ascending
  float* pm;                        // [B,attn_ctas,16]
  float* pl;                        // [B,attn_ctas,16]
  float* po;                        // [B,attn_ctas,16,dv]
  int* cnt;                         // [3,B] last-CTA counters (threshold, indexer, unused)
  DeviceStatus* st;
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// Order-preserving key of an fp32 score: unsigned order of keys = numeric
// order of scores; -0 is folded into +0 so the two compare equal.
__device__ __forceinline__ uint32_t order_key(float f) {
  f = __fadd_rn(f, 0.0f);
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// One row's context: its length, the positions it keeps, whether it keeps
// them all.  A length outside [1, T] is recorded (NSA_ERR_INVALID_ARG, read
// back by nsa_device_status) and the row is read as empty: no position is
// kept, its output is zero, its idx_out row -1.
struct RowGeom {
  int T, kk, all;
};
__device__ __forceinline__ RowGeom row_geom(const DsaArgs& a, int b, DeviceStatus* st) {
  int T = a.lens != nullptr ? __ldg(a.lens + b) : a.T;
  if (T < 1 || T > a.T) {
    record_arg_error(st, NSA_ERR_INVALID_ARG, 500);
    T = 0;
  }
  RowGeom r;
  r.T = T;
  r.kk = min(a.topk, T);
  r.all = r.kk == T;
  return r;
}

__device__ __forceinline__ bool kept(uint32_t key, uint32_t pos, uint32_t Ks, uint32_t Is) {
  return key > Ks || (key == Ks && pos <= Is);
}

// ============================================================ indexer
struct IdxBars {
  uint64_t full[kIdxStages];
  uint64_t empty[kIdxStages];
  int abort_flag;
};

template <int DI>
__global__ void __launch_bounds__(kIdxThreads, 2)
    dsa_index_kernel(const __grid_constant__ CUtensorMap mapKI, const DsaArgs a) {
  constexpr int KB = DI / 64;
  constexpr int kStage = KB * kIdxTile * 128;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint32_t* hs = reinterpret_cast<uint32_t*>(smem + kIdxStages * kStage);
  IdxBars* bars = reinterpret_cast<IdxBars*>(hs + kBins);
  volatile int* abort_flag = &bars->abort_flag;
  const int part = blockIdx.x, b = blockIdx.y;
  const RowGeom rg = row_geom(a, b, part == 0 && threadIdx.x == 0 ? a.st : nullptr);
  const int s0 = part * a.idx_part;
  const int npos = min(a.idx_part, rg.T - s0);
  const int ntiles = npos > 0 ? (npos + kIdxTile - 1) / kIdxTile : 0;
  const int warp = warp_id(), lane = lane_id();
  if (threadIdx.x == 0) {
    for (int s = 0; s < kIdxStages; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 4);
    }
    bars->abort_flag = prior_error(a.st);
    fence_barrier_init();
  }
  for (int i = threadIdx.x; i < kBins; i += kIdxThreads) hs[i] = 0;
  __syncthreads();
  bool ok = *abort_flag == 0;
  if (warp == 4) {
    if (lane == 0 && ok) {
      tma_prefetch_desc(&mapKI);
      int i = 0;
      for (; i < ntiles; ++i) {
        const int slot = i % kIdxStages;
        if (!mbar_wait(&bars->empty[slot], (uint32_t)(((i / kIdxStages) & 1) ^ 1), abort_flag, a.st, 501)) {
          ok = false;
          break;
        }
        uint8_t* dst = smem + slot * kStage;
        mbar_arrive_expect_tx(&bars->full[slot], kStage);
#pragma unroll
        for (int c = 0; c < KB; ++c)
          tma_load_3d(dst + c * kIdxTile * 128, &mapKI, &bars->full[slot], c * 64, s0 + i * kIdxTile, b);
      }
      if (!ok || *abort_flag)
        for (int y = (i > kIdxStages ? i - kIdxStages : 0); y < i; ++y)
          mbar_wait_plain(&bars->full[y % kIdxStages], (uint32_t)((y / kIdxStages) & 1), kWaitLimitNs);
    }
  } else if (ok) {
    const int gq = lane >> 2, tq = lane & 3;
    // B fragments: qI^T (k = dims, n = indexer heads, padded to 8)
    uint32_t qb[DI / 16][2];
    const __nv_bfloat16* qp = a.qI + ((size_t)b * a.HI + gq) * DI;
#pragma unroll
    for (int ks = 0; ks < DI / 16; ++ks) {
      qb[ks][0] = gq < a.HI ? *reinterpret_cast<const uint32_t*>(qp + 16 * ks + 2 * tq) : 0u;
      qb[ks][1] = gq < a.HI ? *reinterpret_cast<const uint32_t*>(qp + 16 * ks + 8 + 2 * tq) : 0u;
    }
    const float w0 = (2 * tq < a.HI) ? __bfloat162float(a.wI[(size_t)b * a.HI + 2 * tq]) : 0.f;
    const float w1 = (2 * tq + 1 < a.HI) ? __bfloat162float(a.wI[(size_t)b * a.HI + 2 * tq + 1]) : 0.f;
    for (int i = 0; i < ntiles; ++i) {
      const int slot = i % kIdxStages;
      if (!mbar_wait(&bars->full[slot], (uint32_t)((i / kIdxStages) & 1), abort_flag, a.st, 502)) break;
      const uint32_t base = smem_u32(smem + slot * kStage);
#pragma unroll
      for (int mt = 0; mt < 2; ++mt) {
        const int r0 = warp * 32 + mt * 16;
        float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int ks = 0; ks < DI / 16; ++ks) {
          uint32_t af[4];
          ldsm_x4(sw128_addr(base + (ks >> 2) * kIdxTile * 128, r0 + (lane & 15), (ks & 3) * 2 + (lane >> 4)),
                  af[0], af[1], af[2], af[3]);
          mma_16816(c, af, qb[ks][0], qb[ks][1]);
        }
        // c0,c1: key r0+gq, heads 2tq, 2tq+1; c2,c3: key r0+gq+8
        float sa = w0 * fmaxf(c[0], 0.f) + w1 * fmaxf(c[1], 0.f);
        float sb = w0 * fmaxf(c[2], 0.f) + w1 * fmaxf(c[3], 0.f);
        sa = quad_sum(sa);
        sb = quad_sum(sb);
        // lanes with tq == 0 own keys r0+gq and r0+gq+8; equal bins within the
        // warp are counted with one shared-memory atomic
        const int pa = s0 + i * kIdxTile + r0 + gq, pb = pa + 8;
        const uint32_t ka = order_key(sa), kb = order_key(sb);
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int pos = e ? pb : pa;
          const uint32_t key = e ? kb : ka;
          const bool mine = tq == 0 && pos < rg.T;
          if (mine) a.keys[(size_t)b * a.T + pos] = key;
          const uint32_t bin = mine ? (key >> 20) : 0xffffffffu;
          const unsigned same = __match_any_sync(0xffffffffu, bin);
          if (mine && (__ffs(same) - 1) == lane) atomicAdd(&hs[bin], (uint32_t)__popc(same));
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->empty[slot]);
    }
  }
  __syncthreads();
  if (*abort_flag) return;
  for (int i = threadIdx.x; i < kBins; i += kIdxThreads)
    if (hs[i]) atomicAdd(&a.hist[(size_t)b * kBins + i], hs[i]);
  // the last CTA of the row finds the boundary bin of the first radix level
  __threadfence();
  __syncthreads();
  __shared__ int s_last;
  if (threadIdx.x == 0) s_last = (atomicAdd(&a.cnt[a.B + b], 1) == (int)gridDim.x - 1) ? 1 : 0;
  __syncthreads();
  if (!s_last || rg.all) return;   // a row that keeps every position needs no cut
  __threadfence();
  // suffix counts over the bins, 16 per thread for the first 256 threads' worth
  uint32_t* hg = hs;   // reuse: copy of the row's histogram
  {
    constexpr int kPer = (kBins + kIdxThreads - 1) / kIdxThreads;
    uint32_t v[kPer];
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int i = threadIdx.x + k * kIdxThreads;
      v[k] = i < kBins ? __ldcg(a.hist + (size_t)b * kBins + i) : 0u;
    }
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int i = threadIdx.x + k * kIdxThreads;
      if (i < kBins) hg[i] = v[k];
    }
  }
  __syncthreads();
  // 128 threads, 32 bins each from the top: warp scans, then the thread whose
  // range holds the kk-th best key walks its bins
  __shared__ uint32_t wtot[4];
  const int t = threadIdx.x;
  uint32_t sum = 0, incl = 0;
  if (t < 128) {
    for (int i = 0; i < 32; ++i) sum += hg[kBins - 32 * t - 1 - i];
    incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) wtot[warp] = incl;
  }
  __syncthreads();
  if (t < 128) {
    for (int k = 0; k < warp; ++k) incl += wtot[k];
    const uint32_t excl = incl - sum;
    if (excl < (uint32_t)rg.kk && incl >= (uint32_t)rg.kk) {
      uint32_t cum = excl;
      for (int i = 0; i < 32; ++i) {
        const int bin = kBins - 32 * t - 1 - i;
        if (cum + hg[bin] >= (uint32_t)rg.kk) {
          a.cut1[(size_t)b * 2] = (uint32_t)bin;
          a.cut1[(size_t)b * 2 + 1] = cum;
          break;
        }
        cum += hg[bin];
      }
    }
  }
}

// ============================================================ threshold
// Block-wide cut over a histogram of ``nbins`` (a multiple of 256) bins read
// through get(i).  from_top: the highest bin B with count(bins >= B) >= need,
// and count(bins > B); otherwise the lowest bin B with count(bins <= B) >=
// need, and count(bins < B).  Needs 256 threads; scan has 256 + 2 words.
template <class Get>
__device__ void block_cut(Get get, int nbins, uint32_t need, bool from_top, uint32_t* scan, uint32_t& bin,
                          uint32_t& before) {
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  const int per = nbins / 256;
  auto bin_of = [&](int i) { return from_top ? nbins - per * t - 1 - i : per * t + i; };
  uint32_t sum = 0;
  for (int i = 0; i < per; ++i) sum += get(bin_of(i));
  // inclusive scan over the 256 threads: within warps by shuffles, then warp totals
  uint32_t incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) scan[w] = incl;
  __syncthreads();
  uint32_t wbase = 0;
  for (int k = 0; k < w; ++k) wbase += scan[k];
  incl += wbase;
  const uint32_t excl = incl - sum;
  if (excl < need && incl >= need) {
    uint32_t cum = excl;
    for (int i = 0; i < per; ++i) {
      const uint32_t c = get(bin_of(i));
      if (cum + c >= need) {
        scan[256] = (uint32_t)bin_of(i);
        scan[257] = cum;
        break;
      }
      cum += c;
    }
  }
  __syncthreads();
  bin = scan[256];
  before = scan[257];
  __syncthreads();
}

// Exact radix select over ``n`` (key, position) elements read through
// elem(i, key, pos) that all share the top-12-bit bin B1: the need-th best
// pair under (key descending, position ascending).  hist: 4096 words.
template <class Elem>
__device__ void radix_resolve(Elem elem, uint32_t n, uint32_t B1, uint32_t need, uint32_t max_pos, uint32_t* hist,
                              uint32_t* scan, uint32_t& Ks, uint32_t& Is) {
  const int t = threadIdx.x;
  uint32_t prefix = B1 << 20, mask = 0xFFF00000u;
  // key bits 19..8 (4096 bins), then 7..0 (256 bins), from the top
  const int shifts[2] = {8, 0};
  const int widths[2] = {12, 8};
  for (int lv = 0; lv < 2; ++lv) {
    const int nb = 1 << widths[lv];
    const uint32_t dmask = (uint32_t)nb - 1;
    for (int i = t; i < nb; i += 256) hist[i] = 0;
    __syncthreads();
    for (uint32_t i = t; i < n; i += 256) {
      uint32_t key, pos;
      elem(i, key, pos);
      if ((key & mask) == prefix) atomicAdd(&hist[(key >> shifts[lv]) & dmask], 1u);
    }
    __syncthreads();
    uint32_t bin, before;
    block_cut([&](int i) { return hist[i]; }, nb, need, true, scan, bin, before);
    prefix |= bin << shifts[lv];
    mask |= dmask << shifts[lv];
    need -= before;
  }
  Ks = prefix;
  // every element equal to K* is kept: no position cut needed
  const uint32_t n_eq = hist[Ks & 255u];
  __syncthreads();
  if (n_eq == need) {
    Is = 0xffffffffu;
    return;
  }
  // among the elements equal to K*, the need-th smallest position (8-bit
  // digits, from the highest digit a position below max_pos can have)
  int top = 0;
  while (top < 24 && (max_pos >> (top + 8)) != 0) top += 8;
  uint32_t pprefix = 0, pmask = 0;
  for (int sh = top; sh >= 0; sh -= 8) {
    for (int i = t; i < 256; i += 256) hist[i] = 0;
    __syncthreads();
    for (uint32_t i = t; i < n; i += 256) {
      uint32_t key, pos;
      elem(i, key, pos);
      if (key == Ks && (pos & pmask) == pprefix) atomicAdd(&hist[(pos >> sh) & 255u], 1u);
    }
    __syncthreads();
    uint32_t bin, before;
    block_cut([&](int i) { return hist[i]; }, 256, need, false, scan, bin, before);
    pprefix |= bin << sh;
    pmask |= 255u << sh;
    need -= before;
  }
  Is = pprefix;
}

__global__ void __launch_bounds__(kSelThreads) dsa_thresh_kernel(const DsaArgs a) {
  extern __shared__ uint8_t dyn[];
  __shared__ uint32_t scan[258];
  __shared__ uint32_t red[8];
  __shared__ int s_last;
  const int part = blockIdx.x, b = blockIdx.y;
  const int t = threadIdx.x, lane = lane_id(), warp = warp_id();
  if (t == 0) s_last = prior_error(a.st);
  __syncthreads();
  if (s_last) return;
  __syncthreads();
  const RowGeom rg = row_geom(a, b, nullptr);
  if (rg.all) return;   // every position kept (or an empty row): no threshold
  const uint32_t* hist = a.hist + (size_t)b * kBins;
  const uint32_t B1 = __ldcg(a.cut1 + (size_t)b * 2), above = __ldcg(a.cut1 + (size_t)b * 2 + 1);
  // this part's keys: count those above the boundary bin, collect the boundary bin
  const int p0 = part * kSelPart, p1 = min(rg.T, p0 + kSelPart);
  const uint32_t* keys = a.keys + (size_t)b * a.T;
  uint32_t gt = 0;
  constexpr int kChunks = kSelPart / kSelThreads;
  uint32_t kv[kChunks];
#pragma unroll
  for (int c = 0; c < kChunks; ++c) {
    const int pos = p0 + c * kSelThreads + t;
    kv[c] = pos < p1 ? __ldcg(keys + pos) : 0u;
  }
#pragma unroll
  for (int c = 0; c < kChunks; ++c) {
    const int pos = p0 + c * kSelThreads + t;
    const uint32_t key = kv[c];
    bool cand = false;
    if (pos < p1) {
      const uint32_t bin = key >> 20;
      gt += bin > B1 ? 1u : 0u;
      cand = bin == B1;
    }
    const unsigned m = __ballot_sync(0xffffffffu, cand);
    if (m) {
      const int leader = __ffs(m) - 1;
      uint32_t base_i = 0;
      if (lane == leader) base_i = atomicAdd(&a.cand_n[b], (uint32_t)__popc(m));
      base_i = __shfl_sync(0xffffffffu, base_i, leader);
      if (cand) {
        const uint32_t r = base_i + __popc(m & ((1u << lane) - 1u));
        if (r < (uint32_t)kCandCap) {
          uint32_t* c = a.cand + ((size_t)b * kCandCap + r) * 2;
          c[0] = key;
          c[1] = (uint32_t)pos;
        }
      }
    }
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) gt += __shfl_xor_sync(0xffffffffu, gt, o);
  if (lane == 0) red[warp] = gt;
  __syncthreads();
  if (t == 0) {
    uint32_t s = 0;
    for (int w = 0; w < kSelThreads / 32; ++w) s += red[w];
    a.gtcnt[(size_t)b * a.nparts + part] = s;
  }
  __threadfence();
  __syncthreads();
  if (t == 0) s_last = (atomicAdd(&a.cnt[b], 1) == (int)gridDim.x - 1) ? 1 : 0;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  // ---------------------------------------------------------- last CTA of the row
  uint32_t* ck = reinterpret_cast<uint32_t*>(dyn);   // [kCandCap]
  uint32_t* cp = ck + kCandCap;                        // [kCandCap]
  uint32_t* h2 = cp + kCandCap;                        // [4096]
  uint32_t* pc = h2 + 4096;                            // [nparts]
  const uint32_t c1 = __ldcg(hist + B1);
  const uint32_t need1 = (uint32_t)rg.kk - above;
  uint32_t Ks, Is;
  const bool fast = c1 <= (uint32_t)kCandCap;
  if (fast) {
    for (uint32_t i = t; i < c1; i += kSelThreads) {
      ck[i] = __ldcg(a.cand + ((size_t)b * kCandCap + i) * 2);
      cp[i] = __ldcg(a.cand + ((size_t)b * kCandCap + i) * 2 + 1);
    }
    __syncthreads();
    radix_resolve([&](uint32_t i, uint32_t& key, uint32_t& pos) { key = ck[i]; pos = cp[i]; }, c1, B1, need1,
                  (uint32_t)(rg.T - 1), h2, scan, Ks, Is);
  } else {
    // more boundary candidates than the buffer holds: resolve over the whole row
    radix_resolve([&](uint32_t i, uint32_t& key, uint32_t& pos) { key = __ldcg(keys + i); pos = i; },
                  (uint32_t)rg.T, B1, need1, (uint32_t)(rg.T - 1), h2, scan, Ks, Is);
  }
  // kept positions per part: above the boundary bin + kept boundary candidates
  for (int p = t; p < a.nparts; p += kSelThreads) pc[p] = __ldcg(a.gtcnt + (size_t)b * a.nparts + p);
  __syncthreads();
  if (fast) {
    for (uint32_t i = t; i < c1; i += kSelThreads)
      if (kept(ck[i], cp[i], Ks, Is)) atomicAdd(&pc[cp[i] / kSelPart], 1u);
  } else {
    for (uint32_t i = t; i < (uint32_t)rg.T; i += kSelThreads) {
      const uint32_t key = __ldcg(keys + i);
      if ((key >> 20) == B1 && kept(key, i, Ks, Is)) atomicAdd(&pc[i / kSelPart], 1u);
    }
  }
  __syncthreads();
  if (t == 0) {
    uint32_t run = 0;
    for (int p = 0; p < a.nparts; ++p) {
      a.offs[(size_t)b * a.nparts + p] = run;
      run += pc[p];
    }
    a.thr[(size_t)b * 2 + 0] = Ks;
    a.thr[(size_t)b * 2 + 1] = Is;
  }
}

// ============================================================ compaction
__global__ void __launch_bounds__(kSelThreads) dsa_compact_kernel(const DsaArgs a) {
  __shared__ uint32_t wc[kSelThreads / 32];
  __shared__ int s_abort;
  const int part = blockIdx.x, b = blockIdx.y;
  const int t = threadIdx.x, lane = lane_id(), warp = warp_id();
  if (t == 0) s_abort = prior_error(a.st);
  __syncthreads();
  if (s_abort) return;
  const RowGeom rg = row_geom(a, b, part == 0 && t == 0 ? a.st : nullptr);
  const int p0 = part * kSelPart, p1 = min(rg.T, p0 + kSelPart);
  uint32_t run = rg.all ? (uint32_t)p0 : __ldcg(a.offs + (size_t)b * a.nparts + part);
  const uint32_t Ks = rg.all ? 0u : __ldcg(a.thr + (size_t)b * 2);
  const uint32_t Is = rg.all ? 0u : __ldcg(a.thr + (size_t)b * 2 + 1);
  const uint32_t* keys = a.keys + (size_t)b * a.T;
  int32_t* dst = a.idx + (size_t)b * a.kk;
  int32_t* dst2 = a.idx_out != nullptr ? a.idx_out + (size_t)b * a.kk : nullptr;
  // a row that keeps fewer than kk positions: its index row ends in -1
  if (part == 0)
    for (int e = rg.kk + t; e < a.kk; e += kSelThreads) {
      dst[e] = -1;
      if (dst2) dst2[e] = -1;
    }
  constexpr int kChunks = kSelPart / kSelThreads;
  bool selv[kChunks];
#pragma unroll
  for (int c = 0; c < kChunks; ++c) {
    const int pos = p0 + c * kSelThreads + t;
    selv[c] = pos < p1 && (rg.all || kept(__ldcg(keys + pos), (uint32_t)pos, Ks, Is));
  }
#pragma unroll
  for (int c = 0; c < kChunks; ++c) {
    const int base = p0 + c * kSelThreads;
    const int pos = base + t;
    const bool sel = selv[c];
    const unsigned m = __ballot_sync(0xffffffffu, sel);
    if (lane == 0) wc[warp] = (uint32_t)__popc(m);
    __syncthreads();
    uint32_t before = 0, total = 0;
#pragma unroll
    for (int w = 0; w < kSelThreads / 32; ++w) {
      before += w < warp ? wc[w] : 0u;
      total += wc[w];
    }
    if (sel) {
      const uint32_t o = run + before + __popc(m & ((1u << lane) - 1u));
      dst[o] = pos;
      if (dst2) dst2[o] = pos;
    }
    run += total;
    __syncthreads();
  }
}

// ============================================================ attention
struct AttnBars {
  uint64_t full[kAttnStages];
  uint64_t empty[kAttnStages];
  int abort_flag;
  int last;
};

struct AttnLayout {
  uint32_t qs, kst, vst, stage, ks_off, vs_off, p_off, red_off, bar_off, total;
};

__host__ __device__ inline AttnLayout attn_layout(int dk, int dv) {
  AttnLayout L;
  L.qs = 2u * dk + 16u;    // padded row strides (bytes): 8 ldmatrix rows hit 8 bank groups
  L.kst = 2u * dk + 16u;
  L.vst = 2u * dv + 16u;
  L.stage = (uint32_t)kAttnTile * (L.kst + L.vst);
  L.ks_off = 16u * L.qs;
  L.vs_off = L.ks_off + (uint32_t)kAttnTile * L.kst;
  L.p_off = L.ks_off + kAttnStages * L.stage;
  L.red_off = L.p_off + 16u * 80u;
  L.bar_off = L.red_off + 2u * 4u * 16u * 4u;
  L.total = L.bar_off + 128u;
  return L;
}

template <int DV>
__global__ void __launch_bounds__(kAttnThreads, 1) dsa_attn_kernel(const DsaArgs a) {
  constexpr int DV4 = DV / 4;   // value columns per compute warp
  extern __shared__ __align__(16) uint8_t smem[];
  const AttnLayout L = attn_layout(a.dk, DV);
  uint8_t* Qs = smem;
  uint8_t* Ps = smem + L.p_off;
  float* red_m = reinterpret_cast<float*>(smem + L.red_off);   // [4][16]
  float* red_l = red_m + 64;                                     // [4][16]
  AttnBars* bars = reinterpret_cast<AttnBars*>(smem + L.bar_off);
  volatile int* abort_flag = &bars->abort_flag;
  const int x = blockIdx.x, b = blockIdx.y;
  const int warp = warp_id(), lane = lane_id();
  const int e0 = x * kAttnTile * kAttnTilesPerCta;
  const int nent = min(kAttnTile * kAttnTilesPerCta, row_geom(a, b, nullptr).kk - e0);
  const int ntiles = nent > 0 ? (nent + kAttnTile - 1) / kAttnTile : 0;
  const int dk = a.dk;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kAttnStages; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 4);
    }
    bars->abort_flag = prior_error(a.st);
    bars->last = 0;
    fence_barrier_init();
  }
  // query rows (heads past H are zero)
  for (int i = threadIdx.x; i < 16 * dk / 8; i += kAttnThreads) {
    const int h = i / (dk / 8), c = i % (dk / 8);
    uint4 v = make_uint4(0, 0, 0, 0);
    if (h < a.H) v = *reinterpret_cast<const uint4*>(a.q + ((size_t)b * a.H + h) * dk + 8 * c);
    *reinterpret_cast<uint4*>(Qs + h * L.qs + 16 * c) = v;
  }
  __syncthreads();
  const int32_t* sel = a.idx + (size_t)b * a.kk + e0;
  bool ok = *abort_flag == 0;
  const int gq = lane >> 2, tq = lane & 3;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  float o[DV4 / 8][4];
#pragma unroll
  for (int i = 0; i < DV4 / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;

  if (warp == 4) {
    // ------------------------------------------------------------ gather warp
    if (ok) {
      int i = 0;
      for (; i < ntiles; ++i) {
        const int slot = i % kAttnStages;
        if (!mbar_wait(&bars->empty[slot], (uint32_t)(((i / kAttnStages) & 1) ^ 1), abort_flag, a.st, 521)) {
          ok = false;
          break;
        }
        uint8_t* ks = smem + L.ks_off + slot * L.stage;
        uint8_t* vs = ks + kAttnTile * L.kst;
        const int nv = min(kAttnTile, nent - i * kAttnTile);
        const int e = i * kAttnTile + lane;
        // with latent KV the value rows are the first DV columns of the key
        // rows: only the keys are fetched
        const uint32_t vbytes = a.v_from_k ? 0u : 2u * DV;
        if (lane >= nv) {   // absent rows read as zeros
          for (int c = 0; c < dk / 8; ++c) *reinterpret_cast<uint4*>(ks + lane * L.kst + 16 * c) = make_uint4(0, 0, 0, 0);
          if (!a.v_from_k)
            for (int c = 0; c < DV / 8; ++c) *reinterpret_cast<uint4*>(vs + lane * L.vst + 16 * c) = make_uint4(0, 0, 0, 0);
          fence_proxy_async_smem();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive_expect_tx(&bars->full[slot], (uint32_t)nv * (2u * dk + vbytes));
        __syncwarp();
        if (lane < nv) {
          const int pos = __ldg(sel + e);
          bulk_load(ks + lane * L.kst, a.k + ((size_t)b * a.T + pos) * dk, 2u * dk, &bars->full[slot]);
          if (!a.v_from_k)
            bulk_load(vs + lane * L.vst, a.v + ((size_t)b * a.T + pos) * DV, 2u * DV, &bars->full[slot]);
        }
      }
      if (lane == 0 && (!ok || *abort_flag))
        for (int y = (i > kAttnStages ? i - kAttnStages : 0); y < i; ++y)
          mbar_wait_plain(&bars->full[y % kAttnStages], (uint32_t)((y / kAttnStages) & 1), kWaitLimitNs);
    }
  } else if (ok) {
    // ------------------------------------------------------------ compute warps
    const uint32_t q_a = smem_u32(Qs);
    for (int i = 0; i < ntiles; ++i) {
      const int slot = i % kAttnStages;
      if (!mbar_wait(&bars->full[slot], (uint32_t)((i / kAttnStages) & 1), abort_flag, a.st, 522)) {
        ok = false;
        break;
      }
      const uint32_t k_a = smem_u32(smem + L.ks_off + slot * L.stage);
      const uint32_t v_a = a.v_from_k ? k_a : k_a + kAttnTile * L.kst;
      const uint32_t vst = a.v_from_k ? L.kst : L.vst;
      const int nv = min(kAttnTile, nent - i * kAttnTile);
      // S[16 heads x 8 keys] for keys 8*warp .. 8*warp+7
      float s[4] = {0.f, 0.f, 0.f, 0.f};
      for (int k0 = 0; k0 < dk; k0 += 32) {
        uint32_t b0, b1, b2, b3, x0[4], x1[4];
        ldsm_x4(k_a + (uint32_t)(8 * warp + (lane & 7)) * L.kst + (uint32_t)(k0 + (lane >> 3) * 8) * 2, b0, b1, b2,
                b3);
        ldsm_x4(q_a + (uint32_t)(lane & 15) * L.qs + (uint32_t)(k0 + (lane >> 4) * 8) * 2, x0[0], x0[1], x0[2],
                x0[3]);
        ldsm_x4(q_a + (uint32_t)(lane & 15) * L.qs + (uint32_t)(k0 + 16 + (lane >> 4) * 8) * 2, x1[0], x1[1],
                x1[2], x1[3]);
        mma_16816(s, x0, b0, b1);
        mma_16816(s, x1, b2, b3);
      }
      const int key0 = 8 * warp + 2 * tq;
      s[0] = key0 < nv ? s[0] * a.sc2 : -INFINITY;
      s[1] = key0 + 1 < nv ? s[1] * a.sc2 : -INFINITY;
      s[2] = key0 < nv ? s[2] * a.sc2 : -INFINITY;
      s[3] = key0 + 1 < nv ? s[3] * a.sc2 : -INFINITY;
      const float mx0 = quad_max(fmaxf(s[0], s[1])), mx1 = quad_max(fmaxf(s[2], s[3]));
      if (tq == 0) {
        red_m[warp * 16 + gq] = mx0;
        red_m[warp * 16 + gq + 8] = mx1;
      }
      named_bar(1, 128);
      const float tm0 = fmaxf(fmaxf(red_m[gq], red_m[16 + gq]), fmaxf(red_m[32 + gq], red_m[48 + gq]));
      const float tm1 =
          fmaxf(fmaxf(red_m[gq + 8], red_m[16 + gq + 8]), fmaxf(red_m[32 + gq + 8], red_m[48 + gq + 8]));
      const float mn0 = fmaxf(m0, tm0), mn1 = fmaxf(m1, tm1);
      const float us0 = mn0 == -INFINITY ? 0.f : mn0, us1 = mn1 == -INFINITY ? 0.f : mn1;
      const float al0 = fast_exp2(m0 - us0), al1 = fast_exp2(m1 - us1);
      const float p0 = fast_exp2(s[0] - us0), p1 = fast_exp2(s[1] - us0);
      const float p2 = fast_exp2(s[2] - us1), p3 = fast_exp2(s[3] - us1);
      const float ps0 = quad_sum(p0 + p1), ps1 = quad_sum(p2 + p3);
      if (tq == 0) {
        red_l[warp * 16 + gq] = ps0;
        red_l[warp * 16 + gq + 8] = ps1;
      }
      *reinterpret_cast<uint32_t*>(Ps + gq * 80 + key0 * 2) = pack_bf16x2(p0, p1);
      *reinterpret_cast<uint32_t*>(Ps + (gq + 8) * 80 + key0 * 2) = pack_bf16x2(p2, p3);
      named_bar(1, 128);
      l0 = l0 * al0 + (red_l[gq] + red_l[16 + gq] + red_l[32 + gq] + red_l[48 + gq]);
      l1 = l1 * al1 + (red_l[gq + 8] + red_l[16 + gq + 8] + red_l[32 + gq + 8] + red_l[48 + gq + 8]);
      m0 = mn0;
      m1 = mn1;
#pragma unroll
      for (int j = 0; j < DV4 / 8; ++j) {
        o[j][0] *= al0;
        o[j][1] *= al0;
        o[j][2] *= al1;
        o[j][3] *= al1;
      }
      const uint32_t p_a = smem_u32(Ps);
#pragma unroll
      for (int kk2 = 0; kk2 < 2; ++kk2) {
        uint32_t pa[4];
        ldsm_x4(p_a + (uint32_t)(lane & 15) * 80u + (uint32_t)(16 * kk2 + (lane >> 4) * 8) * 2, pa[0], pa[1], pa[2],
                pa[3]);
#pragma unroll
        for (int np = 0; np < DV4 / 16; ++np) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(v_a + (uint32_t)(16 * kk2 + (lane & 7) + ((lane >> 3) & 1) * 8) * vst +
                        (uint32_t)(warp * DV4 + 16 * np + (lane >> 4) * 8) * 2,
                    b0, b1, b2, b3);
          mma_16816(o[2 * np], pa, b0, b1);
          mma_16816(o[2 * np + 1], pa, b2, b3);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->empty[slot]);
    }
  }
  __syncthreads();
  if (*abort_flag) return;
  // ---------------------------------------------------------------- partial of this CTA
  const size_t pb = (size_t)b * a.attn_ctas + x;
  if (warp < 4) {
    if (warp == 0 && tq == 0) {
      a.pm[pb * 16 + gq] = m0;
      a.pm[pb * 16 + gq + 8] = m1;
      a.pl[pb * 16 + gq] = l0;
      a.pl[pb * 16 + gq + 8] = l1;
    }
#pragma unroll
    for (int j = 0; j < DV4 / 8; ++j) {
      float* r = a.po + (pb * 16 + gq) * DV + warp * DV4 + 8 * j + 2 * tq;
      r[0] = o[j][0];
      r[1] = o[j][1];
      r[8 * DV] = o[j][2];
      r[8 * DV + 1] = o[j][3];
    }
  }
}

// Merge of a row's attention splits: out[b,h,:] = sum_c w_c O_c / sum_c w_c l_c,
// w_c = exp(m_c - max m).  One CTA per (head, row), one thread per 4 columns.
constexpr int kMergeGroups = 4;   // partial subsets summed in parallel per column

template <int DV>
__global__ void __launch_bounds__(DV / 4 * kMergeGroups) dsa_merge_kernel(const DsaArgs a) {
  constexpr int C4 = DV / 4;            // float4 columns
  const int h = blockIdx.x, b = blockIdx.y;
  const int NC = a.attn_ctas;
  __shared__ float Ms, iLs;
  __shared__ int s_abort;
  __shared__ float4 part[kMergeGroups - 1][C4];
  if (threadIdx.x == 0) s_abort = prior_error(a.st);
  __syncthreads();
  if (s_abort) return;
  const float* pm = a.pm + (size_t)b * NC * 16 + h;
  const float* pl = a.pl + (size_t)b * NC * 16 + h;
  if (threadIdx.x < 32) {
    float M = -INFINITY;
    for (int c = threadIdx.x; c < NC; c += 32) M = fmaxf(M, __ldcg(pm + (size_t)c * 16));
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    const float Mu = M == -INFINITY ? 0.f : M;
    float L = 0.f;
    for (int c = threadIdx.x; c < NC; c += 32)
      L += __ldcg(pl + (size_t)c * 16) * fast_exp2(__ldcg(pm + (size_t)c * 16) - Mu);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
    if (threadIdx.x == 0) {
      Ms = Mu;
      iLs = L > 0.f ? 1.f / L : 0.f;
    }
  }
  __syncthreads();
  const int col = threadIdx.x % C4, grp = threadIdx.x / C4;
  const float* po = a.po + ((size_t)b * NC * 16 + h) * DV + 4 * col;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int c0 = grp * 8; c0 < NC; c0 += 8 * kMergeGroups) {
    float4 v[8];
    float f[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int c = c0 + k;
      v[k] = c < NC ? __ldcg(reinterpret_cast<const float4*>(po + (size_t)c * 16 * DV)) : make_float4(0.f, 0.f, 0.f, 0.f);
      f[k] = c < NC ? __ldcg(pm + (size_t)c * 16) : -INFINITY;
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float ff = fast_exp2(f[k] - Ms);
      acc.x += ff * v[k].x;
      acc.y += ff * v[k].y;
      acc.z += ff * v[k].z;
      acc.w += ff * v[k].w;
    }
  }
  if (grp > 0) part[grp - 1][col] = acc;
  __syncthreads();
  if (grp == 0) {
#pragma unroll
    for (int k = 0; k < kMergeGroups - 1; ++k) {
      const float4 p2 = part[k][col];
      acc.x += p2.x;
      acc.y += p2.y;
      acc.z += p2.z;
      acc.w += p2.w;
    }
    uint2 pk;
    pk.x = pack_bf16x2(acc.x * iLs, acc.y * iLs);
    pk.y = pack_bf16x2(acc.z * iLs, acc.w * iLs);
    *reinterpret_cast<uint2*>(a.out + ((size_t)b * a.H + h) * DV + 4 * col) = pk;
  }
}

// ============================================================ host side
struct DsaWs {
  size_t cnt, hist, cand_n, zero_end, keys, cand, gtcnt, offs, thr, cut1, idx, pm, pl, po, end;
};

struct DsaShape {
  int kk, nparts, attn_ctas, all;
};

DsaShape dsa_shape(const dsa_cfg& c) {
  DsaShape s;
  s.kk = c.topk < c.T ? c.topk : c.T;
  s.all = s.kk == c.T ? 1 : 0;
  s.nparts = (c.T + kSelPart - 1) / kSelPart;
  s.attn_ctas = (s.kk + kAttnTile * kAttnTilesPerCta - 1) / (kAttnTile * kAttnTilesPerCta);
  return s;
}

DsaWs dsa_ws(const dsa_cfg& c) {
  const DsaShape s = dsa_shape(c);
  const size_t B = (size_t)c.B;
  DsaWs w;
  w.cnt = sizeof(DeviceStatus);
  w.cand_n = align_up(w.cnt + sizeof(int) * 3 * B, 256);
  w.hist = align_up(w.cand_n + sizeof(uint32_t) * B, 256);
  w.zero_end = align_up(w.hist + sizeof(uint32_t) * B * kBins, 256);
  w.keys = w.zero_end;
  w.cand = align_up(w.keys + sizeof(uint32_t) * B * (size_t)c.T, 256);
  w.gtcnt = align_up(w.cand + sizeof(uint32_t) * B * kCandCap * 2, 256);
  w.offs = align_up(w.gtcnt + sizeof(uint32_t) * B * s.nparts, 256);
  w.thr = align_up(w.offs + sizeof(uint32_t) * B * s.nparts, 256);
  w.cut1 = align_up(w.thr + sizeof(uint32_t) * B * 2, 256);
  w.idx = align_up(w.cut1 + sizeof(uint32_t) * B * 2, 256);
  w.pm = align_up(w.idx + sizeof(int32_t) * B * (size_t)s.kk, 256);
  w.pl = align_up(w.pm + sizeof(float) * B * s.attn_ctas * 16, 256);
  w.po = align_up(w.pl + sizeof(float) * B * s.attn_ctas * 16, 256);
  w.end = align_up(w.po + sizeof(float) * B * s.attn_ctas * 16 * (size_t)c.dv, 256);
  return w;
}

size_t thresh_smem(const DsaShape& s) {
  return sizeof(uint32_t) * (2 * (size_t)kCandCap + 4096 + (size_t)s.nparts);
}

template <int DI>
int launch_index(const DsaArgs& a, const CUtensorMap& map, cudaStream_t s) {
  constexpr size_t smem = (size_t)kIdxStages * (DI / 64) * kIdxTile * 128 + kBins * 4 + 256 + 1024;
  if (int rc = ensure_smem_attr(reinterpret_cast<const void*>(&dsa_index_kernel<DI>), smem)) return rc;
  prof::begin("dsa_index", s);
  dsa_index_kernel<DI><<<dim3((a.T + a.idx_part - 1) / a.idx_part, a.B), kIdxThreads, smem, s>>>(map, a);
  prof::end(s);
  return cudaPeekAtLastError() == cudaSuccess ? NSA_OK : NSA_ERR_CUDA;
}

template <int DV>
int launch_attn(const DsaArgs& a, cudaStream_t s) {
  const AttnLayout L = attn_layout(a.dk, DV);
  if (int rc = ensure_smem_attr(reinterpret_cast<const void*>(&dsa_attn_kernel<DV>), smem_max())) return rc;
  prof::begin("dsa_attn", s);
  dsa_attn_kernel<DV><<<dim3(a.attn_ctas, a.B), kAttnThreads, L.total, s>>>(a);
  prof::end(s);
  if (cudaPeekAtLastError() != cudaSuccess) return NSA_ERR_CUDA;
  prof::begin("dsa_merge", s);
  dsa_merge_kernel<DV><<<dim3(a.H, a.B), DV / 4 * kMergeGroups, 0, s>>>(a);
  prof::end(s);
  return cudaPeekAtLastError() == cudaSuccess ? NSA_OK : NSA_ERR_CUDA;
}

}  // namespace

int dsa_supported(const dsa_cfg& c) {
  if (c.HI < 1 || c.HI > 8) return NSA_ERR_UNSUPPORTED;
  if (c.dI != 64 && c.dI != 128 && c.dI != 256) return NSA_ERR_UNSUPPORTED;
  if (c.H < 1 || c.H > 16) return NSA_ERR_UNSUPPORTED;
  if (c.dk % 64 != 0 || c.dk > 1024) return NSA_ERR_UNSUPPORTED;
  if (c.dv != 64 && c.dv != 128 && c.dv != 256 && c.dv != 512) return NSA_ERR_UNSUPPORTED;
  if (c.B > 65535 || c.T > (1 << 28)) return NSA_ERR_UNSUPPORTED;
  const DsaShape s = dsa_shape(c);
  if (attn_layout(c.dk, c.dv).total > smem_max()) return NSA_ERR_UNSUPPORTED;
  if (thresh_smem(s) + 2048 > smem_max()) return NSA_ERR_UNSUPPORTED;
  return NSA_OK;
}

size_t dsa_ws_bytes(const dsa_cfg& c) { return dsa_ws(c).end; }
size_t dsa_zero_bytes(const dsa_cfg& c) { return dsa_ws(c).zero_end; }

int launch_dsa(const dsa_cfg& c, const void* qI, const void* wI, const void* kI, const void* q, const void* k,
               const void* v, const int32_t* lens, void* out, int32_t* idx_out, uint8_t* ws, cudaStream_t s) {
  const DsaShape sh = dsa_shape(c);
  const DsaWs w = dsa_ws(c);
  DsaArgs a;
  a.B = c.B;
  a.T = c.T;
  a.HI = c.HI;
  a.dI = c.dI;
  a.H = c.H;
  a.dk = c.dk;
  a.dv = c.dv;
  a.kk = sh.kk;
  a.topk = c.topk;
  a.lens = lens;
  a.nparts = sh.nparts;
  {
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                   cudaSuccess)
      sms = 148;
    const int per_row = (2 * sms + c.B - 1) / c.B;          // two indexer CTAs per SM
    int part = (c.T + per_row - 1) / per_row;
    part = (part + kIdxTile - 1) / kIdxTile * kIdxTile;
    a.idx_part = part < kIdxTile ? kIdxTile : (part > kIdxPartMax ? kIdxPartMax : part);
  }
  a.attn_ctas = sh.attn_ctas;
  a.all = sh.all;
  const float scale = c.scale > 0.f ? c.scale : 1.0f / sqrtf((float)c.dk);
  a.sc2 = scale * 1.4426950408889634f;
  a.qI = static_cast<const __nv_bfloat16*>(qI);
  a.wI = static_cast<const __nv_bfloat16*>(wI);
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.k = static_cast<const __nv_bfloat16*>(k);
  a.v_from_k = v == nullptr ? 1 : 0;
  a.v = static_cast<const __nv_bfloat16*>(v != nullptr ? v : k);
  a.out = static_cast<__nv_bfloat16*>(out);
  a.idx_out = idx_out;
  a.keys = reinterpret_cast<uint32_t*>(ws + w.keys);
  a.hist = reinterpret_cast<uint32_t*>(ws + w.hist);
  a.cand = reinterpret_cast<uint32_t*>(ws + w.cand);
  a.cand_n = reinterpret_cast<uint32_t*>(ws + w.cand_n);
  a.gtcnt = reinterpret_cast<uint32_t*>(ws + w.gtcnt);
  a.offs = reinterpret_cast<uint32_t*>(ws + w.offs);
  a.thr = reinterpret_cast<uint32_t*>(ws + w.thr);
  a.cut1 = reinterpret_cast<uint32_t*>(ws + w.cut1);
  a.idx = reinterpret_cast<int32_t*>(ws + w.idx);
  a.pm = reinterpret_cast<float*>(ws + w.pm);
  a.pl = reinterpret_cast<float*>(ws + w.pl);
  a.po = reinterpret_cast<float*>(ws + w.po);
  a.cnt = reinterpret_cast<int*>(ws + w.cnt);
  a.st = reinterpret_cast<DeviceStatus*>(ws);
  int rc = NSA_OK;
  if (!sh.all) {
    CUtensorMap map;
    const uint64_t dims[3] = {(uint64_t)c.dI, (uint64_t)c.T, (uint64_t)c.B};
    const uint64_t str[2] = {(uint64_t)c.dI * 2, (uint64_t)c.T * c.dI * 2};
    const uint32_t box[3] = {64, (uint32_t)kIdxTile, 1};
    if (!make_tmap_bf16(&map, kI, 3, dims, str, box)) return NSA_ERR_CUDA;
    switch (c.dI) {
      case 64: rc = launch_index<64>(a, map, s); break;
      case 128: rc = launch_index<128>(a, map, s); break;
      case 256: rc = launch_index<256>(a, map, s); break;
      default: return NSA_ERR_UNSUPPORTED;
    }
    if (rc != NSA_OK) return rc;
    // dynamic size actually needed (the kernel also has ~1 KB of static shared memory)
    if ((rc = ensure_smem_attr(reinterpret_cast<const void*>(&dsa_thresh_kernel), thresh_smem(sh))) != NSA_OK)
      return rc;
    prof::begin("dsa_thresh", s);
    dsa_thresh_kernel<<<dim3(sh.nparts, c.B), kSelThreads, thresh_smem(sh), s>>>(a);
    prof::end(s);
    if (cudaPeekAtLastError() != cudaSuccess) return NSA_ERR_CUDA;
  }
  prof::begin("dsa_compact", s);
  dsa_compact_kernel<<<dim3(sh.nparts, c.B), kSelThreads, 0, s>>>(a);
  prof::end(s);
  if (cudaPeekAtLastError() != cudaSuccess) return NSA_ERR_CUDA;
  switch (c.dv) {
    case 64: return launch_attn<64>(a, s);
    case 128: return launch_attn<128>(a, s);
    case 256: return launch_attn<256>(a, s);
    case 512: return launch_attn<512>(a, s);
    default: return NSA_ERR_UNSUPPORTED;
  }
}

}  // namespace nsa
