// dsa.cu -- DSA-style indexed sparse decode [page "딥시크 희소 어텐션 DSA 원리:
// 라이트닝 인덱서와 상위 2048 토큰 선택 구조 해설", section "쉽게 이해하기": a
// lightning indexer scores every past token with a weighted sum of ReLU dot
// products over a few small heads whose keys are shared; the 2048 best tokens
// are kept, independently per query; attention runs over the kept tokens only,
// its softmax normalised over that set].
//
// One query token per batch row b at position T-1.  Four launches:
//   dsa_index   I[s] = sum_h w_h * max(0, qI_h . kI_s) for every s (warp MMA,
//               kI streamed by TMA); writes an order-preserving 32-bit key of
//               the fp32 score and a 4096-bin histogram of the key's top 12
//               bits per row.
//   dsa_select  one thread-block cluster per row: exact radix select of the
//               kk-th best (key, position) pair, ties to the lower position
//               (first level from the histogram, the boundary bin's candidates
//               resolved on 12 + 8 more key bits, then the position), and the
//               ordered compaction of the kept positions (ascending); counts
//               and candidates move through distributed shared memory.
//   dsa_attn    softmax(q K_sel^T * scale) V_sel over the kept positions on
//               tcgen05: rows gathered by TMA tile::gather4, split over CTAs of
//               64 kept positions (two per SM), each leaving (max, sum, O);
//   dsa_merge   merges a row's splits, one CTA per (head, row).
#include "common.cuh"
#include "kernels.hpp"
#include "profiler.hpp"
#include "tmap.hpp"
#include "warp_mma.cuh"

namespace nsa {

namespace {

constexpr int kIdxWarps = 8;        // compute warps: 16 keys of each tile each
constexpr int kIdxThreads = 32 * (kIdxWarps + 1);   // + 1 TMA producer warp
constexpr int kIdxTile = 128;       // keys per indexer tile
constexpr int kIdxStages = 4;
constexpr int kIdxPartMax = 4096;   // most positions per indexer CTA
constexpr int kBins = 4096;         // first radix level: top 12 bits
constexpr int kSelThreads = 512;
constexpr int kCandCap = 4096;      // boundary-bin candidates resolved in shared memory per row

struct DsaArgs {
  int B, T, HI, dI, H, dk, dv, kk;  // B: query rows; T: context capacity; kk = min(topk, T) (row stride of idx)
  int nseq;                         // sequences whose keys the rows read
  int rows_per_seq;                 // 1: one query per sequence (decode); T: every position (prefill)
  int topk;
  const int32_t* lens;              // nullable [B]: context length of each row (query at len-1)
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
  uint32_t* keys;                   // [B,kstride]
  int kstride;                      // T rounded up to 64 keys
  uint32_t* hist;                   // [B,kBins]
  int32_t* idx;                     // [B,kk] kept positions, ascending
  float* pm;                        // [B,attn_ctas,16]
  float* pl;                        // [B,attn_ctas,16]
  float* po;                        // [B,attn_ctas,16,dv]
  DeviceStatus* st;
};

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
  int T;
  if (a.rows_per_seq > 1) {
    T = b % a.rows_per_seq + 1;   // prefill: row b is position b mod T of its sequence
  } else {
    T = a.lens != nullptr ? __ldg(a.lens + b) : a.T;
    if (T < 1 || T > a.T) {
      record_arg_error(st, NSA_ERR_INVALID_ARG, 500);
      T = 0;
    }
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
  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    for (int s = 0; s < kIdxStages; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], kIdxWarps);
    }
    bars->abort_flag = prior_error(a.st);
    fence_barrier_init();
  }
  for (int i = threadIdx.x; i < kBins; i += kIdxThreads) hs[i] = 0;
  __syncthreads();
  bool ok = *abort_flag == 0;
  if (warp == kIdxWarps) {
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
          tma_load_3d(dst + c * kIdxTile * 128, &mapKI, &bars->full[slot], c * 64, s0 + i * kIdxTile,
                      b / a.rows_per_seq);
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
      {
        const int r0 = warp * 16;
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
        // lanes with tq == 0 own keys r0+gq and r0+gq+8
        const int pa = s0 + i * kIdxTile + r0 + gq, pb = pa + 8;
        if (tq == 0) {
          const uint32_t ka = order_key(sa), kb = order_key(sb);
          if (pa < rg.T) {
            a.keys[(size_t)b * a.kstride + pa] = ka;
            atomicAdd(&hs[ka >> 20], 1u);
          }
          if (pb < rg.T) {
            a.keys[(size_t)b * a.kstride + pb] = kb;
            atomicAdd(&hs[kb >> 20], 1u);
          }
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
}

// ============================================================ radix select helpers
// Block-wide cut over a histogram of ``nbins`` bins (a multiple of
// kSelThreads, or fewer) read through get(i).  from_top: the highest bin B with
// count(bins >= B) >= need, and count(bins > B); otherwise the lowest bin B
// with count(bins <= B) >= need, and count(bins < B).  Needs kSelThreads
// threads; scan has 258 words (warp totals, then the result in 256 and 257).
template <class Get>
__device__ void block_cut(Get get, int nbins, uint32_t need, bool from_top, uint32_t* scan, uint32_t& bin,
                          uint32_t& before) {
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  const int per = (nbins + kSelThreads - 1) / kSelThreads;
  auto bin_of = [&](int i) { return from_top ? nbins - per * t - 1 - i : per * t + i; };
  auto count = [&](int i) -> uint32_t {
    const int x = bin_of(i);
    return (x >= 0 && x < nbins) ? get(x) : 0u;
  };
  uint32_t sum = 0;
  for (int i = 0; i < per; ++i) sum += count(i);
  // inclusive scan over the threads: within warps by shuffles, then warp totals
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
      const uint32_t c = count(i);
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
// pair under (key descending, position ascending).  hist: 4096 words.  Once a
// level leaves at most kRankMax elements in the chosen bin, they are ranked
// by direct comparison (positions break key ties), which ends the select.
constexpr uint32_t kRankMax = 256;

template <class Elem>
__device__ void radix_resolve(Elem elem, uint32_t n, uint32_t B1, uint32_t need, uint32_t max_pos, uint32_t* hist,
                              uint32_t* scan, uint32_t& Ks, uint32_t& Is) {
  const int t = threadIdx.x;
  uint32_t prefix = B1 << 20, mask = 0xFFF00000u;
  // key bits 19..12, 11..4 (256 bins each), then 3..0 (16 bins), from the top
  constexpr int kLevels = 3;
  uint32_t last = 0;
  for (int lv = 0; lv < kLevels; ++lv) {
    const int shift = lv == 0 ? 12 : (lv == 1 ? 4 : 0);
    const int nb = lv < 2 ? 256 : 16;
    const uint32_t dmask = (uint32_t)nb - 1;
    for (int i = t; i < nb; i += kSelThreads) hist[i] = 0;
    __syncthreads();
    for (uint32_t i = t; i < n; i += kSelThreads) {
      uint32_t key, pos;
      elem(i, key, pos);
      if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & dmask], 1u);
    }
    __syncthreads();
    uint32_t bin, before;
    block_cut([&](int i) { return hist[i]; }, nb, need, true, scan, bin, before);
    const uint32_t in_bin = hist[bin];
    prefix |= bin << shift;
    mask |= dmask << shift;
    need -= before;
    last = bin;
    if (in_bin <= kRankMax) {
      // the need-th best of the few left: the one with need-1 better pairs
      uint32_t* sk = hist + 1024;
      uint32_t* sp = sk + kRankMax;
      if (t == 0) scan[255] = 0;
      __syncthreads();
      for (uint32_t i = t; i < n; i += kSelThreads) {
        uint32_t key, pos;
        elem(i, key, pos);
        if ((key & mask) == prefix) {
          const uint32_t slot = atomicAdd(&scan[255], 1u);
          sk[slot] = key;
          sp[slot] = pos;
        }
      }
      __syncthreads();
      const uint32_t m = scan[255];
      if ((uint32_t)t < m) {
        const uint32_t k0 = sk[t], p0 = sp[t];
        uint32_t r = 0;
        for (uint32_t u = 0; u < m; ++u) r += (sk[u] > k0 || (sk[u] == k0 && sp[u] < p0)) ? 1u : 0u;
        if (r == need - 1) {
          scan[256] = k0;
          scan[257] = p0;
        }
      }
      __syncthreads();
      Ks = scan[256];
      Is = scan[257];
      __syncthreads();
      return;
    }
  }
  Ks = prefix;
  // every element equal to K* is kept: no position cut needed
  const uint32_t n_eq = hist[last];
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
    for (int i = t; i < 256; i += kSelThreads) hist[i] = 0;
    __syncthreads();
    for (uint32_t i = t; i < n; i += kSelThreads) {
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

// ============================================================ selection
// One cluster of up to kSelCluster CTAs per row turns the row's keys into its kept
// positions, ascending.  Each CTA owns a contiguous range of positions, staged
// in shared memory by bulk copies together with the row's histogram; each
// warp owns a contiguous segment of the staged range:
//   1. every CTA finds the boundary bin B1 of the row's 4096-bin histogram
//      (the bin holding the kk-th best key) and the count above it;
//   2. each warp lists, in position order, its keys at or above B1 (a few
//      per cent of the keys: every kept key and the boundary candidates);
//   3. every CTA stores the boundary candidates of its lists into CTA 0's
//      shared memory (distributed shared memory); CTA 0 resolves the exact
//      kk-th pair (K*, I*) and stores it into every CTA;
//   4. every CTA counts its kept list entries, stores the count into the CTAs
//      after it (their output offsets) and writes its kept positions in order.
// A list that overflows, or a range longer than one staged chunk, switches the
// row to the general path: (K*, I*) resolved over the whole row, then counts
// and writes from full scans of the staged keys.  Every CTA reaches every
// cluster barrier, also after a failed wait.
constexpr int kSelCluster = 8;
constexpr int kSelChunk = 16384;    // keys staged in shared memory at a time
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kWarpList = 256;      // keys at or above B1 listed per warp segment
static_assert(kSelCluster <= kSelThreads, "one thread per cluster CTA stores the shared values");
static_assert(2 * kCandCap >= (kBins / 16) * 17, "the padded histogram fits the candidate buffers");

struct SelShared {
  uint64_t bar;
  uint32_t scan[258];
  uint32_t wcnt[kSelWarps];         // kept positions per warp segment
  uint32_t pre[kSelCluster];        // kept positions of each CTA before this one (stored by them)
  uint32_t gtotal;                  // CTA 0: the row's boundary candidates (stored by every CTA)
  uint32_t spill;                   // CTA 0 collects, then every CTA holds: 1 = general path
  uint32_t ks, is;                  // stored by CTA 0: the kk-th kept pair (K*, I*)
  int abort;
};

size_t select_smem() {
  return sizeof(uint32_t) * ((size_t)kSelChunk + kBins + 2 * (size_t)kCandCap + 2 * kSelWarps * kWarpList) + 1024;
}

__device__ __forceinline__ uint32_t warp_sum_u32(uint32_t v) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__global__ void __launch_bounds__(kSelThreads) dsa_select_kernel(const DsaArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint32_t* kc = reinterpret_cast<uint32_t*>(align1024(smem_raw));   // [kSelChunk] staged keys
  uint32_t* h2 = kc + kSelChunk;                       // [kBins] the row's histogram, then radix scratch
  uint32_t* ck = h2 + kBins;                           // [kCandCap] CTA 0: the row's candidates (keys)
  uint32_t* cp = ck + kCandCap;                        // [kCandCap] their positions
  uint32_t* lk = cp + kCandCap;                        // [kSelWarps][kWarpList] keys >= B1 per warp
  uint32_t* lp = lk + kSelWarps * kWarpList;           // their positions
  __shared__ SelShared sh;
  const uint32_t rank = cluster_rank(), nr = cluster_size();
  const int b = blockIdx.y;
  const int t = threadIdx.x, lane = lane_id(), warp = warp_id();
  const uint32_t lt = (1u << lane) - 1u;
  // this CTA's share of the row by capacity: known before the row's length is
  // read, so the first copy starts at once
  const int per = ((a.T + (int)nr - 1) / (int)nr + 255) / 256 * 256;
  const int c0 = min(a.T, (int)rank * per), c1 = min(a.T, c0 + per);
  const uint32_t* keys = a.keys + (size_t)b * a.kstride;
  if (t == 0) {
    mbar_init(&sh.bar, 1);
    sh.gtotal = 0;
    sh.spill = 0;
    sh.abort = 0;
    fence_barrier_init();
  }
  if (t < kSelCluster) sh.pre[t] = 0;
  pdl_launch_dependents();
  // the keys and the histogram come from the indexer
  pdl_wait();
  __syncthreads();
  // chunk c of the share (with the first, the histogram), copied in whole
  // 16-byte groups (the row stride is a multiple of 64 keys, so the copy stays
  // inside the row); issued by thread 0
  auto issue = [&](int c, bool with_hist) {
    const int s = c0 + c * kSelChunk;
    const int n = max(0, min(kSelChunk, c1 - s));
    const uint32_t bytes = (uint32_t)((n + 3) / 4) * 16u;
    mbar_arrive_expect_tx(&sh.bar, bytes + (with_hist ? kBins * 4u : 0u));
    if (with_hist) bulk_load(h2, a.hist + (size_t)b * kBins, kBins * 4u, &sh.bar);
    for (uint32_t off = 0; off < bytes; off += 16384u)
      bulk_load(kc + off / 4, keys + s + off / 4, min(16384u, bytes - off), &sh.bar);
  };
  if (t == 0) issue(0, true);
  // the status cannot change while this kernel runs (nothing in it records a
  // fail-fast error before its last barrier), so all CTAs of a cluster agree
  const int err = prior_error(a.st);
  const RowGeom rg = row_geom(a, b, rank == 0 && t == 0 ? a.st : nullptr);
  int32_t* dst = a.idx + (size_t)b * a.kk;
  int32_t* dst2 = a.idx_out != nullptr ? a.idx_out + (size_t)b * a.kk : nullptr;
  if (!err) {
    // a row that keeps fewer than kk positions: its index row ends in -1
    if (rank == 0)
      for (int e = rg.kk + t; e < a.kk; e += kSelThreads) {
        dst[e] = -1;
        if (dst2) dst2[e] = -1;
      }
    // a row that keeps every position
    if (rg.all)
      for (int pos = min(rg.T, c0) + t; pos < min(rg.T, c1); pos += kSelThreads) {
        dst[pos] = pos;
        if (dst2) dst2[pos] = pos;
      }
  }
  if (err || rg.all) {
    // the copy lands before the shared memory is released
    if (t == 0) mbar_wait_plain(&sh.bar, 0, kWaitLimitNs);
    return;
  }
  // every CTA's counters are initialised before any CTA stores into them (the
  // matching wait comes before the first remote access)
  cluster_arrive();
  const int p0 = min(rg.T, c0), p1 = min(rg.T, c1);
  const int nchunks = (p1 - p0 + kSelChunk - 1) / kSelChunk;
  bool ok = true;
  uint32_t phase = 0;
  auto wait_copy = [&]() {
    const bool got = mbar_wait(&sh.bar, phase, &sh.abort, a.st, 541);
    // every thread continues on the same outcome; a copy still in flight
    // keeps ``phase`` for the drain at the end
    ok = __syncthreads_and(got ? 1 : 0) != 0;
    if (ok) phase ^= 1u;
  };
  // stage chunk c >= 1 of [p0, p1); returns its valid keys
  auto stage = [&](int c, bool) -> int {
    __syncthreads();   // the previous chunk is no longer read
    if (ok) {
      if (t == 0) issue(c, false);
      wait_copy();
    }
    return min(kSelChunk, p1 - (p0 + c * kSelChunk));
  };
  // warp w's segment of a chunk of n keys: [w*S, min(n, (w+1)*S)), S a multiple of 128
  auto seg_len = [&](int n) { return (n + kSelWarps * 128 - 1) / (kSelWarps * 128) * 128; };
  // the four keys of this lane at chunk index i (i < i1 checked per key; the
  // staged copy covers whole 16-byte groups, so the vector load stays inside it)
  auto load4 = [&](int i, int i1, uint32_t (&k4)[4]) {
    const uint4 v = (ok && i < i1) ? *reinterpret_cast<const uint4*>(kc + i) : make_uint4(0u, 0u, 0u, 0u);
    k4[0] = v.x;
    k4[1] = v.y;
    k4[2] = v.z;
    k4[3] = v.w;
  };

  // ---- 1. boundary bin of the first radix level (through a copy of the
  // histogram padded to 17 words per 16 bins: conflict-free for the cut)
  wait_copy();
  int n_last = nchunks > 0 ? min(kSelChunk, p1 - p0) : 0;
  uint32_t* hp = ck;   // spans ck and cp, both unused until step 3
  for (int j = 0; j < kBins / kSelThreads; ++j) {
    const int f = j * kSelThreads + t;
    hp[(f >> 4) * 17 + (f & 15)] = h2[f];
  }
  __syncthreads();
  uint32_t B1, above;
  block_cut([&](int i) { return hp[(i >> 4) * 17 + (i & 15)]; }, kBins, (uint32_t)rg.kk, true, sh.scan, B1, above);
  // ---- 2. each warp lists its keys at or above B1, in position order
  uint32_t wn = 0;
  for (int c = 0; c < nchunks; ++c) {
    const int n = c == 0 ? n_last : stage(c, false);
    n_last = n;
    const int s = p0 + c * kSelChunk;
    const int S = seg_len(n);
    const int i0 = min(n, warp * S), i1 = min(n, i0 + S);
    for (int base = i0; base < i1; base += 128) {
      const int i = base + 4 * lane;
      uint32_t k4[4];
      load4(i, i1, k4);
      unsigned m[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) m[j] = __ballot_sync(0xffffffffu, ok && i + j < i1 && (k4[j] >> 20) >= B1);
      if (m[0] | m[1] | m[2] | m[3]) {
        uint32_t slot = wn + __popc(m[0] & lt) + __popc(m[1] & lt) + __popc(m[2] & lt) + __popc(m[3] & lt);
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if ((m[j] >> lane) & 1u) {
            if (slot < (uint32_t)kWarpList) {
              lk[warp * kWarpList + slot] = k4[j];
              lp[warp * kWarpList + slot] = (uint32_t)(s + i + j);
            }
            ++slot;
          }
        wn += __popc(m[0]) + __popc(m[1]) + __popc(m[2]) + __popc(m[3]);
      }
    }
  }
  // ---- 3. boundary candidates into CTA 0, which resolves (K*, I*)
  cluster_wait();
  {
    const uint32_t a_tot = dsmem_addr(&sh.gtotal, 0), a_ck = dsmem_addr(ck, 0), a_cp = dsmem_addr(cp, 0);
    if (wn > (uint32_t)kWarpList) {
      if (lane == 0) dsmem_atomic_or_u32(dsmem_addr(&sh.spill, 0), 1u);
    } else {
      for (uint32_t i0 = 0; i0 < wn; i0 += 32) {
        const uint32_t i = i0 + lane;
        const uint32_t key = i < wn ? lk[warp * kWarpList + i] : 0u;
        const bool cand = i < wn && (key >> 20) == B1;
        const unsigned m = __ballot_sync(0xffffffffu, cand);
        if (!m) continue;
        uint32_t slot = 0;
        if (lane == 0) slot = dsmem_atomic_add_u32(a_tot, (uint32_t)__popc(m));
        slot = __shfl_sync(0xffffffffu, slot, 0) + __popc(m & lt);
        if (cand && slot < (uint32_t)kCandCap) {
          dsmem_st_u32(a_ck + 4 * slot, key);
          dsmem_st_u32(a_cp + 4 * slot, lp[warp * kWarpList + i]);
        }
      }
    }
  }
  cluster_sync();
  if (rank == 0) {
    const uint32_t total = sh.gtotal;
    const uint32_t spill = (sh.spill || nchunks > 1 || total > (uint32_t)kCandCap) ? 1u : 0u;
    const uint32_t need1 = (uint32_t)rg.kk - above;
    uint32_t Ks, Is;
    if (!spill) {
      radix_resolve([&](uint32_t i, uint32_t& key, uint32_t& pos) { key = ck[i]; pos = cp[i]; }, total, B1, need1,
                    (uint32_t)(rg.T - 1), h2, sh.scan, Ks, Is);
    } else {
      radix_resolve([&](uint32_t i, uint32_t& key, uint32_t& pos) { key = __ldcg(keys + i); pos = i; },
                    (uint32_t)rg.T, B1, need1, (uint32_t)(rg.T - 1), h2, sh.scan, Ks, Is);
    }
    if (t < (int)nr) {
      dsmem_st_u32(dsmem_addr(&sh.ks, t), Ks);
      dsmem_st_u32(dsmem_addr(&sh.is, t), Is);
      dsmem_st_u32(dsmem_addr(&sh.spill, t), spill);
    }
  }
  cluster_sync();
  const uint32_t Ks = sh.ks, Is = sh.is;
  const bool general = sh.spill != 0;
  // ---- 4. kept positions per warp segment
  // general path: a full scan of a staged chunk
  auto count_chunk = [&](int c, int n) {
    const int s = p0 + c * kSelChunk;
    const int S = seg_len(n);
    const int i0 = min(n, warp * S), i1 = min(n, i0 + S);
    uint32_t cnt = 0;
    for (int base = i0; base < i1; base += 128) {
      const int i = base + 4 * lane;
      uint32_t k4[4];
      load4(i, i1, k4);
#pragma unroll
      for (int j = 0; j < 4; ++j) cnt += (ok && i + j < i1 && kept(k4[j], (uint32_t)(s + i + j), Ks, Is)) ? 1u : 0u;
    }
    cnt = warp_sum_u32(cnt);
    __syncthreads();
    if (lane == 0) sh.wcnt[warp] = cnt;
    __syncthreads();
  };
  uint32_t kept_total = 0;
  if (!general) {
    uint32_t cnt = 0;
    for (uint32_t i = lane; i < wn; i += 32)
      cnt += kept(lk[warp * kWarpList + i], lp[warp * kWarpList + i], Ks, Is) ? 1u : 0u;
    cnt = warp_sum_u32(cnt);
    if (lane == 0) sh.wcnt[warp] = cnt;
    __syncthreads();
#pragma unroll
    for (int w = 0; w < kSelWarps; ++w) kept_total += sh.wcnt[w];
  } else {
    for (int c = 0; c < nchunks; ++c) {
      const int n = nchunks > 1 ? stage(c, false) : n_last;
      count_chunk(c, n);
#pragma unroll
      for (int w = 0; w < kSelWarps; ++w) kept_total += sh.wcnt[w];
    }
  }
  // this CTA's count into the offsets of the CTAs after it
  if (t > (int)rank && t < (int)nr) dsmem_st_u32(dsmem_addr(&sh.pre[rank], t), kept_total);
  cluster_sync();
  uint32_t run = 0;
  for (uint32_t r = 0; r < rank; ++r) run += sh.pre[r];
  // ---- kept positions in order: warp w writes its segment after the segments before it
  auto put = [&](uint32_t e, int pos) {
    if (e < (uint32_t)rg.kk) {
      dst[e] = pos;
      if (dst2) dst2[e] = pos;
    }
  };
  if (!general) {
    uint32_t o = run;
    for (int w = 0; w < warp; ++w) o += sh.wcnt[w];
    for (uint32_t i0 = 0; i0 < wn; i0 += 32) {
      const uint32_t i = i0 + lane;
      const bool k = i < wn && kept(lk[warp * kWarpList + i], lp[warp * kWarpList + i], Ks, Is);
      const unsigned m = __ballot_sync(0xffffffffu, k);
      if (k) put(o + __popc(m & lt), (int)lp[warp * kWarpList + i]);
      o += __popc(m);
    }
  } else {
    for (int c = 0; c < nchunks; ++c) {
      int n = n_last;
      if (nchunks > 1) {
        n = stage(c, false);
        count_chunk(c, n);
      }
      const int s = p0 + c * kSelChunk;
      const int S = seg_len(n);
      const int i0 = min(n, warp * S), i1 = min(n, i0 + S);
      uint32_t o = run;
      for (int w = 0; w < warp; ++w) o += sh.wcnt[w];
      for (int base = i0; base < i1; base += 128) {
        const int i = base + 4 * lane;
        uint32_t k4[4];
        load4(i, i1, k4);
        bool f[4];
        unsigned m[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          f[j] = ok && i + j < i1 && kept(k4[j], (uint32_t)(s + i + j), Ks, Is);
          m[j] = __ballot_sync(0xffffffffu, f[j]);
        }
        uint32_t e = o + __popc(m[0] & lt) + __popc(m[1] & lt) + __popc(m[2] & lt) + __popc(m[3] & lt);
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (f[j]) put(e++, s + i + j);
        o += __popc(m[0]) + __popc(m[1]) + __popc(m[2]) + __popc(m[3]);
      }
#pragma unroll
      for (int w = 0; w < kSelWarps; ++w) run += sh.wcnt[w];
    }
  }
  // a failed copy: wait (bounded) for it before the shared memory is released
  if (!ok && t == 0) mbar_wait_plain(&sh.bar, phase, kWaitLimitNs);
}

// ============================================================ attention (tcgen05)
// One CTA = 64 kept positions of one row, two CTAs per SM: the gather-attention
// design of the selected-block branch, with keys as the M side and the (up to
// 16) heads as N:
//     S^T[key, head] = K_sel[key, :] . q[head, :]           (dk/64 chunks x 4 MMAs)
//     exact softmax of the tile per head (max, exp, sum), P^T bf16 in smem
//     O^T[dv, head] = V_sel^T[dv, key] . P^T[key, head]     (dv/128 tiles x 4 MMAs)
// The kept rows are gathered four at a time by TMA tile::gather4 into the
// 128-byte-swizzled K-major layout the MMAs read; every 64-column chunk of the
// tile's keys stays resident, 8 KB apart.  The QK^T MMAs keep M = 128: rows
// 64..127 of a chunk's operand are the next chunk's rows (the last chunk is
// followed by a spare slot), and their S^T lanes are never read.  Values reuse
// the key slots once the QK^T MMAs have drained them (latent KV: the first
// dv/64 key chunks are the values, so nothing more is fetched).  The tile's
// (max, sum, O^T) goes to the merge.
constexpr int kTcThreads = 192;         // warps 0-1 softmax, 0-3 epilogue, 4 gather, 5 MMA issuer
constexpr int kTcKeys = 64;             // kept positions per CTA
constexpr int kTcMaxChunks = 10;        // resident 64-column chunks: dk <= 640
constexpr int kTcChunk = kTcKeys * 128; // 8 KB

struct TcBars {
  uint64_t q_full;
  uint64_t k_full[kTcMaxChunks];
  uint64_t v_full;
  uint64_t s_full;     // QK^T done: softmax may read S^T
  uint64_t qk_done;    // QK^T done: the gather may overwrite key slots with values
  uint64_t p_full;     // P^T written (2 softmax warps)
  uint64_t o_full;
  uint64_t wg;         // softmax warps' rendezvous
  uint64_t drain;
  uint32_t tmem;
  int abort_flag;
};

struct TcLayout {
  uint32_t k_off, p_off, red_off, rows_off, bar_off, total;
};

__host__ __device__ inline int tc_value_chunks(int dv) { return dv / 64 < 2 ? 2 : dv / 64; }

__host__ __device__ inline TcLayout tc_layout(int dk, int dv) {
  const int nk = dk / 64;
  // key chunks (or value chunks, padded to a pair) plus the spare slot the
  // last chunk's M = 128 operand reads into
  const int nslots = (nk > tc_value_chunks(dv) ? nk : tc_value_chunks(dv)) + 1;
  TcLayout L;
  L.k_off = (uint32_t)(((nk * 2048) + 1023) / 1024 * 1024);   // q: nk chunks of 16 rows x 128 B
  L.p_off = L.k_off + (uint32_t)nslots * kTcChunk;              // P^T: 16 rows x 128 B
  L.red_off = L.p_off + 2048;                                   // [2 m/l][2 warps][16] floats
  L.rows_off = L.red_off + 2 * 2 * 16 * 4;                      // [64] gathered row indices
  L.bar_off = L.rows_off + kTcKeys * 4;
  L.total = L.bar_off + 256 + 1024;                             // + alignment slack
  return L;
}

// Four rows (global row indices r0..r3) of 64 columns starting at column col,
// into 4 consecutive 128-byte swizzled rows.
__device__ __forceinline__ void tma_gather4(void* dst, const CUtensorMap* map, uint64_t* bar, int col, int r0, int r1,
                                            int r2, int r3) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
      "%3, %4, %5, %6}], [%7];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(col), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "r"(smem_u32(bar))
      : "memory");
}

template <int DV>
__global__ void __launch_bounds__(kTcThreads, 2)
    dsa_attn_kernel(const __grid_constant__ CUtensorMap mapQ, const __grid_constant__ CUtensorMap mapK,
                    const __grid_constant__ CUtensorMap mapV, const DsaArgs a) {
  constexpr int kVC = DV / 64 < 2 ? 2 : DV / 64;   // value chunks, padded to one M = 128 pair
  constexpr int kVT = kVC / 2;                        // 128-row value tiles
  constexpr int kG4 = kTcKeys / 4;                    // gather4 copies per chunk
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const TcLayout L = tc_layout(a.dk, DV);
  uint8_t* qs = smem;
  uint8_t* ks = smem + L.k_off;
  uint8_t* ps = smem + L.p_off;
  float* red_m = reinterpret_cast<float*>(smem + L.red_off);   // [2][16]
  float* red_l = red_m + 32;                                     // [2][16]
  int* rows_s = reinterpret_cast<int*>(smem + L.rows_off);
  TcBars* bars = reinterpret_cast<TcBars*>(smem + L.bar_off);
  volatile int* abort_flag = &bars->abort_flag;
  const int x = blockIdx.x, b = blockIdx.y;
  const int warp = warp_id(), lane = lane_id();
  const int nk = a.dk / 64;
  const RowGeom rg = row_geom(a, b, nullptr);
  const int e0 = x * kTcKeys;
  const int nent = min(kTcKeys, rg.kk - e0);
  const size_t pb = (size_t)b * a.attn_ctas + x;
  // a row that keeps fewer positions than this tile starts at has no
  // partial here (the merge reads only a row's own tiles)
  if (nent <= 0) return;
  pdl_launch_dependents();
  // query rows H..15 are never loaded: keep them finite (zero)
  if (a.H < 16)
    for (int i = threadIdx.x; i < nk * 2048 / 16; i += kTcThreads) {
      const int row = (i % 128) / 8;
      if (row >= a.H) reinterpret_cast<uint4*>(qs)[i] = make_uint4(0, 0, 0, 0);
    }
  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    for (int c = 0; c < kTcMaxChunks; ++c) mbar_init(&bars->k_full[c], 1);
    mbar_init(&bars->v_full, 1);
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->qk_done, 1);
    mbar_init(&bars->p_full, 2);
    mbar_init(&bars->o_full, 1);
    mbar_init(&bars->wg, 2);
    mbar_init(&bars->drain, 1);
    fence_barrier_init();
    // the query is an input: its load overlaps the previous kernel's tail
    tma_prefetch_desc(&mapQ);
    tma_prefetch_desc(&mapK);
    mbar_arrive_expect_tx(&bars->q_full, (uint32_t)(nk * a.H * 128));
    for (int c = 0; c < nk; ++c) tma_load_2d(qs + c * 2048, &mapQ, &bars->q_full, c * 64, b * a.H);
  }
  if (warp == 0) {
    tmem_alloc(&bars->tmem, 128);
    tmem_relinquish();
  }
  // the kept positions and the status come from the previous kernels
  pdl_wait();
  if (threadIdx.x == 0) bars->abort_flag = prior_error(a.st);
  // the tile's global row indices; entries past the row's last kept position
  // repeat its first one (finite data, masked out of the softmax)
  const int32_t* sel = a.idx + (size_t)b * a.kk + e0;
  const int seq_row0 = (b / a.rows_per_seq) * a.T;   // the sequence's first key row
  for (int j = threadIdx.x; j < kTcKeys; j += kTcThreads) rows_s[j] = seq_row0 + __ldg(sel + (j < nent ? j : 0));
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem;          // S^T at columns 0..15, O^T tile t at 16 + 16 t
  bool ok = *abort_flag == 0;

  if (!ok) {
    // an earlier CTA failed: only the query load is in flight
    if (threadIdx.x == 0) mbar_wait_plain(&bars->q_full, 0, kWaitLimitNs);
  } else if (warp == 4) {
    // ============================================================ gather (one warp)
    // lane 0 arms every barrier; lane j < kG4 then gathers rows 4j .. 4j+3 of each chunk
    if (lane == 0)
      for (int c = 0; c < nk; ++c) mbar_arrive_expect_tx(&bars->k_full[c], kTcChunk);
    __syncwarp();
    int4 rw = make_int4(0, 0, 0, 0);
    if (lane < kG4) rw = *reinterpret_cast<const int4*>(rows_s + 4 * lane);
    if (lane < kG4)
      for (int c = 0; c < nk; ++c)
        tma_gather4(ks + c * kTcChunk + lane * 512, &mapK, &bars->k_full[c], c * 64, rw.x, rw.y, rw.z, rw.w);
    bool vok = true;
    if (!a.v_from_k) {
      // the value chunks overwrite key slots 0 .. DV/64-1 once QK^T has read them
      if (lane == 0) {
        vok = mbar_wait(&bars->qk_done, 0, abort_flag, a.st, 531);
        if (vok) mbar_arrive_expect_tx(&bars->v_full, (uint32_t)(DV / 64) * kTcChunk);
      }
      vok = __shfl_sync(0xffffffffu, vok ? 1 : 0, 0) != 0;
      if (vok && lane < kG4)
        for (int c = 0; c < DV / 64; ++c)
          tma_gather4(ks + c * kTcChunk + lane * 512, &mapV, &bars->v_full, c * 64, rw.x, rw.y, rw.z, rw.w);
    }
    if (lane == 0 && (!vok || *abort_flag)) {
      // drain every copy issued before the CTA releases its shared memory
      mbar_wait_plain(&bars->q_full, 0, kWaitLimitNs);
      for (int c = 0; c < nk; ++c) mbar_wait_plain(&bars->k_full[c], 0, kWaitLimitNs);
      if (!a.v_from_k && vok) mbar_wait_plain(&bars->v_full, 0, kWaitLimitNs);
    }
  } else if (warp == 5) {
    // ============================================================ MMA issuer (one thread)
    if (lane == 0) {
      const uint32_t idesc_qk = idesc_bf16_f32(128, 16, false, false);
      const uint32_t idesc_pv = idesc_bf16_f32(128, 16, true, false);
      const uint32_t q_a = smem_u32(qs), k_a = smem_u32(ks), p_a = smem_u32(ps);
      bool mok = mbar_wait(&bars->q_full, 0, abort_flag, a.st, 532);
      for (int c = 0; c < nk && mok; ++c) {
        if (!mbar_wait(&bars->k_full[c], 0, abort_flag, a.st, 533)) {
          mok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint64_t ad = sdesc_sw128(k_a + c * kTcChunk + k * 32, 16, 1024);
          const uint64_t bd = sdesc_sw128(q_a + c * 2048 + k * 32, 16, 1024);
          umma_bf16(tmem, ad, bd, idesc_qk, (c > 0 || k > 0) ? 1u : 0u);
        }
      }
      if (mok) {
        umma_commit(&bars->s_full);
        umma_commit(&bars->qk_done);
      }
      if (mok && !mbar_wait(&bars->p_full, 0, abort_flag, a.st, 534)) mok = false;
      if (mok && !a.v_from_k && !mbar_wait(&bars->v_full, 0, abort_flag, a.st, 535)) mok = false;
      if (mok) {
        tc_fence_after();
#pragma unroll
        for (int t = 0; t < kVT; ++t)
#pragma unroll
          for (int k = 0; k < kTcKeys / 16; ++k) {
            // A = V^T: value columns 128 t .. 128 t + 127 as two 64-column
            // chunks one slot apart, keys 16 k .. 16 k + 15 along K
            const uint64_t ad = sdesc_sw128(k_a + 2 * t * kTcChunk + k * 2048, kTcChunk, 1024);
            const uint64_t bd = sdesc_sw128(p_a + k * 32, 16, 1024);
            umma_bf16(tmem + 16 + 16 * t, ad, bd, idesc_pv, k > 0 ? 1u : 0u);
          }
        umma_commit(&bars->o_full);
      }
      if (!mok || *abort_flag) {
        umma_commit(&bars->drain);
        mbar_wait_plain(&bars->drain, 0, kWaitLimitNs);
      }
    }
  } else {
    // ============================================================ softmax (warps 0-1) + epilogue (warps 0-3)
    const int r = warp * 32 + lane;           // TMEM lane: a key of the tile (warps 0-1), a value row
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    if (warp < 2) {
      const bool valid = r < nent;
      uint32_t wg_phase = 0;
      auto wg_sync = [&]() {
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->wg);
        if (!mbar_wait(&bars->wg, wg_phase & 1, abort_flag, a.st, 536)) ok = false;
        ++wg_phase;
      };
      uint32_t sr[16];
      if (!mbar_wait(&bars->s_full, 0, abort_flag, a.st, 537)) ok = false;
      tc_fence_after();
      tmem_ld16(tmem + lane_base, sr);
      tmem_ld_wait(sr);
      float m[16];
#pragma unroll
      for (int h = 0; h < 16; ++h) m[h] = warp_max_f32(valid ? __uint_as_float(sr[h]) * a.sc2 : -INFINITY);
      if (lane == 0)
#pragma unroll
        for (int h = 0; h < 16; ++h) red_m[warp * 16 + h] = m[h];
      wg_sync();
#pragma unroll
      for (int h = 0; h < 16; ++h) {
        m[h] = fmaxf(red_m[h], red_m[16 + h]);
        if (m[h] == -INFINITY) m[h] = 0.f;
      }
      // p = exp2(s * scale - max) as P^T (bf16, key-major rows of heads), sums
      float ls[16];
#pragma unroll
      for (int h = 0; h < 16; ++h) {
        const float e = valid ? fast_exp2(fmaf(__uint_as_float(sr[h]), a.sc2, -m[h])) : 0.f;
        ls[h] = e;
        *reinterpret_cast<__nv_bfloat16*>(ps + sw128_offset(h, r >> 3) + (r & 7) * 2) = __float2bfloat16_rn(e);
      }
      tc_fence_before();
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->p_full);
      const float ws = warp_sum16(ls, lane);
      if ((lane & 1) == 0) red_l[warp * 16 + head_of_lane(lane)] = ws;
      wg_sync();
      if (ok && threadIdx.x < 16) {
        const int h = threadIdx.x;
        const float mh = fmaxf(red_m[h], red_m[16 + h]);
        a.pm[pb * 16 + h] = mh == -INFINITY ? 0.f : mh;
        a.pl[pb * 16 + h] = red_l[h] + red_l[16 + h];
      }
    }
    // unnormalised O^T of the tile: lane r holds value row 128 t + r, 16 heads
    if (ok && mbar_wait(&bars->o_full, 0, abort_flag, a.st, 538)) {
      tc_fence_after();
#pragma unroll
      for (int t = 0; t < kVT; ++t) {
        uint32_t orr[16];
        tmem_ld16(tmem + lane_base + 16 + 16 * t, orr);
        tmem_ld_wait(orr);
        const int d = 128 * t + r;
        if (d < DV) {
          float* dst = a.po + pb * 16 * DV + d;
#pragma unroll
          for (int h = 0; h < 16; ++h) dst[(size_t)h * DV] = __uint_as_float(orr[h]);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, 128);
}

// Merge of a row's attention splits: out[b,h,:] = sum_c w_c O_c / sum_c w_c l_c,
// w_c = exp(m_c - max m).  One CTA per (head, row), one thread per 4 columns.
constexpr int kMergeGroups = 4;   // partial subsets summed in parallel per column

template <int DV>
__global__ void __launch_bounds__(DV / 4 * kMergeGroups) dsa_merge_kernel(const DsaArgs a) {
  constexpr int C4 = DV / 4;            // float4 columns
  const int h = blockIdx.x, b = blockIdx.y;
  const int NC = a.attn_ctas;                                   // partial stride per row
  const int NR = (row_geom(a, b, nullptr).kk + kTcKeys - 1) / kTcKeys;   // this row's partials
  __shared__ float Ms, iLs;
  __shared__ int s_abort;
  __shared__ float4 part[kMergeGroups - 1][C4];
  // the partials come from the attention kernel
  pdl_wait();
  if (threadIdx.x == 0) s_abort = prior_error(a.st);
  __syncthreads();
  if (s_abort) return;
  const float* pm = a.pm + (size_t)b * NC * 16 + h;
  const float* pl = a.pl + (size_t)b * NC * 16 + h;
  if (threadIdx.x < 32) {
    float M = -INFINITY;
    for (int c = threadIdx.x; c < NR; c += 32) M = fmaxf(M, __ldcg(pm + (size_t)c * 16));
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    const float Mu = M == -INFINITY ? 0.f : M;
    float L = 0.f;
    for (int c = threadIdx.x; c < NR; c += 32)
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
  for (int c0 = grp * 8; c0 < NR; c0 += 8 * kMergeGroups) {
    float4 v[8];
    float f[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int c = c0 + k;
      v[k] = c < NR ? __ldcg(reinterpret_cast<const float4*>(po + (size_t)c * 16 * DV)) : make_float4(0.f, 0.f, 0.f, 0.f);
      f[k] = c < NR ? __ldcg(pm + (size_t)c * 16) : -INFINITY;
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
  size_t hist, zero_end, keys, idx, pm, pl, po, end;
};

struct DsaShape {
  int kk, attn_ctas, all, kstride;
};

DsaShape dsa_shape(const dsa_cfg& c) {
  DsaShape s;
  s.kk = c.topk < c.T ? c.topk : c.T;
  s.all = s.kk == c.T ? 1 : 0;
  s.attn_ctas = (s.kk + kTcKeys - 1) / kTcKeys;
  s.kstride = (c.T + 63) / 64 * 64;
  return s;
}

DsaWs dsa_ws(const dsa_cfg& c) {
  const DsaShape s = dsa_shape(c);
  const size_t B = (size_t)c.B;
  DsaWs w;
  w.hist = align_up(sizeof(DeviceStatus), 256);
  w.zero_end = align_up(w.hist + sizeof(uint32_t) * B * kBins, 256);
  w.keys = w.zero_end;
  w.idx = align_up(w.keys + sizeof(uint32_t) * B * (size_t)s.kstride, 256);
  w.pm = align_up(w.idx + sizeof(int32_t) * B * (size_t)s.kk, 256);
  w.pl = align_up(w.pm + sizeof(float) * B * s.attn_ctas * 16, 256);
  w.po = align_up(w.pl + sizeof(float) * B * s.attn_ctas * 16, 256);
  w.end = align_up(w.po + sizeof(float) * B * s.attn_ctas * 16 * (size_t)c.dv, 256);
  return w;
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

int launch_select(const DsaArgs& a, cudaStream_t s) {
  const size_t smem = select_smem();
  if (int rc = ensure_smem_attr(reinterpret_cast<const void*>(&dsa_select_kernel), smem)) return rc;
  // one CTA per staged chunk of the row, at most kSelCluster: a row that fits
  // one chunk (the prefill's short rows) runs on a single CTA
  int cl = (a.T + kSelChunk - 1) / kSelChunk;
  cl = cl < 1 ? 1 : (cl > kSelCluster ? kSelCluster : cl);
  prof::begin("dsa_select", s);
  const int rc = launch_dependent(dsa_select_kernel, dim3(cl, a.B), dim3(kSelThreads), smem, s, cl, a);
  prof::end(s);
  return rc;
}

template <int DV>
int launch_attn(const DsaArgs& a, cudaStream_t s) {
  const TcLayout L = tc_layout(a.dk, DV);
  // each CTA holds 128 TMEM columns: at most 4 may share an SM, so a small
  // layout asks for enough shared memory to keep the count there
  size_t smem = L.total;
  const size_t floor4 = (size_t)smem_max() / 4 + 1024;
  if (smem < floor4) smem = floor4;
  if (int rc = ensure_smem_attr(reinterpret_cast<const void*>(&dsa_attn_kernel<DV>), smem)) return rc;
  // q as [B*H, dk] in boxes of 64 columns x H heads; k and v as [B*T, d] rows
  // fetched one row per gathered coordinate
  CUtensorMap mq, mk, mv;
  {
    const uint64_t dims[2] = {(uint64_t)a.dk, (uint64_t)a.B * a.H};
    const uint64_t str[1] = {(uint64_t)a.dk * 2};
    const uint32_t box[2] = {64, (uint32_t)a.H};
    if (!make_tmap_bf16(&mq, a.q, 2, dims, str, box)) return NSA_ERR_CUDA;
  }
  {
    const uint64_t dims[2] = {(uint64_t)a.dk, (uint64_t)a.nseq * a.T};
    const uint64_t str[1] = {(uint64_t)a.dk * 2};
    const uint32_t box[2] = {64, 1};
    if (!make_tmap_bf16(&mk, a.k, 2, dims, str, box)) return NSA_ERR_CUDA;
  }
  if (a.v_from_k) {
    mv = mk;
  } else {
    const uint64_t dims[2] = {(uint64_t)DV, (uint64_t)a.nseq * a.T};
    const uint64_t str[1] = {(uint64_t)DV * 2};
    const uint32_t box[2] = {64, 1};
    if (!make_tmap_bf16(&mv, a.v, 2, dims, str, box)) return NSA_ERR_CUDA;
  }
  prof::begin("dsa_attn", s);
  int rc = launch_dependent(dsa_attn_kernel<DV>, dim3(a.attn_ctas, a.B), dim3(kTcThreads), smem, s, 1, mq, mk, mv, a);
  prof::end(s);
  if (rc != NSA_OK) return rc;
  prof::begin("dsa_merge", s);
  rc = launch_dependent(dsa_merge_kernel<DV>, dim3(a.H, a.B), dim3(DV / 4 * kMergeGroups), 0, s, 1, a);
  prof::end(s);
  return rc;
}

}  // namespace

int dsa_supported(const dsa_cfg& c) {
  if (c.HI < 1 || c.HI > 8) return NSA_ERR_UNSUPPORTED;
  if (c.dI != 64 && c.dI != 128 && c.dI != 256) return NSA_ERR_UNSUPPORTED;
  if (c.H < 1 || c.H > 16) return NSA_ERR_UNSUPPORTED;
  if (c.dk % 64 != 0 || c.dk > 64 * kTcMaxChunks) return NSA_ERR_UNSUPPORTED;
  if (c.dv != 64 && c.dv != 128 && c.dv != 256 && c.dv != 512) return NSA_ERR_UNSUPPORTED;
  if (c.B > 65535 || c.T > (1 << 28)) return NSA_ERR_UNSUPPORTED;
  if (tc_layout(c.dk, c.dv).total > smem_max()) return NSA_ERR_UNSUPPORTED;
  if (select_smem() + sizeof(SelShared) + 1024 > smem_max()) return NSA_ERR_UNSUPPORTED;
  return NSA_OK;
}

size_t dsa_ws_bytes(const dsa_cfg& c) { return dsa_ws(c).end; }
size_t dsa_zero_bytes(const dsa_cfg& c) { return dsa_ws(c).zero_end; }

int launch_dsa(const dsa_cfg& c, const void* qI, const void* wI, const void* kI, const void* q, const void* k,
               const void* v, const int32_t* lens, void* out, int32_t* idx_out, uint8_t* ws, cudaStream_t s,
               int rows_per_seq) {
  const DsaShape sh = dsa_shape(c);
  const DsaWs w = dsa_ws(c);
  DsaArgs a;
  a.B = c.B;
  a.rows_per_seq = rows_per_seq;
  a.nseq = c.B / rows_per_seq;
  a.T = c.T;
  a.HI = c.HI;
  a.dI = c.dI;
  a.H = c.H;
  a.dk = c.dk;
  a.dv = c.dv;
  a.kk = sh.kk;
  a.topk = c.topk;
  a.lens = lens;
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
  a.kstride = sh.kstride;
  a.hist = reinterpret_cast<uint32_t*>(ws + w.hist);
  a.idx = reinterpret_cast<int32_t*>(ws + w.idx);
  a.pm = reinterpret_cast<float*>(ws + w.pm);
  a.pl = reinterpret_cast<float*>(ws + w.pl);
  a.po = reinterpret_cast<float*>(ws + w.po);
  a.st = reinterpret_cast<DeviceStatus*>(ws);
  int rc = NSA_OK;
  if (!sh.all) {
    CUtensorMap map;
    const uint64_t dims[3] = {(uint64_t)c.dI, (uint64_t)c.T, (uint64_t)a.nseq};
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
  }
  if ((rc = launch_select(a, s)) != NSA_OK) return rc;
  switch (c.dv) {
    case 64: return launch_attn<64>(a, s);
    case 128: return launch_attn<128>(a, s);
    case 256: return launch_attn<256>(a, s);
    case 512: return launch_attn<512>(a, s);
    default: return NSA_ERR_UNSUPPORTED;
  }
}

}  // namespace nsa
