// prefill_cmp_win.cu -- NSA prefill, per (sequence, KV group, tile of queries):
//   0. sliding-window attention over (t-w, t] [P2 II.3; P3], one pass with an
//      online softmax: both softmax warpgroups share each row's reference max
//      (exchanged once per key tile) and rescale their half of O, while O is
//      idle, when the max grows by more than 2^8; at the end O is scaled by
//      g_win / sum.  The window runs first so that these rescales never touch
//      the compressed branch's part of O;
//   1. compressed attention [P2 II.1; P3 token compression], two passes over
//      the compressed keys: pass 1 finds each row's softmax max and sum, pass 2
//      recomputes the scores, forms the exactly normalised probabilities p,
//      accumulates O_cmp and the block importance scores
//          S[t,j] = sum_{h in group} sum_i w(i,j) p[t,h,i]
//      (w = d-token chunks shared by compressed block i and selection block j);
//   2. top-n block selection [P2 II: n blocks incl. block 0 and the 2 local
//      blocks; P3 token selection], ties to the lower block index.
// Dense mode (``dense``): step 0 alone with w >= T and gate 1, i.e. exact
// causal full attention -- the comparison the pages quote NSA's speed-ups
// against [P2 III.3] -- written straight to the output.
// The gates are folded into the probabilities (P' = g * p), so one TMEM
// accumulator holds g_cmp*O_cmp + g_win*O_win; that partial sum is written in
// fp32 (an accumulation intermediate: the output is rounded to bf16 once) and
// the selected-attention kernel adds g_slc*O_slc to it.
//
// Rows of the MMA are (query, head) pairs of ONE GQA group: 128/HPG queries x
// HPG heads share every K/V tile (group-centric loading).  Warp roles:
//   warps 0-3, 4-7  softmax / scores / top-k; thread = one row (TMEM lane),
//                   warpgroup 0 takes key columns 0-63 of every S tile,
//                   warpgroup 1 columns 64-127 (per-row max/sum are merged
//                   between the two at the end of a statistics pass)
//   warp  8         TMA producer: Q once, then the key chunks (16 KB ring)
//   warp  9         QK^T issuer (single thread), ahead by the two S buffers
//   warp 10         TMA producer: the value chunks (16 KB ring)
//   warp 11         PV issuer (single thread), P read from tensor memory
// TMEM: S double buffer (2 x 128 columns), O (dv <= 128 columns), P as bf16
// pairs (64 columns, the A operand of PV).
#include "common.cuh"
#include "kernels.hpp"
#include "profiler.hpp"
#include "tmap.hpp"

namespace nsa {

namespace {

constexpr int kRingK = 5;      // key chunks in flight
constexpr int kRingV = 3;      // value chunks in flight
static_assert(kRingV >= 2, "a tile's two value chunks must fit the ring");
constexpr int kSlot = 16384;   // 128 rows x 128 bytes
constexpr int kThreads = 384;
constexpr int kTile = 128;     // keys (or compressed blocks) per S tile

struct CmpWinArgs {
  int T, H, G, dk, dv, n, w, Nc, QT, nbs, dense;
  int R, qoff;                     // query rows; row r sits at position qoff + r
  int hm;                          // k/v head-major [B,G,T,d] (else [B,T,G,d])
  float sc2;                       // softmax scale * log2(e)
  const __nv_bfloat16* gates;      // [B,T,H,3]
  void* part;                      // [B,R,H,dv]: fp32 partial (NSA), bf16 output (dense)
  int32_t* idx;                    // [B,T,G,n]
  DeviceStatus* st;
  uint32_t off_kring, off_vring, off_scores, off_red, off_bar;
};

struct Bars {
  uint64_t q_full;
  // a tile's chunks complete on ONE barrier (one arrival with its bytes per
  // chunk), so the MMA issuers wait once per tile: key tile u on
  // kt_full[u % kRingK], value tile u on vt_full[u % kRingV].  One barrier per
  // ring slot: tile u's first slot was last used by tile u - ceil(R / chunks
  // per tile) >= u - R, which the issuer waited for before freeing the slot,
  // so a barrier is re-armed only after its previous phase was consumed.
  uint64_t kt_full[kRingK];
  uint64_t k_empty[kRingK];
  uint64_t vt_full[kRingV];
  uint64_t v_empty[kRingV];
  uint64_t s_full[2];
  uint64_t s_free[2];
  uint64_t p_full;
  uint64_t p_free;
  uint64_t o_full;
  uint64_t drain[2];
  uint64_t all8;        // rendezvous of the 8 softmax warps
  uint32_t tmem;
  int abort_flag;
};

__device__ __forceinline__ int visible_cmp(int t, int Nc) {
  // compressed block i is visible once its last token 16*i+31 <= t
  if (t < 31) return 0;
  const int nv = (t - 31) / 16 + 1;
  return nv < Nc ? nv : Nc;
}

// Butterfly reduce-scatter of 16 values over groups of HPG lanes (HPG <= 16):
// afterwards lane holds 16/HPG group sums in v[0..], original indices base+k.
template <int HPG>
__device__ __forceinline__ int reduce_scatter16(float (&v)[16], int lane) {
  int base = 0;
#pragma unroll
  for (int m = HPG / 2, n = 8; m >= 1; m >>= 1, n >>= 1) {
    const bool up = (lane & m) != 0;
#pragma unroll
    for (int k = 0; k < n; ++k) {
      const float send = up ? v[k] : v[k + n];
      const float keep = up ? v[k + n] : v[k];
      v[k] = keep + __shfl_xor_sync(0xffffffffu, send, m);
    }
    if (up) base += n;
  }
  return base;
}

__device__ __forceinline__ uint32_t warp_min_u32(uint32_t x) {
  uint32_t r;
  asm volatile("redux.sync.min.u32 %0, %1, 0xffffffff;" : "=r"(r) : "r"(x));
  return r;
}

template <int HPG>
__device__ __forceinline__ float allreduce_group(float x) {
#pragma unroll
  for (int m = HPG / 2; m >= 1; m >>= 1) x += __shfl_xor_sync(0xffffffffu, x, m);
  return x;
}

// 64 consecutive fp32 columns of one TMEM lane (four loads, one wait).
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float (&x)[64]) {
  uint32_t rs[4][16];
#pragma unroll
  for (int c = 0; c < 4; ++c) tmem_ld16(taddr + c * 16, rs[c]);
  tmem_ld_wait(rs[0]);
#pragma unroll
  for (int c = 1; c < 4; ++c) tmem_reg_fence(rs[c]);
#pragma unroll
  for (int c = 0; c < 4; ++c)
#pragma unroll
    for (int i = 0; i < 16; ++i) x[c * 16 + i] = __uint_as_float(rs[c][i]);
}

// kDense: exact causal full attention (window covering the prefix, gate 1,
// no compressed branch, no selection), a separate instance of the kernel.
template <int HPG, bool kDense>
__global__ void __launch_bounds__(kThreads, 1)
    cmp_win_kernel(const __grid_constant__ CUtensorMap mapQ, const __grid_constant__ CUtensorMap mapKc,
                   const __grid_constant__ CUtensorMap mapVc, const __grid_constant__ CUtensorMap mapK,
                   const __grid_constant__ CUtensorMap mapV, const CmpWinArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* qs = smem;
  uint8_t* kring = smem + a.off_kring;
  uint8_t* vring = smem + a.off_vring;
  float* scores = reinterpret_cast<float*>(smem + a.off_scores);
  Bars* bars = reinterpret_cast<Bars*>(smem + a.off_bar);
  volatile int* abort_flag = &bars->abort_flag;

  const int QT = a.QT;
  // the last query tiles see the most keys: launch them first
  const int t0 = (gridDim.x - 1 - blockIdx.x) * QT;   // first row of the tile
  const int p0 = a.qoff + t0;                          // its position
  const int g = blockIdx.y;
  const int b = blockIdx.z;
  const int warp = warp_id();
  const int lane = lane_id();
  const int kcs = a.dk / 64;   // 64-column chunks of a key row
  const int vcs = a.dv / 64;

  // per-CTA schedule (identical in every role)
  const int t_last = a.qoff + min(t0 + QT - 1, a.R - 1);
  const int nmax = visible_cmp(t_last, a.Nc);
  const int ntc = (nmax + kTile - 1) / kTile;
  const int s_lo = max(0, p0 - a.w + 1);
  const int ntw = (t_last - s_lo) / kTile + 1;

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    for (int s = 0; s < kRingK; ++s) {
      mbar_init(&bars->k_empty[s], 1);
      mbar_init(&bars->kt_full[s], kcs);
    }
    for (int s = 0; s < kRingV; ++s) {
      mbar_init(&bars->v_empty[s], 1);
      mbar_init(&bars->vt_full[s], vcs);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars->s_full[s], 1);
      mbar_init(&bars->s_free[s], 8);
    }
    mbar_init(&bars->p_full, 8);
    mbar_init(&bars->p_free, 1);
    mbar_init(&bars->o_full, 1);
    mbar_init(&bars->drain[0], 1);
    mbar_init(&bars->drain[1], 1);
    mbar_init(&bars->all8, 8);
    bars->abort_flag = prior_error(a.st);
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(&bars->tmem, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem;
  const uint32_t tmem_s = tmem;          // S buffers at columns 0 and 128
  const uint32_t tmem_o = tmem + 256;    // O at columns 256 .. 256+dv (dv <= 128)
  const uint32_t tmem_p = tmem + 384;    // P (bf16 pairs): 64 columns, the A operand of PV

  if (*abort_flag) {
    // an earlier CTA failed: do nothing
  } else if (warp == 8 || warp == 10) {
    // =============================================================== producers
    // warp 8: Q, then the key chunks of every QK^T tile in issue order;
    // warp 10: the value chunks of every PV tile
    if (lane == 0) {
      const bool keys = warp == 8;
      if (keys) {
        tma_prefetch_desc(&mapQ);
        tma_prefetch_desc(&mapKc);
        tma_prefetch_desc(&mapK);
        mbar_arrive_expect_tx(&bars->q_full, (uint32_t)(kcs * kSlot));
        for (int c = 0; c < kcs; ++c) tma_load_4d(qs + c * kSlot, &mapQ, &bars->q_full, c * 64, g * HPG, t0, b);
      } else {
        tma_prefetch_desc(&mapVc);
        tma_prefetch_desc(&mapV);
      }
      const int nring = keys ? kRingK : kRingV;
      const int nc = keys ? kcs : vcs;         // chunks per tile
      uint8_t* rbase = keys ? kring : vring;
      uint64_t* tile_full = keys ? bars->kt_full : bars->vt_full;
      uint64_t* empty = keys ? bars->k_empty : bars->v_empty;
      int v = 0, ut = 0;                       // chunks and tiles pushed
      bool ok = true;
      // chunk c of tile ut, completing on the tile's barrier
      auto push = [&](int c, const CUtensorMap* map, int c0, int c1, int c2, int c3) {
        if (!ok) return;
        uint64_t* tf = &tile_full[ut % nring];
        const int slot = v % nring;
        const uint32_t round = (uint32_t)(v / nring);
        if (!mbar_wait(&empty[slot], (round & 1) ^ 1, abort_flag, a.st, keys ? 201 : 202)) {
          // complete the tile's arrivals so its phase ends once the chunks
          // already issued have landed (the drain below waits for it)
          for (int x = c; x < nc; ++x) mbar_arrive(tf);
          ++ut;
          ok = false;
          return;
        }
        mbar_arrive_expect_tx(tf, kSlot);
        tma_load_4d(rbase + slot * kSlot, map, tf, c0, c1, c2, c3);
        ++v;
        if (c == nc - 1) ++ut;
      };
      if (keys) {
        // window keys once (online softmax), then compressed keys twice
        // (statistics pass, exact pass)
        for (int j = 0; j < ntw; ++j)
          for (int c = 0; c < kcs; ++c) {
            if (a.hm) push(c, &mapK, c * 64, s_lo + j * kTile, g, b);
            else push(c, &mapK, c * 64, g, s_lo + j * kTile, b);
          }
        for (int pass = 0; pass < 2; ++pass)
          for (int j = 0; j < ntc; ++j)
            for (int c = 0; c < kcs; ++c) push(c, &mapKc, c * 64, j * kTile, g, b);
      } else {
        // with two value chunks a tile's PV is one N = 128 MMA per key step,
        // whose B operand takes dv 0..63 from the lower of the tile's two
        // slots: a tile that straddles the ring end (slots kRingV-1, 0) loads
        // dv 64..127 first
        for (int j = 0; j < ntc + ntw; ++j) {
          const bool swap = vcs == 2 && v % kRingV == kRingV - 1;   // tile's first slot
          for (int c = 0; c < vcs; ++c) {
            const int cc = swap ? 1 - c : c;
            if (j >= ntw) push(c, &mapVc, cc * 64, (j - ntw) * kTile, g, b);
            else if (a.hm) push(c, &mapV, cc * 64, s_lo + j * kTile, g, b);
            else push(c, &mapV, cc * 64, g, s_lo + j * kTile, b);
          }
        }
      }
      if (!ok || *abort_flag) {
        if (keys) mbar_wait_plain(&bars->q_full, 0, kWaitLimitNs);
        // only the last nring started tiles can still have copies in flight
        for (int x = (ut > nring ? ut - nring : 0); x < ut; ++x)
          mbar_wait_plain(&tile_full[x % nring], (uint32_t)((x / nring) & 1), kWaitLimitNs);
      }
    }
  } else if (warp == 9 || warp == 11) {
    // =============================================================== MMA issuers
    // warp 9: QK^T of every tile (statistics and exact passes), limited only
    // by the two S buffers; warp 11: PV of every exact-pass tile, as soon as
    // its P is in tensor memory
    if (lane == 0) {
      bool ok = true;
      if (warp == 9) {
        const uint32_t idesc_qk = idesc_bf16_f32(128, kTile, false, false);
        const uint32_t qs_a = smem_u32(qs), k_a = smem_u32(kring);
        ok = mbar_wait(&bars->q_full, 0, abort_flag, a.st, 211);
        const int ntiles = ntw + 2 * ntc;
        int kv = 0;
        for (int u = 0; u < ntiles && ok; ++u) {
          const int sb = u & 1;
          const uint32_t use = (uint32_t)(u >> 1);
          if (!mbar_wait(&bars->s_free[sb], (use & 1) ^ 1, abort_flag, a.st, 213)) {
            ok = false;
            break;
          }
          if (!mbar_wait(&bars->kt_full[u % kRingK], (uint32_t)((u / kRingK) & 1), abort_flag, a.st, 212)) {
            ok = false;
            break;
          }
          tc_fence_after();
          for (int c = 0; c < kcs; ++c) {
            const int slot = kv % kRingK;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint64_t ad = sdesc_sw128(qs_a + c * kSlot + k * 32, 16, 1024);
              const uint64_t bd = sdesc_sw128(k_a + slot * kSlot + k * 32, 16, 1024);
              umma_bf16(tmem_s + sb * kTile, ad, bd, idesc_qk, (c > 0 || k > 0) ? 1u : 0u);
            }
            umma_commit(&bars->k_empty[slot]);
            ++kv;
          }
          if (ok) umma_commit(&bars->s_full[sb]);
        }
        if (!ok || *abort_flag) {
          umma_commit(&bars->drain[0]);
          mbar_wait_plain(&bars->drain[0], 0, kWaitLimitNs);
        }
      } else {
        const uint32_t idesc_pv = idesc_bf16_f32(128, 64, false, true);
        const uint32_t v_a = smem_u32(vring);
        const int npv = ntc + ntw;
        int vv = 0;
        const uint32_t idesc_pv2 = idesc_bf16_f32(128, 128, false, true);
        for (int pv = 0; pv < npv && ok; ++pv) {
          if (!mbar_wait(&bars->p_full, (uint32_t)(pv & 1), abort_flag, a.st, 214) ||
              !mbar_wait(&bars->vt_full[pv % kRingV], (uint32_t)((pv / kRingV) & 1), abort_flag, a.st, 215)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (vcs == 2) {
            // both dv halves in one N = 128 MMA per key step: dv 0..63 sit in
            // the lower of the tile's two slots, dv 64..127 LBO bytes above
            const int s0 = vv % kRingV, s1 = (vv + 1) % kRingV;
            const int lo = s0 < s1 ? s0 : s1;
            const uint32_t lbo = (uint32_t)((s0 < s1 ? s1 - s0 : s0 - s1) * kSlot);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const uint64_t bd = sdesc_sw128(v_a + lo * kSlot + k * 2048, lbo, 1024);
              umma_bf16_ts(tmem_o, tmem_p + 8 * k, bd, idesc_pv2, (pv == 0 && k == 0) ? 0u : 1u);
            }
            umma_commit(&bars->v_empty[s0]);
            umma_commit(&bars->v_empty[s1]);
            vv += 2;
            if (ok) umma_commit(&bars->p_free);
            continue;
          }
          for (int c = 0; c < vcs; ++c) {
            const int slot = vv % kRingV;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              // A = P from tensor memory (keys 16k .. 16k+15 = columns 8k .. 8k+7)
              const uint64_t bd = sdesc_sw128(v_a + slot * kSlot + k * 2048, kSlot, 1024);
              umma_bf16_ts(tmem_o + c * 64, tmem_p + 8 * k, bd, idesc_pv, (pv == 0 && k == 0) ? 0u : 1u);
            }
            umma_commit(&bars->v_empty[slot]);
            ++vv;
          }
          if (ok) umma_commit(&bars->p_free);
        }
        if (ok) umma_commit(&bars->o_full);
        if (!ok || *abort_flag) {
          umma_commit(&bars->drain[1]);
          mbar_wait_plain(&bars->drain[1], 0, kWaitLimitNs);
        }
      }
    }
  } else if (warp < 8) {
    // =============================================================== softmax warpgroups
    const int wg = warp >> 2;                // key columns 64*wg .. 64*wg+63 of every tile
    const int lw = warp & 3;
    const int r = lw * 32 + lane;            // row = TMEM lane
    const int qi = r / HPG;
    const int h = r % HPG;
    const int row = t0 + qi;
    const int t = p0 + qi;                   // position of the query
    const bool row_ok = row < a.R;
    const int head = g * HPG + h;
    const int n_t = row_ok ? visible_cmp(t, a.Nc) : 0;
    float g_c = 0.f, g_w = kDense ? 1.f : 0.f;
    if (row_ok && !kDense) {
      const __nv_bfloat16* gp = a.gates + (((size_t)b * a.R + row) * a.H + head) * 3;
      g_c = __bfloat162float(gp[0]);
      g_w = __bfloat162float(gp[2]);
    }
    const uint32_t lane_base = (uint32_t)(lw * 32) << 16;
    const int c0 = 64 * wg;                  // first column of this warpgroup
    float* red = reinterpret_cast<float*>(smem + a.off_red);   // [2 wg][2 m/l][128 rows]
    float* xmax = red + 2 * 2 * 128;                            // [2 tiles][2 wg][128 rows]
    bool ok = true;
    int u = 0, pv = 0;
    uint32_t all_phase = 0;

    auto sync8 = [&]() {
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->all8);
      if (!mbar_wait(&bars->all8, all_phase & 1, abort_flag, a.st, 221)) ok = false;
      ++all_phase;
    };
    // loads this warpgroup's 64 columns of the next S tile and releases it
    auto consume_s = [&](float (&x)[64]) -> bool {
      const int sb = u & 1;
      const uint32_t use = (uint32_t)(u >> 1);
      ++u;
      if (!mbar_wait(&bars->s_full[sb], use & 1, abort_flag, a.st, 222)) return false;
      tc_fence_after();
      tmem_ld64(tmem_s + lane_base + sb * kTile + c0, x);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->s_free[sb]);
      return true;
    };
    const int half = a.dv / 2;               // O columns of this warpgroup: wg*half ..
    // multiplies this row's half of O by f; O must be idle (no PV in flight)
    auto scale_o = [&](float f) {
      for (int cc = wg * half; cc < (wg + 1) * half; cc += 16) {
        uint32_t rr[16];
        tmem_ld16(tmem_o + lane_base + cc, rr);
        tmem_ld_wait(rr);
#pragma unroll
        for (int k = 0; k < 16; k += 2) {
          const float2 y = __fmul2_rn(make_float2(__uint_as_float(rr[k]), __uint_as_float(rr[k + 1])), make_float2(f, f));
          rr[k] = __float_as_uint(y.x);
          rr[k + 1] = __float_as_uint(y.y);
        }
        tmem_st16(tmem_o + lane_base + cc, rr);
      }
    };
    // waits until every PV issued so far has completed: O is then idle until
    // this thread's next P arrives (the PV issuer waits for all 8 warps' P)
    auto wait_o_idle = [&]() -> bool {
      if (!mbar_wait(&bars->p_free, (uint32_t)((pv & 1) ^ 1), abort_flag, a.st, 223)) return false;
      tc_fence_after();
      return true;
    };
    // P (times ``gate``) of the next PV tile; when oscale != 1 this row's half
    // of O is first multiplied by it (O is idle at that point)
    auto put_p = [&](const float (&p)[64], float gate, float oscale) -> bool {
      if (!wait_o_idle()) return false;
      if (oscale != 1.f && pv > 0) scale_o(oscale);
      ++pv;
      // this row's 64 keys of the warpgroup's half, as bf16 pairs, into
      // columns 32*wg .. 32*wg+31 of P in tensor memory
      {
        uint32_t pk[16];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float2 gp = __fmul2_rn(make_float2(p[32 * hh + 2 * j], p[32 * hh + 2 * j + 1]), make_float2(gate, gate));
            pk[j] = pack_bf16x2(gp.x, gp.y);
          }
          tmem_st16(tmem_p + lane_base + 32 * wg + 16 * hh, pk);
        }
        tmem_st_wait();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->p_full);
      return true;
    };
    // online max / sum over this warpgroup's columns; x holds raw scores
    // (-inf where masked), m is kept in log2 units (scores * scale * log2 e)
    const float2 sc2x2 = make_float2(a.sc2, a.sc2);
    auto stats_add = [&](float (&x)[64], float& m, float& l) {
      float mt = -INFINITY;
#pragma unroll
      for (int i = 0; i < 64; ++i) mt = fmaxf(mt, x[i]);
      const float mn = fmaxf(m, mt * a.sc2);
      if (mn == -INFINITY) return;
      // pairs of columns through the packed f32x2 FMA / add
      const float2 nm = make_float2(-mn, -mn);
      float2 sm = make_float2(0.f, 0.f);
#pragma unroll
      for (int i = 0; i < 64; i += 2) {
        const float2 y = __ffma2_rn(make_float2(x[i], x[i + 1]), sc2x2, nm);
        sm = __fadd2_rn(sm, make_float2(fast_exp2(y.x), fast_exp2(y.y)));
      }
      l = l * fast_exp2(m - mn) + (sm.x + sm.y);
      m = mn;
    };
    // p = exp2(x * scale - mu) for 64 columns, pairs through the packed FMA
    auto exp_cols = [&](float (&x)[64], float mu) {
      const float2 nm = make_float2(-mu, -mu);
#pragma unroll
      for (int i = 0; i < 64; i += 2) {
        const float2 y = __ffma2_rn(make_float2(x[i], x[i + 1]), sc2x2, nm);
        x[i] = fast_exp2(y.x);
        x[i + 1] = fast_exp2(y.y);
      }
    };
    // merge with the other warpgroup: afterwards m = max + log2(sum) of the
    // row (p = exp2(s*scale - m) is then normalised), +inf if the row is empty
    auto merge_stats = [&](float& m, float l, float& il) {
      red[(wg * 2 + 0) * 128 + r] = m;
      red[(wg * 2 + 1) * 128 + r] = l;
      sync8();
      const float mo = red[((1 - wg) * 2 + 0) * 128 + r];
      const float lo = red[((1 - wg) * 2 + 1) * 128 + r];
      const float M = fmaxf(m, mo);
      float L = 0.f;
      if (M != -INFINITY) L = l * fast_exp2(m - M) + lo * fast_exp2(mo - M);
      m = (L > 0.f) ? M + __log2f(L) : INFINITY;
      il = L > 0.f ? 1.f / L : 0.f;
      sync8();   // both warpgroups have read before the area is reused
    };

    // zero the block-score rows
    if (!kDense) {
      for (int i = wg * 128 + r; i < QT * a.nbs; i += 256) scores[i] = 0.f;
      sync8();
    }
    float x[64];
    // ---------------- phase 0: window, online softmax
    // mref: this row's reference max (log2 units, shared by both warpgroups),
    // p = exp2(s*scale - mref); O and the sum follow mref when it moves up
    {
      const int w_lo = t - a.w + 1;
      float mref = -INFINITY, lw = 0.f;
      for (int j = 0; j < ntw && ok; ++j) {
        if (!consume_s(x)) { ok = false; break; }
        const int s0 = s_lo + j * kTile + c0;
        if (!(row_ok && s0 >= w_lo && s0 + 63 <= t)) {   // interior tiles need no mask
#pragma unroll
          for (int i = 0; i < 64; ++i) {
            const int sx = s0 + i;
            x[i] = (row_ok && sx >= w_lo && sx <= t) ? x[i] : -INFINITY;
          }
        }
        float mt = -INFINITY;
#pragma unroll
        for (int i = 0; i < 64; ++i) mt = fmaxf(mt, x[i]);
        float* xm = xmax + (j & 1) * 256;
        xm[wg * 128 + r] = mt;
        sync8();
        if (!ok) break;
        const float mtile = fmaxf(mt, xm[(1 - wg) * 128 + r]) * a.sc2;
        float fac = 1.f;
        if (mtile > mref + 8.f) {     // also the first finite tile (mref = -inf)
          fac = fast_exp2(mref - mtile);
          lw *= fac;
          mref = mtile;
        }
        if (mref == -INFINITY) {
#pragma unroll
          for (int i = 0; i < 64; ++i) x[i] = 0.f;
        } else {
          exp_cols(x, mref);
        }
        float2 sm = make_float2(0.f, 0.f);
#pragma unroll
        for (int i = 0; i < 64; i += 2) sm = __fadd2_rn(sm, make_float2(x[i], x[i + 1]));
        lw += sm.x + sm.y;
        if (!put_p(x, 1.f, fac)) { ok = false; break; }
      }
      // O <- O * g_win / sum, once every window PV has completed
      red[wg * 128 + r] = lw;
      sync8();
      const float L = lw + red[(1 - wg) * 128 + r];
      sync8();
      if (ok && pv > 0) {
        if (!wait_o_idle()) ok = false;
        else {
          scale_o(L > 0.f ? g_w / L : 0.f);
          tmem_st_wait();
          tc_fence_before();
        }
      }
    }
    // ---------------- phase 1: compressed max / sum
    float m = -INFINITY, l = 0.f, inv_l = 0.f;
    for (int j = 0; j < ntc && ok; ++j) {
      if (!consume_s(x)) { ok = false; break; }
      if (j * kTile + c0 + 64 > n_t) {   // only a row's last visible tile is masked
#pragma unroll
        for (int i = 0; i < 64; ++i) x[i] = (j * kTile + c0 + i < n_t) ? x[i] : -INFINITY;
      }
      stats_add(x, m, l);
    }
    merge_stats(m, l, inv_l);
    // ---------------- phase 2: exact p, O_cmp, block scores
    float* srow = scores + (size_t)qi * a.nbs;
    const bool lead = (lane % HPG) == 0;
    for (int j = 0; j < ntc && ok; ++j) {
      if (!consume_s(x)) { ok = false; break; }
      if (j * kTile + c0 + 64 > n_t) {
#pragma unroll
        for (int i = 0; i < 64; ++i) x[i] = (j * kTile + c0 + i < n_t) ? fast_exp2(fmaf(x[i], a.sc2, -m)) : 0.f;
      } else {
        exp_cols(x, m);
      }
      // block importance: selection block 32j+16wg+uu collects compressed
      // blocks 4u-1 (one chunk), 4u..4u+2 (two chunks each), 4u+3 (one chunk);
      // entry 4u-1 of the first block is added by whoever holds it (the
      // previous column half), as the carry below
      float vsum[16];
#pragma unroll
      for (int uu = 0; uu < 16; ++uu)
        vsum[uu] = (uu > 0 ? x[4 * uu - 1] : 0.f) + 2.f * (x[4 * uu] + x[4 * uu + 1] + x[4 * uu + 2]) +
                   x[4 * uu + 3];
      const float carry = allreduce_group<HPG>(x[63]);
      const int base = reduce_scatter16<HPG>(vsum, lane);
      if (row_ok) {
        // every block receives at most two additions (its own columns and the
        // carry of the columns before it), so the sums are order-independent
#pragma unroll
        for (int k = 0; k < 16 / HPG; ++k) atomicAdd(&srow[32 * j + 16 * wg + base + k], vsum[k]);
        if (lead) atomicAdd(&srow[32 * j + 16 * wg + 16], carry);
      }
      if (!put_p(x, g_c, 1.f)) { ok = false; break; }
    }
    // ---------------- top-n selection (one warp per query)
    sync8();
    if (ok && !kDense) {
      for (int qq = warp; qq < QT; qq += 8) {
        const int tq = p0 + qq;
        if (t0 + qq >= a.R) continue;
        const int jt = tq / 64;
        int32_t* out = a.idx + (((size_t)b * a.R + t0 + qq) * a.G + g) * a.n;
        if (jt + 1 <= a.n) {
          if (lane < a.n) out[lane] = lane <= jt ? lane : -1;
          continue;
        }
        const float* sq = scores + (size_t)qq * a.nbs;
        // candidates 1 .. jt-2 (blocks 0, jt-1, jt are forced): each lane
        // keeps its 8 best (higher score, then lower block) in a sorted list;
        // a round's winner is a warp max reduction, ties to the lowest block,
        // and only its owner lane pops (and refills after giving all 8)
        float tv[8];
        int tj[8];
        auto fill = [&]() {
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            tv[k] = -INFINITY;
            tj[k] = 0x7fffffff;
          }
          for (int jj = 1 + lane; jj <= jt - 2; jj += 32) {
            float cv = sq[jj];
            if (!(cv > tv[7])) continue;
            int cj = jj;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const bool sw = cv > tv[k];
              const float t0v = tv[k];
              const int t0j = tj[k];
              tv[k] = sw ? cv : t0v;
              tj[k] = sw ? cj : t0j;
              cv = sw ? t0v : cv;
              cj = sw ? t0j : cj;
            }
          }
        };
        fill();
        int mine = -1;
        const int nfree = a.n - 3;
        for (int rnd = 0; rnd < nfree; ++rnd) {
          const float gv = warp_max_f32(tv[0]);
          const uint32_t gj = warp_min_u32(tv[0] == gv ? (uint32_t)tj[0] : 0x7fffffffu);
          if (lane == rnd) mine = (gv == -INFINITY) ? 0x7fffffff : (int)gj;
          if (gv != -INFINITY && (uint32_t)tj[0] == gj) {
            // taken: mark it, pop the head
            const_cast<float*>(sq)[gj] = -INFINITY;
#pragma unroll
            for (int k = 0; k < 7; ++k) {
              tv[k] = tv[k + 1];
              tj[k] = tj[k + 1];
            }
            tv[7] = -INFINITY;
            tj[7] = 0x7fffffff;
            if (tv[0] == -INFINITY) fill();
          }
        }
        if (lane == nfree) mine = 0;
        if (lane == nfree + 1) mine = jt - 1;
        if (lane == nfree + 2) mine = jt;
        int rank = 0;
        for (int k = 0; k < a.n; ++k) {
          const int o = __shfl_sync(0xffffffffu, mine, k);
          rank += (o < mine) ? 1 : 0;
        }
        if (lane < a.n) out[rank] = mine;
      }
    }
    // ---------------- epilogue: O -> fp32 partial (NSA) or bf16 output
    // (dense), each warpgroup half the columns
    if (ok && mbar_wait(&bars->o_full, 0, abort_flag, a.st, 224)) {
      tc_fence_after();
      const size_t off = (((size_t)b * a.R + row) * a.H + head) * a.dv;
      for (int cc = wg * half; cc < (wg + 1) * half; cc += 16) {
        uint32_t rr[16];
        tmem_ld16(tmem_o + lane_base + cc, rr);
        tmem_ld_wait(rr);
        if (row_ok && kDense) {
          uint32_t pk[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) pk[k] = pack_bf16x2(__uint_as_float(rr[2 * k]), __uint_as_float(rr[2 * k + 1]));
          uint4* d4 = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.part) + off + cc);
          d4[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          d4[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
        } else if (row_ok) {
          uint4* d4 = reinterpret_cast<uint4*>(static_cast<float*>(a.part) + off + cc);
#pragma unroll
          for (int k = 0; k < 4; ++k) d4[k] = make_uint4(rr[4 * k], rr[4 * k + 1], rr[4 * k + 2], rr[4 * k + 3]);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

struct Layout {
  uint32_t off_kring, off_vring, off_scores, off_red, off_bar, total;
};

Layout layout_for(int dk, int QT, int nbs) {
  Layout L;
  L.off_kring = (uint32_t)(dk / 64) * kSlot;
  L.off_vring = L.off_kring + kRingK * kSlot;
  L.off_scores = L.off_vring + kRingV * kSlot;
  L.off_red = (uint32_t)align_up(L.off_scores + (size_t)QT * nbs * sizeof(float), 256);
  // red: [2 wg][2 m/l][128 rows] statistics, then [2 tiles][2 wg][128 rows] window tile maxima
  L.off_bar = (uint32_t)align_up(L.off_red + 4 * 2 * 128 * sizeof(float), 1024);
  L.total = L.off_bar + (uint32_t)align_up(sizeof(Bars), 256) + 1024;  // + alignment slack
  return L;
}

int scores_stride(int T, int Nc) {
  const int ntc = (Nc + kTile - 1) / kTile;
  const int nb = (T + 63) / 64;
  const int s = (32 * ntc + 1 > nb ? 32 * ntc + 1 : nb) + 1;
  return (s + 3) & ~3;
}

template <int HPG, bool kDense>
int launch_inst(const CmpWinArgs& a0, int B, const CUtensorMap* maps, size_t smem, cudaStream_t s) {
  if (int rc = ensure_smem_attr(reinterpret_cast<const void*>(&cmp_win_kernel<HPG, kDense>), smem_max())) return rc;
  dim3 grid((a0.R + a0.QT - 1) / a0.QT, a0.G, B);
  prof::begin(kDense ? "full_attn" : "cmp_win", s);
  cmp_win_kernel<HPG, kDense><<<grid, kThreads, smem, s>>>(maps[0], maps[1], maps[2], maps[3], maps[4], a0);
  prof::end(s);
  return cudaPeekAtLastError() == cudaSuccess ? NSA_OK : NSA_ERR_CUDA;
}

template <int HPG>
int launch_hpg(const CmpWinArgs& a0, int B, const CUtensorMap* maps, size_t smem, cudaStream_t s) {
  return a0.dense ? launch_inst<HPG, true>(a0, B, maps, smem, s) : launch_inst<HPG, false>(a0, B, maps, smem, s);
}

}  // namespace

size_t cmp_win_smem_bytes(const nsa_cfg& c, bool dense) {
  const int hpg = c.H / c.G;
  const int QT = 128 / hpg;
  const int Nc = c.T < c.l ? 0 : (c.T - c.l) / c.d + 1;
  return layout_for(c.dk, QT, dense ? 0 : scores_stride(c.T, Nc)).total;
}

int launch_cmp_win(const nsa_cfg& c, const void* q, const void* k, const void* v, const void* kc, const void* vc,
                   const void* gates, void* part, int32_t* idx, DeviceStatus* st, cudaStream_t s, bool dense,
                   const QueryRows& rows) {
  const int R = rows.R > 0 ? rows.R : c.T;
  const int hpg = c.H / c.G;
  const int QT = 128 / hpg;
  // dense: no compressed branch, a window covering the whole prefix
  const int Nc = dense || c.T < c.l ? 0 : (c.T - c.l) / c.d + 1;
  const int nbs = dense ? 0 : scores_stride(c.T, Nc);
  const Layout L = layout_for(c.dk, QT, nbs);
  if (L.total > smem_max()) return NSA_ERR_UNSUPPORTED;
  const uint64_t e = 2;
  CUtensorMap maps[5];
  {  // q [B,R,H,dk]: box (64, hpg heads, QT query rows)
    const uint64_t dims[4] = {(uint64_t)c.dk, (uint64_t)c.H, (uint64_t)R, (uint64_t)c.B};
    const uint64_t str[3] = {c.dk * e, (uint64_t)c.H * c.dk * e, (uint64_t)R * c.H * c.dk * e};
    const uint32_t box[4] = {64, (uint32_t)hpg, (uint32_t)QT, 1};
    if (!make_tmap_bf16(&maps[0], q, 4, dims, str, box)) return NSA_ERR_CUDA;
  }
  const int Ncm = Nc > 0 ? Nc : 1;
  {  // kc [B,G,Nc,dk]
    const uint64_t dims[4] = {(uint64_t)c.dk, (uint64_t)Ncm, (uint64_t)c.G, (uint64_t)c.B};
    const uint64_t str[3] = {c.dk * e, (uint64_t)Ncm * c.dk * e, (uint64_t)c.G * Ncm * c.dk * e};
    const uint32_t box[4] = {64, 128, 1, 1};
    if (!make_tmap_bf16(&maps[1], Nc > 0 ? kc : k, 4, dims, str, box)) return NSA_ERR_CUDA;
  }
  {  // vc [B,G,Nc,dv]
    const uint64_t dims[4] = {(uint64_t)c.dv, (uint64_t)Ncm, (uint64_t)c.G, (uint64_t)c.B};
    const uint64_t str[3] = {c.dv * e, (uint64_t)Ncm * c.dv * e, (uint64_t)c.G * Ncm * c.dv * e};
    const uint32_t box[4] = {64, 128, 1, 1};
    if (!make_tmap_bf16(&maps[2], Nc > 0 ? vc : v, 4, dims, str, box)) return NSA_ERR_CUDA;
  }
  if (!make_kv_map(&maps[3], k, c.B, c.T, c.G, c.dk, 128, rows.head_major)) return NSA_ERR_CUDA;
  if (!make_kv_map(&maps[4], v, c.B, c.T, c.G, c.dv, 128, rows.head_major)) return NSA_ERR_CUDA;
  CmpWinArgs a;
  a.T = c.T;
  a.H = c.H;
  a.G = c.G;
  a.dk = c.dk;
  a.dv = c.dv;
  a.n = c.n;
  a.w = dense ? c.T : c.w;
  a.Nc = Nc;
  a.QT = QT;
  a.nbs = nbs;
  a.dense = dense ? 1 : 0;
  a.R = R;
  a.qoff = rows.qoff;
  a.hm = rows.head_major ? 1 : 0;
  const float scale = c.scale > 0.f ? c.scale : 1.0f / sqrtf((float)c.dk);
  a.sc2 = scale * 1.4426950408889634f;
  a.gates = static_cast<const __nv_bfloat16*>(gates);
  a.part = part;
  a.idx = idx;
  a.st = st;
  a.off_kring = L.off_kring;
  a.off_vring = L.off_vring;
  a.off_scores = L.off_scores;
  a.off_red = L.off_red;
  a.off_bar = L.off_bar;
  switch (hpg) {
    case 1: return launch_hpg<1>(a, c.B, maps, L.total, s);
    case 2: return launch_hpg<2>(a, c.B, maps, L.total, s);
    case 4: return launch_hpg<4>(a, c.B, maps, L.total, s);
    case 8: return launch_hpg<8>(a, c.B, maps, L.total, s);
    case 16: return launch_hpg<16>(a, c.B, maps, L.total, s);
    default: return NSA_ERR_UNSUPPORTED;
  }
}

}  // namespace nsa
