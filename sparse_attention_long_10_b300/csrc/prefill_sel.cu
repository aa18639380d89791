// prefill_sel.cu -- NSA selected-block attention + gated combine [P2 II.2;
// P3 token-selection paragraph: the kept blocks are re-read at full
// resolution; blockwise selection keeps the memory access contiguous].
//
// One work item = one query t of one KV group g (all HPG heads of the group
// share the n kept blocks: group-centric loading, each 64-token block fetched
// once per group).  The MMA is "swapped": keys are the M side, heads the N
// side, so a 128-row tcgen05 tile is two kept blocks against the group's
// heads:
//     S^T[key, head] = K_pair[key, :] . Q_t[head, :]        (M=128, N=NP)
//     O^T[dv, head] += V_pair^T[dv, key] . P^T[key, head]    (M=128, N=NP)
// All n*l' scores of the item sit in TMEM at once, so the softmax over the
// kept keys is exact: one pass over TMEM finds each head's max, a second forms
// p = exp(s - max) (unnormalised, bf16) and the sums.  The epilogue applies
// g_slc / sum and adds the cmp+win partial sum (fp32) from prefill_cmp_win.cu:
//     out = bf16(part + g_slc * O_slc)
//
// Warp roles (12 warps):
//   warps 0-3, 4-7  two softmax + epilogue warpgroups, taking alternate items
//                   (thread = TMEM lane = one key of a pair, or one value dim)
//   warp 8          TMA producer of Q and the key chunks
//   warp 9          QK^T MMA issuer
//   warp 10         TMA producer of the value pairs
//   warp 11         PV MMA issuer
// TMEM: S^T double buffer (2 x 8 pairs x NP columns), O^T in 4 buffers.
#include "common.cuh"
#include "kernels.hpp"
#include "profiler.hpp"
#include "tmap.hpp"

namespace nsa {

namespace {

constexpr int kThreads = 384;
constexpr int NP = 16;           // MMA N: heads of the group, padded to 16
constexpr int kRingK = 5;        // 16 KB: one 64-column chunk of a block pair
constexpr int kRingV = 2;        // 32 KB: both 64-column chunks of a value pair
constexpr int kSlotK = 16384;
constexpr int kSlotV = 32768;
constexpr int kQBuf = 2048;      // one 64-column chunk of NP query rows
constexpr int kPBuf = 32768;     // P^T of one item: 8 pairs x 2 chunks x 2 KB
constexpr int kItemsPerCta = 64;

struct SelArgs {
  int T, H, G, dk, dv, n, hpg, QPC;
  int R, qoff;                     // query rows; row r sits at position qoff + r
  int hm;                          // k/v head-major [B,G,T,d] (else [B,T,G,d])
  float sc2;
  const int32_t* idx;              // [B,T,G,n]
  const __nv_bfloat16* gates;      // [B,T,H,3]
  const float* part;               // [B,R,H,dv] fp32
  __nv_bfloat16* out;              // [B,T,H,dv]
  float* slc_lse;                  // kSave: [B,R,H] log2-domain log-sum-exp of s*scale
  float* slc_o;                    // kSave: [B,R,H,dv] O_slc (fp32, before the gate)
  DeviceStatus* st;
  uint32_t off_kring, off_vring, off_pt, off_red, off_bar;
};

struct Bars {
  uint64_t q_full[2], q_empty[2];
  uint64_t k_full[kRingK], k_empty[kRingK];
  uint64_t v_full[kRingV], v_empty[kRingV];
  uint64_t s_full[2], s_free[2];
  uint64_t p_full[2], p_free[2];
  uint64_t o_full[4], o_free[4];
  uint64_t wg[2];
  uint64_t drain[2];
  uint32_t tmem;
  int abort_flag;
};

// token coordinate of block ``blk`` for a TMA load; an absent block reads
// zeros from a negative coordinate
__device__ __forceinline__ int block_token(int blk) { return blk >= 0 ? blk * 64 : -128; }

// one 64-token box of K or V (see make_kv_map for the coordinate order)
__device__ __forceinline__ void tma_kv(void* dst, const CUtensorMap* map, uint64_t* bar, int col, int g, int tok,
                                       int b, bool head_major) {
  if (head_major) tma_load_4d(dst, map, bar, col, tok, g, b);
  else tma_load_4d(dst, map, bar, col, g, tok, b);
}

// The n (<= 16) kept blocks of one item, -1 past n: issued as independent
// loads (four 16-byte loads when n == 16) so they cost one memory round trip.
__device__ __forceinline__ void load_blocks(const int32_t* blk, int n, int (&bk)[16]) {
  if (n == 16 && (reinterpret_cast<uintptr_t>(blk) & 15u) == 0) {
    const int4* p4 = reinterpret_cast<const int4*>(blk);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int4 v = __ldg(p4 + k);
      bk[4 * k + 0] = v.x;
      bk[4 * k + 1] = v.y;
      bk[4 * k + 2] = v.z;
      bk[4 * k + 3] = v.w;
    }
  } else {
#pragma unroll
    for (int k = 0; k < 16; ++k) bk[k] = k < n ? __ldg(blk + k) : -1;
  }
}

// kMulti: query rows at positions qoff + row against head-major caches (a
// multi-token decode); otherwise one row per position of token-major inputs
// (the prefill), with those values known at compile time.  kSave: also write
// the branch's log-sum-exp and its output O_slc, which the backward pass
// reads instead of recomputing them.
template <bool kMulti, bool kSave>
__global__ void __launch_bounds__(kThreads, 1)
    sel_kernel(const __grid_constant__ CUtensorMap mapQ, const __grid_constant__ CUtensorMap mapK,
               const __grid_constant__ CUtensorMap mapV, const SelArgs a) {
  const int R = kMulti ? a.R : a.T;
  const int qoff = kMulti ? a.qoff : 0;
  constexpr bool hm = kMulti;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* qbuf = smem;                        // 2 items x kcs chunks x 2 KB
  uint8_t* kring = smem + a.off_kring;
  uint8_t* vring = smem + a.off_vring;
  uint8_t* pt = smem + a.off_pt;               // P^T: 2 buffers x 8 pairs x 2 chunks x 2 KB
  float* red = reinterpret_cast<float*>(smem + a.off_red);   // [2 wg][2 max/sum][4 warps][NP]
  Bars* bars = reinterpret_cast<Bars*>(smem + a.off_bar);
  volatile int* abort_flag = &bars->abort_flag;

  const int g = blockIdx.y;
  const int b = blockIdx.z;
  const int t0 = blockIdx.x * a.QPC;          // first row of the CTA
  const int nitems = min(a.QPC, R - t0);
  const int warp = warp_id();
  const int lane = lane_id();
  const int kcs = a.dk / 64;
  const int vcs = a.dv / 64;
  const int npairs = (a.n + 1) / 2;
  const int SC = npairs * NP;                  // TMEM columns of one S^T buffer

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->q_full[i], 1);
      mbar_init(&bars->q_empty[i], 1);
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->s_free[i], 4);
      mbar_init(&bars->p_full[i], 4);
      mbar_init(&bars->p_free[i], 1);
      mbar_init(&bars->wg[i], 4);
      mbar_init(&bars->drain[i], 1);
    }
    for (int i = 0; i < 4; ++i) {
      mbar_init(&bars->o_full[i], 1);
      mbar_init(&bars->o_free[i], 4);
    }
    for (int i = 0; i < kRingK; ++i) {
      mbar_init(&bars->k_full[i], 1);
      mbar_init(&bars->k_empty[i], 1);
    }
    for (int i = 0; i < kRingV; ++i) {
      mbar_init(&bars->v_full[i], 1);
      mbar_init(&bars->v_empty[i], 1);
    }
    bars->abort_flag = prior_error(a.st);
    fence_barrier_init();
  }
  // query rows hpg..NP-1 are never loaded: keep them finite (zero)
  for (int i = threadIdx.x; i < 2 * kcs * kQBuf / 16; i += kThreads)
    reinterpret_cast<uint4*>(qbuf)[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  if (warp == 0) {
    tmem_alloc(&bars->tmem, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem;
  const uint32_t tmem_s = tmem;                   // 2 x SC columns
  const uint32_t tmem_o = tmem + 2 * SC;          // 4 x NP columns

  if (*abort_flag) {
    // an earlier CTA failed: do nothing
  } else if (warp == 8 || warp == 10) {
    // =============================================================== producers
    // warp 8 streams Q and the key chunks, warp 10 the value pairs, so both
    // rings stay in flight at once
    if (lane == 0) {
      tma_prefetch_desc(&mapQ);
      tma_prefetch_desc(&mapK);
      tma_prefetch_desc(&mapV);
      bool ok = true;
      int kv = 0, vv = 0, nq = 0;
      auto load_q = [&](int i) {
        if (!ok) return;
        const int qb = i & 1;
        if (!mbar_wait(&bars->q_empty[qb], (uint32_t)(((i >> 1) & 1) ^ 1), abort_flag, a.st, 301)) {
          ok = false;
          return;
        }
        mbar_arrive_expect_tx(&bars->q_full[qb], (uint32_t)(kcs * a.hpg * 128));
        for (int c = 0; c < kcs; ++c)
          tma_load_4d(qbuf + (qb * kcs + c) * kQBuf, &mapQ, &bars->q_full[qb], c * 64, g * a.hpg, t0 + i, b);
        ++nq;
      };
      auto load_k = [&](int i) {
        int bks[16];
        load_blocks(a.idx + (((size_t)b * R + t0 + i) * a.G + g) * a.n, a.n, bks);
#pragma unroll
        for (int p = 0; p < 8; ++p) {
          if (p >= npairs || !ok) break;
          const int tk0 = block_token(bks[2 * p]);
          const int tk1 = block_token(bks[2 * p + 1]);
          for (int c = 0; c < kcs; ++c) {
            const int slot = kv % kRingK;
            if (!mbar_wait(&bars->k_empty[slot], (uint32_t)(((kv / kRingK) & 1) ^ 1), abort_flag, a.st, 302)) {
              ok = false;
              return;
            }
            uint8_t* dst = kring + slot * kSlotK;
            mbar_arrive_expect_tx(&bars->k_full[slot], kSlotK);
            tma_kv(dst, &mapK, &bars->k_full[slot], c * 64, g, tk0, b, hm);
            tma_kv(dst + 8192, &mapK, &bars->k_full[slot], c * 64, g, tk1, b, hm);
            ++kv;
          }
        }
      };
      auto load_v = [&](int i) {
        int bks[16];
        load_blocks(a.idx + (((size_t)b * R + t0 + i) * a.G + g) * a.n, a.n, bks);
#pragma unroll
        for (int p = 0; p < 8; ++p) {
          if (p >= npairs || !ok) break;
          const int tk0 = block_token(bks[2 * p]);
          const int tk1 = block_token(bks[2 * p + 1]);
          const int slot = vv % kRingV;
          if (!mbar_wait(&bars->v_empty[slot], (uint32_t)(((vv / kRingV) & 1) ^ 1), abort_flag, a.st, 303)) {
            ok = false;
            return;
          }
          uint8_t* dst = vring + slot * kSlotV;
          mbar_arrive_expect_tx(&bars->v_full[slot], (uint32_t)(vcs * 16384));
          for (int c = 0; c < vcs; ++c) {
            tma_kv(dst + c * 16384, &mapV, &bars->v_full[slot], c * 64, g, tk0, b, hm);
            tma_kv(dst + c * 16384 + 8192, &mapV, &bars->v_full[slot], c * 64, g, tk1, b, hm);
          }
          ++vv;
        }
      };
      if (warp == 8) {
        for (int i = 0; i < nitems && ok; ++i) {
          load_q(i);
          load_k(i);
        }
      } else {
        for (int i = 0; i < nitems && ok; ++i) load_v(i);
      }
      if (!ok || *abort_flag) {
        for (int x = (nq > 2 ? nq - 2 : 0); x < nq; ++x)
          mbar_wait_plain(&bars->q_full[x & 1], (uint32_t)((x >> 1) & 1), kWaitLimitNs);
        for (int x = (kv > kRingK ? kv - kRingK : 0); x < kv; ++x)
          mbar_wait_plain(&bars->k_full[x % kRingK], (uint32_t)((x / kRingK) & 1), kWaitLimitNs);
        for (int x = (vv > kRingV ? vv - kRingV : 0); x < vv; ++x)
          mbar_wait_plain(&bars->v_full[x % kRingV], (uint32_t)((x / kRingV) & 1), kWaitLimitNs);
      }
    }
  } else if (warp == 9 || warp == 11) {
    // =============================================================== MMA issuers
    // warp 9 issues QK^T of every item, warp 11 PV; they use separate TMEM
    // accumulators, so the key and value streams are consumed concurrently
    if (lane == 0) {
      const uint32_t idesc_qk = idesc_bf16_f32(128, NP, false, false);
      const uint32_t idesc_pv = idesc_bf16_f32(128, NP, true, false);
      const uint32_t q_a = smem_u32(qbuf), k_a = smem_u32(kring), v_a = smem_u32(vring), p_a = smem_u32(pt);
      bool ok = true;
      int kv = 0, vv = 0;
      auto issue_qk = [&](int i) {
        if (!ok) return;
        const int sb = i & 1;
        const uint32_t par = (uint32_t)((i >> 1) & 1);
        if (!mbar_wait(&bars->s_free[sb], par ^ 1, abort_flag, a.st, 311) ||
            !mbar_wait(&bars->q_full[sb], par, abort_flag, a.st, 312)) {
          ok = false;
          return;
        }
        tc_fence_after();
        for (int p = 0; p < npairs; ++p) {
          for (int c = 0; c < kcs; ++c) {
            const int slot = kv % kRingK;
            if (!mbar_wait(&bars->k_full[slot], (uint32_t)((kv / kRingK) & 1), abort_flag, a.st, 313)) {
              ok = false;
              return;
            }
            tc_fence_after();
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint64_t ad = sdesc_sw128(k_a + slot * kSlotK + k * 32, 16, 1024);
              const uint64_t bd = sdesc_sw128(q_a + (sb * kcs + c) * kQBuf + k * 32, 16, 1024);
              umma_bf16(tmem_s + sb * SC + p * NP, ad, bd, idesc_qk, (c > 0 || k > 0) ? 1u : 0u);
            }
            umma_commit(&bars->k_empty[slot]);
            ++kv;
          }
        }
        umma_commit(&bars->s_full[sb]);
        umma_commit(&bars->q_empty[sb]);
      };
      auto issue_pv = [&](int i) {
        if (!ok) return;
        const int pb = i & 1, ob = i & 3;
        if (!mbar_wait(&bars->o_free[ob], (uint32_t)(((i >> 2) & 1) ^ 1), abort_flag, a.st, 314) ||
            !mbar_wait(&bars->p_full[pb], (uint32_t)((i >> 1) & 1), abort_flag, a.st, 315)) {
          ok = false;
          return;
        }
        tc_fence_after();
        for (int p = 0; p < npairs; ++p) {
          const int slot = vv % kRingV;
          if (!mbar_wait(&bars->v_full[slot], (uint32_t)((vv / kRingV) & 1), abort_flag, a.st, 316)) {
            ok = false;
            return;
          }
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            // A = V^T (dv-major rows of keys), B = P^T (head rows, keys along K)
            const uint64_t ad = sdesc_sw128(v_a + slot * kSlotV + k * 2048, 16384, 1024);
            const uint64_t bd =
                sdesc_sw128(p_a + pb * kPBuf + (p * 2 + (k >> 2)) * kQBuf + (k & 3) * 32, 16, 1024);
            umma_bf16(tmem_o + ob * NP, ad, bd, idesc_pv, (p > 0 || k > 0) ? 1u : 0u);
          }
          umma_commit(&bars->v_empty[slot]);
          ++vv;
        }
        umma_commit(&bars->p_free[pb]);
        umma_commit(&bars->o_full[ob]);
      };
      if (warp == 9) {
        for (int i = 0; i < nitems; ++i) issue_qk(i);
      } else {
        for (int i = 0; i < nitems; ++i) issue_pv(i);
      }
      if (!ok || *abort_flag) {
        // wait for every MMA this thread issued before the CTA releases TMEM
        umma_commit(&bars->drain[warp == 9 ? 0 : 1]);
        mbar_wait_plain(&bars->drain[warp == 9 ? 0 : 1], 0, kWaitLimitNs);
      }
    }
  } else if (warp < 8) {
    // =============================================================== softmax + epilogue
    const int wg = warp >> 2;                 // warpgroup: items i with i % 2 == wg
    const int lw = warp & 3;
    const int r = lw * 32 + lane;             // TMEM lane: key of a pair / value dim
    const uint32_t lane_base = (uint32_t)(lw * 32) << 16;
    const bool hi_half = (r >> 6) != 0;
    const int kk = r & 63;
    uint8_t* my_pt = pt + wg * kPBuf;
    float* red_m = red + wg * 2 * 4 * NP;     // [4][NP]
    float* red_l = red_m + 4 * NP;            // [4][NP]
    bool ok = true;
    uint32_t wg_phase = 0;
    auto wg_sync = [&]() {
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->wg[wg]);
      if (!mbar_wait(&bars->wg[wg], wg_phase & 1, abort_flag, a.st, 321)) ok = false;
      ++wg_phase;
    };
    float coef[NP];   // g_slc / sum of the item whose epilogue is pending
    float linv[NP];   // kSave: 1 / sum of that item

    // softmax of item i: P^T (unnormalised) into this warpgroup's buffer and
    // coef[h] = g_slc[h] / sum[h]
    auto softmax = [&](int i) {
      if (!ok) return;
      const int row = t0 + i;
      const int t = qoff + row;               // position of the query
      const int sb = i & 1;
      const uint32_t par = (uint32_t)((i >> 1) & 1);
      int bks[16];
      load_blocks(a.idx + (((size_t)b * R + row) * a.G + g) * a.n, a.n, bks);
      float gsl[NP];
      {
        const __nv_bfloat16* gp = a.gates + (((size_t)b * R + row) * a.H + g * a.hpg) * 3 + 1;
#pragma unroll
        for (int h = 0; h < NP; ++h) gsl[h] = h < a.hpg ? __bfloat162float(gp[3 * h]) : 0.f;
      }
      if (!mbar_wait(&bars->s_full[sb], par, abort_flag, a.st, 322)) {
        ok = false;
        return;
      }
      tc_fence_after();
      // pass 1: per-head max of the raw scores over the valid kept keys
      float mx[NP];
#pragma unroll
      for (int h = 0; h < NP; ++h) mx[h] = -INFINITY;
#pragma unroll
      for (int p = 0; p < 8; ++p) {
        if (p < npairs) {
          uint32_t rr[16];
          tmem_ld16(tmem_s + lane_base + sb * SC + p * NP, rr);
          tmem_ld_wait(rr);
          const int bk = hi_half ? bks[2 * p + 1] : bks[2 * p];
          const bool valid = bk >= 0 && bk * 64 + kk <= t;
#pragma unroll
          for (int h = 0; h < NP; ++h) mx[h] = fmaxf(mx[h], valid ? __uint_as_float(rr[h]) : -INFINITY);
        }
      }
#pragma unroll
      for (int h = 0; h < NP; ++h) mx[h] = warp_max_f32(mx[h]);
      if (lane == 0)
#pragma unroll
        for (int h = 0; h < NP; ++h) red_m[lw * NP + h] = mx[h];
      wg_sync();
      if (!ok) return;
#pragma unroll
      for (int h = 0; h < NP; ++h) {
        const float m = fmaxf(fmaxf(red_m[h], red_m[NP + h]), fmaxf(red_m[2 * NP + h], red_m[3 * NP + h]));
        mx[h] = (m == -INFINITY) ? 0.f : m * a.sc2;
      }
      // pass 2: p = exp(s*scale - max), sums, P^T (bf16) for the PV MMA
      if (!mbar_wait(&bars->p_free[sb], par ^ 1, abort_flag, a.st, 323)) {
        ok = false;
        return;
      }
      tc_fence_after();
      float ls[NP];
#pragma unroll
      for (int h = 0; h < NP; ++h) ls[h] = 0.f;
#pragma unroll
      for (int p = 0; p < 8; ++p) {
        if (p < npairs) {
          uint32_t rr[16];
          tmem_ld16(tmem_s + lane_base + sb * SC + p * NP, rr);
          tmem_ld_wait(rr);
          const int bk = hi_half ? bks[2 * p + 1] : bks[2 * p];
          const bool valid = bk >= 0 && bk * 64 + kk <= t;
          uint8_t* chunk = my_pt + (p * 2 + (hi_half ? 1 : 0)) * kQBuf + (kk & 7) * 2;
#pragma unroll
          for (int h = 0; h < NP; ++h) {
            const float e = valid ? fast_exp2(fmaf(__uint_as_float(rr[h]), a.sc2, -mx[h])) : 0.f;
            ls[h] += e;
            *reinterpret_cast<__nv_bfloat16*>(chunk + sw128_offset(h, kk >> 3)) = __float2bfloat16_rn(e);
          }
        }
      }
      tc_fence_before();
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&bars->s_free[sb]);
        mbar_arrive(&bars->p_full[sb]);
      }
      // sums per head over the warpgroup (off the MMA's critical path)
      const float ws = warp_sum16(ls, lane);
      if ((lane & 1) == 0) red_l[lw * NP + head_of_lane(lane)] = ws;
      wg_sync();
      if (!ok) return;
#pragma unroll
      for (int h = 0; h < NP; ++h) {
        const float l = red_l[h] + red_l[NP + h] + red_l[2 * NP + h] + red_l[3 * NP + h];
        coef[h] = (l > 0.f) ? __fdividef(gsl[h], l) : 0.f;
        if constexpr (kSave) linv[h] = (l > 0.f) ? __fdividef(1.f, l) : 0.f;
      }
      if constexpr (kSave) {
        // thread r < hpg: head r's log-sum-exp, m * sc2 + log2(l) in the
        // exp2 domain the kernel uses (the max and the sums as above)
        // (the maxima come from this thread's registers: the red_m rows may
        // already hold a later item's maxima)
        if (lw == 0 && lane < a.hpg) {
          const int hh = lane;
          float mm = 0.f;
#pragma unroll
          for (int h = 0; h < NP; ++h)
            if (h == hh) mm = mx[h];
          const float l = red_l[hh] + red_l[NP + hh] + red_l[2 * NP + hh] + red_l[3 * NP + hh];
          a.slc_lse[((size_t)b * R + row) * a.H + g * a.hpg + hh] = l > 0.f ? mm + __log2f(l) : INFINITY;
        }
      }
    };

    auto epilogue = [&](int i, const float (&cf)[NP], const float (&li)[NP]) {
      if (!ok) return;
      const int ob = i & 3;
      const int d = r;
      const size_t rowbase = ((size_t)b * R + t0 + i) * a.H + g * a.hpg;
      // the cmp+win partial sum of this item, read before waiting for O
      float prt[NP];
#pragma unroll
      for (int h = 0; h < NP; ++h)
        prt[h] = (h < a.hpg && d < a.dv) ? a.part[(rowbase + h) * a.dv + d] : 0.f;
      if (!mbar_wait(&bars->o_full[ob], (uint32_t)((i >> 2) & 1), abort_flag, a.st, 324)) {
        ok = false;
        return;
      }
      tc_fence_after();
      uint32_t rr[16];
      tmem_ld16(tmem_o + lane_base + ob * NP, rr);
      tmem_ld_wait(rr);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->o_free[ob]);
      if (d < a.dv) {
#pragma unroll
        for (int h = 0; h < NP; ++h) {
          if (h < a.hpg) {
            a.out[(rowbase + h) * a.dv + d] = __float2bfloat16_rn(fmaf(cf[h], __uint_as_float(rr[h]), prt[h]));
            if constexpr (kSave) a.slc_o[(rowbase + h) * a.dv + d] = li[h] * __uint_as_float(rr[h]);
          }
        }
      }
    };

    // items wg, wg+2, ...: softmax(next) overlaps the PV of the current item,
    // whose epilogue follows
    float cprev[NP], lprev[NP];
    if (wg < nitems) {
      softmax(wg);
#pragma unroll
      for (int h = 0; h < NP; ++h) {
        cprev[h] = coef[h];
        if constexpr (kSave) lprev[h] = linv[h];
      }
    }
    for (int i = wg; i < nitems; i += 2) {
      if (i + 2 < nitems) softmax(i + 2);
      epilogue(i, cprev, lprev);
#pragma unroll
      for (int h = 0; h < NP; ++h) {
        cprev[h] = coef[h];
        if constexpr (kSave) lprev[h] = linv[h];
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

struct Layout {
  uint32_t off_kring, off_vring, off_pt, off_red, off_bar, total;
};

Layout layout_for(int dk, int n) {
  Layout L;
  (void)n;
  L.off_kring = (uint32_t)align_up((size_t)2 * (dk / 64) * kQBuf, 1024);
  L.off_vring = L.off_kring + kRingK * kSlotK;
  L.off_pt = L.off_vring + kRingV * kSlotV;
  L.off_red = L.off_pt + 2 * kPBuf;
  L.off_bar = (uint32_t)align_up(L.off_red + 2 * 2 * 4 * NP * sizeof(float), 256);
  L.total = L.off_bar + (uint32_t)align_up(sizeof(Bars), 256) + 1024;
  return L;
}

}  // namespace

size_t sel_smem_bytes(const nsa_cfg& c) { return layout_for(c.dk, c.n).total; }

int launch_sel(const nsa_cfg& c, const void* q, const void* k, const void* v, const void* gates, const int32_t* idx,
               const void* part, void* out, DeviceStatus* st, cudaStream_t s, const QueryRows& rows, float* slc_lse,
               float* slc_o) {
  const int R = rows.R > 0 ? rows.R : c.T;
  const int hpg = c.H / c.G;
  if (hpg > NP || c.n > 16 || (c.dv != 64 && c.dv != 128)) return NSA_ERR_UNSUPPORTED;
  const Layout L = layout_for(c.dk, c.n);
  if (L.total > smem_max()) return NSA_ERR_UNSUPPORTED;
  const uint64_t e = 2;
  CUtensorMap mq, mk, mv;
  {  // q [B,R,H,dk]: box (64, hpg heads, 1 query row)
    const uint64_t dims[4] = {(uint64_t)c.dk, (uint64_t)c.H, (uint64_t)R, (uint64_t)c.B};
    const uint64_t str[3] = {c.dk * e, (uint64_t)c.H * c.dk * e, (uint64_t)R * c.H * c.dk * e};
    const uint32_t box[4] = {64, (uint32_t)hpg, 1, 1};
    if (!make_tmap_bf16(&mq, q, 4, dims, str, box)) return NSA_ERR_CUDA;
  }
  // k, v: boxes of 64 columns x 64 tokens (one selection block) of one head
  if (!make_kv_map(&mk, k, c.B, c.T, c.G, c.dk, 64, rows.head_major)) return NSA_ERR_CUDA;
  if (!make_kv_map(&mv, v, c.B, c.T, c.G, c.dv, 64, rows.head_major)) return NSA_ERR_CUDA;
  SelArgs a;
  a.T = c.T;
  a.H = c.H;
  a.G = c.G;
  a.dk = c.dk;
  a.dv = c.dv;
  a.n = c.n;
  a.hpg = hpg;
  a.QPC = kItemsPerCta;
  a.R = R;
  a.qoff = rows.qoff;
  a.hm = rows.head_major ? 1 : 0;
  const float scale = c.scale > 0.f ? c.scale : 1.0f / sqrtf((float)c.dk);
  a.sc2 = scale * 1.4426950408889634f;
  a.idx = idx;
  a.gates = static_cast<const __nv_bfloat16*>(gates);
  a.part = static_cast<const float*>(part);
  a.out = static_cast<__nv_bfloat16*>(out);
  a.slc_lse = slc_lse;
  a.slc_o = slc_o;
  a.st = st;
  a.off_kring = L.off_kring;
  a.off_vring = L.off_vring;
  a.off_pt = L.off_pt;
  a.off_red = L.off_red;
  a.off_bar = L.off_bar;
  dim3 grid((R + a.QPC - 1) / a.QPC, c.G, c.B);
  const bool save = slc_lse != nullptr && slc_o != nullptr;
  if (rows.head_major) {
    if (save) return NSA_ERR_UNSUPPORTED;
    if (int rc = ensure_smem_attr(reinterpret_cast<const void*>(&sel_kernel<true, false>), smem_max())) return rc;
    prof::begin("sel_multi", s);
    sel_kernel<true, false><<<grid, kThreads, L.total, s>>>(mq, mk, mv, a);
  } else {
    if (rows.R > 0 && rows.R != c.T) return NSA_ERR_UNSUPPORTED;   // token-major rows are positions
    if (save) {
      if (int rc = ensure_smem_attr(reinterpret_cast<const void*>(&sel_kernel<false, true>), smem_max())) return rc;
      prof::begin("sel_save", s);
      sel_kernel<false, true><<<grid, kThreads, L.total, s>>>(mq, mk, mv, a);
    } else {
      if (int rc = ensure_smem_attr(reinterpret_cast<const void*>(&sel_kernel<false, false>), smem_max())) return rc;
      prof::begin("sel", s);
      sel_kernel<false, false><<<grid, kThreads, L.total, s>>>(mq, mk, mv, a);
    }
  }
  prof::end(s);
  return cudaPeekAtLastError() == cudaSuccess ? NSA_OK : NSA_ERR_CUDA;
}

}  // namespace nsa
