// backward.cu -- NSA backward pass over whole sequences: gradients of
// <dout, out> for the prefill forward (three branches and the gated combine
// [P2 II; P3 token compression / selection / sliding window], the pages'
// 6.0x training-speed figure [P2 III.3]).
//
// The pages give no backward formula; the gradients are those of the forward
// under three readings: the kept blocks are constants (top-n has no
// gradient), the bf16 rounding of the compressed cache passes gradients
// unchanged, and W_c / PE gradients sum over the KV heads.  Each branch is
// softmax attention, so its backward is the textbook one: with
// P = softmax(s), dO_b = g_b * dout,
//     dV_j += P_j dO_b,   dS_j = P_j (dO_b . V_j - dO_b . O_b),
//     dq += scale sum_j dS_j K_j,   dK_j += scale dS_j q,
// and dg_b = dout . O_b = sum_j P_j (dout . V_j).
//
// Kernels (in launch order):
//  1. bwd_dq_kernel     one item = one query t of one KV group g (the group's
//                       16 heads on the MMA N side, keys on M, as in the
//                       forward's selected-block kernel).  Per branch: pass 0
//                       streams the keys once for the log-sum-exp and dg_b
//                       (per-thread online max / sum, merged across the 128
//                       key lanes at the end); pass 1 streams them again for
//                       dS and accumulates dQ^T = K^T dS^T in TMEM over all
//                       three branches.  Writes dq, dgates and, per branch,
//                       the log-sum-exp and dg of every (t, h) row.
//  2. slc_count / build_units / slc_fill: for the selected branch the
//                       inverse of the kept-block lists (per (b, g, block):
//                       the queries that kept it); for every branch a list of
//                       work units (b, g, key tile, query range).
//  3. bwd_dkv_kernel<BR> key-outer, one CTA per unit at a time: a 128-key tile
//                       (K and V loaded once) against chunks of 4 queries x 16
//                       heads (64 MMA columns):
//                           S^T  = K Q^T,   dP'^T = V dout^T          (tcgen05, TMEM)
//                           P^T g, dS^T  -> bf16 in TMEM
//                           dV  += (g P)^T dout,  dK += dS^T Q         (A from TMEM)
//                       The unit's dK / dV are added to global memory with
//                       fp32 reductions (units of one key tile may overlap).
//  4. compression backward on CUDA cores in fp32: dX overlap-add of
//     dB_i = dXc_i W^T into dk / dv, dPE = (sum_i dXc_i) W_r^T per offset r,
//     dW = sum_i flatten(X_i + PE)^T dXc_i.
#include <algorithm>

#include "common.cuh"
#include "kernels.hpp"
#include "profiler.hpp"
#include "tmap.hpp"

namespace nsa {

namespace {

constexpr int NP = 16;              // MMA N of one item: the group's heads, padded
constexpr int kQB = 2048;           // one 64-column chunk of NP rows (bf16, 128-B swizzle)
constexpr int kChunk = 16384;       // one 64-column chunk of 128 key rows
constexpr int kRowsPerUnit = 1024;  // queries per key-outer work unit
constexpr int kDqRingK = 3;         // bwd_dq_kernel: key-pair slots (held until the dQ MMA)

constexpr int kBrCmp = 0, kBrSlc = 1, kBrWin = 2;

// ============================================================================
// branch key lists of one query (shared by every role of bwd_dq_kernel)
// ============================================================================
struct BranchKeys {
  int np;      // 128-row key tiles ("pairs")
  int start;   // cmp: visible entries nc; win: first token of the window
};

__device__ __forceinline__ int visible_compressed(int t, int Nc) {
  // entries i with 16 i + 31 <= t (l = 32, d = 16)
  return t >= 31 ? min(Nc, (t - 31) / 16 + 1) : 0;
}

__device__ __forceinline__ BranchKeys branch_keys(int br, int t, int Nc, int n, int w) {
  BranchKeys k;
  if (br == kBrCmp) {
    k.start = visible_compressed(t, Nc);
    k.np = (k.start + 127) / 128;
  } else if (br == kBrSlc) {
    k.start = 0;
    k.np = (n + 1) / 2;
  } else {
    k.start = max(0, t - w + 1);
    k.np = (t - k.start + 1 + 127) / 128;
  }
  return k;
}

// The n (<= 16) kept blocks of query t, -1 past n.
__device__ __forceinline__ void load_kept(const int32_t* blk, int n, int (&bk)[16]) {
#pragma unroll
  for (int k = 0; k < 16; ++k) bk[k] = k < n ? __ldg(blk + k) : -1;
}

__device__ __forceinline__ int block_token(int blk) { return blk >= 0 ? blk * 64 : -128; }

// ============================================================================
// 1. dQ, dgates, per-branch log-sum-exp and dg
// ============================================================================
struct DqArgs {
  int T, H, G, dk, dv, n, w, hpg, Nc, QPC;
  int br_lo, br_hi;                // branches handled (cmp 0, slc 1, win 2)
  int acc_dq;                      // add to dq (another kernel wrote the other branches)
  float sc2, scale;
  const int32_t* idx;              // [B,T,G,n]
  const float* slc_lse;            // nullable: the forward's selected-branch log-sum-exp [B,T,H]
  const float* slc_o;              // and O_slc [B,T,H,dv]: the statistics pass is skipped
  const __nv_bfloat16* dout;       // [B,T,H,dv]
  const __nv_bfloat16* gates;      // [B,T,H,3]
  float* dq;                       // [B,T,H,dk]
  float* dgates;                   // [B,T,H,3]
  float* lse;                      // [3][B,T,H]  log2-domain log-sum-exp of s*scale
  float* dgw;                      // [3][B,T,H]  dout . O_b
  DeviceStatus* st;
  uint32_t off_kv, off_ds, off_red, off_bar;
};

struct DqBars {
  uint64_t q_full[2], q_empty[2];
  uint64_t k_full[kDqRingK], k_empty[kDqRingK];
  uint64_t v_full, v_empty;
  uint64_t s_full[4], s_free[4];
  uint64_t ds_full[2], ds_free[2];
  uint64_t dq_full[2], dq_free[2];
  uint64_t wg[2];
  uint64_t drain;
  uint32_t tmem;
  int abort_flag;
};

constexpr int kDqThreads = 320;   // warps 0-7 softmax (two warpgroups), 8 producer, 9 MMA

__global__ void __launch_bounds__(kDqThreads, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap mapQ, const __grid_constant__ CUtensorMap mapDO,
                  const __grid_constant__ CUtensorMap mapK, const __grid_constant__ CUtensorMap mapV,
                  const __grid_constant__ CUtensorMap mapKc, const __grid_constant__ CUtensorMap mapVc,
                  const DqArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const int kcs = a.dk / 64, vcs = a.dv / 64, cs = kcs + vcs;
  const int kslot_bytes = kcs * kChunk;
  uint8_t* qbuf = smem;                         // 2 items x (kcs Q + vcs dout) chunks x 2 KB
  uint8_t* kring = smem + a.off_kv;             // kDqRingK slots x kcs K chunks x 16 KB
  uint8_t* vbuf = kring + kDqRingK * kslot_bytes;   // vcs V chunks x 16 KB
  uint8_t* dsbuf = smem + a.off_ds;             // 2 x dS^T (2 chunks x 2 KB)
  float* red = reinterpret_cast<float*>(smem + a.off_red);   // [2 warpgroups][3][4 warps][NP / 2]
  DqBars* bars = reinterpret_cast<DqBars*>(smem + a.off_bar);
  volatile int* abort_flag = &bars->abort_flag;

  const int g = blockIdx.y, b = blockIdx.z;
  const int t0 = blockIdx.x * a.QPC;
  const int nitems = min(a.QPC, a.T - t0);
  const int warp = warp_id(), lane = lane_id();
  const int nm = (a.dk + 127) / 128;            // M=128 tiles of dQ^T (dk rows)

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->q_full[i], 1);
      mbar_init(&bars->q_empty[i], 1);
      mbar_init(&bars->ds_full[i], 8);
      mbar_init(&bars->ds_free[i], 1);
      mbar_init(&bars->dq_full[i], 1);
      mbar_init(&bars->dq_free[i], 8);
      mbar_init(&bars->wg[i], 4);
    }
    for (int i = 0; i < 4; ++i) {
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->s_free[i], 8);
    }
    for (int i = 0; i < kDqRingK; ++i) {
      mbar_init(&bars->k_full[i], 1);
      mbar_init(&bars->k_empty[i], 1);
    }
    mbar_init(&bars->v_full, 1);
    mbar_init(&bars->v_empty, 1);
    mbar_init(&bars->drain, 1);
    bars->abort_flag = prior_error(a.st);
    fence_barrier_init();
  }
  // query / dout rows hpg..NP-1 are never loaded: keep them zero
  for (int i = threadIdx.x; i < 2 * cs * kQB / 16; i += kDqThreads)
    reinterpret_cast<uint4*>(qbuf)[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  if (warp == 0) {
    tmem_alloc(&bars->tmem, 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem;
  const uint32_t tmem_sd = tmem;          // 4 x (S^T 16 + dP'^T 16) columns
  const uint32_t tmem_dq = tmem + 128;    // 2 x (nm x 16) columns

  if (*abort_flag) {
  } else if (warp == 8) {
    // ===================================================================== producer
    if (lane == 0) {
      tma_prefetch_desc(&mapQ);
      tma_prefetch_desc(&mapDO);
      tma_prefetch_desc(&mapK);
      tma_prefetch_desc(&mapV);
      bool ok = true;
      int jp = 0, nq = 0, nv = 0;
      for (int i = 0; i < nitems && ok; ++i) {
        const int t = t0 + i;
        const int qb = i & 1;
        if (!mbar_wait(&bars->q_empty[qb], (uint32_t)(((i >> 1) & 1) ^ 1), abort_flag, a.st, 801)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&bars->q_full[qb], (uint32_t)(cs * a.hpg * 128));
        for (int c = 0; c < kcs; ++c)
          tma_load_4d(qbuf + (qb * cs + c) * kQB, &mapQ, &bars->q_full[qb], c * 64, g * a.hpg, t, b);
        for (int c = 0; c < vcs; ++c)
          tma_load_4d(qbuf + (qb * cs + kcs + c) * kQB, &mapDO, &bars->q_full[qb], c * 64, g * a.hpg, t, b);
        ++nq;
        int bks[16];
        load_kept(a.idx + (((size_t)b * a.T + t) * a.G + g) * a.n, a.n, bks);
        for (int br = a.br_lo; br <= a.br_hi && ok; ++br) {
          const BranchKeys bk = branch_keys(br, t, a.Nc, a.n, a.w);
          for (int pass = (br == kBrSlc && a.slc_lse != nullptr) ? 1 : 0; pass < 2 && ok; ++pass) {
            for (int p = 0; p < bk.np; ++p) {
              const int ks = jp % kDqRingK;
              if (!mbar_wait(&bars->k_empty[ks], (uint32_t)(((jp / kDqRingK) & 1) ^ 1), abort_flag, a.st, 802)) {
                ok = false;
                break;
              }
              int tk0, tk1;   // first row of each 64-row half (entries for cmp, tokens otherwise)
              if (br == kBrCmp) {
                tk0 = 128 * p;
                tk1 = tk0 + 64;
              } else if (br == kBrSlc) {
                int b0 = -1, b1 = -1;
#pragma unroll
                for (int q = 0; q < 8; ++q)
                  if (q == p) {
                    b0 = bks[2 * q];
                    b1 = bks[2 * q + 1];
                  }
                tk0 = block_token(b0);
                tk1 = block_token(b1);
              } else {
                tk0 = bk.start + 128 * p;
                tk1 = tk0 + 64;
              }
              auto load_half = [&](uint8_t* dst, const CUtensorMap* m, uint64_t* bar, int col, int row) {
                if (br == kBrCmp) tma_load_4d(dst, m, bar, col, row, g, b);
                else tma_load_4d(dst, m, bar, col, g, row, b);
              };
              {
                uint8_t* dst = kring + ks * kslot_bytes;
                uint64_t* bar = &bars->k_full[ks];
                const CUtensorMap* m = br == kBrCmp ? &mapKc : &mapK;
                mbar_arrive_expect_tx(bar, (uint32_t)kslot_bytes);
                for (int c = 0; c < kcs; ++c) {
                  load_half(dst + c * kChunk, m, bar, c * 64, tk0);
                  load_half(dst + c * kChunk + 8192, m, bar, c * 64, tk1);
                }
              }
              if (!mbar_wait(&bars->v_empty, (uint32_t)((jp & 1) ^ 1), abort_flag, a.st, 803)) {
                ok = false;
                ++jp;
                break;
              }
              {
                const CUtensorMap* m = br == kBrCmp ? &mapVc : &mapV;
                mbar_arrive_expect_tx(&bars->v_full, (uint32_t)(vcs * kChunk));
                for (int c = 0; c < vcs; ++c) {
                  load_half(vbuf + c * kChunk, m, &bars->v_full, c * 64, tk0);
                  load_half(vbuf + c * kChunk + 8192, m, &bars->v_full, c * 64, tk1);
                }
              }
              ++jp;
              ++nv;
            }
          }
        }
      }
      if (!ok || *abort_flag) {
        for (int x = (nq > 2 ? nq - 2 : 0); x < nq; ++x)
          mbar_wait_plain(&bars->q_full[x & 1], (uint32_t)((x >> 1) & 1), kWaitLimitNs);
        for (int x = (jp > kDqRingK ? jp - kDqRingK : 0); x < jp; ++x)
          mbar_wait_plain(&bars->k_full[x % kDqRingK], (uint32_t)((x / kDqRingK) & 1), kWaitLimitNs);
        if (nv > 0) mbar_wait_plain(&bars->v_full, (uint32_t)((nv - 1) & 1), kWaitLimitNs);
      }
    }
  } else if (warp == 9) {
    // ===================================================================== MMA issuer
    if (lane == 0) {
      const uint32_t idesc_s = idesc_bf16_f32(128, NP, false, false);
      const uint32_t idesc_dq = idesc_bf16_f32(128, NP, true, false);
      const uint32_t q_a = smem_u32(qbuf), k_a = smem_u32(kring), v_a = smem_u32(vbuf), ds_a = smem_u32(dsbuf);
      // first 64-row chunk of each dQ^T tile: 0, then dk - 128 (overlapping rows discarded)
      const int mchunk1 = (a.dk - 128) / 64;
      bool ok = true;
      int jp = 0, jd = 0;
      for (int i = 0; i < nitems && ok; ++i) {
        const int t = t0 + i;
        const int qb = i & 1;
        const int qq = i & 1;
        if (!mbar_wait(&bars->q_full[qb], (uint32_t)((i >> 1) & 1), abort_flag, a.st, 811) ||
            !mbar_wait(&bars->dq_free[qq], (uint32_t)(((i >> 1) & 1) ^ 1), abort_flag, a.st, 812)) {
          ok = false;
          break;
        }
        tc_fence_after();
        bool dq_started = false;
        // dQ^T of a dS pass pair is issued after the next pair's S^T / dP'^T,
        // so those run while the rows form this pair's dS
        int pend_slot = -1, pend_db = 0;
        auto issue_dq = [&]() -> bool {
          if (!mbar_wait(&bars->ds_full[pend_db], (uint32_t)((jd >> 1) & 1), abort_flag, a.st, 815)) return false;
          tc_fence_after();
          const uint32_t kvs = k_a + pend_slot * kslot_bytes;
          for (int m = 0; m < nm; ++m) {
            const int mc = m == 0 ? 0 : mchunk1;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              // A = K^T (dk-major rows of keys), B = dS^T (head rows, keys along K)
              const uint64_t ad = sdesc_sw128(kvs + mc * kChunk + k * 2048, kChunk, 1024);
              const uint64_t bd = sdesc_sw128(ds_a + pend_db * 2 * kQB + (k >> 2) * kQB + (k & 3) * 32, 16, 1024);
              umma_bf16(tmem_dq + qq * 32 + m * 16, ad, bd, idesc_dq, (dq_started || k > 0) ? 1u : 0u);
            }
          }
          dq_started = true;
          umma_commit(&bars->ds_free[pend_db]);
          umma_commit(&bars->k_empty[pend_slot]);
          ++jd;
          pend_slot = -1;
          return true;
        };
        for (int br = a.br_lo; br <= a.br_hi && ok; ++br) {
          const BranchKeys bk = branch_keys(br, t, a.Nc, a.n, a.w);
          for (int pass = (br == kBrSlc && a.slc_lse != nullptr) ? 1 : 0; pass < 2 && ok; ++pass) {
            for (int p = 0; p < bk.np; ++p) {
              const int slot = jp % kDqRingK, sb = jp & 3;
              if (!mbar_wait(&bars->k_full[slot], (uint32_t)((jp / kDqRingK) & 1), abort_flag, a.st, 813) ||
                  !mbar_wait(&bars->s_free[sb], (uint32_t)(((jp >> 2) & 1) ^ 1), abort_flag, a.st, 814)) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint32_t kvs = k_a + slot * kslot_bytes;
              for (int c = 0; c < kcs; ++c) {
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                  const uint64_t ad = sdesc_sw128(kvs + c * kChunk + k * 32, 16, 1024);
                  const uint64_t bd = sdesc_sw128(q_a + (qb * cs + c) * kQB + k * 32, 16, 1024);
                  umma_bf16(tmem_sd + sb * 32, ad, bd, idesc_s, (c > 0 || k > 0) ? 1u : 0u);
                }
              }
              if (!mbar_wait(&bars->v_full, (uint32_t)(jp & 1), abort_flag, a.st, 816)) {
                ok = false;
                break;
              }
              tc_fence_after();
              for (int c = 0; c < vcs; ++c) {
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                  const uint64_t ad = sdesc_sw128(v_a + c * kChunk + k * 32, 16, 1024);
                  const uint64_t bd = sdesc_sw128(q_a + (qb * cs + kcs + c) * kQB + k * 32, 16, 1024);
                  umma_bf16(tmem_sd + sb * 32 + 16, ad, bd, idesc_s, (c > 0 || k > 0) ? 1u : 0u);
                }
              }
              umma_commit(&bars->v_empty);
              umma_commit(&bars->s_full[sb]);
              if (pend_slot >= 0 && !issue_dq()) {
                ok = false;
                break;
              }
              if (pass == 1) {
                pend_slot = slot;
                pend_db = jd & 1;
              } else {
                umma_commit(&bars->k_empty[slot]);
              }
              ++jp;
            }
          }
        }
        if (ok && pend_slot >= 0 && !issue_dq()) ok = false;
        if (!ok) break;
        umma_commit(&bars->q_empty[qb]);
        umma_commit(&bars->dq_full[qq]);
      }
      if (!ok || *abort_flag) {
        umma_commit(&bars->drain);
        mbar_wait_plain(&bars->drain, 0, kWaitLimitNs);
      }
    }
  } else {
    // ===================================================================== softmax + epilogue
    // two warpgroups on the same 128 lanes, warpgroup wg taking heads
    // 8 wg .. 8 wg + 7 of every tile (the heads' statistics are independent)
    constexpr int HW = NP / 2;
    const int wg = warp >> 2, lw = warp & 3;
    const int h0 = wg * HW;
    const int r = lw * 32 + lane;             // TMEM lane: key row of a tile / dk row of dQ^T
    const uint32_t lane_base = (uint32_t)(lw * 32) << 16;
    float* red_m = red + wg * 3 * 4 * HW;     // [4][HW]
    float* red_l = red_m + 4 * HW;            // [4][HW]
    float* red_a = red_l + 4 * HW;            // [4][HW]
    bool ok = true;
    uint32_t wg_phase = 0;
    auto wg_sync = [&]() {
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->wg[wg]);
      if (!mbar_wait(&bars->wg[wg], wg_phase & 1, abort_flag, a.st, 821)) ok = false;
      ++wg_phase;
    };
    auto warp_sum = [](float x) {
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
      return x;
    };
    // this warpgroup's 8 columns of S^T and dP'^T in score buffer sb
    auto load_sd = [&](int sb, uint32_t (&sr)[HW], uint32_t (&dr)[HW]) {
      const uint32_t base = tmem_sd + lane_base + sb * 32 + h0;
      asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                   : "=r"(sr[0]), "=r"(sr[1]), "=r"(sr[2]), "=r"(sr[3]), "=r"(sr[4]), "=r"(sr[5]), "=r"(sr[6]),
                     "=r"(sr[7])
                   : "r"(base));
      asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                   : "=r"(dr[0]), "=r"(dr[1]), "=r"(dr[2]), "=r"(dr[3]), "=r"(dr[4]), "=r"(dr[5]), "=r"(dr[6]),
                     "=r"(dr[7])
                   : "r"(base + 16));
      asm volatile("tcgen05.wait::ld.sync.aligned;"
                   : "+r"(sr[0]), "+r"(sr[1]), "+r"(sr[2]), "+r"(sr[3]), "+r"(sr[4]), "+r"(sr[5]), "+r"(sr[6]),
                     "+r"(sr[7]), "+r"(dr[0]), "+r"(dr[1]), "+r"(dr[2]), "+r"(dr[3]), "+r"(dr[4]), "+r"(dr[5]),
                     "+r"(dr[6]), "+r"(dr[7])
                   :
                   : "memory");
    };
    const int mchunk1 = (a.dk - 128) / 64;
    int jp = 0, jd = 0;
    for (int i = 0; i < nitems && ok; ++i) {
      const int t = t0 + i;
      const int qq = i & 1;
      const size_t rowbase = ((size_t)b * a.T + t) * a.H + g * a.hpg;
      int bks[16];
      load_kept(a.idx + (((size_t)b * a.T + t) * a.G + g) * a.n, a.n, bks);
      bool any = false;
      for (int br = a.br_lo; br <= a.br_hi && ok; ++br) {
        const BranchKeys bk = branch_keys(br, t, a.Nc, a.n, a.w);
        float gs[HW];
#pragma unroll
        for (int hh = 0; hh < HW; ++hh)
          gs[hh] = h0 + hh < a.hpg ? __bfloat162float(a.gates[(rowbase + h0 + hh) * 3 + br]) : 0.f;
        float lse2[HW], dg[HW];
        // head h0 + lane (lane < HW) writes its row's statistics
        auto write_row = [&](float lv, float dv) {
          if (lw == 0 && lane < HW && h0 + lane < a.hpg) {
            const size_t row = rowbase + h0 + lane;
            a.dgates[row * 3 + br] = dv;
            a.lse[(size_t)br * a.T * a.H * gridDim.z + row] = lv;
            a.dgw[(size_t)br * a.T * a.H * gridDim.z + row] = dv;
          }
        };
        if (br == kBrSlc && a.slc_lse != nullptr) {
          // ---- the forward's statistics: lse as saved, dg = dout . O_slc
          // (thread r takes value dim r of each head; sums over the 128 lanes)
#pragma unroll
          for (int hh = 0; hh < HW; ++hh) {
            const size_t e = (rowbase + h0 + hh) * a.dv + r;
            const float v = (h0 + hh < a.hpg && r < a.dv) ? __bfloat162float(a.dout[e]) * a.slc_o[e] : 0.f;
            const float vw = warp_sum(v);
            if (lane == 0) red_a[lw * HW + hh] = vw;
            lse2[hh] = h0 + hh < a.hpg ? a.slc_lse[rowbase + h0 + hh] : INFINITY;
          }
          wg_sync();
          if (!ok) break;
          float mine_l = 0.f, mine_d = 0.f;
#pragma unroll
          for (int hh = 0; hh < HW; ++hh) {
            dg[hh] = red_a[hh] + red_a[HW + hh] + red_a[2 * HW + hh] + red_a[3 * HW + hh];
            if (hh == lane) {
              mine_l = lse2[hh];
              mine_d = dg[hh];
            }
          }
          write_row(mine_l, mine_d);
          wg_sync();   // the reduction array is reused by the next item
          if (!ok) break;
        } else {
          // ---- pass 0: per-thread online max / sum / sum of p * dP' over this lane's keys
          float m[HW], l[HW], s1[HW];
#pragma unroll
          for (int hh = 0; hh < HW; ++hh) {
            m[hh] = -INFINITY;
            l[hh] = 0.f;
            s1[hh] = 0.f;
          }
          for (int p = 0; p < bk.np; ++p) {
            const int sb = jp & 3;
            if (!mbar_wait(&bars->s_full[sb], (uint32_t)((jp >> 2) & 1), abort_flag, a.st, 822)) {
              ok = false;
              break;
            }
            tc_fence_after();
            uint32_t sr[HW], dr[HW];
            load_sd(sb, sr, dr);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->s_free[sb]);
            ++jp;
            bool valid;
            if (br == kBrCmp) {
              valid = 128 * p + r < bk.start;
            } else if (br == kBrSlc) {
              int blk = -1;
#pragma unroll
              for (int q = 0; q < 8; ++q)
                if (q == p) blk = (r >> 6) ? bks[2 * q + 1] : bks[2 * q];
              valid = blk >= 0 && blk * 64 + (r & 63) <= t;
            } else {
              valid = bk.start + 128 * p + r <= t;
            }
            if (valid) {
#pragma unroll
              for (int hh = 0; hh < HW; ++hh) {
                const float sv = __uint_as_float(sr[hh]) * a.sc2;
                const float dp = __uint_as_float(dr[hh]);
                if (sv > m[hh]) {
                  const float f = fast_exp2(m[hh] - sv);   // 0 when m = -inf
                  l[hh] = fmaf(l[hh], f, 1.f);
                  s1[hh] = fmaf(s1[hh], f, dp);
                  m[hh] = sv;
                } else {
                  const float e = fast_exp2(sv - m[hh]);
                  l[hh] += e;
                  s1[hh] = fmaf(e, dp, s1[hh]);
                }
              }
            }
          }
          if (!ok) break;
          // merge across the 128 key lanes: per warp, then across the 4 warps
#pragma unroll
          for (int hh = 0; hh < HW; ++hh) {
            const float mw = warp_max_f32(m[hh]);
            const float f = (m[hh] == -INFINITY) ? 0.f : fast_exp2(m[hh] - mw);
            const float lw_ = warp_sum(l[hh] * f);
            const float aw_ = warp_sum(s1[hh] * f);
            if (lane == 0) {
              red_m[lw * HW + hh] = mw;
              red_l[lw * HW + hh] = lw_;
              red_a[lw * HW + hh] = aw_;
            }
          }
          wg_sync();
          if (!ok) break;
          float mine_l = 0.f, mine_d = 0.f;
#pragma unroll
          for (int hh = 0; hh < HW; ++hh) {
            float M = -INFINITY;
#pragma unroll
            for (int x = 0; x < 4; ++x) M = fmaxf(M, red_m[x * HW + hh]);
            float L = 0.f, A = 0.f;
            if (M != -INFINITY) {
#pragma unroll
              for (int x = 0; x < 4; ++x) {
                const float mx = red_m[x * HW + hh];
                const float f = (mx == -INFINITY) ? 0.f : fast_exp2(mx - M);
                L = fmaf(red_l[x * HW + hh], f, L);
                A = fmaf(red_a[x * HW + hh], f, A);
              }
            }
            lse2[hh] = L > 0.f ? M + __log2f(L) : INFINITY;
            dg[hh] = L > 0.f ? __fdividef(A, L) : 0.f;
            if (hh == lane) {
              mine_l = lse2[hh];
              mine_d = dg[hh];
            }
          }
          write_row(mine_l, mine_d);
          wg_sync();   // the reduction arrays are reused by the next branch
          if (!ok) break;
        }
        // ---- pass 1: dS^T -> shared memory (bf16) for dQ^T += K^T dS^T
        for (int p = 0; p < bk.np; ++p) {
          const int sb = jp & 3;
          const int db = jd & 1;
          if (!mbar_wait(&bars->s_full[sb], (uint32_t)((jp >> 2) & 1), abort_flag, a.st, 823)) {
            ok = false;
            break;
          }
          tc_fence_after();
          uint32_t sr[HW], dr[HW];
          load_sd(sb, sr, dr);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars->s_free[sb]);
          ++jp;
          bool valid;
          if (br == kBrCmp) {
            valid = 128 * p + r < bk.start;
          } else if (br == kBrSlc) {
            int blk = -1;
#pragma unroll
            for (int q = 0; q < 8; ++q)
              if (q == p) blk = (r >> 6) ? bks[2 * q + 1] : bks[2 * q];
            valid = blk >= 0 && blk * 64 + (r & 63) <= t;
          } else {
            valid = bk.start + 128 * p + r <= t;
          }
          if (!mbar_wait(&bars->ds_free[db], (uint32_t)(((jd >> 1) & 1) ^ 1), abort_flag, a.st, 824)) {
            ok = false;
            break;
          }
          const int kk = r & 63;
          uint8_t* chunk = dsbuf + db * 2 * kQB + (r >> 6) * kQB + (kk & 7) * 2;
#pragma unroll
          for (int hh = 0; hh < HW; ++hh) {
            float ds = 0.f;
            if (valid) {
              const float pr = fast_exp2(fmaf(__uint_as_float(sr[hh]), a.sc2, -lse2[hh]));
              ds = gs[hh] * a.scale * pr * (__uint_as_float(dr[hh]) - dg[hh]);
            }
            *reinterpret_cast<__nv_bfloat16*>(chunk + sw128_offset(h0 + hh, kk >> 3)) = __float2bfloat16_rn(ds);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars->ds_full[db]);
          ++jd;
          any = true;
        }
      }
      if (!ok) break;
      // ---- epilogue: dq rows of this item (fp32), this warpgroup's heads
      if (!mbar_wait(&bars->dq_full[qq], (uint32_t)((i >> 1) & 1), abort_flag, a.st, 825)) {
        ok = false;
        break;
      }
      tc_fence_after();
      for (int m = 0; m < nm; ++m) {
        uint32_t rr[HW];
        asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                     : "=r"(rr[0]), "=r"(rr[1]), "=r"(rr[2]), "=r"(rr[3]), "=r"(rr[4]), "=r"(rr[5]), "=r"(rr[6]),
                       "=r"(rr[7])
                     : "r"(tmem_dq + lane_base + qq * 32 + m * 16 + h0));
        asm volatile("tcgen05.wait::ld.sync.aligned;"
                     : "+r"(rr[0]), "+r"(rr[1]), "+r"(rr[2]), "+r"(rr[3]), "+r"(rr[4]), "+r"(rr[5]), "+r"(rr[6]),
                       "+r"(rr[7])
                     :
                     : "memory");
        const int drow = (m == 0 ? 0 : mchunk1 * 64) + r;
        const bool own = drow < a.dk && (m == 0 || drow >= 128);
        if (own) {
#pragma unroll
          for (int hh = 0; hh < HW; ++hh)
            if (h0 + hh < a.hpg) {
              float* o = a.dq + (rowbase + h0 + hh) * a.dk + drow;
              const float v = any ? __uint_as_float(rr[hh]) : 0.f;
              *o = a.acc_dq ? *o + v : v;
            }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->dq_free[qq]);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, 256);
}

// ============================================================================
// 1b. dQ of the compressed and window branches, query-tile form
// ============================================================================
// One CTA = 8 consecutive queries of one KV group: 128 rows (query, head) on
// the MMA M side against 128-key tiles, so every key tile is read once for 8
// queries (the compressed and window keys of neighbouring queries coincide):
//     S   = Q K^T,  dP' = dout V^T                  (M=128 rows, N=128 keys)
//     dQ += dS K      (dS bf16 in tensor memory as the A operand, N = dk)
// Thread = TMEM lane = one (query, head) row, so a row's statistics need no
// cross-thread reduction.  Per branch a statistics pass and a dS pass, as in
// bwd_dq_kernel.  Writes dq (fp32, overwritten), dgates and the branch rows
// of lse / dg.
constexpr int kTileQ = 8;
constexpr int kTileThreads = 320;     // warps 0-7 rows (two warpgroups), 8 producer, 9 MMA

struct TileArgs {
  int T, H, G, dk, dv, w, hpg, Nc;
  float sc2, scale;
  const __nv_bfloat16* gates;     // [B,T,H,3]
  float* dq;                      // [B,T,H,dk]
  float* dgates;                  // [B,T,H,3]
  float* lse;                     // [3][B,T,H]
  float* dgw;                     // [3][B,T,H]
  DeviceStatus* st;
  uint32_t off_do, off_k, off_v, off_x, off_bar;
};

struct TileBars {
  uint64_t q_full;
  uint64_t k_full[2], k_empty[2];
  uint64_t v_full, v_empty;
  uint64_t s_full, s_free;
  uint64_t ds_full, ds_free;
  uint64_t dq_full;
  uint64_t xbar[2];
  uint64_t drain;
  uint32_t tmem;
  int abort_flag;
};

struct TileKeys {
  int ntiles;   // 128-key tiles of the CTA's 8 queries
  int base;     // cmp: first entry (0); win: first token
};

__device__ __forceinline__ TileKeys tile_keys(int br, int t0, int t_last, int Nc, int w) {
  TileKeys k;
  if (br == kBrCmp) {
    k.base = 0;
    k.ntiles = (visible_compressed(t_last, Nc) + 127) / 128;
  } else {
    k.base = max(0, t0 - w + 1);
    k.ntiles = (t_last - k.base + 1 + 127) / 128;
  }
  return k;
}

__global__ void __launch_bounds__(kTileThreads, 1)
    bwd_dq_tile_kernel(const __grid_constant__ CUtensorMap mapQ, const __grid_constant__ CUtensorMap mapDO,
                       const __grid_constant__ CUtensorMap mapK, const __grid_constant__ CUtensorMap mapV,
                       const __grid_constant__ CUtensorMap mapKc, const __grid_constant__ CUtensorMap mapVc,
                       const TileArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const int kcs = a.dk / 64, vcs = a.dv / 64;
  uint8_t* qt = smem;                       // Q tile: kcs chunks x 16 KB (128 rows x 64 columns)
  uint8_t* dot = smem + a.off_do;           // dout tile: vcs chunks x 16 KB
  uint8_t* kring = smem + a.off_k;          // 2 x kcs chunks x 16 KB
  uint8_t* vbuf = smem + a.off_v;           // vcs chunks x 16 KB
  TileBars* bars = reinterpret_cast<TileBars*>(smem + a.off_bar);
  volatile int* abort_flag = &bars->abort_flag;
  const int g = blockIdx.y, b = blockIdx.z;
  const int t0 = blockIdx.x * kTileQ;
  const int t_last = min(a.T - 1, t0 + kTileQ - 1);
  const int warp = warp_id(), lane = lane_id();
  const int kslot = kcs * kChunk;

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->k_full[i], 1);
      mbar_init(&bars->k_empty[i], 1);
    }
    mbar_init(&bars->v_full, 1);
    mbar_init(&bars->v_empty, 1);
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->s_free, 8);
    mbar_init(&bars->ds_full, 8);
    mbar_init(&bars->xbar[0], 8);
    mbar_init(&bars->xbar[1], 8);
    mbar_init(&bars->ds_free, 1);
    mbar_init(&bars->dq_full, 1);
    mbar_init(&bars->drain, 1);
    bars->abort_flag = prior_error(a.st);
    fence_barrier_init();
  }
  // query / dout rows of heads hpg..15 are never loaded: keep them zero
  for (int i = threadIdx.x; i < (int)(a.off_k / 16); i += kTileThreads)
    reinterpret_cast<uint4*>(smem)[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  if (warp == 0) {
    tmem_alloc(&bars->tmem, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem;
  const uint32_t tm_s = tmem, tm_dp = tmem + 128, tm_ds = tmem + 256, tm_dq = tmem + 320;

  if (*abort_flag) {
  } else if (warp == 8) {
    // ===================================================================== producer
    if (lane == 0) {
      tma_prefetch_desc(&mapQ);
      tma_prefetch_desc(&mapDO);
      bool ok = true;
      mbar_arrive_expect_tx(&bars->q_full, (uint32_t)(kTileQ * (kcs + vcs) * a.hpg * 128));
      for (int k = 0; k < kTileQ; ++k) {
        for (int c = 0; c < kcs; ++c)
          tma_load_4d(qt + c * kChunk + k * kQB, &mapQ, &bars->q_full, c * 64, g * a.hpg, t0 + k, b);
        for (int c = 0; c < vcs; ++c)
          tma_load_4d(dot + c * kChunk + k * kQB, &mapDO, &bars->q_full, c * 64, g * a.hpg, t0 + k, b);
      }
      int jk = 0, jv = 0;
      for (int br = kBrCmp; br <= kBrWin && ok; br += kBrWin - kBrCmp) {
        const TileKeys tk = tile_keys(br, t0, t_last, a.Nc, a.w);
        const CUtensorMap* mk = br == kBrCmp ? &mapKc : &mapK;
        const CUtensorMap* mv = br == kBrCmp ? &mapVc : &mapV;
        for (int pass = 0; pass < 2 && ok; ++pass) {
          for (int kt = 0; kt < tk.ntiles; ++kt) {
            const int r0 = tk.base + 128 * kt;
            const int slot = jk & 1;
            if (!mbar_wait(&bars->k_empty[slot], (uint32_t)(((jk >> 1) & 1) ^ 1), abort_flag, a.st, 861)) {
              ok = false;
              break;
            }
            uint8_t* kd = kring + slot * kslot;
            mbar_arrive_expect_tx(&bars->k_full[slot], (uint32_t)kslot);
            for (int c = 0; c < kcs; ++c) {
              if (br == kBrCmp) {
                tma_load_4d(kd + c * kChunk, mk, &bars->k_full[slot], c * 64, r0, g, b);
                tma_load_4d(kd + c * kChunk + 8192, mk, &bars->k_full[slot], c * 64, r0 + 64, g, b);
              } else {
                tma_load_4d(kd + c * kChunk, mk, &bars->k_full[slot], c * 64, g, r0, b);
                tma_load_4d(kd + c * kChunk + 8192, mk, &bars->k_full[slot], c * 64, g, r0 + 64, b);
              }
            }
            ++jk;
            if (!mbar_wait(&bars->v_empty, (uint32_t)((jv & 1) ^ 1), abort_flag, a.st, 862)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&bars->v_full, (uint32_t)(vcs * kChunk));
            for (int c = 0; c < vcs; ++c) {
              if (br == kBrCmp) {
                tma_load_4d(vbuf + c * kChunk, mv, &bars->v_full, c * 64, r0, g, b);
                tma_load_4d(vbuf + c * kChunk + 8192, mv, &bars->v_full, c * 64, r0 + 64, g, b);
              } else {
                tma_load_4d(vbuf + c * kChunk, mv, &bars->v_full, c * 64, g, r0, b);
                tma_load_4d(vbuf + c * kChunk + 8192, mv, &bars->v_full, c * 64, g, r0 + 64, b);
              }
            }
            ++jv;
          }
        }
      }
      if (!ok || *abort_flag) {
        mbar_wait_plain(&bars->q_full, 0, kWaitLimitNs);
        for (int x = (jk > 2 ? jk - 2 : 0); x < jk; ++x)
          mbar_wait_plain(&bars->k_full[x & 1], (uint32_t)((x >> 1) & 1), kWaitLimitNs);
        if (jv > 0) mbar_wait_plain(&bars->v_full, (uint32_t)((jv - 1) & 1), kWaitLimitNs);
      }
    }
  } else if (warp == 9) {
    // ===================================================================== MMA issuer
    if (lane == 0) {
      const uint32_t idesc_s = idesc_bf16_f32(128, 128, false, false);
      const uint32_t idesc_dq = idesc_bf16_f32(128, a.dk, false, true);
      const uint32_t q_a = smem_u32(qt), do_a = smem_u32(dot), k_a = smem_u32(kring), v_a = smem_u32(vbuf);
      bool ok = mbar_wait(&bars->q_full, 0, abort_flag, a.st, 871);
      tc_fence_after();
      int jk = 0, jv = 0, jt = 0, jd = 0;
      bool dq_started = false;
      for (int br = kBrCmp; br <= kBrWin && ok; br += kBrWin - kBrCmp) {
        const TileKeys tk = tile_keys(br, t0, t_last, a.Nc, a.w);
        for (int pass = 0; pass < 2 && ok; ++pass) {
          for (int kt = 0; kt < tk.ntiles; ++kt) {
            const int slot = jk & 1;
            const uint32_t ks = k_a + slot * kslot;
            if (!mbar_wait(&bars->k_full[slot], (uint32_t)((jk >> 1) & 1), abort_flag, a.st, 872) ||
                !mbar_wait(&bars->s_free, (uint32_t)((jt & 1) ^ 1), abort_flag, a.st, 873)) {
              ok = false;
              break;
            }
            tc_fence_after();
            for (int c = 0; c < kcs; ++c) {
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const uint64_t ad = sdesc_sw128(q_a + c * kChunk + k * 32, 16, 1024);
                const uint64_t bd = sdesc_sw128(ks + c * kChunk + k * 32, 16, 1024);
                umma_bf16(tm_s, ad, bd, idesc_s, (c > 0 || k > 0) ? 1u : 0u);
              }
            }
            if (!mbar_wait(&bars->v_full, (uint32_t)(jv & 1), abort_flag, a.st, 874)) {
              ok = false;
              break;
            }
            tc_fence_after();
            for (int c = 0; c < vcs; ++c) {
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const uint64_t ad = sdesc_sw128(do_a + c * kChunk + k * 32, 16, 1024);
                const uint64_t bd = sdesc_sw128(v_a + c * kChunk + k * 32, 16, 1024);
                umma_bf16(tm_dp, ad, bd, idesc_s, (c > 0 || k > 0) ? 1u : 0u);
              }
            }
            umma_commit(&bars->v_empty);
            umma_commit(&bars->s_full);
            ++jv;
            ++jt;
            if (pass == 1) {
              if (!mbar_wait(&bars->ds_full, (uint32_t)(jd & 1), abort_flag, a.st, 875)) {
                ok = false;
                break;
              }
              tc_fence_after();
#pragma unroll
              for (int k = 0; k < 8; ++k) {
                // B = K rows (keys) along K, head dims along N (N-major, 16 KB per 64 columns)
                const uint64_t bd = sdesc_sw128(ks + k * 2048, kChunk, 1024);
                umma_bf16_ts(tm_dq, tm_ds + 8 * k, bd, idesc_dq, (dq_started || k > 0) ? 1u : 0u);
              }
              dq_started = true;
              umma_commit(&bars->ds_free);
              ++jd;
            }
            umma_commit(&bars->k_empty[slot]);
            ++jk;
          }
        }
      }
      if (ok) umma_commit(&bars->dq_full);
      if (!ok || *abort_flag) {
        umma_commit(&bars->drain);
        mbar_wait_plain(&bars->drain, 0, kWaitLimitNs);
      }
    }
  } else {
    // ===================================================================== rows
    // two warpgroups on the same 128 rows: warpgroup wg takes key columns
    // 64 wg .. 64 wg + 63 of every tile; a row's statistics are the merge of
    // the two halves (exchanged through shared memory, one buffer per branch)
    const int wg = warp >> 2, lw = warp & 3;
    const int r = lw * 32 + lane;
    const uint32_t lane_base = (uint32_t)(lw * 32) << 16;
    const int t = t0 + (r >> 4), h = r & 15;
    const bool row_ok = t < a.T && h < a.hpg;
    const size_t row = ((size_t)b * a.T + (row_ok ? t : 0)) * a.H + g * a.hpg + (row_ok ? h : 0);
    const size_t plane = (size_t)gridDim.z * a.T * a.H;
    float* xchg = reinterpret_cast<float*>(smem + a.off_x);   // [2 branches][2 warpgroups][3][128]
    bool ok = true;
    int jt = 0, jd = 0;
    bool any = false;
    for (int br = kBrCmp; br <= kBrWin && ok; br += kBrWin - kBrCmp) {
      const int bi = br == kBrCmp ? 0 : 1;
      const TileKeys tk = tile_keys(br, t0, t_last, a.Nc, a.w);
      const float gs = row_ok ? __bfloat162float(a.gates[row * 3 + br]) : 0.f;
      // visible keys of this row, as positions inside the branch's key range
      int lo, hi;
      if (br == kBrCmp) {
        lo = 0;
        hi = t >= 31 ? min(a.Nc - 1, (t - 31) / 16) : -1;
      } else {
        lo = max(0, t - a.w + 1) - tk.base;
        hi = t - tk.base;
      }
      float lse2 = INFINITY, dg = 0.f;
      for (int pass = 0; pass < 2 && ok; ++pass) {
        float m = -INFINITY, l = 0.f, s1 = 0.f;
        for (int kt = 0; kt < tk.ntiles; ++kt) {
          if (!mbar_wait(&bars->s_full, (uint32_t)(jt & 1), abort_flag, a.st, 881)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (pass == 1 && !mbar_wait(&bars->ds_free, (uint32_t)((jd & 1) ^ 1), abort_flag, a.st, 882)) {
            ok = false;
            break;
          }
          const int kb = 128 * kt;
          for (int gi = 0; gi < 4; ++gi) {
            const int grp = 4 * wg + gi;
            uint32_t sr[16], dr[16];
            tmem_ld16(tm_s + lane_base + grp * 16, sr);
            tmem_ld16(tm_dp + lane_base + grp * 16, dr);
            tmem_ld_wait(sr);
            tmem_reg_fence(dr);
            const int j0 = kb + grp * 16;
            if (pass == 0) {
              float gm = -INFINITY;
#pragma unroll
              for (int e = 0; e < 16; ++e) {
                const bool vis = j0 + e >= lo && j0 + e <= hi;
                if (vis) gm = fmaxf(gm, __uint_as_float(sr[e]) * a.sc2);
              }
              if (gm != -INFINITY) {
                const float mn = fmaxf(m, gm);
                const float f = fast_exp2(m - mn);
                l *= f;
                s1 *= f;
                m = mn;
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                  const bool vis = j0 + e >= lo && j0 + e <= hi;
                  if (vis) {
                    const float p = fast_exp2(fmaf(__uint_as_float(sr[e]), a.sc2, -m));
                    l += p;
                    s1 = fmaf(p, __uint_as_float(dr[e]), s1);
                  }
                }
              }
            } else {
              uint32_t pk[8];
#pragma unroll
              for (int e = 0; e < 16; e += 2) {
                float d2[2];
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                  const bool vis = j0 + e + u >= lo && j0 + e + u <= hi;
                  float d = 0.f;
                  if (vis) {
                    const float p = fast_exp2(fmaf(__uint_as_float(sr[e + u]), a.sc2, -lse2));
                    d = gs * a.scale * p * (__uint_as_float(dr[e + u]) - dg);
                  }
                  d2[u] = d;
                }
                pk[e / 2] = pack_bf16x2(d2[0], d2[1]);
              }
              // 8 columns of packed bf16 pairs per 16 keys
              asm volatile(
                  "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(
                      tm_ds + lane_base + grp * 8),
                  "r"(pk[0]), "r"(pk[1]), "r"(pk[2]), "r"(pk[3]), "r"(pk[4]), "r"(pk[5]), "r"(pk[6]), "r"(pk[7])
                  : "memory");
            }
          }
          if (pass == 1) tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(&bars->s_free);
            if (pass == 1) mbar_arrive(&bars->ds_full);
          }
          ++jt;
          if (pass == 1) {
            ++jd;
            any = true;
          }
        }
        if (!ok) break;
        if (pass == 0) {
          // merge the two warpgroups' halves of the row, in a fixed order
          float* xb = xchg + bi * 2 * 3 * 128;
          xb[(wg * 3 + 0) * 128 + r] = m;
          xb[(wg * 3 + 1) * 128 + r] = l;
          xb[(wg * 3 + 2) * 128 + r] = s1;
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars->xbar[bi]);
          if (!mbar_wait(&bars->xbar[bi], 0, abort_flag, a.st, 884)) {
            ok = false;
            break;
          }
          const float m0 = xb[0 * 128 + r], l0 = xb[1 * 128 + r], a0 = xb[2 * 128 + r];
          const float m1 = xb[3 * 128 + r], l1 = xb[4 * 128 + r], a1 = xb[5 * 128 + r];
          const float mm = fmaxf(m0, m1);
          float L = 0.f, A = 0.f;
          if (mm != -INFINITY) {
            const float f0 = m0 == -INFINITY ? 0.f : fast_exp2(m0 - mm);
            const float f1 = m1 == -INFINITY ? 0.f : fast_exp2(m1 - mm);
            L = fmaf(l0, f0, l1 * f1);
            A = fmaf(a0, f0, a1 * f1);
          }
          lse2 = L > 0.f ? mm + __log2f(L) : INFINITY;
          dg = L > 0.f ? __fdividef(A, L) : 0.f;
          if (row_ok && wg == 0) {
            a.dgates[row * 3 + br] = dg;
            a.lse[(size_t)br * plane + row] = lse2;
            a.dgw[(size_t)br * plane + row] = dg;
          }
        }
      }
    }
    // ---- epilogue: this row's dq (cmp + win), fp32; warpgroup wg writes half the columns
    if (ok && mbar_wait(&bars->dq_full, 0, abort_flag, a.st, 883)) {
      tc_fence_after();
      for (int c0 = wg * a.dk / 2; c0 < (wg + 1) * a.dk / 2; c0 += 16) {
        uint32_t rr[16];
        tmem_ld16(tm_dq + lane_base + c0, rr);
        tmem_ld_wait(rr);
        if (row_ok) {
          float4* o = reinterpret_cast<float4*>(a.dq + row * a.dk + c0);
#pragma unroll
          for (int e = 0; e < 16; e += 4)
            o[e / 4] = any ? make_float4(__uint_as_float(rr[e]), __uint_as_float(rr[e + 1]),
                                         __uint_as_float(rr[e + 2]), __uint_as_float(rr[e + 3]))
                           : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

// ============================================================================
// 2. selected-branch inverse lists and work units
// ============================================================================
// one thread per kept-block entry of idx [B,T,G,n]
__global__ void slc_count_kernel(const int32_t* __restrict__ idx, int B, int T, int G, int n, int nblk,
                                 int* __restrict__ cnt) {
  const size_t e = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  const size_t total = (size_t)B * T * G * n;
  if (e >= total) return;
  const int blk = idx[e];
  const size_t btg = e / n;
  const int g = (int)(btg % G);
  const int b = (int)(btg / ((size_t)T * G));
  if (blk >= 0 && blk < nblk) atomicAdd(&cnt[((size_t)b * G + g) * nblk + blk], 1);
}

__global__ void slc_fill_kernel(const int32_t* __restrict__ idx, int B, int T, int G, int n, int nblk,
                                const int* __restrict__ offs, int* __restrict__ fill, int* __restrict__ inv) {
  const size_t e = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  const size_t total = (size_t)B * T * G * n;
  if (e >= total) return;
  const int blk = idx[e];
  const size_t btg = e / n;
  const int g = (int)(btg % G);
  const int t = (int)((btg / G) % T);
  const int b = (int)(btg / ((size_t)T * G));
  if (blk < 0 || blk >= nblk) return;
  const size_t list = ((size_t)b * G + g) * nblk + blk;
  const int pos = atomicAdd(&fill[list], 1);
  inv[offs[list] + pos] = t;
}

struct UnitArgs {
  int B, T, G, Nc, w, nblk;
  int ntc, ntw;                 // 128-entry tiles of the compressed cache / 128-token tiles
  const int* cnt;               // [B*G*nblk] selected-branch list lengths
  int* offs;                    // [B*G*nblk] out: list starts in inv
  int4* units[3];               // out: {b*G+g, first key, query lo, query hi}
  int cap[3];
  int* nunits;                  // out: [3]
};

// Exclusive scan of one value per thread over the CTA (1024 threads); returns
// the thread's prefix and writes the CTA total to *total.
__device__ int cta_exclusive_scan(int v, int* sh, int* total) {
  const int lane = lane_id(), warp = warp_id();
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sh[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int s = lane < (int)(blockDim.x >> 5) ? sh[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    sh[32 + lane] = s;
  }
  __syncthreads();
  const int before = (warp > 0 ? sh[32 + warp - 1] : 0) + x - v;
  *total = sh[32 + (blockDim.x >> 5) - 1];
  __syncthreads();
  return before;
}

// One CTA of 1024 threads: list starts of the selected branch, and the work
// units of all three branches (each list cut into pieces of kRowsPerUnit).
__global__ void __launch_bounds__(1024) build_units_kernel(const UnitArgs a) {
  __shared__ int sh[64];
  // selected-branch list starts
  const int nl_s = a.B * a.G * a.nblk;
  int carry = 0;
  for (int base = 0; base < nl_s; base += blockDim.x) {
    const int l = base + threadIdx.x;
    const int v = l < nl_s ? a.cnt[l] : 0;
    int tot;
    const int pre = cta_exclusive_scan(v, sh, &tot);
    if (l < nl_s) a.offs[l] = carry + pre;
    carry += tot;
  }
  __syncthreads();
  // compressed branch: every compressed tile is seen by most queries, so its
  // units are listed query range first (ranges of kRowsPerUnit on a fixed
  // grid, then every tile that range sees): the CTAs running at one time
  // share their query rows through L2 instead of each reading them from HBM
  {
    const int nqr = (a.T + kRowsPerUnit - 1) / kRowsPerUnit;
    const int nl = a.B * a.G * nqr;
    int ucarry = 0;
    for (int base = 0; base < nl; base += blockDim.x) {
      const int l = base + threadIdx.x;
      const int qlo = (l % nqr) * kRowsPerUnit;
      const int qhi = min(a.T, qlo + kRowsPerUnit);
      int nu = 0;
      if (l < nl)
        for (int tile = 0; tile < a.ntc; ++tile) nu += 16 * 128 * tile + 31 < qhi ? 1 : 0;
      int tot;
      const int pre = cta_exclusive_scan(nu, sh, &tot);
      for (int tile = 0; tile < nu; ++tile) {
        const int u = ucarry + pre + tile;
        if (u < a.cap[kBrCmp])
          a.units[kBrCmp][u] = make_int4(l / nqr, 128 * tile, max(qlo, 16 * 128 * tile + 31), qhi);
      }
      ucarry += tot;
    }
    if (threadIdx.x == 0) a.nunits[kBrCmp] = min(ucarry, a.cap[kBrCmp]);
    __syncthreads();
  }
  for (int br = kBrSlc; br <= kBrWin; ++br) {
    const int per = br == kBrWin ? a.ntw : a.nblk;
    const int nl = a.B * a.G * per;
    int ucarry = 0;
    for (int base = 0; base < nl; base += blockDim.x) {
      const int l = base + threadIdx.x;
      int key0 = 0, lo = 0, hi = 0;
      if (l < nl) {
        const int tile = l % per;
        if (br == kBrWin) {
          key0 = 128 * tile;
          lo = key0;
          hi = min(a.T, key0 + 127 + a.w);
        } else {
          key0 = 64 * tile;
          lo = a.offs[l];
          hi = lo + a.cnt[l];
        }
      }
      const int nu = hi > lo ? (hi - lo + kRowsPerUnit - 1) / kRowsPerUnit : 0;
      int tot;
      const int pre = cta_exclusive_scan(nu, sh, &tot);
      for (int k = 0; k < nu; ++k) {
        const int u = ucarry + pre + k;
        if (u < a.cap[br])
          a.units[br][u] = make_int4(l / per, key0, lo + k * kRowsPerUnit, min(hi, lo + (k + 1) * kRowsPerUnit));
      }
      ucarry += tot;
    }
    if (threadIdx.x == 0) a.nunits[br] = min(ucarry, a.cap[br]);
    __syncthreads();
  }
}

// ============================================================================
// 3. key-outer dK / dV of one branch
// ============================================================================
struct DkvArgs {
  int T, H, G, dk, dv, w, hpg, Nc;
  float sc2, scale;
  const __nv_bfloat16* gates;  // [B,T,H,3]
  const float* lse;            // [B,T,H] of this branch
  const float* dgw;            // [B,T,H] of this branch
  const int* inv;              // selected branch: query lists
  const int4* units;
  const int* nunits;           // device count of this branch's units
  float* dK;                   // cmp: [B,G,Nc,dk]; slc/win: [B,T,G,dk]  (fp32, reduced into)
  float* dV;
  DeviceStatus* st;
  uint32_t off_q, off_col, off_bar;
};

constexpr int kDkvQBuf = 3;        // query-chunk buffers in flight

struct DkvBars {
  uint64_t kv_full, kv_empty;
  uint64_t q_full[kDkvQBuf], q_empty[kDkvQBuf];
  uint64_t col_full[kDkvQBuf], col_free[kDkvQBuf];
  uint64_t s_full, s_free;
  uint64_t p_full, p_free;
  uint64_t acc_full, acc_free;
  uint64_t drain;
  uint32_t tmem;
  int abort_flag;
};

struct ColInfo {
  int t;        // query position, -1 for a padded column
  float lse2;   // log2-domain log-sum-exp of the row
  float dg;     // dout . O_b of the row
  float gs;     // gate of the branch
};

constexpr int kDkvThreads = 320;   // warps 0-7 softmax / epilogue, 8 producer, 9 MMA
constexpr int kQChunk = 8192;      // one 64-column chunk of 4 queries x 16 heads

template <int BR>
__global__ void __launch_bounds__(kDkvThreads, 1)
    bwd_dkv_kernel(const __grid_constant__ CUtensorMap mapQ, const __grid_constant__ CUtensorMap mapDO,
                   const __grid_constant__ CUtensorMap mapK, const __grid_constant__ CUtensorMap mapV,
                   const DkvArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const int kcs = a.dk / 64, vcs = a.dv / 64, cs = kcs + vcs;
  uint8_t* kv = smem;                                   // kcs K + vcs V chunks x 16 KB
  uint8_t* qb_base = smem + a.off_q;                    // kDkvQBuf x (kcs Q + vcs dout) chunks x 8 KB
  ColInfo* cols = reinterpret_cast<ColInfo*>(smem + a.off_col);   // [kDkvQBuf][64]
  DkvBars* bars = reinterpret_cast<DkvBars*>(smem + a.off_bar);
  volatile int* abort_flag = &bars->abort_flag;
  const int warp = warp_id(), lane = lane_id();
  const int nunits = *a.nunits;

  if (threadIdx.x == 0) {
    mbar_init(&bars->kv_full, 1);
    mbar_init(&bars->kv_empty, 1);
    for (int i = 0; i < kDkvQBuf; ++i) {
      mbar_init(&bars->q_full[i], 1);
      mbar_init(&bars->q_empty[i], 1);
      mbar_init(&bars->col_full[i], 32);
      mbar_init(&bars->col_free[i], 8);
    }
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->s_free, 8);
    mbar_init(&bars->p_full, 8);
    mbar_init(&bars->p_free, 1);
    mbar_init(&bars->acc_full, 1);
    mbar_init(&bars->acc_free, 8);
    mbar_init(&bars->drain, 1);
    bars->abort_flag = prior_error(a.st);
    fence_barrier_init();
  }
  // key rows never loaded (the upper half of a selected-branch tile) and query
  // rows hpg..15 stay zero
  for (int i = threadIdx.x; i < (int)(a.off_col / 16); i += kDkvThreads)
    reinterpret_cast<uint4*>(smem)[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  if (warp == 0) {
    tmem_alloc(&bars->tmem, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem;
  const uint32_t tm_s = tmem, tm_dp = tmem + 64, tm_pg = tmem + 128, tm_ds = tmem + 160;
  const uint32_t tm_dk = tmem + 192, tm_dv = tmem + 192 + a.dk;

  if (*abort_flag) {
  } else if (warp == 8) {
    // ===================================================================== producer
    if (lane == 0) {
      tma_prefetch_desc(&mapQ);
      tma_prefetch_desc(&mapDO);
      tma_prefetch_desc(&mapK);
      tma_prefetch_desc(&mapV);
    }
    bool ok = true;
    int jc = 0, ju = 0;
    for (int u = blockIdx.x; u < nunits && ok; u += gridDim.x, ++ju) {
      const int4 un = a.units[u];
      const int b = un.x / a.G, g = un.x % a.G, key0 = un.y;
      const int nq = un.w - un.z;
      const int nch = (nq + 3) / 4;
      if (lane == 0) {
        if (!mbar_wait(&bars->kv_empty, (uint32_t)((ju & 1) ^ 1), abort_flag, a.st, 831)) ok = false;
        if (ok) {
          const uint32_t rows_bytes = BR == kBrSlc ? 8192u : 16384u;
          mbar_arrive_expect_tx(&bars->kv_full, (uint32_t)cs * rows_bytes);
          for (int c = 0; c < cs; ++c) {
            const CUtensorMap* m = c < kcs ? &mapK : &mapV;
            const int col = (c < kcs ? c : c - kcs) * 64;
            uint8_t* dst = kv + c * kChunk;
            if (BR == kBrCmp) {
              tma_load_4d(dst, m, &bars->kv_full, col, key0, g, b);
              tma_load_4d(dst + 8192, m, &bars->kv_full, col, key0 + 64, g, b);
            } else {
              tma_load_4d(dst, m, &bars->kv_full, col, g, key0, b);
              if (BR != kBrSlc) tma_load_4d(dst + 8192, m, &bars->kv_full, col, g, key0 + 64, b);
            }
          }
        }
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      for (int ci = 0; ci < nch && ok; ++ci, ++jc) {
        const int qb = jc % kDkvQBuf;
        const uint32_t par = (uint32_t)(((jc / kDkvQBuf) & 1) ^ 1);
        if (lane == 0) {
          if (!mbar_wait(&bars->q_empty[qb], par, abort_flag, a.st, 832) ||
              !mbar_wait(&bars->col_free[qb], par, abort_flag, a.st, 833))
            ok = false;
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok) break;
        // the chunk's 4 query positions
        int tq[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int e = un.z + 4 * ci + k;
          tq[k] = e < un.w ? (BR == kBrSlc ? __ldg(a.inv + e) : e) : -1;
        }
        if (lane == 0) {
          uint8_t* qd = qb_base + qb * cs * kQChunk;
          mbar_arrive_expect_tx(&bars->q_full[qb], (uint32_t)(4 * cs * a.hpg * 128));
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            for (int c = 0; c < kcs; ++c)
              tma_load_4d(qd + c * kQChunk + k * kQB, &mapQ, &bars->q_full[qb], c * 64, g * a.hpg, tq[k], b);
            for (int c = 0; c < vcs; ++c)
              tma_load_4d(qd + (kcs + c) * kQChunk + k * kQB, &mapDO, &bars->q_full[qb], c * 64, g * a.hpg,
                          tq[k], b);
          }
        }
        // per-column data: column 16 k + h is head h of query k
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          const int col = lane + 32 * x;
          const int k = col >> 4, h = col & 15;
          int tk = -1;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            if (kk == k) tk = tq[kk];
          ColInfo ci_;
          ci_.t = -1;
          ci_.lse2 = INFINITY;
          ci_.dg = 0.f;
          ci_.gs = 0.f;
          if (tk >= 0 && h < a.hpg) {
            const size_t row = ((size_t)b * a.T + tk) * a.H + g * a.hpg + h;
            ci_.t = tk;
            ci_.lse2 = a.lse[row];
            ci_.dg = a.dgw[row];
            ci_.gs = __bfloat162float(a.gates[row * 3 + BR]);
          }
          cols[qb * 64 + col] = ci_;
        }
        mbar_arrive(&bars->col_full[qb]);
      }
    }
    if (lane == 0 && (!ok || *abort_flag)) {
      for (int x = (jc > kDkvQBuf ? jc - kDkvQBuf : 0); x < jc; ++x)
        mbar_wait_plain(&bars->q_full[x % kDkvQBuf], (uint32_t)((x / kDkvQBuf) & 1), kWaitLimitNs);
      if (ju > 0) mbar_wait_plain(&bars->kv_full, (uint32_t)((ju - 1) & 1), kWaitLimitNs);
    }
  } else if (warp == 9) {
    // ===================================================================== MMA issuer
    if (lane == 0) {
      const uint32_t idesc_s = idesc_bf16_f32(128, 64, false, false);
      const uint32_t idesc_dv = idesc_bf16_f32(128, a.dv, false, true);
      const uint32_t idesc_dk = idesc_bf16_f32(128, a.dk, false, true);
      const uint32_t kv_a = smem_u32(kv), q_a = smem_u32(qb_base);
      bool ok = true;
      int jc = 0, ju = 0;
      for (int u = blockIdx.x; u < nunits && ok; u += gridDim.x, ++ju) {
        const int4 un = a.units[u];
        const int nch = (un.w - un.z + 3) / 4;
        if (!mbar_wait(&bars->kv_full, (uint32_t)(ju & 1), abort_flag, a.st, 841) ||
            !mbar_wait(&bars->acc_free, (uint32_t)((ju & 1) ^ 1), abort_flag, a.st, 842)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // S^T / dP'^T of chunk j into the (single) score buffer once the rows
        // have read chunk j-1's scores, so they run while the rows compute
        // chunk j-1's gP / dS; then dV / dK of chunk j-1
        auto issue_s = [&](int j) -> bool {
          const int qb = j % kDkvQBuf;
          const uint32_t qd = q_a + qb * cs * kQChunk;
          if (!mbar_wait(&bars->q_full[qb], (uint32_t)((j / kDkvQBuf) & 1), abort_flag, a.st, 843) ||
              !mbar_wait(&bars->s_free, (uint32_t)((j & 1) ^ 1), abort_flag, a.st, 844))
            return false;
          tc_fence_after();
          for (int c = 0; c < kcs; ++c) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint64_t ad = sdesc_sw128(kv_a + c * kChunk + k * 32, 16, 1024);
              const uint64_t bd = sdesc_sw128(qd + c * kQChunk + k * 32, 16, 1024);
              umma_bf16(tm_s, ad, bd, idesc_s, (c > 0 || k > 0) ? 1u : 0u);
            }
          }
          for (int c = 0; c < vcs; ++c) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint64_t ad = sdesc_sw128(kv_a + (kcs + c) * kChunk + k * 32, 16, 1024);
              const uint64_t bd = sdesc_sw128(qd + (kcs + c) * kQChunk + k * 32, 16, 1024);
              umma_bf16(tm_dp, ad, bd, idesc_s, (c > 0 || k > 0) ? 1u : 0u);
            }
          }
          umma_commit(&bars->s_full);
          return true;
        };
        if (nch > 0 && !issue_s(jc)) {
          ok = false;
          break;
        }
        for (int ci = 0; ci < nch; ++ci, ++jc) {
          const int qb = jc % kDkvQBuf;
          const uint32_t qd = q_a + qb * cs * kQChunk;
          if (ci + 1 < nch && !issue_s(jc + 1)) {
            ok = false;
            break;
          }
          if (!mbar_wait(&bars->p_full, (uint32_t)(jc & 1), abort_flag, a.st, 845)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            // B = dout / Q rows (t, h) along K, head dims along N (N-major, 8 KB per 64 columns)
            const uint64_t bdo = sdesc_sw128(qd + kcs * kQChunk + k * 2048, kQChunk, 1024);
            umma_bf16_ts(tm_dv, tm_pg + 8 * k, bdo, idesc_dv, (ci > 0 || k > 0) ? 1u : 0u);
            const uint64_t bq = sdesc_sw128(qd + k * 2048, kQChunk, 1024);
            umma_bf16_ts(tm_dk, tm_ds + 8 * k, bq, idesc_dk, (ci > 0 || k > 0) ? 1u : 0u);
          }
          umma_commit(&bars->q_empty[qb]);
          umma_commit(&bars->p_free);
        }
        if (!ok) break;
        umma_commit(&bars->kv_empty);
        umma_commit(&bars->acc_full);
      }
      if (!ok || *abort_flag) {
        umma_commit(&bars->drain);
        mbar_wait_plain(&bars->drain, 0, kWaitLimitNs);
      }
    }
  } else {
    // ===================================================================== softmax + epilogue
    // two warpgroups on the same 128 key lanes: warpgroup wg takes score
    // columns 32 wg .. 32 wg + 31 (queries 2 wg, 2 wg + 1) and, in the
    // epilogue, half of the dK and dV columns
    const int wg = warp >> 2, lw = warp & 3;
    const int r = lw * 32 + lane;             // TMEM lane = key row of the tile
    const uint32_t lane_base = (uint32_t)(lw * 32) << 16;
    bool ok = true;
    int jc = 0, ju = 0;
    for (int u = blockIdx.x; u < nunits && ok; u += gridDim.x, ++ju) {
      const int4 un = a.units[u];
      const int b = un.x / a.G, g = un.x % a.G, key0 = un.y;
      const int nch = (un.w - un.z + 3) / 4;
      // this lane's key: compressed entry or token position
      const int key = key0 + r;
      const bool key_ok = BR == kBrCmp ? key < a.Nc : (BR == kBrSlc ? (r < 64 && key < a.T) : key < a.T);
      const int vis_from = BR == kBrCmp ? 16 * key + 31 : key;   // first query that sees the key
      for (int ci = 0; ci < nch; ++ci, ++jc) {
        const int qb = jc % kDkvQBuf;
        const uint32_t par = (uint32_t)((jc / kDkvQBuf) & 1);
        if (!mbar_wait(&bars->col_full[qb], par, abort_flag, a.st, 851) ||
            !mbar_wait(&bars->s_full, (uint32_t)(jc & 1), abort_flag, a.st, 852)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const ColInfo* cc = cols + qb * 64;
        uint32_t pg[16], dsv[16];
#pragma unroll
        for (int gi = 0; gi < 2; ++gi) {
          const int grp = 2 * wg + gi;
          uint32_t sr[16], dr[16];
          tmem_ld16(tm_s + lane_base + grp * 16, sr);
          tmem_ld16(tm_dp + lane_base + grp * 16, dr);
          tmem_ld_wait(sr);
          tmem_reg_fence(dr);
#pragma unroll
          for (int h = 0; h < 16; h += 2) {
            float pv[2], dv2[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const ColInfo c = cc[grp * 16 + h + e];
              bool vis = key_ok && c.t >= 0 && c.t >= vis_from;
              if (BR == kBrWin) vis = vis && key > c.t - a.w;
              float p = 0.f, d = 0.f;
              if (vis) {
                p = fast_exp2(fmaf(__uint_as_float(sr[h + e]), a.sc2, -c.lse2));
                d = c.gs * a.scale * p * (__uint_as_float(dr[h + e]) - c.dg);
                p *= c.gs;
              }
              pv[e] = p;
              dv2[e] = d;
            }
            pg[gi * 8 + h / 2] = pack_bf16x2(pv[0], pv[1]);
            dsv[gi * 8 + h / 2] = pack_bf16x2(dv2[0], dv2[1]);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&bars->s_free);
          mbar_arrive(&bars->col_free[qb]);
        }
        if (!mbar_wait(&bars->p_free, (uint32_t)((jc & 1) ^ 1), abort_flag, a.st, 853)) {
          ok = false;
          break;
        }
        tc_fence_after();
        tmem_st16(tm_pg + lane_base + wg * 16, pg);
        tmem_st16(tm_ds + lane_base + wg * 16, dsv);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->p_full);
      }
      if (!ok) break;
      // ---- epilogue: this unit's dK / dV rows reduced into global memory
      if (!mbar_wait(&bars->acc_full, (uint32_t)(ju & 1), abort_flag, a.st, 854)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float* dkrow = nullptr;
      float* dvrow = nullptr;
      if (key_ok) {
        if (BR == kBrCmp) {
          dkrow = a.dK + (((size_t)b * a.G + g) * a.Nc + key) * a.dk;
          dvrow = a.dV + (((size_t)b * a.G + g) * a.Nc + key) * a.dv;
        } else {
          dkrow = a.dK + (((size_t)b * a.T + key) * a.G + g) * a.dk;
          dvrow = a.dV + (((size_t)b * a.T + key) * a.G + g) * a.dv;
        }
      }
      for (int c0 = wg * a.dk / 2; c0 < (wg + 1) * a.dk / 2; c0 += 16) {
        uint32_t rr[16];
        tmem_ld16(tm_dk + lane_base + c0, rr);
        tmem_ld_wait(rr);
        if (dkrow != nullptr)
#pragma unroll
          for (int e = 0; e < 16; ++e) atomicAdd(dkrow + c0 + e, __uint_as_float(rr[e]));
      }
      for (int c0 = wg * a.dv / 2; c0 < (wg + 1) * a.dv / 2; c0 += 16) {
        uint32_t rr[16];
        tmem_ld16(tm_dv + lane_base + c0, rr);
        tmem_ld_wait(rr);
        if (dvrow != nullptr)
#pragma unroll
          for (int e = 0; e < 16; ++e) atomicAdd(dvrow + c0 + e, __uint_as_float(rr[e]));
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->acc_free);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

// ============================================================================
// 4. compression backward (fp32, CUDA cores)
// ============================================================================
// s[e] = sum over (b, g, i) of dXc[b,g,i,e]
__global__ void colsum_kernel(const float* __restrict__ dxc, size_t rows, int D, float* __restrict__ s) {
  const int e = threadIdx.x;   // blockDim.x == D
  float acc = 0.f;
  for (size_t r = blockIdx.x; r < rows; r += gridDim.x) acc += dxc[r * D + e];
  atomicAdd(s + e, acc);
}

// dPE[r, c] = sum_e s[e] W[r*D + c, e]   (one CTA per offset r, one thread per c)
__global__ void dpe_kernel(const float* __restrict__ s, const __nv_bfloat16* __restrict__ W, int D,
                           float* __restrict__ dpe) {
  const int r = blockIdx.x, c = threadIdx.x;
  const __nv_bfloat16* wr = W + ((size_t)r * D + c) * D;
  float acc = 0.f;
  for (int e = 0; e < D; ++e) acc = fmaf(s[e], __bfloat162float(wr[e]), acc);
  dpe[(size_t)r * D + c] = acc;
}

// dX[b, 16 i + rr, g, c] += sum_{q in {0,1}} sum_e dXc[b,g,i-q,e] W[(rr + 16 q) D + c, e]
// for rr in [0,16): tile of 64 entries i x 64 columns c, 256 threads x (4 x 4).
// X is token-major [B,T,G,D] (fp32, the dk / dv output, added into).
__global__ void __launch_bounds__(256) dx_kernel(const float* __restrict__ dxc, const __nv_bfloat16* __restrict__ W,
                                                 int B, int T, int G, int Nc, int D, float* __restrict__ dX) {
  __shared__ float sa[16][65];   // [e][i]
  __shared__ float sw[16][65];   // [e][c]
  const int i0 = blockIdx.x * 64, c0 = blockIdx.y * 64;
  const int rr = blockIdx.z % 16, bg = blockIdx.z / 16;
  const int b = bg / G, g = bg % G;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  float acc[4][4];
#pragma unroll
  for (int x = 0; x < 4; ++x)
#pragma unroll
    for (int y = 0; y < 4; ++y) acc[x][y] = 0.f;
  const float* base = dxc + (size_t)bg * Nc * D;
  for (int q = 0; q < 2; ++q) {
    const int wrow = (rr + 16 * q) * D;
    for (int e0 = 0; e0 < D; e0 += 16) {
      for (int x = threadIdx.x; x < 16 * 64; x += 256) {
        const int ii = x / 16, e = x % 16;
        const int ent = i0 + ii - q;
        sa[e][ii] = (ent >= 0 && ent < Nc) ? base[(size_t)ent * D + e0 + e] : 0.f;
        sw[e][ii] = __bfloat162float(W[(size_t)(wrow + c0 + ii) * D + e0 + e]);
      }
      __syncthreads();
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        float av[4], wv[4];
#pragma unroll
        for (int x = 0; x < 4; ++x) av[x] = sa[e][ty * 4 + x];
#pragma unroll
        for (int y = 0; y < 4; ++y) wv[y] = sw[e][tx * 4 + y];
#pragma unroll
        for (int x = 0; x < 4; ++x)
#pragma unroll
          for (int y = 0; y < 4; ++y) acc[x][y] = fmaf(av[x], wv[y], acc[x][y]);
      }
      __syncthreads();
    }
  }
#pragma unroll
  for (int x = 0; x < 4; ++x) {
    const int tok = 16 * (i0 + ty * 4 + x) + rr;
    if (tok >= T) continue;
    float* o = dX + (((size_t)b * T + tok) * G + g) * D + c0 + tx * 4;
#pragma unroll
    for (int y = 0; y < 4; ++y) o[y] += acc[x][y];
  }
}

// dW[r*D + c, e] += sum over rows rho = (b, g, i) of (X[b, 16 i + r, g, c] + PE[r, c]) dXc[rho, e]:
// tile 64 c x 64 e, rows split in pieces of 256, fp32 reductions into dW.
__global__ void __launch_bounds__(256) dw_kernel(const __nv_bfloat16* __restrict__ X,
                                                 const __nv_bfloat16* __restrict__ PE,
                                                 const float* __restrict__ dxc, int B, int T, int G, int Nc, int D,
                                                 float* __restrict__ dW) {
  __shared__ float sx[16][65];   // [row][c]
  __shared__ float sd[16][65];   // [row][e]
  const int c0 = blockIdx.x * 64, e0 = blockIdx.y * 64;
  const int r = blockIdx.z % 32, piece = blockIdx.z / 32;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const size_t rows = (size_t)B * G * Nc;
  const size_t r_lo = (size_t)piece * 256, r_hi = min(rows, r_lo + 256);
  float acc[4][4];
#pragma unroll
  for (int x = 0; x < 4; ++x)
#pragma unroll
    for (int y = 0; y < 4; ++y) acc[x][y] = 0.f;
  for (size_t rb = r_lo; rb < r_hi; rb += 16) {
    for (int x = threadIdx.x; x < 16 * 64; x += 256) {
      const int rw = x / 64, cc = x % 64;
      const size_t rho = rb + rw;
      float xv = 0.f, dv = 0.f;
      if (rho < r_hi) {
        const int i = (int)(rho % Nc);
        const size_t bg = rho / Nc;
        const int g = (int)(bg % G), b = (int)(bg / G);
        xv = __bfloat162float(X[(((size_t)b * T + 16 * i + r) * G + g) * D + c0 + cc]) +
             __bfloat162float(PE[(size_t)r * D + c0 + cc]);
        dv = dxc[rho * D + e0 + cc];
      }
      sx[rw][cc] = xv;
      sd[rw][cc] = dv;
    }
    __syncthreads();
#pragma unroll
    for (int rw = 0; rw < 16; ++rw) {
      float xv[4], dv[4];
#pragma unroll
      for (int x = 0; x < 4; ++x) xv[x] = sx[rw][ty * 4 + x];
#pragma unroll
      for (int y = 0; y < 4; ++y) dv[y] = sd[rw][tx * 4 + y];
#pragma unroll
      for (int x = 0; x < 4; ++x)
#pragma unroll
        for (int y = 0; y < 4; ++y) acc[x][y] = fmaf(xv[x], dv[y], acc[x][y]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int x = 0; x < 4; ++x)
#pragma unroll
    for (int y = 0; y < 4; ++y)
      atomicAdd(dW + ((size_t)r * D + c0 + ty * 4 + x) * D + e0 + tx * 4 + y, acc[x][y]);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
struct DqLayout {
  uint32_t off_kv, off_ds, off_red, off_bar, total;
};
DqLayout dq_layout(int dk, int dv) {
  const int cs = dk / 64 + dv / 64;
  DqLayout L;
  L.off_kv = (uint32_t)align_up((size_t)2 * cs * kQB, 1024);
  L.off_ds = L.off_kv + (kDqRingK * (dk / 64) + dv / 64) * kChunk;
  L.off_red = L.off_ds + 2 * 2 * kQB;
  L.off_bar = (uint32_t)align_up(L.off_red + 3 * 4 * NP * sizeof(float), 256);
  L.total = L.off_bar + (uint32_t)align_up(sizeof(DqBars), 256) + 1024;
  return L;
}

struct TileLayout {
  uint32_t off_do, off_k, off_v, off_x, off_bar, total;
};
TileLayout tile_layout(int dk, int dv) {
  TileLayout L;
  L.off_do = (uint32_t)(dk / 64 * kChunk);
  L.off_k = L.off_do + (uint32_t)(dv / 64 * kChunk);
  L.off_v = L.off_k + (uint32_t)(2 * (dk / 64) * kChunk);
  L.off_x = L.off_v + (uint32_t)(dv / 64 * kChunk);
  L.off_bar = L.off_x + (uint32_t)(2 * 2 * 3 * 128 * sizeof(float));
  L.total = L.off_bar + (uint32_t)align_up(sizeof(TileBars), 256) + 1024;
  return L;
}

struct DkvLayout {
  uint32_t off_q, off_col, off_bar, total;
};
DkvLayout dkv_layout(int dk, int dv) {
  const int cs = dk / 64 + dv / 64;
  DkvLayout L;
  L.off_q = (uint32_t)(cs * kChunk);
  L.off_col = L.off_q + kDkvQBuf * cs * kQChunk;
  L.off_bar = (uint32_t)align_up(L.off_col + kDkvQBuf * 64 * sizeof(ColInfo), 256);
  L.total = L.off_bar + (uint32_t)align_up(sizeof(DkvBars), 256) + 1024;
  return L;
}

// q-like tensor [B,T,H,d]: boxes of 64 columns x hpg heads x 1 row
bool make_rows_map(CUtensorMap* m, const void* p, int B, int T, int H, int d, int hpg) {
  const uint64_t e = 2;
  const uint64_t dims[4] = {(uint64_t)d, (uint64_t)H, (uint64_t)T, (uint64_t)B};
  const uint64_t str[3] = {d * e, (uint64_t)H * d * e, (uint64_t)T * H * d * e};
  const uint32_t box[4] = {64, (uint32_t)hpg, 1, 1};
  return make_tmap_bf16(m, p, 4, dims, str, box);
}

}  // namespace

int bwd_supported(const nsa_cfg& c) {
  const int hpg = c.H / c.G;
  if (hpg > NP || c.n > 16 || (c.dk != 128 && c.dk != 192) || (c.dv != 64 && c.dv != 128)) return NSA_ERR_UNSUPPORTED;
  if (c.T > 65536 || c.B > 65535) return NSA_ERR_UNSUPPORTED;
  // grid limits of the compression-backward launches
  const long long Nc = c.T < 32 ? 0 : (c.T - 32) / 16 + 1;
  if (16ll * c.B * c.G > 65535 || 32ll * ((c.B * c.G * Nc + 255) / 256) > 65535) return NSA_ERR_UNSUPPORTED;
  if (dq_layout(c.dk, c.dv).total > smem_max() || dkv_layout(c.dk, c.dv).total > smem_max() ||
      tile_layout(c.dk, c.dv).total > smem_max())
    return NSA_ERR_UNSUPPORTED;
  return NSA_OK;
}

BwdWs bwd_ws(const nsa_cfg& c, size_t header) {
  const int Nc = c.T < 32 ? 0 : (c.T - 32) / 16 + 1;
  const int nblk = (c.T + 63) / 64;
  const size_t rows = (size_t)c.B * c.T * c.H;
  const size_t lists = (size_t)c.B * c.G * nblk;
  const int ntc = (Nc + 127) / 128, ntw = (c.T + 127) / 128;
  BwdWs w;
  w.cap[kBrCmp] = (size_t)c.B * c.G * ntc * ((c.T + kRowsPerUnit - 1) / kRowsPerUnit);
  w.cap[kBrWin] = (size_t)c.B * c.G * ntw * ((127 + c.w + kRowsPerUnit - 1) / kRowsPerUnit + 1);
  w.cap[kBrSlc] = lists + (size_t)c.B * c.T * c.G * c.n / kRowsPerUnit + 1;
  size_t o = header;
  w.lse = o;   o = align_up(o + 3 * rows * sizeof(float), 256);
  w.dgw = o;   o = align_up(o + 3 * rows * sizeof(float), 256);
  w.dkc = o;   o = align_up(o + (size_t)c.B * c.G * Nc * c.dk * sizeof(float), 256);
  w.dvc = o;   o = align_up(o + (size_t)c.B * c.G * Nc * c.dv * sizeof(float), 256);
  w.zero_begin = o;
  w.cnt = o;   o = align_up(o + lists * sizeof(int), 256);
  w.fill = o;  o = align_up(o + lists * sizeof(int), 256);
  w.csum = o;  o = align_up(o + (size_t)(c.dk + c.dv) * sizeof(float), 256);
  w.zero_end = o;
  w.offs = o;  o = align_up(o + lists * sizeof(int), 256);
  w.nunits = o; o = align_up(o + 4 * sizeof(int), 256);
  w.inv = o;   o = align_up(o + (size_t)c.B * c.T * c.G * c.n * sizeof(int), 256);
  for (int br = 0; br < 3; ++br) {
    w.units[br] = o;
    o = align_up(o + w.cap[br] * sizeof(int4), 256);
  }
  w.end = o;
  return w;
}

int launch_prefill_bwd(const nsa_cfg& c, const BwdPtrs& p, uint8_t* ws, const BwdWs& w, cudaStream_t s) {
  DeviceStatus* st = reinterpret_cast<DeviceStatus*>(ws);
  const int hpg = c.H / c.G;
  const int Nc = c.T < 32 ? 0 : (c.T - 32) / 16 + 1;
  const int nblk = (c.T + 63) / 64;
  const float scale = c.scale > 0.f ? c.scale : 1.0f / sqrtf((float)c.dk);
  const float sc2 = scale * 1.4426950408889634f;
  float* lse = reinterpret_cast<float*>(ws + w.lse);
  float* dgw = reinterpret_cast<float*>(ws + w.dgw);
  float* dkc = reinterpret_cast<float*>(ws + w.dkc);
  float* dvc = reinterpret_cast<float*>(ws + w.dvc);
  const size_t rows = (size_t)c.B * c.T * c.H;

  // zeroed outputs and counters
  if (cudaMemsetAsync(p.dk, 0, sizeof(float) * (size_t)c.B * c.T * c.G * c.dk, s) != cudaSuccess ||
      cudaMemsetAsync(p.dv, 0, sizeof(float) * (size_t)c.B * c.T * c.G * c.dv, s) != cudaSuccess ||
      cudaMemsetAsync(p.dw_k, 0, sizeof(float) * (size_t)32 * c.dk * c.dk, s) != cudaSuccess ||
      cudaMemsetAsync(p.dw_v, 0, sizeof(float) * (size_t)32 * c.dv * c.dv, s) != cudaSuccess ||
      cudaMemsetAsync(p.dpe_k, 0, sizeof(float) * (size_t)32 * c.dk, s) != cudaSuccess ||
      cudaMemsetAsync(p.dpe_v, 0, sizeof(float) * (size_t)32 * c.dv, s) != cudaSuccess ||
      cudaMemsetAsync(ws + w.dkc, 0, w.zero_begin - w.dkc, s) != cudaSuccess ||
      cudaMemsetAsync(ws + w.zero_begin, 0, w.zero_end - w.zero_begin, s) != cudaSuccess)
    return NSA_ERR_CUDA;

  CUtensorMap mq, mdo, mk, mv, mkc, mvc;
  if (!make_rows_map(&mq, p.q, c.B, c.T, c.H, c.dk, hpg) || !make_rows_map(&mdo, p.dout, c.B, c.T, c.H, c.dv, hpg) ||
      !make_kv_map(&mk, p.k, c.B, c.T, c.G, c.dk, 64, false) || !make_kv_map(&mv, p.v, c.B, c.T, c.G, c.dv, 64, false))
    return NSA_ERR_CUDA;
  // the compressed cache as a head-major [B,G,Nc,d] tensor (a 1-row stand-in when empty)
  const int ncr = Nc > 0 ? Nc : 1;
  if (!make_kv_map(&mkc, Nc > 0 ? p.kc : p.k, c.B, ncr, c.G, c.dk, 64, true) ||
      !make_kv_map(&mvc, Nc > 0 ? p.vc : p.v, c.B, ncr, c.G, c.dv, 64, true))
    return NSA_ERR_CUDA;

  // ---- 1. dq, dgates, per-branch statistics: the compressed and window
  // branches in query tiles, then the selected branch per (query, group)
  {
    const TileLayout L = tile_layout(c.dk, c.dv);
    TileArgs a;
    a.T = c.T;
    a.H = c.H;
    a.G = c.G;
    a.dk = c.dk;
    a.dv = c.dv;
    a.w = c.w;
    a.hpg = hpg;
    a.Nc = Nc;
    a.sc2 = sc2;
    a.scale = scale;
    a.gates = static_cast<const __nv_bfloat16*>(p.gates);
    a.dq = p.dq;
    a.dgates = p.dgates;
    a.lse = lse;
    a.dgw = dgw;
    a.st = st;
    a.off_do = L.off_do;
    a.off_k = L.off_k;
    a.off_v = L.off_v;
    a.off_x = L.off_x;
    a.off_bar = L.off_bar;
    if (int rc = ensure_smem_attr(reinterpret_cast<const void*>(&bwd_dq_tile_kernel), L.total)) return rc;
    dim3 grid((c.T + kTileQ - 1) / kTileQ, c.G, c.B);
    prof::begin("bwd_dq_tile", s);
    bwd_dq_tile_kernel<<<grid, kTileThreads, L.total, s>>>(mq, mdo, mk, mv, mkc, mvc, a);
    prof::end(s);
    if (cudaPeekAtLastError() != cudaSuccess) return NSA_ERR_CUDA;
  }
  {
    const DqLayout L = dq_layout(c.dk, c.dv);
    DqArgs a;
    a.br_lo = kBrSlc;
    a.br_hi = kBrSlc;
    a.acc_dq = 1;
    a.slc_lse = p.slc_lse;
    a.slc_o = p.slc_o;
    a.dout = static_cast<const __nv_bfloat16*>(p.dout);
    a.T = c.T;
    a.H = c.H;
    a.G = c.G;
    a.dk = c.dk;
    a.dv = c.dv;
    a.n = c.n;
    a.w = c.w;
    a.hpg = hpg;
    a.Nc = Nc;
    a.QPC = 16;
    a.sc2 = sc2;
    a.scale = scale;
    a.idx = p.idx;
    a.gates = static_cast<const __nv_bfloat16*>(p.gates);
    a.dq = p.dq;
    a.dgates = p.dgates;
    a.lse = lse;
    a.dgw = dgw;
    a.st = st;
    a.off_kv = L.off_kv;
    a.off_ds = L.off_ds;
    a.off_red = L.off_red;
    a.off_bar = L.off_bar;
    if (int rc = ensure_smem_attr(reinterpret_cast<const void*>(&bwd_dq_kernel), L.total)) return rc;
    dim3 grid((c.T + a.QPC - 1) / a.QPC, c.G, c.B);
    prof::begin("bwd_dq_slc", s);
    bwd_dq_kernel<<<grid, kDqThreads, L.total, s>>>(mq, mdo, mk, mv, mkc, mvc, a);
    prof::end(s);
    if (cudaPeekAtLastError() != cudaSuccess) return NSA_ERR_CUDA;
  }

  // ---- 2. selected-branch inverse lists, work units
  int* cnt = reinterpret_cast<int*>(ws + w.cnt);
  int* fill = reinterpret_cast<int*>(ws + w.fill);
  int* offs = reinterpret_cast<int*>(ws + w.offs);
  int* inv = reinterpret_cast<int*>(ws + w.inv);
  int* nunits = reinterpret_cast<int*>(ws + w.nunits);
  {
    const size_t entries = (size_t)c.B * c.T * c.G * c.n;
    const unsigned nb = (unsigned)((entries + 255) / 256);
    prof::begin("bwd_lists", s);
    slc_count_kernel<<<nb, 256, 0, s>>>(p.idx, c.B, c.T, c.G, c.n, nblk, cnt);
    UnitArgs ua;
    ua.B = c.B;
    ua.T = c.T;
    ua.G = c.G;
    ua.Nc = Nc;
    ua.w = c.w;
    ua.nblk = nblk;
    ua.ntc = (Nc + 127) / 128;
    ua.ntw = (c.T + 127) / 128;
    ua.cnt = cnt;
    ua.offs = offs;
    for (int br = 0; br < 3; ++br) {
      ua.units[br] = reinterpret_cast<int4*>(ws + w.units[br]);
      ua.cap[br] = (int)w.cap[br];
    }
    ua.nunits = nunits;
    build_units_kernel<<<1, 1024, 0, s>>>(ua);
    slc_fill_kernel<<<nb, 256, 0, s>>>(p.idx, c.B, c.T, c.G, c.n, nblk, offs, fill, inv);
    prof::end(s);
    if (cudaPeekAtLastError() != cudaSuccess) return NSA_ERR_CUDA;
  }

  // ---- 3. key-outer dK / dV per branch
  {
    const DkvLayout L = dkv_layout(c.dk, c.dv);
    int nsm = 148;
    {
      int dev = 0;
      if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    }
    for (int br = 0; br < 3; ++br) {
      if (br == kBrCmp && Nc == 0) continue;
      DkvArgs a;
      a.T = c.T;
      a.H = c.H;
      a.G = c.G;
      a.dk = c.dk;
      a.dv = c.dv;
      a.w = c.w;
      a.hpg = hpg;
      a.Nc = Nc;
      a.sc2 = sc2;
      a.scale = scale;
      a.gates = static_cast<const __nv_bfloat16*>(p.gates);
      a.lse = lse + (size_t)br * rows;
      a.dgw = dgw + (size_t)br * rows;
      a.inv = inv;
      a.units = reinterpret_cast<const int4*>(ws + w.units[br]);
      a.nunits = nunits + br;
      a.dK = br == kBrCmp ? dkc : p.dk;
      a.dV = br == kBrCmp ? dvc : p.dv;
      a.st = st;
      a.off_q = L.off_q;
      a.off_col = L.off_col;
      a.off_bar = L.off_bar;
      const unsigned grid = (unsigned)std::min<size_t>((size_t)nsm, std::max<size_t>(1, w.cap[br]));
      if (br == kBrCmp) {
        if (int rc = ensure_smem_attr(reinterpret_cast<const void*>(&bwd_dkv_kernel<kBrCmp>), L.total)) return rc;
        prof::begin("bwd_dkv_cmp", s);
        bwd_dkv_kernel<kBrCmp><<<grid, kDkvThreads, L.total, s>>>(mq, mdo, mkc, mvc, a);
      } else if (br == kBrSlc) {
        if (int rc = ensure_smem_attr(reinterpret_cast<const void*>(&bwd_dkv_kernel<kBrSlc>), L.total)) return rc;
        prof::begin("bwd_dkv_slc", s);
        bwd_dkv_kernel<kBrSlc><<<grid, kDkvThreads, L.total, s>>>(mq, mdo, mk, mv, a);
      } else {
        if (int rc = ensure_smem_attr(reinterpret_cast<const void*>(&bwd_dkv_kernel<kBrWin>), L.total)) return rc;
        prof::begin("bwd_dkv_win", s);
        bwd_dkv_kernel<kBrWin><<<grid, kDkvThreads, L.total, s>>>(mq, mdo, mk, mv, a);
      }
      prof::end(s);
      if (cudaPeekAtLastError() != cudaSuccess) return NSA_ERR_CUDA;
    }
  }

  // ---- 4. compression backward
  if (Nc > 0) {
    float* csum = reinterpret_cast<float*>(ws + w.csum);
    const size_t crow = (size_t)c.B * c.G * Nc;
    prof::begin("bwd_compress", s);
    for (int kvs = 0; kvs < 2; ++kvs) {
      const int D = kvs == 0 ? c.dk : c.dv;
      const float* dxc = kvs == 0 ? dkc : dvc;
      float* sv = csum + (kvs == 0 ? 0 : c.dk);
      const __nv_bfloat16* W = static_cast<const __nv_bfloat16*>(kvs == 0 ? c.w_k : c.w_v);
      const __nv_bfloat16* PE = static_cast<const __nv_bfloat16*>(kvs == 0 ? c.pe_k : c.pe_v);
      const __nv_bfloat16* X = static_cast<const __nv_bfloat16*>(kvs == 0 ? p.k : p.v);
      colsum_kernel<<<(unsigned)std::min<size_t>(crow, 1184), D, 0, s>>>(dxc, crow, D, sv);
      dpe_kernel<<<32, D, 0, s>>>(sv, W, D, kvs == 0 ? p.dpe_k : p.dpe_v);
      dim3 gx((unsigned)((c.T + 16 * 64 - 1) / (16 * 64)), (unsigned)(D / 64), (unsigned)(16 * c.B * c.G));
      dx_kernel<<<gx, 256, 0, s>>>(dxc, W, c.B, c.T, c.G, Nc, D, kvs == 0 ? p.dk : p.dv);
      dim3 gw((unsigned)(D / 64), (unsigned)(D / 64), (unsigned)(32 * ((crow + 255) / 256)));
      dw_kernel<<<gw, 256, 0, s>>>(X, PE, dxc, c.B, c.T, c.G, Nc, D, kvs == 0 ? p.dw_k : p.dw_v);
    }
    prof::end(s);
    if (cudaPeekAtLastError() != cudaSuccess) return NSA_ERR_CUDA;
  }
  return NSA_OK;
}

}  // namespace nsa
