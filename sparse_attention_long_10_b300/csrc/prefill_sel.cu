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
// kept keys is exact (one max, one sum), and the slc gate is folded into P.
// The epilogue adds the cmp+win partial sum from prefill_cmp_win.cu:
//     out = part + g_slc * O_slc          (bf16)
//
// Warp roles: warps 0-3 softmax + epilogue (thread = TMEM lane = one key of
// a pair, or one value dimension), warp 4 TMA producer, warp 5 MMA issuer.
#include "common.cuh"
#include "kernels.hpp"
#include "profiler.hpp"
#include "tmap.hpp"

namespace nsa {

namespace {

constexpr int kThreads = 192;
constexpr int NP = 16;           // MMA N: heads of the group, padded to 16
constexpr int kRingK = 6;        // 16 KB: one 64-column chunk of a block pair
constexpr int kRingV = 2;        // 32 KB: both 64-column chunks of a value pair
constexpr int kSlotK = 16384;
constexpr int kSlotV = 32768;
constexpr int kQBuf = 2048;      // one 64-column chunk of NP query rows

struct SelArgs {
  int T, H, G, dk, dv, n, hpg, QPC;
  float sc2;
  const int32_t* idx;              // [B,T,G,n]
  const __nv_bfloat16* gates;      // [B,T,H,3]
  const __nv_bfloat16* part;       // [B,T,H,dv]
  __nv_bfloat16* out;              // [B,T,H,dv]
  DeviceStatus* st;
  uint32_t off_kring, off_vring, off_pt, off_red, off_bar;
};

struct Bars {
  uint64_t q_full[2], q_empty[2];
  uint64_t k_full[kRingK], k_empty[kRingK];
  uint64_t v_full[kRingV], v_empty[kRingV];
  uint64_t s_full[2], s_free[2];
  uint64_t p_full, p_free;
  uint64_t o_full[2], o_free[2];
  uint64_t wg;
  uint64_t drain;
  uint32_t tmem;
  int abort_flag;
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// token coordinate of block ``blk`` for a TMA load; an absent block reads
// zeros from a negative coordinate
__device__ __forceinline__ int block_token(int blk) { return blk >= 0 ? blk * 64 : -128; }

__global__ void __launch_bounds__(kThreads, 1)
    sel_kernel(const __grid_constant__ CUtensorMap mapQ, const __grid_constant__ CUtensorMap mapK,
               const __grid_constant__ CUtensorMap mapV, const SelArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* qbuf = smem;                        // 2 items x kcs chunks x 2 KB
  uint8_t* kring = smem + a.off_kring;
  uint8_t* vring = smem + a.off_vring;
  uint8_t* pt = smem + a.off_pt;               // P^T: npairs*2 chunks x 2 KB
  float* red = reinterpret_cast<float*>(smem + a.off_red);   // [2][4][NP]
  Bars* bars = reinterpret_cast<Bars*>(smem + a.off_bar);
  volatile int* abort_flag = &bars->abort_flag;

  const int g = blockIdx.y;
  const int b = blockIdx.z;
  const int t0 = blockIdx.x * a.QPC;
  const int nitems = min(a.QPC, a.T - t0);
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
    mbar_init(&bars->p_full, 4);
    mbar_init(&bars->p_free, 1);
    mbar_init(&bars->wg, 4);
    mbar_init(&bars->drain, 1);
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
  const uint32_t tmem_o = tmem + 2 * SC;          // 2 x NP columns

  if (*abort_flag) {
    // an earlier CTA failed: do nothing
  } else if (warp == 4) {
    // =============================================================== producer
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
        const int32_t* blk = a.idx + (((size_t)b * a.T + t0 + i) * a.G + g) * a.n;
        for (int p = 0; p < npairs && ok; ++p) {
          const int tk0 = block_token(__ldg(blk + 2 * p));
          const int tk1 = block_token(2 * p + 1 < a.n ? __ldg(blk + 2 * p + 1) : -1);
          for (int c = 0; c < kcs; ++c) {
            const int slot = kv % kRingK;
            if (!mbar_wait(&bars->k_empty[slot], (uint32_t)(((kv / kRingK) & 1) ^ 1), abort_flag, a.st, 302)) {
              ok = false;
              return;
            }
            uint8_t* dst = kring + slot * kSlotK;
            mbar_arrive_expect_tx(&bars->k_full[slot], kSlotK);
            tma_load_4d(dst, &mapK, &bars->k_full[slot], c * 64, g, tk0, b);
            tma_load_4d(dst + 8192, &mapK, &bars->k_full[slot], c * 64, g, tk1, b);
            ++kv;
          }
        }
      };
      auto load_v = [&](int i) {
        const int32_t* blk = a.idx + (((size_t)b * a.T + t0 + i) * a.G + g) * a.n;
        for (int p = 0; p < npairs && ok; ++p) {
          const int tk0 = block_token(__ldg(blk + 2 * p));
          const int tk1 = block_token(2 * p + 1 < a.n ? __ldg(blk + 2 * p + 1) : -1);
          const int slot = vv % kRingV;
          if (!mbar_wait(&bars->v_empty[slot], (uint32_t)(((vv / kRingV) & 1) ^ 1), abort_flag, a.st, 303)) {
            ok = false;
            return;
          }
          uint8_t* dst = vring + slot * kSlotV;
          mbar_arrive_expect_tx(&bars->v_full[slot], (uint32_t)(vcs * 16384));
          for (int c = 0; c < vcs; ++c) {
            tma_load_4d(dst + c * 16384, &mapV, &bars->v_full[slot], c * 64, g, tk0, b);
            tma_load_4d(dst + c * 16384 + 8192, &mapV, &bars->v_full[slot], c * 64, g, tk1, b);
          }
          ++vv;
        }
      };
      load_q(0);
      load_k(0);
      for (int i = 0; i < nitems && ok; ++i) {
        if (i + 1 < nitems) {
          load_q(i + 1);
          load_k(i + 1);
        }
        load_v(i);
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
  } else if (warp == 5) {
    // =============================================================== MMA issuer
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
        const int ob = i & 1;
        if (!mbar_wait(&bars->o_free[ob], (uint32_t)(((i >> 1) & 1) ^ 1), abort_flag, a.st, 314) ||
            !mbar_wait(&bars->p_full, (uint32_t)(i & 1), abort_flag, a.st, 315)) {
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
            const uint64_t bd = sdesc_sw128(p_a + (p * 2 + (k >> 2)) * kQBuf + (k & 3) * 32, 16, 1024);
            umma_bf16(tmem_o + ob * NP, ad, bd, idesc_pv, (p > 0 || k > 0) ? 1u : 0u);
          }
          umma_commit(&bars->v_empty[slot]);
          ++vv;
        }
        umma_commit(&bars->p_free);
        umma_commit(&bars->o_full[ob]);
      };
      issue_qk(0);
      for (int i = 0; i < nitems; ++i) {
        if (i + 1 < nitems) issue_qk(i + 1);
        issue_pv(i);
      }
      if (!ok || *abort_flag) {
        // wait for every MMA issued so far before the CTA releases TMEM
        umma_commit(&bars->drain);
        mbar_wait_plain(&bars->drain, 0, kWaitLimitNs);
      }
    }
  } else {
    // =============================================================== softmax + epilogue
    const int r = threadIdx.x;          // key lane within a pair / value dim
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    bool ok = true;
    uint32_t wg_phase = 0;
    auto wg_sync = [&]() {
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->wg);
      if (!mbar_wait(&bars->wg, wg_phase & 1, abort_flag, a.st, 321)) ok = false;
      ++wg_phase;
    };
    float x[8][NP];    // [pair][head] (n <= 16 -> at most 8 pairs)

    auto softmax = [&](int i) {
      if (!ok) return;
      const int t = t0 + i;
      const int sb = i & 1;
      const uint32_t par = (uint32_t)((i >> 1) & 1);
      if (!mbar_wait(&bars->s_full[sb], par, abort_flag, a.st, 322)) {
        ok = false;
        return;
      }
      tc_fence_after();
      const int32_t* blk = a.idx + (((size_t)b * a.T + t) * a.G + g) * a.n;
#pragma unroll
      for (int p = 0; p < 8; ++p) {
        if (p < npairs) {
          uint32_t rr[16];
          tmem_ld16(tmem_s + lane_base + sb * SC + p * NP, rr);
          tmem_ld_wait(rr);
          const int bi = 2 * p + (r >> 6);
          const int bk = bi < a.n ? __ldg(blk + bi) : -1;
          const int s = bk * 64 + (r & 63);
          const bool valid = bk >= 0 && s <= t;
#pragma unroll
          for (int h = 0; h < NP; ++h) x[p][h] = valid ? __uint_as_float(rr[h]) * a.sc2 : -INFINITY;
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->s_free[sb]);
      // max over the kept keys, per head
      float mh[NP], lh[NP];
#pragma unroll
      for (int h = 0; h < NP; ++h) {
        float m = -INFINITY;
#pragma unroll
        for (int p = 0; p < 8; ++p)
          if (p < npairs) m = fmaxf(m, x[p][h]);
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        mh[h] = m;
      }
      float* rd = red + (wg_phase & 1) * 4 * NP;
      if (lane == 0)
#pragma unroll
        for (int h = 0; h < NP; ++h) rd[warp * NP + h] = mh[h];
      wg_sync();
#pragma unroll
      for (int h = 0; h < NP; ++h) mh[h] = fmaxf(fmaxf(rd[h], rd[NP + h]), fmaxf(rd[2 * NP + h], rd[3 * NP + h]));
      // sum
#pragma unroll
      for (int h = 0; h < NP; ++h) {
        float s = 0.f;
#pragma unroll
        for (int p = 0; p < 8; ++p)
          if (p < npairs) {
            x[p][h] = (mh[h] == -INFINITY) ? 0.f : fast_exp2(x[p][h] - mh[h]);
            s += x[p][h];
          }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        lh[h] = s;
      }
      rd = red + (wg_phase & 1) * 4 * NP;
      if (lane == 0)
#pragma unroll
        for (int h = 0; h < NP; ++h) rd[warp * NP + h] = lh[h];
      wg_sync();
      float coef[NP];
#pragma unroll
      for (int h = 0; h < NP; ++h) {
        const float l = rd[h] + rd[NP + h] + rd[2 * NP + h] + rd[3 * NP + h];
        float gs = 0.f;
        if (h < a.hpg) gs = __bfloat162float(a.gates[(((size_t)b * a.T + t) * a.H + g * a.hpg + h) * 3 + 1]);
        coef[h] = (l > 0.f) ? gs / l : 0.f;
      }
      // P^T (K-major: row = head, keys along K) for the PV MMA
      if (!mbar_wait(&bars->p_free, (uint32_t)((i & 1) ^ 1), abort_flag, a.st, 323)) {
        ok = false;
        return;
      }
      tc_fence_after();
      const int kk = r & 63;
#pragma unroll
      for (int p = 0; p < 8; ++p) {
        if (p < npairs) {
          uint8_t* chunk = pt + (p * 2 + (r >> 6)) * kQBuf;
#pragma unroll
          for (int h = 0; h < NP; ++h) {
            const __nv_bfloat16 v = __float2bfloat16_rn(x[p][h] * coef[h]);
            *reinterpret_cast<__nv_bfloat16*>(chunk + sw128_offset(h, kk >> 3) + (kk & 7) * 2) = v;
          }
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->p_full);
    };

    auto epilogue = [&](int i) {
      if (!ok) return;
      const int t = t0 + i;
      const int ob = i & 1;
      if (!mbar_wait(&bars->o_full[ob], (uint32_t)((i >> 1) & 1), abort_flag, a.st, 324)) {
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
      const int d = r;
      if (d < a.dv) {
        const size_t rowbase = ((size_t)b * a.T + t) * a.H + g * a.hpg;
#pragma unroll
        for (int h = 0; h < NP; ++h) {
          if (h < a.hpg) {
            const size_t o = (rowbase + h) * a.dv + d;
            a.out[o] = __float2bfloat16_rn(__bfloat162float(a.part[o]) + __uint_as_float(rr[h]));
          }
        }
      }
    };

    softmax(0);
    for (int i = 0; i < nitems; ++i) {
      if (i + 1 < nitems) softmax(i + 1);
      epilogue(i);
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
  const int npairs = (n + 1) / 2;
  L.off_kring = (uint32_t)align_up((size_t)2 * (dk / 64) * kQBuf, 1024);
  L.off_vring = L.off_kring + kRingK * kSlotK;
  L.off_pt = L.off_vring + kRingV * kSlotV;
  L.off_red = L.off_pt + (uint32_t)(npairs * 2 * kQBuf);
  L.off_bar = (uint32_t)align_up(L.off_red + 2 * 4 * NP * sizeof(float), 256);
  L.total = L.off_bar + (uint32_t)align_up(sizeof(Bars), 256) + 1024;
  return L;
}

}  // namespace

size_t sel_smem_bytes(const nsa_cfg& c) { return layout_for(c.dk, c.n).total; }

int launch_sel(const nsa_cfg& c, const void* q, const void* k, const void* v, const void* gates, const int32_t* idx,
               const void* part, void* out, DeviceStatus* st, cudaStream_t s) {
  const int hpg = c.H / c.G;
  if (hpg > NP || c.n > 16 || (c.dv != 64 && c.dv != 128)) return NSA_ERR_UNSUPPORTED;
  const Layout L = layout_for(c.dk, c.n);
  if (L.total > smem_max()) return NSA_ERR_UNSUPPORTED;
  const uint64_t e = 2;
  CUtensorMap mq, mk, mv;
  {  // q [B,T,H,dk]: box (64, hpg heads, 1 query)
    const uint64_t dims[4] = {(uint64_t)c.dk, (uint64_t)c.H, (uint64_t)c.T, (uint64_t)c.B};
    const uint64_t str[3] = {c.dk * e, (uint64_t)c.H * c.dk * e, (uint64_t)c.T * c.H * c.dk * e};
    const uint32_t box[4] = {64, (uint32_t)hpg, 1, 1};
    if (!make_tmap_bf16(&mq, q, 4, dims, str, box)) return NSA_ERR_CUDA;
  }
  {  // k [B,T,G,dk]: box (64, 1 group, 64 tokens = one selection block)
    const uint64_t dims[4] = {(uint64_t)c.dk, (uint64_t)c.G, (uint64_t)c.T, (uint64_t)c.B};
    const uint64_t str[3] = {c.dk * e, (uint64_t)c.G * c.dk * e, (uint64_t)c.T * c.G * c.dk * e};
    const uint32_t box[4] = {64, 1, 64, 1};
    if (!make_tmap_bf16(&mk, k, 4, dims, str, box)) return NSA_ERR_CUDA;
  }
  {
    const uint64_t dims[4] = {(uint64_t)c.dv, (uint64_t)c.G, (uint64_t)c.T, (uint64_t)c.B};
    const uint64_t str[3] = {c.dv * e, (uint64_t)c.G * c.dv * e, (uint64_t)c.T * c.G * c.dv * e};
    const uint32_t box[4] = {64, 1, 64, 1};
    if (!make_tmap_bf16(&mv, v, 4, dims, str, box)) return NSA_ERR_CUDA;
  }
  SelArgs a;
  a.T = c.T;
  a.H = c.H;
  a.G = c.G;
  a.dk = c.dk;
  a.dv = c.dv;
  a.n = c.n;
  a.hpg = hpg;
  a.QPC = 16;
  const float scale = c.scale > 0.f ? c.scale : 1.0f / sqrtf((float)c.dk);
  a.sc2 = scale * 1.4426950408889634f;
  a.idx = idx;
  a.gates = static_cast<const __nv_bfloat16*>(gates);
  a.part = static_cast<const __nv_bfloat16*>(part);
  a.out = static_cast<__nv_bfloat16*>(out);
  a.st = st;
  a.off_kring = L.off_kring;
  a.off_vring = L.off_vring;
  a.off_pt = L.off_pt;
  a.off_red = L.off_red;
  a.off_bar = L.off_bar;
  static bool attr = false;
  if (!attr) {
    if (cudaFuncSetAttribute(sel_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_max()) != cudaSuccess)
      return NSA_ERR_CUDA;
    attr = true;
  }
  dim3 grid((c.T + a.QPC - 1) / a.QPC, c.G, c.B);
  prof::begin("sel", s);
  sel_kernel<<<grid, kThreads, L.total, s>>>(mq, mk, mv, a);
  prof::end(s);
  return cudaPeekAtLastError() == cudaSuccess ? NSA_OK : NSA_ERR_CUDA;
}

}  // namespace nsa
