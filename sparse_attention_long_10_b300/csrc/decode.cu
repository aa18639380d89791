// decode.cu -- NSA single-token decode step [P2 section II (three paths,
// n=16 blocks incl. block 0 and the 2 local blocks, w=512) and III.3 (a 64k
// decode step reads 5,632 tokens' worth of KV instead of 65,536); P3
// token-compression, token-selection and sliding-window paragraphs].
//
// The query sits at t = T-1 (the caches already hold the new token), so every
// compressed entry and every cached token is causal.  Per (sequence b, KV
// group g) the step reads the Nc compressed entries, the n kept selection
// blocks and the w-token window once, for all hpg <= 16 query heads of the
// group at the same time (group-centric loading).
//
// Two launches, split-KV:
//   dec_kernel<MODE 0>  grid (cmp splits + 1, B*G)
//       split x < splits: compressed attention over 8 tiles of 64 entries;
//       split x = splits: window attention over (T-w, T-1].
//       Each CTA leaves a partial (running max m, sum l, unnormalised O) per
//       head, and the cmp splits also leave the per-quarter (16 entries)
//       block-score partials u/c with their reference max.  The last CTA of
//       a group (atomic counter, no waiting) merges the cmp partials into the
//       exact softmax, normalises O_cmp, forms the block importance
//           S[j] = sum_h sum_i w(i,j) p[h,i]
//       (w = 16-token chunks shared by compressed entry i and block j) and
//       picks blocks 0, j_t, j_t-1 plus the top n-3 others, ties to the lower
//       index.
//   dec_kernel<MODE 1>  grid (ceil(n/4), B*G)
//       each CTA attends over 4 kept blocks; the last CTA of the group merges
//       them, adds the window and compressed outputs with the gates and
//       writes out = g_cmp*O_cmp + g_slc*O_slc + g_win*O_win (bf16).
//
// Data movement: 64-row x 64-column 128B-swizzled TMA boxes (one 16-byte
// aligned row of 128 B per key), a 2-stage ring per CTA, two CTAs per SM.
// Math: one warp takes 16 keys of each 64-key tile; QK^T and PV are
// mma.sync m16n8k16 with the 16 heads as the M side (fp32 accumulation),
// online softmax in registers.
#include "common.cuh"
#include "kernels.hpp"
#include "profiler.hpp"
#include "tmap.hpp"
#include "warp_mma.cuh"

namespace nsa {

namespace {

constexpr int kThreads = 160;        // warps 0-3 compute, warp 4 TMA producer
constexpr int kStages = 2;
constexpr int kBox = 8192;           // 64 rows x 128 bytes
constexpr int kTilesPerSplit = 8;    // 64-entry tiles per compressed split
constexpr int kBlocksPerSelCta = 4;  // kept blocks per selection CTA

struct DecArgs {
  int B, T, H, G, BG, hpg, n, w;
  int Nc, nq, ntc;                   // compressed entries, 16-entry quarters, 64-entry tiles
  int splits, tps, sel_splits, bps, NS;
  float sc2;                         // softmax scale * log2(e)
  const __nv_bfloat16* q;            // [B,H,dk]
  const __nv_bfloat16* gates;        // [B,H,3]
  __nv_bfloat16* out;                // [B,H,dv]
  int32_t* idx_out;                  // nullable [B,G,n]
  float* pm;                         // [BG][NS][16]
  float* pl;                         // [BG][NS][16]
  float* po;                         // [BG][NS][16][dv]
  float* u;                          // [BG][4*nq][16]
  float* cc;                         // [BG][nq+1][16]
  float* mref;                       // [BG][nq][16]
  float* stats;                      // [BG][32]: compressed-branch max (log2 units) and 1/sum per head
  int32_t* idx;                      // [BG][n]
  int* cnt;                          // [2][BG]
  DeviceStatus* st;
};

struct DecBars {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  int abort_flag;
  int last;
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

__device__ __forceinline__ float ldcg_f(const float* p) { return __ldcg(p); }

// Block-score partials of one head for the warp's 16 entries (quarter qd):
// group k (entries 4k..4k+3) feeds block 4qd+k with 2*sum - last + prev_last,
// and its last entry's second chunk feeds block 4qd+4 (the carry c).  All 16
// head slots are written (heads past hpg see a zero query and stay finite);
// the selection step weights them by zero.
__device__ __forceinline__ void block_partials(const float (&p)[2][4], int eo, int head, int qd, float mref_val,
                                               int tq, int bg, const DecArgs& a) {
  float last[2], gs[2];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    const float pair = p[nt][eo] + p[nt][eo + 1];
    gs[nt] = pair + __shfl_xor_sync(0xffffffffu, pair, 1);
    const float y = __shfl_xor_sync(0xffffffffu, p[nt][eo + 1], 1);
    last[nt] = (tq & 1) ? p[nt][eo + 1] : y;
  }
  const float sx0 = __shfl_xor_sync(0xffffffffu, last[0], 2);
  const float sx1 = __shfl_xor_sync(0xffffffffu, last[1], 2);
  const bool hi = (tq >> 1) != 0;
  const float prev0 = hi ? sx0 : 0.f;
  const float prev1 = hi ? sx1 : sx0;
  const float u0 = 2.f * gs[0] - last[0] + prev0;
  const float u1 = 2.f * gs[1] - last[1] + prev1;
  float* ub = a.u + ((size_t)bg * (4 * a.nq) + 4 * qd) * 16 + head;
  if ((tq & 1) == 0) {
    ub[(tq >> 1) * 16] = u0;
    ub[(2 + (tq >> 1)) * 16] = u1;
  }
  if (tq == 2) a.cc[((size_t)bg * (a.nq + 1) + qd + 1) * 16 + head] = last[1];
  if (tq == 0) a.mref[((size_t)bg * a.nq + qd) * 16 + head] = mref_val;
}

__device__ __forceinline__ float dot16(const float* f, const float4* v) {
  const float4 a = v[0], b = v[1], c = v[2], d = v[3];
  return f[0] * a.x + f[1] * a.y + f[2] * a.z + f[3] * a.w + f[4] * b.x + f[5] * b.y + f[6] * b.z + f[7] * b.w +
         f[8] * c.x + f[9] * c.y + f[10] * c.z + f[11] * c.w + f[12] * d.x + f[13] * d.y + f[14] * d.z +
         f[15] * d.w;
}

__device__ __forceinline__ float4 ldcg4(const float* p) { return __ldcg(reinterpret_cast<const float4*>(p)); }

// Selection step, run by the last CTA of a group after every compressed and
// window split has left its partial: exact softmax statistics of the
// compressed branch (kept in ``stats`` for the final combine), block
// importance S[j] for every causal block, top-n.
__device__ void select_step(const DecArgs& a, int bg, uint8_t* smem) {
  const int tid = threadIdx.x;
  const int warp = warp_id(), lane = lane_id();
  const int NSc = a.splits;
  float* Mh = reinterpret_cast<float*>(smem);      // 16
  float* iL = Mh + 16;                              // 16
  float* wv = iL + 16;                              // [4][32] winner scores
  int* wj = reinterpret_cast<int*>(wv + 128);       // [4][32] winner blocks
  float* sp = reinterpret_cast<float*>(wj + 128);   // [NSc][2][16] partial m, l
  float* fsm = sp + 32 * NSc;                       // [nq][16]
  float* Ssm = fsm + (size_t)a.nq * 16;             // [jt+1]
  for (int e = tid; e < NSc * 16; e += kThreads) {
    const size_t o = ((size_t)bg * a.NS + e / 16) * 16 + (e & 15);
    sp[(e / 16) * 32 + (e & 15)] = ldcg_f(a.pm + o);
    sp[(e / 16) * 32 + 16 + (e & 15)] = ldcg_f(a.pl + o);
  }
  __syncthreads();
  if (tid < 16) {
    float M = -INFINITY;
    for (int s = 0; s < NSc; ++s) M = fmaxf(M, sp[s * 32 + tid]);
    const float Mu = (M == -INFINITY) ? 0.f : M;
    float L = 0.f;
    for (int s = 0; s < NSc; ++s) L += sp[s * 32 + 16 + tid] * fast_exp2(sp[s * 32 + tid] - Mu);
    const float il = (L > 0.f && tid < a.hpg) ? 1.f / L : 0.f;
    Mh[tid] = Mu;
    iL[tid] = il;
    a.stats[(size_t)bg * 32 + tid] = Mu;
    a.stats[(size_t)bg * 32 + 16 + tid] = il;
  }
  const int jt = (a.T - 1) / 64;
  const int n = a.n;
  int32_t* idx = a.idx + (size_t)bg * n;
  int32_t* idx_out = a.idx_out != nullptr ? a.idx_out + (size_t)bg * n : nullptr;
  if (jt + 1 <= n) {
    if (tid < n) {
      const int v = tid <= jt ? tid : -1;
      idx[tid] = v;
      if (idx_out) idx_out[tid] = v;
    }
    return;
  }
  __syncthreads();
  // per-quarter normalisation factors exp(mref - M) / L
  {
    const float* mr = a.mref + (size_t)bg * a.nq * 16;
    for (int e4 = tid; e4 < a.nq * 4; e4 += kThreads) {
      const float4 m4 = ldcg4(mr + 4 * e4);
      const int h = (4 * e4) & 15;
      float4 f;
      f.x = fast_exp2(m4.x - Mh[h + 0]) * iL[h + 0];
      f.y = fast_exp2(m4.y - Mh[h + 1]) * iL[h + 1];
      f.z = fast_exp2(m4.z - Mh[h + 2]) * iL[h + 2];
      f.w = fast_exp2(m4.w - Mh[h + 3]) * iL[h + 3];
      reinterpret_cast<float4*>(fsm)[e4] = f;
    }
  }
  __syncthreads();
  // block importance S[j], j <= jt
  {
    const float* ub = a.u + (size_t)bg * (4 * a.nq) * 16;
    const float* cb = a.cc + (size_t)bg * (a.nq + 1) * 16;
    for (int j = tid; j <= jt; j += kThreads) {
      const int qq = j >> 2;
      float s = 0.f;
      if (qq < a.nq) {
        float4 v[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) v[k] = ldcg4(ub + (size_t)j * 16 + 4 * k);
        s = dot16(fsm + qq * 16, v);
      }
      if ((j & 3) == 0 && qq >= 1 && qq <= a.nq) {
        float4 v[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) v[k] = ldcg4(cb + (size_t)qq * 16 + 4 * k);
        s += dot16(fsm + (qq - 1) * 16, v);
      }
      Ssm[j] = s;
    }
  }
  __syncthreads();
  // top-(n-3) among the free blocks 1 .. jt-2: each of 4 warps finds the best
  // of its quarter of the range, warp 0 merges.  Order: higher score, then
  // lower block index.  Scores are >= 0; -2 marks a taken block.
  const int kfree = n - 3;
  const int ncand = jt - 2;
  if (warp < 4) {
    const int per = (ncand + 3) / 4;
    const int lo = 1 + warp * per;
    const int hi = min(1 + ncand, lo + per);
    for (int rnd = 0; rnd < kfree; ++rnd) {
      float best = -1.f;
      int bj = 0x7fffffff;
      for (int j = lo + lane; j < hi; j += 32) {
        const float v = Ssm[j];
        if (v > best) {
          best = v;
          bj = j;
        }
      }
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, best, o);
        const int oj = __shfl_xor_sync(0xffffffffu, bj, o);
        if (ov > best || (ov == best && oj < bj)) {
          best = ov;
          bj = oj;
        }
      }
      if (lane == 0) {
        wv[warp * 32 + rnd] = best;
        wj[warp * 32 + rnd] = bj;
        if (bj != 0x7fffffff) Ssm[bj] = -2.f;
      }
      __syncwarp();
    }
  }
  __syncthreads();
  if (warp == 0) {
    // lane holds candidates c = lane + 32k of the 4*kfree winners
    float cv[4];
    int cj[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int c = lane + 32 * k;
      if (c < 4 * kfree) {
        cv[k] = wv[(c / kfree) * 32 + c % kfree];
        cj[k] = wj[(c / kfree) * 32 + c % kfree];
      } else {
        cv[k] = -1.f;
        cj[k] = 0x7fffffff;
      }
    }
    int mine = -1;
    for (int rnd = 0; rnd < kfree; ++rnd) {
      float best = -1.f;
      int bj = 0x7fffffff;
#pragma unroll
      for (int k = 0; k < 4; ++k)
        if (cv[k] > best || (cv[k] == best && cj[k] < bj)) {
          best = cv[k];
          bj = cj[k];
        }
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, best, o);
        const int oj = __shfl_xor_sync(0xffffffffu, bj, o);
        if (ov > best || (ov == best && oj < bj)) {
          best = ov;
          bj = oj;
        }
      }
#pragma unroll
      for (int k = 0; k < 4; ++k)
        if (cj[k] == bj) cv[k] = -2.f;
      if (lane == rnd) mine = bj;
    }
    if (lane == kfree) mine = 0;
    if (lane == kfree + 1) mine = jt - 1;
    if (lane == kfree + 2) mine = jt;
    int rank = 0;
    for (int k = 0; k < n; ++k) {
      const int o = __shfl_sync(0xffffffffu, mine, k);
      rank += (o < mine) ? 1 : 0;
    }
    if (lane < n) {
      idx[rank] = mine;
      if (idx_out) idx_out[rank] = mine;
    }
  }
}

// Final combine, run by the last selection CTA of a group:
//   out = g_cmp * O_cmp + g_slc * O_slc + g_win * O_win
// with each branch's partials weighted by exp(m_split - M) / L.
template <int DV>
__device__ void combine_step(const DecArgs& a, int bg, uint8_t* smem) {
  const int tid = threadIdx.x;
  const int b = bg / a.G, g = bg % a.G;
  const int NS = a.NS;
  const int win = a.splits, s0 = a.splits + 1;
  float* sp = reinterpret_cast<float*>(smem);    // [NS][2][16] partial m, l
  float* fac = sp + 32 * NS;                     // [NS][16] weight of each partial
  float* gt = fac + 16 * NS;                     // [16][3]
  for (int e = tid; e < NS * 16; e += kThreads) {
    const size_t o = ((size_t)bg * NS + e / 16) * 16 + (e & 15);
    sp[(e / 16) * 32 + (e & 15)] = ldcg_f(a.pm + o);
    sp[(e / 16) * 32 + 16 + (e & 15)] = ldcg_f(a.pl + o);
  }
  if (tid < 16 && tid < a.hpg) {
    const __nv_bfloat16* gp = a.gates + ((size_t)b * a.H + g * a.hpg + tid) * 3;
    gt[tid * 3 + 0] = __bfloat162float(gp[0]);
    gt[tid * 3 + 1] = __bfloat162float(gp[1]);
    gt[tid * 3 + 2] = __bfloat162float(gp[2]);
  }
  __syncthreads();
  if (tid < 16) {
    const int h = tid;
    // compressed: statistics from the selection step, folded with g_cmp
    const float Mc = ldcg_f(a.stats + (size_t)bg * 32 + h);
    const float iLc = ldcg_f(a.stats + (size_t)bg * 32 + 16 + h);
    const float gc = h < a.hpg ? gt[h * 3 + 0] : 0.f;
    const float gs = h < a.hpg ? gt[h * 3 + 1] : 0.f;
    const float gw = h < a.hpg ? gt[h * 3 + 2] : 0.f;
    for (int s = 0; s < a.splits; ++s) fac[s * 16 + h] = gc * fast_exp2(sp[s * 32 + h] - Mc) * iLc;
    const float lw = sp[win * 32 + 16 + h];
    fac[win * 16 + h] = lw > 0.f ? gw / lw : 0.f;
    float M = -INFINITY;
    for (int s = s0; s < NS; ++s) M = fmaxf(M, sp[s * 32 + h]);
    const float Mu = (M == -INFINITY) ? 0.f : M;
    float L = 0.f;
    for (int s = s0; s < NS; ++s) L += sp[s * 32 + 16 + h] * fast_exp2(sp[s * 32 + h] - Mu);
    const float il = L > 0.f ? gs / L : 0.f;
    for (int s = s0; s < NS; ++s) fac[s * 16 + h] = fast_exp2(sp[s * 32 + h] - Mu) * il;
  }
  __syncthreads();
  const float* po = a.po + (size_t)bg * NS * 16 * DV;
  for (int e4 = tid; e4 < a.hpg * DV / 4; e4 += kThreads) {
    const int h = (4 * e4) / DV;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    int s = 0;
    for (; s + 4 <= NS; s += 4) {
      float4 v[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) v[k] = ldcg4(po + ((size_t)(s + k) * 16) * DV + 4 * e4);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float f = fac[(s + k) * 16 + h];
        acc.x += f * v[k].x;
        acc.y += f * v[k].y;
        acc.z += f * v[k].z;
        acc.w += f * v[k].w;
      }
    }
    for (; s < NS; ++s) {
      const float4 v = ldcg4(po + ((size_t)s * 16) * DV + 4 * e4);
      const float f = fac[s * 16 + h];
      acc.x += f * v.x;
      acc.y += f * v.y;
      acc.z += f * v.z;
      acc.w += f * v.w;
    }
    uint2 pk;
    pk.x = pack_bf16x2(acc.x, acc.y);
    pk.y = pack_bf16x2(acc.z, acc.w);
    *reinterpret_cast<uint2*>(a.out + ((size_t)b * a.H + g * a.hpg) * DV + 4 * e4) = pk;
  }
}

template <int DK, int DV, int MODE>
__global__ void __launch_bounds__(kThreads, 2)
    dec_kernel(const __grid_constant__ CUtensorMap mK0, const __grid_constant__ CUtensorMap mV0,
               const __grid_constant__ CUtensorMap mK1, const __grid_constant__ CUtensorMap mV1,
               const DecArgs a, uint32_t off_bars) {
  constexpr int KB = DK / 64, VB = DV / 64;
  constexpr int kStageBytes = (KB + VB) * kBox;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  DecBars* bars = reinterpret_cast<DecBars*>(smem + off_bars);
  volatile int* abort_flag = &bars->abort_flag;
  const int x = blockIdx.x, bg = blockIdx.y;
  const int b = bg / a.G, g = bg % a.G;
  const int warp = warp_id(), lane = lane_id();

  // this CTA's tiles: kind 0 compressed entries, 1 window tokens, 2 kept blocks
  int kind, first, ntiles;
  if (MODE == 0) {
    if (x < a.splits) {
      kind = 0;
      first = x * a.tps;
      ntiles = min(a.tps, a.ntc - first);
    } else {
      kind = 1;
      first = max(0, a.T - a.w);
      ntiles = (a.T - first + 63) / 64;
    }
  } else {
    kind = 2;
    first = x * a.bps;
    ntiles = min(a.bps, a.n - first);
  }
  const CUtensorMap* mapK = (kind == 1) ? &mK1 : &mK0;
  const CUtensorMap* mapV = (kind == 1) ? &mV1 : &mV0;
  const int limit = (kind == 0) ? a.Nc : a.T;
  auto tile_row = [&](int i) -> int {  // first map row of tile i, -1 = absent
    if (kind == 0) return 64 * (first + i);
    if (kind == 1) return first + 64 * i;
    const int blk = a.idx[(size_t)bg * a.n + first + i];
    return blk >= 0 ? 64 * blk : -1;
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 4);
    }
    bars->abort_flag = prior_error(a.st);
    bars->last = 0;
    fence_barrier_init();
  }
  __syncthreads();

  const int gq = lane >> 2, tq = lane & 3;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  float o[DV / 8][4];
#pragma unroll
  for (int i = 0; i < DV / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  bool ok = *abort_flag == 0;

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && ok) {
      tma_prefetch_desc(mapK);
      tma_prefetch_desc(mapV);
      int v = 0;
      for (int i = 0; i < ntiles && ok; ++i) {
        const int row = tile_row(i);
        if (row < 0) continue;
        const int slot = v % kStages;
        if (!mbar_wait(&bars->empty[slot], (uint32_t)(((v / kStages) & 1) ^ 1), abort_flag, a.st, 401)) {
          ok = false;
          break;
        }
        uint8_t* dst = smem + slot * kStageBytes;
        mbar_arrive_expect_tx(&bars->full[slot], kStageBytes);
#pragma unroll
        for (int c = 0; c < KB; ++c) tma_load_3d(dst + c * kBox, mapK, &bars->full[slot], c * 64, row, bg);
#pragma unroll
        for (int c = 0; c < VB; ++c) tma_load_3d(dst + (KB + c) * kBox, mapV, &bars->full[slot], c * 64, row, bg);
        ++v;
      }
      if (!ok || *abort_flag) {
        for (int y = (v > kStages ? v - kStages : 0); y < v; ++y)
          mbar_wait_plain(&bars->full[y % kStages], (uint32_t)((y / kStages) & 1), kWaitLimitNs);
      }
    }
  } else if (ok) {
    // ------------------------------------------------------------ compute warps
    uint32_t qa[DK / 16][4];
    {
      const __nv_bfloat16* qb = a.q + ((size_t)b * a.H + (size_t)g * a.hpg) * DK;
#pragma unroll
      for (int ks = 0; ks < DK / 16; ++ks) {
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          const int row = gq + 8 * hf;
          uint32_t lo = 0, hi = 0;
          if (row < a.hpg) {
            lo = *reinterpret_cast<const uint32_t*>(qb + (size_t)row * DK + 16 * ks + 2 * tq);
            hi = *reinterpret_cast<const uint32_t*>(qb + (size_t)row * DK + 16 * ks + 8 + 2 * tq);
          }
          qa[ks][hf] = lo;
          qa[ks][2 + hf] = hi;
        }
      }
    }
    const int r0 = warp * 16;
    int v = 0;
    for (int i = 0; i < ntiles; ++i) {
      const int row = tile_row(i);
      if (row < 0) continue;
      const int slot = v % kStages;
      if (!mbar_wait(&bars->full[slot], (uint32_t)((v / kStages) & 1), abort_flag, a.st, 402)) {
        ok = false;
        break;
      }
      const uint32_t kbase = smem_u32(smem + slot * kStageBytes);
      const uint32_t vbase = kbase + KB * kBox;
      float s[2][4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
      for (int ks = 0; ks < DK / 16; ++ks) {
        const int rr = r0 + (lane & 7) + ((lane >> 4) << 3);
        const int unit = (ks & 3) * 2 + ((lane >> 3) & 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(sw128_addr(kbase + (ks >> 2) * kBox, rr, unit), b0, b1, b2, b3);
        mma_16816(s[0], qa[ks], b0, b1);
        mma_16816(s[1], qa[ks], b2, b3);
      }
      // mask + online softmax (rows gq and gq+8 = two heads)
      float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const bool valid = row + r0 + 8 * nt + 2 * tq + e < limit;
          s[nt][e] = valid ? s[nt][e] * a.sc2 : -INFINITY;
          s[nt][2 + e] = valid ? s[nt][2 + e] * a.sc2 : -INFINITY;
          mx0 = fmaxf(mx0, s[nt][e]);
          mx1 = fmaxf(mx1, s[nt][2 + e]);
        }
      mx0 = quad_max(mx0);
      mx1 = quad_max(mx1);
      const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
      const float us0 = (mn0 == -INFINITY) ? 0.f : mn0;
      const float us1 = (mn1 == -INFINITY) ? 0.f : mn1;
      const float al0 = fast_exp2(m0 - us0), al1 = fast_exp2(m1 - us1);
      float p[2][4];
      float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          p[nt][e] = fast_exp2(s[nt][e] - us0);
          p[nt][2 + e] = fast_exp2(s[nt][2 + e] - us1);
          rs0 += p[nt][e];
          rs1 += p[nt][2 + e];
        }
      l0 = l0 * al0 + rs0;
      l1 = l1 * al1 + rs1;
      m0 = mn0;
      m1 = mn1;
#pragma unroll
      for (int k = 0; k < DV / 8; ++k) {
        o[k][0] *= al0;
        o[k][1] *= al0;
        o[k][2] *= al1;
        o[k][3] *= al1;
      }
      if (MODE == 0 && kind == 0) {
        const int qd = 4 * (first + i) + warp;
        if (qd < a.nq) {
          block_partials(p, 0, gq, qd, mn0, tq, bg, a);
          block_partials(p, 2, gq + 8, qd, mn1, tq, bg, a);
        }
      }
      uint32_t pa[4];
      pa[0] = pack_bf16x2(p[0][0], p[0][1]);
      pa[1] = pack_bf16x2(p[0][2], p[0][3]);
      pa[2] = pack_bf16x2(p[1][0], p[1][1]);
      pa[3] = pack_bf16x2(p[1][2], p[1][3]);
#pragma unroll
      for (int np = 0; np < DV / 16; ++np) {
        const int rr = r0 + (lane & 7) + (((lane >> 3) & 1) << 3);
        const int unit = (np & 3) * 2 + (lane >> 4);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(sw128_addr(vbase + (np >> 2) * kBox, rr, unit), b0, b1, b2, b3);
        mma_16816(o[2 * np], pa, b0, b1);
        mma_16816(o[2 * np + 1], pa, b2, b3);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->empty[slot]);
      ++v;
    }
    l0 = quad_sum(l0);
    l1 = quad_sum(l1);
  }

  // ---------------------------------------------------------------- merge the 4 warps
  __syncthreads();
  if (*abort_flag) return;
  float* mw = reinterpret_cast<float*>(smem);   // [4][16]
  float* lw = mw + 64;                          // [4][16]
  float* fw = lw + 64;                          // [4][16]
  float* ow = fw + 64;                          // [4][16][DV]
  if (warp < 4) {
    if (tq == 0) {
      mw[warp * 16 + gq] = m0;
      mw[warp * 16 + gq + 8] = m1;
      lw[warp * 16 + gq] = l0;
      lw[warp * 16 + gq + 8] = l1;
    }
#pragma unroll
    for (int k = 0; k < DV / 8; ++k) {
      float* r = ow + (size_t)(warp * 16 + gq) * DV + 8 * k + 2 * tq;
      r[0] = o[k][0];
      r[1] = o[k][1];
      r[8 * DV] = o[k][2];
      r[8 * DV + 1] = o[k][3];
    }
  }
  __syncthreads();
  const int slot_id = (MODE == 0) ? x : (a.splits + 1 + x);
  const size_t pbase = (size_t)bg * a.NS + slot_id;
  if (threadIdx.x < 16) {
    const int h = threadIdx.x;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < 4; ++w) M = fmaxf(M, mw[w * 16 + h]);
    const float Mu = (M == -INFINITY) ? 0.f : M;
    float L = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const float f = fast_exp2(mw[w * 16 + h] - Mu);
      fw[w * 16 + h] = f;
      L += lw[w * 16 + h] * f;
    }
    a.pm[pbase * 16 + h] = M;
    a.pl[pbase * 16 + h] = L;
  }
  __syncthreads();
  for (int e = threadIdx.x; e < 16 * DV; e += kThreads) {
    const int h = e / DV;
    float acc = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) acc += fw[w * 16 + h] * ow[(size_t)w * 16 * DV + e];
    a.po[pbase * 16 * DV + e] = acc;
  }

  // ---------------------------------------------------------------- last CTA of the group
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const int old = atomicAdd(&a.cnt[MODE * a.BG + bg], 1);
    bars->last = (old == (int)gridDim.x - 1) ? 1 : 0;
  }
  __syncthreads();
  if (!bars->last) return;
  __threadfence();
  if (MODE == 0)
    select_step(a, bg, smem);
  else
    combine_step<DV>(a, bg, smem);
}

// ------------------------------------------------------------------ host side
struct DecWs {
  size_t cnt, pm, pl, po, u, cc, mref, stats, idx, end;
};

struct DecShape {
  int Nc, nq, ntc, splits, sel_splits, NS, BG;
};

DecShape dec_shape(const nsa_cfg& c) {
  DecShape s;
  s.Nc = c.T < c.l ? 0 : (c.T - c.l) / c.d + 1;
  s.nq = (s.Nc + 15) / 16;
  s.ntc = (s.Nc + 63) / 64;
  s.splits = (s.ntc + kTilesPerSplit - 1) / kTilesPerSplit;
  s.sel_splits = (c.n + kBlocksPerSelCta - 1) / kBlocksPerSelCta;
  s.NS = s.splits + 1 + s.sel_splits;
  s.BG = c.B * c.G;
  return s;
}

DecWs dec_ws(const nsa_cfg& c) {
  const DecShape s = dec_shape(c);
  const size_t BG = (size_t)s.BG;
  DecWs w;
  w.cnt = sizeof(DeviceStatus);
  w.pm = align_up(w.cnt + sizeof(int) * 2 * BG, 256);
  w.pl = align_up(w.pm + sizeof(float) * BG * s.NS * 16, 256);
  w.po = align_up(w.pl + sizeof(float) * BG * s.NS * 16, 256);
  w.u = align_up(w.po + sizeof(float) * BG * s.NS * 16 * c.dv, 256);
  w.cc = align_up(w.u + sizeof(float) * BG * 16 * 4 * (size_t)s.nq, 256);
  w.mref = align_up(w.cc + sizeof(float) * BG * 16 * (size_t)(s.nq + 1), 256);
  w.stats = align_up(w.mref + sizeof(float) * BG * (size_t)s.nq * 16, 256);
  w.idx = align_up(w.stats + sizeof(float) * BG * 32, 256);
  w.end = align_up(w.idx + sizeof(int32_t) * BG * c.n, 256);
  return w;
}

struct DecSmem {
  uint32_t off_bars, total;
};

DecSmem dec_smem(const nsa_cfg& c) {
  const DecShape s = dec_shape(c);
  const size_t ring = (size_t)kStages * (c.dk / 64 + c.dv / 64) * kBox;
  const size_t merge = sizeof(float) * (3 * 64 + 4 * 16 * (size_t)c.dv);
  const size_t jt1 = (size_t)(c.T - 1) / 64 + 1;
  const size_t select = sizeof(float) * (32 + 256 + 32 * (size_t)s.splits + 16 * (size_t)s.nq + jt1);
  const size_t combine = sizeof(float) * (48 * (size_t)s.NS + 48);
  size_t body = ring;
  if (merge > body) body = merge;
  if (select > body) body = select;
  if (combine > body) body = combine;
  DecSmem m;
  m.off_bars = (uint32_t)align_up(body, 256);
  m.total = m.off_bars + (uint32_t)align_up(sizeof(DecBars), 256) + 1024;
  return m;
}

template <int DK, int DV, int MODE>
int launch_one(const DecArgs& a, dim3 grid, const CUtensorMap* maps, uint32_t off_bars, uint32_t smem,
               cudaStream_t s, const char* name) {
  static bool attr = false;
  if (!attr) {
    if (cudaFuncSetAttribute(dec_kernel<DK, DV, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem_max()) != cudaSuccess)
      return NSA_ERR_CUDA;
    attr = true;
  }
  prof::begin(name, s);
  dec_kernel<DK, DV, MODE><<<grid, kThreads, smem, s>>>(maps[0], maps[1], maps[2], maps[3], a, off_bars);
  prof::end(s);
  return cudaPeekAtLastError() == cudaSuccess ? NSA_OK : NSA_ERR_CUDA;
}

template <int DK, int DV>
int launch_dims(const DecArgs& a, const DecShape& sh, const CUtensorMap* maps_cmp, const CUtensorMap* maps_sel,
                const DecSmem& m, cudaStream_t s) {
  int rc = launch_one<DK, DV, 0>(a, dim3(sh.splits + 1, sh.BG), maps_cmp, m.off_bars, m.total, s, "dec_cmp_win");
  if (rc != NSA_OK) return rc;
  return launch_one<DK, DV, 1>(a, dim3(sh.sel_splits, sh.BG), maps_sel, m.off_bars, m.total, s, "dec_sel");
}

}  // namespace

int decode_supported(const nsa_cfg& c) {
  const int hpg = c.H / c.G;
  if (hpg > 16) return NSA_ERR_UNSUPPORTED;
  if (c.dk != 64 && c.dk != 128 && c.dk != 192 && c.dk != 256) return NSA_ERR_UNSUPPORTED;
  if (c.dv != 64 && c.dv != 128) return NSA_ERR_UNSUPPORTED;
  if ((size_t)c.B * c.G > 65535) return NSA_ERR_UNSUPPORTED;
  if (dec_smem(c).total > smem_max()) return NSA_ERR_UNSUPPORTED;
  return NSA_OK;
}

size_t decode_ws_bytes(const nsa_cfg& c) { return dec_ws(c).end; }

size_t decode_zero_bytes(const nsa_cfg& c) { return dec_ws(c).pm; }

int launch_decode(const nsa_cfg& c, const void* q, const void* kcache, const void* vcache, const void* kc,
                  const void* vc, const void* gates, void* out, int32_t* idx_out, uint8_t* ws, cudaStream_t s) {
  const DecShape sh = dec_shape(c);
  const DecWs w = dec_ws(c);
  const DecSmem m = dec_smem(c);
  const uint64_t e = 2;
  const uint64_t BG = (uint64_t)sh.BG;
  CUtensorMap maps_cmp[4], maps_sel[4];
  const int Ncm = sh.Nc > 0 ? sh.Nc : 1;
  auto map3 = [&](CUtensorMap* mp, const void* base, int d, uint64_t rows) -> bool {
    const uint64_t dims[3] = {(uint64_t)d, rows, BG};
    const uint64_t str[2] = {(uint64_t)d * e, rows * d * e};
    const uint32_t box[3] = {64, 64, 1};
    return make_tmap_bf16(mp, base, 3, dims, str, box);
  };
  if (!map3(&maps_cmp[0], sh.Nc > 0 ? kc : kcache, c.dk, (uint64_t)Ncm)) return NSA_ERR_CUDA;
  if (!map3(&maps_cmp[1], sh.Nc > 0 ? vc : vcache, c.dv, (uint64_t)Ncm)) return NSA_ERR_CUDA;
  if (!map3(&maps_cmp[2], kcache, c.dk, (uint64_t)c.T)) return NSA_ERR_CUDA;
  if (!map3(&maps_cmp[3], vcache, c.dv, (uint64_t)c.T)) return NSA_ERR_CUDA;
  maps_sel[0] = maps_cmp[2];
  maps_sel[1] = maps_cmp[3];
  maps_sel[2] = maps_cmp[2];
  maps_sel[3] = maps_cmp[3];

  DecArgs a;
  a.B = c.B;
  a.T = c.T;
  a.H = c.H;
  a.G = c.G;
  a.BG = sh.BG;
  a.hpg = c.H / c.G;
  a.n = c.n;
  a.w = c.w;
  a.Nc = sh.Nc;
  a.nq = sh.nq;
  a.ntc = sh.ntc;
  a.splits = sh.splits;
  a.tps = kTilesPerSplit;
  a.sel_splits = sh.sel_splits;
  a.bps = kBlocksPerSelCta;
  a.NS = sh.NS;
  const float scale = c.scale > 0.f ? c.scale : 1.0f / sqrtf((float)c.dk);
  a.sc2 = scale * 1.4426950408889634f;
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.gates = static_cast<const __nv_bfloat16*>(gates);
  a.out = static_cast<__nv_bfloat16*>(out);
  a.idx_out = idx_out;
  a.pm = reinterpret_cast<float*>(ws + w.pm);
  a.pl = reinterpret_cast<float*>(ws + w.pl);
  a.po = reinterpret_cast<float*>(ws + w.po);
  a.u = reinterpret_cast<float*>(ws + w.u);
  a.cc = reinterpret_cast<float*>(ws + w.cc);
  a.mref = reinterpret_cast<float*>(ws + w.mref);
  a.stats = reinterpret_cast<float*>(ws + w.stats);
  a.idx = reinterpret_cast<int32_t*>(ws + w.idx);
  a.cnt = reinterpret_cast<int*>(ws + w.cnt);
  a.st = reinterpret_cast<DeviceStatus*>(ws);

#define NSA_DEC_CASE(DK_, DV_) \
  if (c.dk == DK_ && c.dv == DV_) return launch_dims<DK_, DV_>(a, sh, maps_cmp, maps_sel, m, s);
  NSA_DEC_CASE(64, 64)
  NSA_DEC_CASE(64, 128)
  NSA_DEC_CASE(128, 64)
  NSA_DEC_CASE(128, 128)
  NSA_DEC_CASE(192, 64)
  NSA_DEC_CASE(192, 128)
  NSA_DEC_CASE(256, 64)
  NSA_DEC_CASE(256, 128)
#undef NSA_DEC_CASE
  return NSA_ERR_UNSUPPORTED;
}

}  // namespace nsa
