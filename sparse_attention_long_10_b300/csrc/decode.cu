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
// Work is cut into units of up to 2 pairs of 64-row key/value blocks (256
// keys) of one group; one CTA takes one unit, two CTAs share an SM:
//     S^T[key, head] = K_pair[key, :] . q[head, :]         (tcgen05, M=128, N=16)
//     exact softmax over the unit's keys (max pass, then exp pass over TMEM)
//     O^T[dv, head] += V_pair^T[dv, key] . P^T[key, head]  (tcgen05, M=128, N=16)
// and leaves the unit's (max, sum, unnormalised O) per head in the workspace.
// Two launches:
//   dec_kernel<MODE 0>  grid (compressed units + window units, B*G)
//       compressed units also leave block-importance partials: for every
//       selection block j the sum over its compressed entries i of
//       w(i,j) p[h,i] (w = 16-token chunks shared), relative to the unit's
//       max; the last CTA of a group (atomic counter, no waiting) normalises
//       them, forms S[j] = sum_h ..., and keeps blocks 0, j_t, j_t-1 plus the
//       top n-3 others, ties to the lower index.
//   dec_kernel<MODE 1>  grid (selected units, B*G)
//       the kept blocks; the last CTA of a group merges every unit and writes
//       out = g_cmp*O_cmp + g_slc*O_slc + g_win*O_win (bf16).
#include <algorithm>

#include "common.cuh"
#include "kernels.hpp"
#include "profiler.hpp"
#include "tmap.hpp"

namespace nsa {

namespace {

constexpr int kThreads = 192;        // warps 0-3 softmax, 4 TMA producer, 5 MMA issuer
constexpr int NP = 16;               // MMA N: heads of the group, padded to 16
constexpr int kPairs = 2;            // block pairs per unit (256 keys)
constexpr int kUnitKeys = 128 * kPairs;
constexpr int kUnitBlocks = kUnitKeys / 4;   // selection blocks fed by one compressed unit
constexpr int kUnitChunks = kUnitKeys / 32;  // 32-entry chunks of one compressed unit
constexpr int kRingK = 3;            // 16 KB: one 64-column chunk of a pair
constexpr int kRingV = 1;            // 32 KB: both 64-column chunks of a value pair
constexpr int kSlotK = 16384;
constexpr int kSlotV = 32768;
constexpr int kQBuf = 2048;          // one 64-column chunk of NP query rows
constexpr int kPBuf = kPairs * 2 * kQBuf;

struct DecArgs {
  int B, T, H, G, BG, hpg, n, w;     // T: cache capacity (row stride of the caches)
  int Nc, ncu, nwu, nsu, NS;         // at capacity: compressed / window / selected units per group, slots
  float sc2;                         // softmax scale * log2(e)
  const int32_t* lens;               // nullable [B]: tokens of each sequence (query at len-1)
  const __nv_bfloat16* gates;        // [B,H,3]
  __nv_bfloat16* out;                // [B,H,dv]
  int32_t* idx_out;                  // nullable [B,G,n]
  float* pm;                         // [BG][NS][16] unit max (log2 units, -inf if empty)
  float* pl;                         // [BG][NS][16] unit sum
  float* po;                         // [BG][NS][16][dv] unit O (unnormalised)
  float* u;                          // [BG][ncu*kUnitBlocks][16] block partials within a 32-entry chunk
  float* cc;                         // [BG][ncu*kUnitChunks][16] carry of each chunk's last entry
  float* stats;                      // [BG][32] compressed-branch max and 1/sum per head
  int32_t* idx;                      // [BG][n]
  int* cnt;                          // [2][BG]
  DeviceStatus* st;
  int sel_cap, part_cap;             // last-CTA staging capacity: blocks, 16 x dv partials
  uint32_t off_kring, off_vring, off_pt, off_red, off_bar;
};

struct Bars {
  uint64_t q_full;
  uint64_t k_full[kRingK], k_empty[kRingK];
  uint64_t v_full[kRingV], v_empty[kRingV];
  uint64_t s_full, p_full, o_full;
  uint64_t wg;
  uint64_t drain;
  uint32_t tmem;
  int abort_flag;
  int last;
};

// This sequence's length, its compressed-entry count and window start.  A
// length outside [1, T] is recorded as NSA_ERR_INVALID_ARG and the sequence
// is treated as empty (nothing of it is read; its output is zero).
struct SeqGeom {
  int len, Nc, win0;
};
__device__ __forceinline__ SeqGeom seq_geom(const DecArgs& a, int b, DeviceStatus* st) {
  int len = a.lens != nullptr ? __ldg(a.lens + b) : a.T;
  if (len < 1 || len > a.T) {
    record_arg_error(st, NSA_ERR_INVALID_ARG, 400);
    len = 0;
  }
  SeqGeom s;
  s.len = len;
  s.Nc = len < 32 ? 0 : min((len - 32) / 16 + 1, a.Nc);
  s.win0 = len - min(a.w, len);
  return s;
}

__device__ __forceinline__ float ldcg_f(const float* p) { return __ldcg(p); }
__device__ __forceinline__ float4 ldcg4(const float* p) { return __ldcg(reinterpret_cast<const float4*>(p)); }

__device__ __forceinline__ float dot16(const float* f, const float4* v) {
  const float4 a = v[0], b = v[1], c = v[2], d = v[3];
  return f[0] * a.x + f[1] * a.y + f[2] * a.z + f[3] * a.w + f[4] * b.x + f[5] * b.y + f[6] * b.z + f[7] * b.w +
         f[8] * c.x + f[9] * c.y + f[10] * c.z + f[11] * c.w + f[12] * d.x + f[13] * d.y + f[14] * d.z +
         f[15] * d.w;
}

__device__ __forceinline__ uint32_t warp_min_u32(uint32_t x) {
  uint32_t r;
  asm volatile("redux.sync.min.u32 %0, %1, 0xffffffff;" : "=r"(r) : "r"(x));
  return r;
}
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_all;" ::: "memory");
}
// Copies n16 16-byte pieces global -> shared, spread over the CTA.
__device__ __forceinline__ void stage(void* dst, const void* src, int n16) {
  for (int i = threadIdx.x; i < n16; i += kThreads)
    cp_async16(static_cast<uint8_t*>(dst) + 16 * (size_t)i, static_cast<const uint8_t*>(src) + 16 * (size_t)i);
}
// (max, sum) of the 16 heads of partial slots [s0, s1) of group bg into sp[r][32]
__device__ __forceinline__ void stage_stats(const DecArgs& a, int bg, int s0, int s1, float* sp) {
  for (int e = threadIdx.x; e < (s1 - s0) * 8; e += kThreads) {
    const int r = e >> 3, q = e & 7;   // q < 4: max, q >= 4: sum
    const float* src = (q < 4 ? a.pm : a.pl) + ((size_t)bg * a.NS + s0 + r) * 16 + 4 * (q & 3);
    cp_async16(sp + r * 32 + (q < 4 ? 0 : 16) + 4 * (q & 3), src);
  }
}

// Per-lane sorted list of the 8 best (score, block) candidates: higher score
// first, equal scores in arrival order (lower block first).
struct Top8 {
  float v[8];
  int j[8];
  __device__ __forceinline__ void clear() {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      v[k] = -1.f;
      j[k] = 0x7fffffff;
    }
  }
  __device__ __forceinline__ void insert(float cv, int cj) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const bool sw = cv > v[k];
      const float t = v[k];
      const int u = j[k];
      v[k] = sw ? cv : t;
      j[k] = sw ? cj : u;
      cv = sw ? t : cv;
      cj = sw ? u : cj;
    }
  }
  __device__ __forceinline__ void pop() {
#pragma unroll
    for (int k = 0; k < 7; ++k) {
      v[k] = v[k + 1];
      j[k] = j[k + 1];
    }
    v[7] = -1.f;
    j[7] = 0x7fffffff;
  }
};

// Shared-memory plan of the selection step (floats).
struct SelStage {
  int sp, fsm, car, cc, S, ub, misc, total;
};
__host__ __device__ inline SelStage sel_stage(int ncu, int jt, int cap) {
  SelStage L;
  L.sp = 0;                                  // [ncu][32] unit max, sum
  L.fsm = 32 * ncu;                          // [ncu][16] factors exp2(m_unit - M) / L
  L.car = L.fsm + 16 * ncu;                  // [ncu*kUnitChunks] carry term of each chunk
  L.cc = (L.car + kUnitChunks * ncu + 3) & ~3;   // [ncu*kUnitChunks][16] last entry of each chunk
  L.S = L.cc + 16 * kUnitChunks * ncu;       // [jt+1] block importance
  L.ub = (L.S + jt + 1 + 3) & ~3;            // [cap][16] block partials
  L.misc = L.ub + 16 * cap;                  // Mh[16], iL[16], wv[128], wj[128]
  L.total = L.misc + 32 + 256;
  return L;
}

// Selection step, run by the last compressed/window CTA of a group: exact
// softmax statistics of the compressed branch (kept in ``stats`` for the
// final combine), block importance S[j] for every causal block, top-n.
// Its inputs are staged into shared memory with asynchronous copies, so
// they cost one round trip through L2 for caches up to sel_cap*64 tokens.
__device__ void select_step(const DecArgs& a, int bg, uint8_t* smem) {
  const int tid = threadIdx.x;
  const int warp = warp_id(), lane = lane_id();
  const int ncu = a.ncu, n = a.n;
  const SeqGeom sg = seq_geom(a, bg / a.G, nullptr);
  const int Nc = sg.Nc;
  const int jt = sg.len > 0 ? (sg.len - 1) / 64 : -1;   // -1: empty sequence, nothing kept
  const bool trivial = jt + 1 <= n;
  const SelStage L = sel_stage(ncu, jt, a.sel_cap);
  float* st = reinterpret_cast<float*>(smem);
  float* sp = st + L.sp;
  float* fsm = st + L.fsm;
  float* car = st + L.car;
  float* ccs = st + L.cc;
  float* Ssm = st + L.S;
  float* ubuf = st + L.ub;
  float* Mh = st + L.misc;
  float* iL = Mh + 16;
  float* wv = iL + 16;
  int* wj = reinterpret_cast<int*>(wv + 128);
  const int nblk = min(jt + 1, (Nc + 3) / 4);     // blocks holding compressed entries
  const float* ub = a.u + (size_t)bg * ncu * kUnitBlocks * 16;
  stage_stats(a, bg, 0, ncu, sp);
  if (!trivial) {
    stage(ccs, a.cc + (size_t)bg * ncu * kUnitChunks * 16, ncu * kUnitChunks * 4);
    stage(ubuf, ub, min(nblk, a.sel_cap) * 4);
  }
  cp_async_wait_all();
  __syncthreads();
  if (tid < 16) {
    float M = -INFINITY;
    for (int s = 0; s < ncu; ++s) M = fmaxf(M, sp[s * 32 + tid]);
    const float Mu = (M == -INFINITY) ? 0.f : M;
    float Ls = 0.f;
    for (int s = 0; s < ncu; ++s) Ls += sp[s * 32 + 16 + tid] * fast_exp2(sp[s * 32 + tid] - Mu);
    const float il = (Ls > 0.f && tid < a.hpg) ? 1.f / Ls : 0.f;
    Mh[tid] = Mu;
    iL[tid] = il;
    a.stats[(size_t)bg * 32 + tid] = Mu;
    a.stats[(size_t)bg * 32 + 16 + tid] = il;
  }
  int32_t* idx = a.idx + (size_t)bg * n;
  int32_t* idx_out = a.idx_out != nullptr ? a.idx_out + (size_t)bg * n : nullptr;
  if (trivial) {
    if (tid < n) {
      const int v = tid <= jt ? tid : -1;
      idx[tid] = v;
      if (idx_out) idx_out[tid] = v;
    }
    return;
  }
  __syncthreads();
  for (int e = tid; e < ncu * 16; e += kThreads) fsm[e] = fast_exp2(sp[(e >> 4) * 32 + (e & 15)] - Mh[e & 15]) * iL[e & 15];
  __syncthreads();
  // block importance: block j takes the partial of its four entries (unit
  // j/kUnitBlocks); blocks 8k+8 also take the carry of chunk k (entry 32k+31)
  for (int k = tid; k < ncu * kUnitChunks; k += kThreads)
    car[k] = (32 * k < Nc) ? dot16(fsm + (k / kUnitChunks) * 16, reinterpret_cast<const float4*>(ccs + 16 * k))
                             : 0.f;
  for (int c0 = 0; c0 <= jt; c0 += a.sel_cap) {
    if (c0 > 0) {
      __syncthreads();   // the previous chunk is consumed
      if (c0 < nblk) stage(ubuf, ub + (size_t)c0 * 16, min(nblk - c0, a.sel_cap) * 4);
      cp_async_wait_all();
      __syncthreads();
    }
    const int c1 = min(jt + 1, c0 + a.sel_cap);
#pragma unroll 4
    for (int j = c0 + tid; j < c1; j += kThreads)
      Ssm[j] = (j < nblk) ? dot16(fsm + (j / kUnitBlocks) * 16, reinterpret_cast<const float4*>(ubuf + 16 * (j - c0)))
                          : 0.f;
  }
  __syncthreads();
  for (int k = tid; 8 * k + 8 <= jt; k += kThreads)
    if (32 * k < Nc) Ssm[8 * k + 8] += car[k];
  __syncthreads();
  // top-(n-3) among the free blocks 1 .. jt-2: each of 4 warps finds the best
  // of its quarter of the range, warp 0 merges.  Order: higher score, then
  // lower block index.  Scores are >= 0; -2 marks a taken block.  Each lane
  // keeps its 8 best candidates sorted; a round's winner is a warp max
  // reduction, ties to the lowest index, and only its owner lane pops.
  const int kfree = n - 3;
  const int ncand = jt - 2;
  if (warp < 4) {
    const int per = (ncand + 3) / 4;
    const int lo = 1 + warp * per;
    const int hi = min(1 + ncand, lo + per);
    Top8 t;
    auto fill = [&]() {
      t.clear();
      for (int j = lo + lane; j < hi; j += 32) {
        const float v = Ssm[j];
        if (v > t.v[7]) t.insert(v, j);
      }
    };
    fill();
    for (int rnd = 0; rnd < kfree; ++rnd) {
      const float gv = warp_max_f32(t.v[0]);
      const int gj = (int)warp_min_u32(t.v[0] == gv ? (uint32_t)t.j[0] : 0x7fffffffu);
      if (lane == 0) {
        wv[warp * 32 + rnd] = gv;
        wj[warp * 32 + rnd] = gj;
      }
      if (gj != 0x7fffffff && t.j[0] == gj) {   // owner lane: candidates j = lo + lane (mod 32)
        Ssm[gj] = -2.f;
        t.pop();
        if (t.v[0] < 0.f) fill();   // this lane gave all 8: refill from the untaken rest
      }
    }
  }
  __syncthreads();
  if (warp == 0) {
    // lane holds candidates c = lane + 32k of the 4*kfree winners
    Top8 t;
    t.clear();
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int c = lane + 32 * k;
      if (c < 4 * kfree) t.insert(wv[(c / kfree) * 32 + c % kfree], wj[(c / kfree) * 32 + c % kfree]);
    }
    int mine = -1;
    for (int rnd = 0; rnd < kfree; ++rnd) {
      const float gv = warp_max_f32(t.v[0]);
      const int gj = (int)warp_min_u32(t.v[0] == gv ? (uint32_t)t.j[0] : 0x7fffffffu);
      if (t.j[0] == gj) t.pop();
      if (lane == rnd) mine = gj;
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
// with each branch's unit partials weighted by exp(m_unit - M) / L.  The
// statistics, the gates and part_cap partials at a time are staged into
// shared memory with asynchronous copies.
template <int DV>
__device__ void combine_step(const DecArgs& a, int bg, uint8_t* smem) {
  const int tid = threadIdx.x;
  const int b = bg / a.G, g = bg % a.G;
  const int NS = a.NS;
  constexpr int kE4 = (16 * DV / 4 + kThreads - 1) / kThreads;   // float4 elements per thread
  float* sp = reinterpret_cast<float*>(smem);    // [NS][2][16] unit max, sum
  float* fac = sp + 32 * NS;                     // [NS][16] weight of each partial
  float* gt = fac + 16 * NS;                     // [16][3]
  float* cst = gt + 48;                          // [32] compressed statistics
  float* pos = reinterpret_cast<float*>(smem) + ((48 * NS + 48 + 32 + 31) & ~31);   // [part_cap][16][DV]
  const float* po = a.po + (size_t)bg * NS * 16 * DV;
  stage_stats(a, bg, 0, NS, sp);
  stage(cst, a.stats + (size_t)bg * 32, 8);
  const int pb = a.part_cap;
  for (int r = 0; r < pb && r < NS; ++r) stage(pos + (size_t)r * 16 * DV, po + (size_t)r * 16 * DV, 16 * DV / 4);
  if (tid < 16) {
    const bool hv = tid < a.hpg;
    const __nv_bfloat16* gp = a.gates + ((size_t)b * a.H + g * a.hpg + (hv ? tid : 0)) * 3;
    gt[tid * 3 + 0] = hv ? __bfloat162float(gp[0]) : 0.f;
    gt[tid * 3 + 1] = hv ? __bfloat162float(gp[1]) : 0.f;
    gt[tid * 3 + 2] = hv ? __bfloat162float(gp[2]) : 0.f;
  }
  cp_async_wait_all();
  __syncthreads();
  if (tid < 16) {
    const int h = tid;
    // compressed: statistics from the selection step, folded with g_cmp
    const float Mc = cst[h], iLc = cst[16 + h];
    for (int s = 0; s < a.ncu; ++s) fac[s * 16 + h] = gt[h * 3 + 0] * fast_exp2(sp[s * 32 + h] - Mc) * iLc;
    // window and selected: merge their units here
    auto branch = [&](int s0, int s1, float gate) {
      float M = -INFINITY;
      for (int s = s0; s < s1; ++s) M = fmaxf(M, sp[s * 32 + h]);
      const float Mu = (M == -INFINITY) ? 0.f : M;
      float L = 0.f;
      for (int s = s0; s < s1; ++s) L += sp[s * 32 + 16 + h] * fast_exp2(sp[s * 32 + h] - Mu);
      const float il = L > 0.f ? gate / L : 0.f;
      for (int s = s0; s < s1; ++s) fac[s * 16 + h] = fast_exp2(sp[s * 32 + h] - Mu) * il;
    };
    branch(a.ncu, a.ncu + a.nwu, gt[h * 3 + 2]);
    branch(a.ncu + a.nwu, NS, gt[h * 3 + 1]);
  }
  __syncthreads();
  float4 acc[kE4];
#pragma unroll
  for (int k = 0; k < kE4; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int b0 = 0; b0 < NS; b0 += pb) {
    const int nb = min(pb, NS - b0);
    if (b0 > 0) {
      __syncthreads();   // the previous batch is consumed
      for (int r = 0; r < nb; ++r)
        stage(pos + (size_t)r * 16 * DV, po + (size_t)(b0 + r) * 16 * DV, 16 * DV / 4);
      cp_async_wait_all();
      __syncthreads();
    }
    for (int r = 0; r < nb; ++r) {
      const float4* src = reinterpret_cast<const float4*>(pos + (size_t)r * 16 * DV);
#pragma unroll
      for (int k = 0; k < kE4; ++k) {
        const int e4 = tid + kThreads * k;
        if (e4 < a.hpg * DV / 4) {
          const float f = fac[(b0 + r) * 16 + (4 * e4) / DV];
          const float4 v = src[e4];
          acc[k].x += f * v.x;
          acc[k].y += f * v.y;
          acc[k].z += f * v.z;
          acc[k].w += f * v.w;
        }
      }
    }
  }
#pragma unroll
  for (int k = 0; k < kE4; ++k) {
    const int e4 = tid + kThreads * k;
    if (e4 < a.hpg * DV / 4) {
      uint2 pk;
      pk.x = pack_bf16x2(acc[k].x, acc[k].y);
      pk.y = pack_bf16x2(acc[k].z, acc[k].w);
      *reinterpret_cast<uint2*>(a.out + ((size_t)b * a.H + g * a.hpg) * DV + 4 * e4) = pk;
    }
  }
}

// One unit: up to kPairs pairs of 64-row blocks of one group against the
// group's query heads.
//   MODE 0: x < ncu     compressed entries [U x, U x + U) (limit Nc)
//           x >= ncu    window tokens win0 + U (x-ncu) + [0, U) (limit T)
//           (U = kUnitKeys = 256)
//   MODE 1: x           kept blocks idx[4x .. 4x+3] (token rows 64*blk)
template <int DK, int DV, int MODE>
__global__ void __launch_bounds__(kThreads, 2)
    dec_kernel(const __grid_constant__ CUtensorMap mapQ, const __grid_constant__ CUtensorMap mK0,
               const __grid_constant__ CUtensorMap mV0, const __grid_constant__ CUtensorMap mK1,
               const __grid_constant__ CUtensorMap mV1, const DecArgs a) {
  constexpr int kcs = DK / 64, vcs = DV / 64;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* qbuf = smem;                        // kcs chunks x 2 KB
  uint8_t* kring = smem + a.off_kring;
  uint8_t* vring = smem + a.off_vring;
  uint8_t* pt = smem + a.off_pt;               // P^T: kPairs x 2 chunks x 2 KB
  float* red = reinterpret_cast<float*>(smem + a.off_red);   // [2 max/sum][4 warps][NP]
  Bars* bars = reinterpret_cast<Bars*>(smem + a.off_bar);
  volatile int* abort_flag = &bars->abort_flag;
  const int x = blockIdx.x, bg = blockIdx.y;
  const int b = bg / a.G, g = bg % a.G;
  const int warp = warp_id(), lane = lane_id();

  // ------------------------------------------------------------ unit geometry
  // (the grid is sized for the cache capacity; a shorter sequence leaves some
  // units empty: npairs = 0)
  const SeqGeom sg = seq_geom(a, b, threadIdx.x == 0 && x == 0 ? a.st : nullptr);
  const bool cmp_unit = MODE == 0 && x < a.ncu;
  int base = 0, limit = sg.len, npairs = kPairs, sel0 = 0;
  if (MODE == 0) {
    if (cmp_unit) {
      base = kUnitKeys * x;
      limit = sg.Nc;
      npairs = min(kPairs, (sg.Nc - base + 127) / 128);
    } else {
      base = sg.win0 + kUnitKeys * (x - a.ncu);
      limit = sg.len;
      npairs = min(kPairs, (sg.len - base + 127) / 128);
    }
  } else {
    sel0 = 2 * kPairs * x;
    npairs = sg.len > 0 ? min(kPairs, (a.n - sel0 + 1) / 2) : 0;
  }
  npairs = max(npairs, 0);
  const CUtensorMap* mapK = cmp_unit ? &mK0 : &mK1;
  const CUtensorMap* mapV = cmp_unit ? &mV0 : &mV1;
  // first map row of block 2p+hb of this unit; -1 if absent (reads zeros)
  auto block_row = [&](int p, int hb) -> int {
    if (MODE == 0) return base + 128 * p + 64 * hb;
    const int e = sel0 + 2 * p + hb;
    const int blk = e < a.n ? a.idx[(size_t)bg * a.n + e] : -1;
    return blk >= 0 ? 64 * blk : -1;
  };

  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    for (int i = 0; i < kRingK; ++i) {
      mbar_init(&bars->k_full[i], 1);
      mbar_init(&bars->k_empty[i], 1);
    }
    for (int i = 0; i < kRingV; ++i) {
      mbar_init(&bars->v_full[i], 1);
      mbar_init(&bars->v_empty[i], 1);
    }
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->p_full, 4);
    mbar_init(&bars->o_full, 1);
    mbar_init(&bars->wg, 4);
    mbar_init(&bars->drain, 1);
    bars->last = 0;
    fence_barrier_init();
  }
  // query rows hpg..NP-1 are never loaded: keep them finite (zero)
  for (int i = threadIdx.x; i < kcs * kQBuf / 16; i += kThreads)
    reinterpret_cast<uint4*>(qbuf)[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  if (warp == 0) {
    tmem_alloc(&bars->tmem, 128);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // the query is an input: its load overlaps the previous kernel's tail
  if (threadIdx.x == 0) {
    tma_prefetch_desc(&mapQ);
    tma_prefetch_desc(mapK);
    tma_prefetch_desc(mapV);
    mbar_arrive_expect_tx(&bars->q_full, (uint32_t)(kcs * a.hpg * 128));
    for (int c = 0; c < kcs; ++c) tma_load_3d(qbuf + c * kQBuf, &mapQ, &bars->q_full, c * 64, g * a.hpg, b);
  }
  // the kept blocks, the partials and the status come from the previous kernel
  pdl_wait();
  if (threadIdx.x == 0) bars->abort_flag = prior_error(a.st);
  __syncthreads();
  const uint32_t tmem = bars->tmem;
  const uint32_t tmem_s = tmem;                 // kPairs x NP columns
  const uint32_t tmem_o = tmem + kPairs * NP;   // NP columns

  bool ok = *abort_flag == 0;

  if (!ok) {
    // an earlier CTA failed: only the query load is in flight
    if (threadIdx.x == 0) mbar_wait_plain(&bars->q_full, 0, kWaitLimitNs);
  } else if (warp == 4) {
    // =============================================================== producer
    if (lane == 0) {
      int kv = 0, vv = 0;
      for (int p = 0; p < npairs && ok; ++p) {
        const int r0 = block_row(p, 0), r1 = block_row(p, 1);
        for (int c = 0; c < kcs; ++c) {
          const int slot = kv % kRingK;
          if (!mbar_wait(&bars->k_empty[slot], (uint32_t)(((kv / kRingK) & 1) ^ 1), abort_flag, a.st, 401)) {
            ok = false;
            break;
          }
          uint8_t* dst = kring + slot * kSlotK;
          mbar_arrive_expect_tx(&bars->k_full[slot], kSlotK);
          tma_load_3d(dst, mapK, &bars->k_full[slot], c * 64, r0 >= 0 ? r0 : -128, bg);
          tma_load_3d(dst + 8192, mapK, &bars->k_full[slot], c * 64, r1 >= 0 ? r1 : -128, bg);
          ++kv;
        }
      }
      for (int p = 0; p < npairs && ok; ++p) {
        const int r0 = block_row(p, 0), r1 = block_row(p, 1);
        const int slot = vv % kRingV;
        if (!mbar_wait(&bars->v_empty[slot], (uint32_t)(((vv / kRingV) & 1) ^ 1), abort_flag, a.st, 402)) {
          ok = false;
          break;
        }
        uint8_t* dst = vring + slot * kSlotV;
        mbar_arrive_expect_tx(&bars->v_full[slot], (uint32_t)(vcs * 16384));
        for (int c = 0; c < vcs; ++c) {
          tma_load_3d(dst + c * 16384, mapV, &bars->v_full[slot], c * 64, r0 >= 0 ? r0 : -128, bg);
          tma_load_3d(dst + c * 16384 + 8192, mapV, &bars->v_full[slot], c * 64, r1 >= 0 ? r1 : -128, bg);
        }
        ++vv;
      }
      if (!ok || *abort_flag) {
        mbar_wait_plain(&bars->q_full, 0, kWaitLimitNs);
        for (int y = (kv > kRingK ? kv - kRingK : 0); y < kv; ++y)
          mbar_wait_plain(&bars->k_full[y % kRingK], (uint32_t)((y / kRingK) & 1), kWaitLimitNs);
        for (int y = (vv > kRingV ? vv - kRingV : 0); y < vv; ++y)
          mbar_wait_plain(&bars->v_full[y % kRingV], (uint32_t)((y / kRingV) & 1), kWaitLimitNs);
      }
    }
  } else if (warp == 5) {
    // =============================================================== MMA issuer
    if (lane == 0) {
      const uint32_t idesc_qk = idesc_bf16_f32(128, NP, false, false);
      const uint32_t idesc_pv = idesc_bf16_f32(128, NP, true, false);
      const uint32_t q_a = smem_u32(qbuf), k_a = smem_u32(kring), v_a = smem_u32(vring), p_a = smem_u32(pt);
      int kv = 0, vv = 0;
      if (!mbar_wait(&bars->q_full, 0, abort_flag, a.st, 411)) ok = false;
      tc_fence_after();
      for (int p = 0; p < npairs && ok; ++p) {
        for (int c = 0; c < kcs; ++c) {
          const int slot = kv % kRingK;
          if (!mbar_wait(&bars->k_full[slot], (uint32_t)((kv / kRingK) & 1), abort_flag, a.st, 412)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint64_t ad = sdesc_sw128(k_a + slot * kSlotK + k * 32, 16, 1024);
            const uint64_t bd = sdesc_sw128(q_a + c * kQBuf + k * 32, 16, 1024);
            umma_bf16(tmem_s + p * NP, ad, bd, idesc_qk, (c > 0 || k > 0) ? 1u : 0u);
          }
          umma_commit(&bars->k_empty[slot]);
          ++kv;
        }
      }
      if (ok) umma_commit(&bars->s_full);
      if (ok && !mbar_wait(&bars->p_full, 0, abort_flag, a.st, 413)) ok = false;
      tc_fence_after();
      for (int p = 0; p < npairs && ok; ++p) {
        const int slot = vv % kRingV;
        if (!mbar_wait(&bars->v_full[slot], (uint32_t)((vv / kRingV) & 1), abort_flag, a.st, 414)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          // A = V^T (dv-major rows of keys), B = P^T (head rows, keys along K)
          const uint64_t ad = sdesc_sw128(v_a + slot * kSlotV + k * 2048, 16384, 1024);
          const uint64_t bd = sdesc_sw128(p_a + (p * 2 + (k >> 2)) * kQBuf + (k & 3) * 32, 16, 1024);
          umma_bf16(tmem_o, ad, bd, idesc_pv, (p > 0 || k > 0) ? 1u : 0u);
        }
        umma_commit(&bars->v_empty[slot]);
        ++vv;
      }
      if (ok) umma_commit(&bars->o_full);
      if (!ok || *abort_flag) {
        umma_commit(&bars->drain);
        mbar_wait_plain(&bars->drain, 0, kWaitLimitNs);
      }
    }
  } else {
    // =============================================================== softmax (warps 0-3)
    const int r = warp * 32 + lane;       // TMEM lane: key of a pair / value dim
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const bool hi_half = (r >> 6) != 0;
    const int kk = r & 63;
    float* red_m = red;                    // [4][NP]
    float* red_l = red + 4 * NP;           // [4][NP]
    uint32_t wg_phase = 0;
    auto wg_sync = [&]() {
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->wg);
      if (!mbar_wait(&bars->wg, wg_phase & 1, abort_flag, a.st, 421)) ok = false;
      ++wg_phase;
    };
    // first map row of this lane's block in each pair (-1 if absent)
    int rows[kPairs];
#pragma unroll
    for (int p = 0; p < kPairs; ++p) rows[p] = p < npairs ? block_row(p, hi_half ? 1 : 0) : -1;
    if (!mbar_wait(&bars->s_full, 0, abort_flag, a.st, 422)) ok = false;
    tc_fence_after();
    // pass 1: per-head max of the raw scores over the valid keys
    float mrow[NP];
#pragma unroll
    for (int h = 0; h < NP; ++h) mrow[h] = -INFINITY;
    if (ok) {
#pragma unroll
      for (int p = 0; p < kPairs; ++p) {
        if (p < npairs) {
          uint32_t rr[16];
          tmem_ld16(tmem_s + lane_base + p * NP, rr);
          tmem_ld_wait(rr);
          const bool v = rows[p] >= 0 && rows[p] + kk < limit;
#pragma unroll
          for (int h = 0; h < NP; ++h) mrow[h] = fmaxf(mrow[h], v ? __uint_as_float(rr[h]) : -INFINITY);
        }
      }
#pragma unroll
      for (int h = 0; h < NP; ++h) mrow[h] = warp_max_f32(mrow[h]);
      if (lane == 0)
#pragma unroll
        for (int h = 0; h < NP; ++h) red_m[warp * NP + h] = mrow[h];
    }
    wg_sync();
    float mu[NP];
#pragma unroll
    for (int h = 0; h < NP; ++h) {
      const float m = fmaxf(fmaxf(red_m[h], red_m[NP + h]), fmaxf(red_m[2 * NP + h], red_m[3 * NP + h]));
      mrow[h] = (m == -INFINITY) ? -INFINITY : m * a.sc2;
      mu[h] = (m == -INFINITY) ? 0.f : m * a.sc2;
    }
    // pass 2: p = exp(s*scale - max), sums, P^T, block-score partials
    float lrow[NP];
#pragma unroll
    for (int h = 0; h < NP; ++h) lrow[h] = 0.f;
    if (ok) {
#pragma unroll
      for (int p = 0; p < kPairs; ++p) {
        if (p < npairs) {
          uint32_t rr[16];
          tmem_ld16(tmem_s + lane_base + p * NP, rr);
          tmem_ld_wait(rr);
          const bool v = rows[p] >= 0 && rows[p] + kk < limit;
          float e[NP];
          uint8_t* chunk = pt + (p * 2 + (hi_half ? 1 : 0)) * kQBuf + (kk & 7) * 2;
#pragma unroll
          for (int h = 0; h < NP; ++h) {
            e[h] = v ? fast_exp2(fmaf(__uint_as_float(rr[h]), a.sc2, -mu[h])) : 0.f;
            lrow[h] += e[h];
            *reinterpret_cast<__nv_bfloat16*>(chunk + sw128_offset(h, kk >> 3)) = __float2bfloat16_rn(e[h]);
          }
          if (cmp_unit) {
            // entries 4q..4q+3 of this warp's 32 feed block (entry/4) with
            // 2*sum - last + last of the previous group; the warp's last entry
            // carries one chunk into the block of the next 32 entries
            float uq[NP];
#pragma unroll
            for (int h = 0; h < NP; ++h) {
              float gsum = e[h] + __shfl_xor_sync(0xffffffffu, e[h], 1);
              gsum += __shfl_xor_sync(0xffffffffu, gsum, 2);
              const float last = __shfl_sync(0xffffffffu, e[h], lane | 3);
              const float prev = __shfl_up_sync(0xffffffffu, last, 4);
              uq[h] = 2.f * gsum - last + (lane >= 4 ? prev : 0.f);
            }
            const int entry0 = base + 128 * p + 32 * warp;   // first entry of this warp
            if ((lane & 3) == 0) {
              float4* dst =
                  reinterpret_cast<float4*>(a.u + ((size_t)bg * a.ncu * kUnitBlocks + (entry0 + lane) / 4) * 16);
#pragma unroll
              for (int k = 0; k < 4; ++k) dst[k] = make_float4(uq[4 * k], uq[4 * k + 1], uq[4 * k + 2], uq[4 * k + 3]);
            }
            if (lane == 31) {
              float4* dst = reinterpret_cast<float4*>(a.cc + ((size_t)bg * a.ncu * kUnitChunks + entry0 / 32) * 16);
#pragma unroll
              for (int k = 0; k < 4; ++k) dst[k] = make_float4(e[4 * k], e[4 * k + 1], e[4 * k + 2], e[4 * k + 3]);
            }
          }
        }
      }
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars->p_full);
    // sums per head over the unit
    const float ws = warp_sum16(lrow, lane);
    if ((lane & 1) == 0) red_l[warp * NP + head_of_lane(lane)] = ws;
    wg_sync();
    // unit partial: max, sum, unnormalised O^T (lane = value dim)
    const int slot_id = (MODE == 0) ? x : (a.ncu + a.nwu + x);
    const size_t pbase = (size_t)bg * a.NS + slot_id;
    if (ok && r < NP) {
      a.pm[pbase * 16 + r] = mrow[r];
      a.pl[pbase * 16 + r] = red_l[r] + red_l[NP + r] + red_l[2 * NP + r] + red_l[3 * NP + r];
    }
    if (ok && mbar_wait(&bars->o_full, 0, abort_flag, a.st, 423)) {
      tc_fence_after();
      uint32_t rr[16];
      tmem_ld16(tmem_o + lane_base, rr);
      tmem_ld_wait(rr);
      if (npairs == 0) {   // no MMA wrote O: the unit's partial is zero
#pragma unroll
        for (int h = 0; h < NP; ++h) rr[h] = 0u;
      }
      if (r < DV) {
        float* dst = a.po + pbase * 16 * DV + r;
#pragma unroll
        for (int h = 0; h < NP; ++h) dst[(size_t)h * DV] = __uint_as_float(rr[h]);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, 128);
  if (*abort_flag) return;

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
struct DecShape {
  int Nc, ncu, nwu, nsu, NS, BG, win0, win_len;
};

DecShape dec_shape(const nsa_cfg& c) {
  DecShape s;
  s.Nc = c.T < c.l ? 0 : (c.T - c.l) / c.d + 1;
  s.ncu = (s.Nc + kUnitKeys - 1) / kUnitKeys;
  s.win_len = c.w < c.T ? c.w : c.T;
  s.win0 = c.T - s.win_len;
  s.nwu = (s.win_len + kUnitKeys - 1) / kUnitKeys;
  s.nsu = (c.n + 2 * kPairs - 1) / (2 * kPairs);
  s.NS = s.ncu + s.nwu + s.nsu;
  s.BG = c.B * c.G;
  return s;
}

struct DecWs {
  size_t cnt, pm, pl, po, u, cc, stats, idx, end;
};

DecWs dec_ws(const nsa_cfg& c) {
  const DecShape s = dec_shape(c);
  const size_t BG = (size_t)s.BG;
  DecWs w;
  w.cnt = sizeof(DeviceStatus);
  w.pm = align_up(w.cnt + sizeof(int) * 2 * BG, 256);
  w.pl = align_up(w.pm + sizeof(float) * BG * s.NS * 16, 256);
  w.po = align_up(w.pl + sizeof(float) * BG * s.NS * 16, 256);
  w.u = align_up(w.po + sizeof(float) * BG * s.NS * 16 * c.dv, 256);
  w.cc = align_up(w.u + sizeof(float) * BG * (size_t)s.ncu * kUnitBlocks * 16, 256);
  w.stats = align_up(w.cc + sizeof(float) * BG * (size_t)s.ncu * kUnitChunks * 16, 256);
  w.idx = align_up(w.stats + sizeof(float) * BG * 32, 256);
  w.end = align_up(w.idx + sizeof(int32_t) * BG * c.n, 256);
  return w;
}

struct DecLayout {
  uint32_t off_kring, off_vring, off_pt, off_red, off_bar, total;
  int sel_cap, part_cap;
};

DecLayout dec_layout(const nsa_cfg& c) {
  const DecShape s = dec_shape(c);
  DecLayout L;
  L.off_kring = (uint32_t)align_up((size_t)(c.dk / 64) * kQBuf, 1024);
  L.off_vring = L.off_kring + kRingK * kSlotK;
  L.off_pt = L.off_vring + kRingV * kSlotV;
  L.off_red = L.off_pt + kPBuf;
  const size_t body = L.off_red + 2 * 4 * NP * sizeof(float);
  // The last-CTA steps reuse the start of shared memory as staging: at least
  // 1,024 blocks (or all) of selection inputs and 4 (or all) partials, more if
  // the pipeline area is larger.
  const int jt = (c.T - 1) / 64;
  const int nblk = s.Nc > 0 ? std::min(jt + 1, (s.Nc + 3) / 4) : 1;
  const long sel_fixed = sel_stage(s.ncu, jt, 0).total;
  const long head = (48L * s.NS + 48 + 32 + 31) & ~31L;
  const long need_sel = sel_fixed + 16L * std::min(((long)nblk + 3) & ~3L, 1024L);
  const long need_comb = head + 16L * c.dv * std::min(s.NS, 4);
  size_t end = std::max<size_t>(body, 4 * (size_t)std::max(need_sel, need_comb));
  L.off_bar = (uint32_t)align_up(end, 256);
  const long avail_f = L.off_bar / 4;
  long cap = (avail_f - sel_fixed) / 16;
  cap = std::min<long>(cap, ((long)nblk + 3) & ~3L) & ~3L;
  L.sel_cap = (int)std::max(cap, 4L);
  L.part_cap = (int)std::max(1L, std::min<long>((avail_f - head) / (16L * c.dv), s.NS));
  L.total = L.off_bar + (uint32_t)align_up(sizeof(Bars), 256) + 1024;
  return L;
}

template <int DK, int DV, int MODE>
int launch_one(const DecArgs& a, dim3 grid, const CUtensorMap* maps, uint32_t smem, cudaStream_t s,
               const char* name) {
  if (int rc = ensure_smem_attr(reinterpret_cast<const void*>(&dec_kernel<DK, DV, MODE>), smem_max())) return rc;
  prof::begin(name, s);
  int rc = NSA_OK;
  if (MODE == 0) {
    dec_kernel<DK, DV, MODE><<<grid, kThreads, smem, s>>>(maps[0], maps[1], maps[2], maps[3], maps[4], a);
    rc = cudaPeekAtLastError() == cudaSuccess ? NSA_OK : NSA_ERR_CUDA;
  } else {
    // may start while the compressed / window kernel finishes (pdl_wait)
    rc = launch_dependent(dec_kernel<DK, DV, MODE>, grid, dim3(kThreads), smem, s, 1, maps[0], maps[1], maps[2],
                          maps[3], maps[4], a);
  }
  prof::end(s);
  return rc;
}

template <int DK, int DV>
int launch_dims(const DecArgs& a, const DecShape& sh, const CUtensorMap* maps, uint32_t smem, cudaStream_t s) {
  int rc = launch_one<DK, DV, 0>(a, dim3(sh.ncu + sh.nwu, sh.BG), maps, smem, s, "dec_cmp_win");
  if (rc != NSA_OK) return rc;
  return launch_one<DK, DV, 1>(a, dim3(sh.nsu, sh.BG), maps, smem, s, "dec_sel");
}

}  // namespace

int decode_supported(const nsa_cfg& c) {
  const int hpg = c.H / c.G;
  if (hpg > NP) return NSA_ERR_UNSUPPORTED;
  if (c.dk != 64 && c.dk != 128 && c.dk != 192 && c.dk != 256) return NSA_ERR_UNSUPPORTED;
  if (c.dv != 64 && c.dv != 128) return NSA_ERR_UNSUPPORTED;
  if ((size_t)c.B * c.G > 65535) return NSA_ERR_UNSUPPORTED;
  if (dec_layout(c).total > smem_max()) return NSA_ERR_UNSUPPORTED;
  return NSA_OK;
}

size_t decode_ws_bytes(const nsa_cfg& c) { return dec_ws(c).end; }

size_t decode_zero_bytes(const nsa_cfg& c) { return dec_ws(c).pm; }

int launch_decode(const nsa_cfg& c, const void* q, const void* kcache, const void* vcache, const void* kc,
                  const void* vc, const int32_t* lens, const void* gates, void* out, int32_t* idx_out, uint8_t* ws,
                  cudaStream_t s) {
  const DecShape sh = dec_shape(c);
  const DecWs w = dec_ws(c);
  const DecLayout L = dec_layout(c);
  const uint64_t e = 2;
  const uint64_t BG = (uint64_t)sh.BG;
  CUtensorMap maps[5];
  const int Ncm = sh.Nc > 0 ? sh.Nc : 1;
  auto map3 = [&](CUtensorMap* mp, const void* base, int d, uint64_t rows) -> bool {
    const uint64_t dims[3] = {(uint64_t)d, rows, BG};
    const uint64_t str[2] = {(uint64_t)d * e, rows * d * e};
    const uint32_t box[3] = {64, 64, 1};
    return make_tmap_bf16(mp, base, 3, dims, str, box);
  };
  {  // q [B,H,dk]: box (64 columns, hpg heads, 1)
    const uint64_t dims[3] = {(uint64_t)c.dk, (uint64_t)c.H, (uint64_t)c.B};
    const uint64_t str[2] = {(uint64_t)c.dk * e, (uint64_t)c.H * c.dk * e};
    const uint32_t box[3] = {64, (uint32_t)(c.H / c.G), 1};
    if (!make_tmap_bf16(&maps[0], q, 3, dims, str, box)) return NSA_ERR_CUDA;
  }
  if (!map3(&maps[1], sh.Nc > 0 ? kc : kcache, c.dk, (uint64_t)Ncm)) return NSA_ERR_CUDA;
  if (!map3(&maps[2], sh.Nc > 0 ? vc : vcache, c.dv, (uint64_t)Ncm)) return NSA_ERR_CUDA;
  if (!map3(&maps[3], kcache, c.dk, (uint64_t)c.T)) return NSA_ERR_CUDA;
  if (!map3(&maps[4], vcache, c.dv, (uint64_t)c.T)) return NSA_ERR_CUDA;

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
  a.ncu = sh.ncu;
  a.nwu = sh.nwu;
  a.nsu = sh.nsu;
  a.NS = sh.NS;
  a.lens = lens;
  const float scale = c.scale > 0.f ? c.scale : 1.0f / sqrtf((float)c.dk);
  a.sc2 = scale * 1.4426950408889634f;
  a.gates = static_cast<const __nv_bfloat16*>(gates);
  a.out = static_cast<__nv_bfloat16*>(out);
  a.idx_out = idx_out;
  a.pm = reinterpret_cast<float*>(ws + w.pm);
  a.pl = reinterpret_cast<float*>(ws + w.pl);
  a.po = reinterpret_cast<float*>(ws + w.po);
  a.u = reinterpret_cast<float*>(ws + w.u);
  a.cc = reinterpret_cast<float*>(ws + w.cc);
  a.stats = reinterpret_cast<float*>(ws + w.stats);
  a.idx = reinterpret_cast<int32_t*>(ws + w.idx);
  a.cnt = reinterpret_cast<int*>(ws + w.cnt);
  a.st = reinterpret_cast<DeviceStatus*>(ws);
  a.off_kring = L.off_kring;
  a.off_vring = L.off_vring;
  a.off_pt = L.off_pt;
  a.off_red = L.off_red;
  a.off_bar = L.off_bar;
  a.sel_cap = L.sel_cap;
  a.part_cap = L.part_cap;

#define NSA_DEC_CASE(DK_, DV_) \
  if (c.dk == DK_ && c.dv == DV_) return launch_dims<DK_, DV_>(a, sh, maps, L.total, s);
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
