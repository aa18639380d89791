// compress.cu -- token compression phi as a tcgen05 GEMM [P2 section II.1;
// P3 token-compression paragraph].
//
// For one KV head, compressed block i is flatten(X[d*i : d*i+l] + PE) @ W.
// Split W into l row-slices W_r [dX, N]:
//     Xc_i = sum_r X[d*i + r] @ W_r  +  bias,      bias = flatten(PE) @ W
// so the GEMM's A operand is "row i of X shifted by r tokens": a strided view
// of X that one 5-D TMA box per (r, 64-column chunk) fetches directly from the
// K/V tensor (tokens split as 16*a + b).  No im2col copy is ever written.
//
//   M = 128 compressed blocks per CTA, N = dout (<= 256), K = l*dX in steps
//   of 64 (one 128-byte swizzle row), 4-stage TMA -> tcgen05 pipeline,
//   fp32 accumulator in TMEM, bias + bf16 epilogue from TMEM.
#include "common.cuh"
#include "kernels.hpp"
#include "profiler.hpp"
#include "tmap.hpp"

namespace nsa {

namespace {

constexpr int kStages = 4;
constexpr int kTileM = 128;

struct CompressArgs {
  int Nc;          // compressed blocks per head
  int N;           // output dim (multiple of 64, <= 256)
  int nkb;         // K blocks of 64: l * dX / 64
  int cpr;         // 64-column chunks per token row: dX / 64
  int layout;      // NSA_LAYOUT_*
  int G;
  int stall;              // test hook: CTA (0,0,0) withholds stage 1 (NSA_FLAG_TEST_STALL)
  const float* bias;      // [N]
  __nv_bfloat16* out;     // [B, G, Nc, N]
  DeviceStatus* st;
};

// bias[n] = sum_r pe_flat[r] * W[r, n], r < rows = l*dX  (fp32).
// A cluster of kBiasSplit CTAs shares 32 columns: CTA c sums its slice of the
// rows, and CTA 0 adds the slices' partials from the other CTAs' shared
// memory (distributed shared memory) in a fixed order, so the result does not
// depend on scheduling.
constexpr int kBiasSplit = 8;
constexpr int kBiasRowsY = 16;

__global__ void __cluster_dims__(1, kBiasSplit, 1) __launch_bounds__(32 * kBiasRowsY)
    phi_bias_kernel(const __nv_bfloat16* __restrict__ pe, const __nv_bfloat16* __restrict__ w, int rows, int N,
                    float* __restrict__ bias) {
  __shared__ float red[kBiasRowsY][33];
  __shared__ float part[32];
  const int n = blockIdx.x * 32 + threadIdx.x;
  const int per = (rows + kBiasSplit - 1) / kBiasSplit;
  const int r0 = blockIdx.y * per, r1 = min(rows, r0 + per);
  float acc = 0.f;
  if (n < N) {
#pragma unroll 4
    for (int r = r0 + threadIdx.y; r < r1; r += kBiasRowsY)
      acc = fmaf(__bfloat162float(pe[r]), __bfloat162float(w[(size_t)r * N + n]), acc);
  }
  red[threadIdx.y][threadIdx.x] = acc;
  __syncthreads();
  if (threadIdx.y == 0) {
    float sum = 0.f;
#pragma unroll
    for (int y = 0; y < kBiasRowsY; ++y) sum += red[y][threadIdx.x];
    part[threadIdx.x] = sum;
  }
  // every CTA's partial is in its shared memory before CTA 0 reads them
  cluster_sync();
  if (blockIdx.y == 0 && threadIdx.y == 0) {
    float sum = 0.f;
    for (int c = 0; c < kBiasSplit; ++c) sum += __uint_as_float(dsmem_ld_u32(dsmem_addr(&part[threadIdx.x], c)));
    if (n < N) bias[n] = sum;
  }
  // no CTA leaves while CTA 0 may still read its shared memory
  cluster_sync();
}

__global__ void __launch_bounds__(128, 1)
    compress_gemm_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
                         const CompressArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const int nchunk = a.N / 64;
  const uint32_t a_bytes = kTileM * 128;
  const uint32_t b_bytes = (uint32_t)nchunk * 64 * 128;
  const uint32_t stage_bytes = a_bytes + b_bytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * stage_bytes);
  uint64_t* empty = full + kStages;
  uint64_t* done = empty + kStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int i0 = blockIdx.x * kTileM;
  const int g = blockIdx.y;
  const int b = blockIdx.z;
  const int warp = warp_id();
  const int lane = lane_id();

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(done, 1);
    *abort_flag = prior_error(a.st);
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const bool skip = *abort_flag != 0;

  if (skip) {
  } else if (warp == 0 && lane == 0) {
    // ---------------- TMA producer
    tma_prefetch_desc(&mapA);
    tma_prefetch_desc(&mapB);
    int issued = 0;
    for (int kb = 0; kb < a.nkb; ++kb) {
      const int s = kb % kStages;
      const uint32_t ph = (kb / kStages) & 1;
      if (!mbar_wait(&empty[s], ph ^ 1, abort_flag, a.st, 101)) break;
      if (a.stall && kb == 1 && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0) {
        // test hook: this stage is never armed, so the MMA issuer's bounded
        // wait for it runs out (and the drain below gives up on it)
        ++issued;
        continue;
      }
      const int r = kb / a.cpr;            // token offset inside the block
      const int c = kb % a.cpr;            // 64-column chunk of the token row
      uint8_t* sa = smem + s * stage_bytes;
      uint8_t* sb = sa + a_bytes;
      mbar_arrive_expect_tx(&full[s], stage_bytes);
      // token of row i is 16*(i + r/16) + r%16
      if (a.layout == NSA_LAYOUT_BTGD)
        tma_load_5d(sa, &mapA, &full[s], c * 64, g, r & 15, i0 + (r >> 4), b);
      else
        tma_load_5d(sa, &mapA, &full[s], c * 64, r & 15, i0 + (r >> 4), g, b);
      for (int n = 0; n < nchunk; ++n) tma_load_2d(sb + n * 8192, &mapB, &full[s], n * 64, kb * 64);
      ++issued;
    }
    if (*abort_flag) {
      // drain the loads still landing in shared memory before the CTA exits
      for (int kb = (issued > kStages ? issued - kStages : 0); kb < issued; ++kb)
        mbar_wait_plain(&full[kb % kStages], (kb / kStages) & 1, kWaitLimitNs);
    }
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer (single thread)
    const uint32_t idesc = idesc_bf16_f32(kTileM, a.N, false, true);
    for (int kb = 0; kb < a.nkb; ++kb) {
      const int s = kb % kStages;
      const uint32_t ph = (kb / kStages) & 1;
      if (!mbar_wait(&full[s], ph, abort_flag, a.st, 102)) break;
      tc_fence_after();
      const uint32_t sa = smem_u32(smem + s * stage_bytes);
      const uint32_t sb = sa + a_bytes;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint64_t ad = sdesc_sw128(sa + k * 32, 16, 1024);
        const uint64_t bd = sdesc_sw128(sb + k * 2048, 8192, 1024);
        umma_bf16(tmem, ad, bd, idesc, (kb > 0 || k > 0) ? 1u : 0u);
      }
      umma_commit(&empty[s]);
    }
    umma_commit(done);
  }
  __syncwarp();

  // ---------------- epilogue: TMEM -> +bias -> bf16 -> global
  const bool ok = !skip && mbar_wait(done, 0, abort_flag, a.st, 103);
  tc_fence_after();
  if (ok && !*abort_flag) {
    const int row = warp * 32 + lane;
    const int i = i0 + row;
    __nv_bfloat16* dst = a.out + (((size_t)b * a.G + g) * a.Nc + i) * a.N;
    for (int c0 = 0; c0 < a.N; c0 += 16) {
      uint32_t r[16];
      tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)c0, r);
      tmem_ld_wait(r);
      if (i < a.Nc) {
        uint32_t pk[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
          pk[j] = pack_bf16x2(__uint_as_float(r[2 * j]) + __ldg(a.bias + c0 + 2 * j),
                              __uint_as_float(r[2 * j + 1]) + __ldg(a.bias + c0 + 2 * j + 1));
        uint4* d4 = reinterpret_cast<uint4*>(dst + c0);
        d4[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        d4[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 256);
}

}  // namespace

size_t compress_smem_bytes(int N) {
  return (size_t)kStages * (kTileM * 128 + (size_t)(N / 64) * 8192) + 1024 + 256;
}

int launch_compress_one(const nsa_cfg& c, int layout, const void* X, int dX, const void* pe, const void* W,
                        void* out, float* bias_ws, DeviceStatus* st, cudaStream_t stream) {
  const int Nc = (c.T < c.l) ? 0 : (c.T - c.l) / c.d + 1;
  if (Nc == 0) return NSA_OK;
  const int N = dX;
  // bias = flatten(PE) @ W
  {
    dim3 grid((N + 31) / 32, kBiasSplit), block(32, kBiasRowsY);
    prof::begin("phi_bias", stream);
    phi_bias_kernel<<<grid, block, 0, stream>>>(static_cast<const __nv_bfloat16*>(pe),
                                                static_cast<const __nv_bfloat16*>(W), c.l * dX, N, bias_ws);
    prof::end(stream);
  }
  CUtensorMap mapA, mapB;
  const uint64_t T16 = (uint64_t)c.T / 16;
  const uint64_t e = 2;  // bytes per element
  if (layout == NSA_LAYOUT_BTGD) {
    const uint64_t dims[5] = {(uint64_t)dX, (uint64_t)c.G, 16, T16, (uint64_t)c.B};
    const uint64_t str[4] = {dX * e, (uint64_t)c.G * dX * e, 16ull * c.G * dX * e, (uint64_t)c.T * c.G * dX * e};
    const uint32_t box[5] = {64, 1, 1, kTileM, 1};
    if (!make_tmap_bf16(&mapA, X, 5, dims, str, box)) return NSA_ERR_CUDA;
  } else {
    const uint64_t dims[5] = {(uint64_t)dX, 16, T16, (uint64_t)c.G, (uint64_t)c.B};
    const uint64_t str[4] = {dX * e, 16ull * dX * e, (uint64_t)c.T * dX * e, (uint64_t)c.G * c.T * dX * e};
    const uint32_t box[5] = {64, 1, kTileM, 1, 1};
    if (!make_tmap_bf16(&mapA, X, 5, dims, str, box)) return NSA_ERR_CUDA;
  }
  {
    const uint64_t dims[2] = {(uint64_t)N, (uint64_t)c.l * dX};
    const uint64_t str[1] = {(uint64_t)N * e};
    const uint32_t box[2] = {64, 64};
    if (!make_tmap_bf16(&mapB, W, 2, dims, str, box)) return NSA_ERR_CUDA;
  }
  CompressArgs a;
  a.Nc = Nc;
  a.N = N;
  a.cpr = dX / 64;
  a.nkb = c.l * a.cpr;
  a.layout = layout;
  a.G = c.G;
  a.stall = (c.flags & NSA_FLAG_TEST_STALL) != 0 ? 1 : 0;
  a.bias = bias_ws;
  a.out = static_cast<__nv_bfloat16*>(out);
  a.st = st;
  const size_t smem = compress_smem_bytes(N);
  if (int rc = ensure_smem_attr(reinterpret_cast<const void*>(&compress_gemm_kernel), smem_max())) return rc;
  dim3 grid((Nc + kTileM - 1) / kTileM, c.G, c.B);
  prof::begin("compress_gemm", stream);
  compress_gemm_kernel<<<grid, 128, smem, stream>>>(mapA, mapB, a);
  prof::end(stream);
  return cudaPeekAtLastError() == cudaSuccess ? NSA_OK : NSA_ERR_CUDA;
}

}  // namespace nsa
