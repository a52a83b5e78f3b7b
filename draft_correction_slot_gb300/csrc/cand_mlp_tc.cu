// cand_mlp_tc.cu -- per-candidate LayerNorms, fuse map and layer-1 partial
// products on the tensor cores.
//
// DCOCO page ("Contextual Correction of Parallel Drafts for Speculative
// Decoding"), Method step details (2) and (4):
//   b = LN(W_cand E[c])                       (non-affine; W_cand E[c] = cand_proj)
//   z = gamma * LN(W_fuse[:, :r] b + W_fuse[:, r:] g_i) + beta
//   U = W1[:, r:2r] z + W1[:, 3r] l(c),  V = W1[:, 2r:3r] z + W1[:, 3r+1] l(c)
// (U feeds the candidate's transitions as predecessor, V as successor.)
//
// One CTA per (128-candidate tile, half): half 0 writes U, half 1 writes V;
// both recompute z (a 128x128 map, cheap).  Both maps are dense 128-deep
// contractions: A (b, then z) is split in registers into bf16 hi + lo and
// stored 128B-swizzled, the weights come pre-split through TMA, and three MMA
// passes (hi.hi + hi.lo + lo.hi) accumulate in fp32 tensor memory, which
// keeps fp32-level accuracy.  Warps 0-3 own one candidate row per thread
// (= tensor-memory lane); one thread of warp 4 issues the TMA copies and
// MMAs.  Every wait is bounded in time (kErrTimeout in the status word).
#include <cuda_bf16.h>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace dc {
namespace {

using namespace tc;

constexpr int kR = 128, kH = 256;
constexpr int kRows = 128;                 // candidates per CTA (MMA M)
constexpr int kKBlk = 128 * 64 * 2;        // 128 rows x 64 k of bf16: 16 KB
constexpr int kMat = 2 * kKBlk;            // 128 rows x 128 k: 32 KB
// shared memory: A (hi, lo) | W0: W_fuse[:, :r] (hi, lo), later W1 chunk 1 | W1: W1 chunk 0
constexpr int kOffA = 0, kOffW0 = 2 * kMat, kOffW1 = 4 * kMat;
constexpr int kSmemBytes = 6 * kMat + 1024;
constexpr int kThreads = 160;
constexpr uint32_t kTmemCols = 512;        // [0,128) fuse, [128,256) chunk 0, [256,384) chunk 1
constexpr uint32_t kIdesc = idesc_bf16(128, 128);
constexpr uint32_t kWTx = 2 * kMat;        // one matrix pair (hi + lo): 64 KB

__device__ __forceinline__ uint32_t bf16_rn_bits(float f) {
  return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// Store row r (128 values) as bf16 hi and lo into the 128B-swizzled K-major
// A tiles (two 64-wide k-blocks each).
__device__ __forceinline__ void store_split_row(uint8_t *a_hi, uint8_t *a_lo, int r, const float (&x)[kR]) {
#pragma unroll
  for (int kb = 0; kb < 2; ++kb) {
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      uint32_t hw[4], lw[4];
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        const float v0 = x[kb * 64 + c * 8 + 2 * p], v1 = x[kb * 64 + c * 8 + 2 * p + 1];
        const uint32_t h0 = bf16_rn_bits(v0), h1 = bf16_rn_bits(v1);
        const uint32_t l0 = bf16_rn_bits(v0 - __uint_as_float(h0 << 16));
        const uint32_t l1 = bf16_rn_bits(v1 - __uint_as_float(h1 << 16));
        hw[p] = h0 | (h1 << 16);
        lw[p] = l0 | (l1 << 16);
      }
      const int off = kb * kKBlk + (r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) * 16);
      *reinterpret_cast<uint4 *>(a_hi + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
      *reinterpret_cast<uint4 *>(a_lo + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
    }
  }
}

__device__ __forceinline__ void ln0_inplace(float (&x)[kR], float eps) {
  float s = 0.f;
#pragma unroll
  for (int k = 0; k < kR; ++k) s += x[k];
  const float mean = s * (1.0f / kR);
  float q = 0.f;
#pragma unroll
  for (int k = 0; k < kR; ++k) {
    x[k] -= mean;
    q = fmaf(x[k], x[k], q);
  }
  const float inv = rsqrtf(q * (1.0f / kR) + eps);
#pragma unroll
  for (int k = 0; k < kR; ++k) x[k] *= inv;
}

// 3-pass split product of one 128-deep contraction into tmem columns `col`.
__device__ __forceinline__ void mma_split(uint32_t tmem, uint32_t a_hi, uint32_t a_lo, uint32_t w_hi,
                                          uint32_t w_lo) {
#pragma unroll
  for (int kb = 0; kb < 2; ++kb)
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t o = kb * kKBlk + k * 32;
      const uint64_t ah = sw128_desc(a_hi + o), al = sw128_desc(a_lo + o);
      mma_bf16(tmem, ah, sw128_desc(w_hi + o), kIdesc, (kb | k) ? 1u : 0u);
      mma_bf16(tmem, ah, sw128_desc(w_lo + o), kIdesc, 1u);
      mma_bf16(tmem, al, sw128_desc(w_hi + o), kIdesc, 1u);
    }
}

__global__ void __launch_bounds__(kThreads, 1)
k_cand_mlp_tc(const __grid_constant__ CUtensorMap map_fb_hi, const __grid_constant__ CUtensorMap map_fb_lo,
              const __grid_constant__ CUtensorMap map_w1_hi, const __grid_constant__ CUtensorMap map_w1_lo,
              const float *__restrict__ cand_proj, const float *__restrict__ Gf,
              const float *__restrict__ topk_val, const float *__restrict__ gamma,
              const float *__restrict__ beta, const float *__restrict__ w_la,
              const float *__restrict__ w_lb, int K, int M, float eps, float *__restrict__ U,
              float *__restrict__ Vout, int *err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  __shared__ __align__(8) unsigned long long bar_w0, bar_w1, bar_w2, bar_a, bar_fuse, bar_a2, bar_uv0,
      bar_uv1;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int half = blockIdx.x, m0 = blockIdx.y * kRows;
  const uint32_t sb = smem_u32(smem);
  const uint32_t a_hi = sb + kOffA, a_lo = sb + kOffA + kMat;
  const uint32_t w0_hi = sb + kOffW0, w0_lo = sb + kOffW0 + kMat;
  const uint32_t w1_hi = sb + kOffW1, w1_lo = sb + kOffW1 + kMat;

  if (tid == 0) {
    mbar_init(smem_u32(&bar_w0), 1);
    mbar_init(smem_u32(&bar_w1), 1);
    mbar_init(smem_u32(&bar_w2), 1);
    mbar_init(smem_u32(&bar_a), kRows);
    mbar_init(smem_u32(&bar_fuse), 1);
    mbar_init(smem_u32(&bar_a2), kRows);
    mbar_init(smem_u32(&bar_uv0), 1);
    mbar_init(smem_u32(&bar_uv1), 1);
    s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 4) tmem_alloc(smem_u32(&s_tmem), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  const int wrow0 = half * kH;  // first W1 row of this half (W1_a or W1_b block)
  bool w2_issued = false;

  if (warp == 4) {
    if (lane == 0) {
      // ------------------------------------------------------------ control thread
      mbar_arrive_expect_tx(smem_u32(&bar_w0), kWTx);
      for (int kb = 0; kb < 2; ++kb) {
        tma_load_2d(w0_hi + kb * kKBlk, &map_fb_hi, kb * 64, 0, smem_u32(&bar_w0));
        tma_load_2d(w0_lo + kb * kKBlk, &map_fb_lo, kb * 64, 0, smem_u32(&bar_w0));
      }
      mbar_arrive_expect_tx(smem_u32(&bar_w1), kWTx);
      for (int kb = 0; kb < 2; ++kb) {
        tma_load_2d(w1_hi + kb * kKBlk, &map_w1_hi, kb * 64, wrow0, smem_u32(&bar_w1));
        tma_load_2d(w1_lo + kb * kKBlk, &map_w1_lo, kb * 64, wrow0, smem_u32(&bar_w1));
      }
      // y = W_fuse[:, :r] b
      if (mbar_wait(smem_u32(&bar_w0), 0, &s_abort, err) && mbar_wait(smem_u32(&bar_a), 0, &s_abort, err)) {
        tc_fence_after();
        mma_split(tmem, a_hi, a_lo, w0_hi, w0_lo);
      }
      mma_commit(smem_u32(&bar_fuse));
      // once the fuse MMAs have read W0, bring W1 chunk 1 into it
      if (mbar_wait(smem_u32(&bar_fuse), 0, &s_abort, err)) {
        mbar_arrive_expect_tx(smem_u32(&bar_w2), kWTx);
        for (int kb = 0; kb < 2; ++kb) {
          tma_load_2d(w0_hi + kb * kKBlk, &map_w1_hi, kb * 64, wrow0 + 128, smem_u32(&bar_w2));
          tma_load_2d(w0_lo + kb * kKBlk, &map_w1_lo, kb * 64, wrow0 + 128, smem_u32(&bar_w2));
        }
        w2_issued = true;
      }
      // chunk 0 and chunk 1 of this half of layer 1
      if (mbar_wait(smem_u32(&bar_a2), 0, &s_abort, err) && mbar_wait(smem_u32(&bar_w1), 0, &s_abort, err)) {
        tc_fence_after();
        mma_split(tmem + 128, a_hi, a_lo, w1_hi, w1_lo);
      }
      mma_commit(smem_u32(&bar_uv0));
      if (w2_issued && mbar_wait(smem_u32(&bar_w2), 0, &s_abort, err)) {
        tc_fence_after();
        mma_split(tmem + 256, a_hi, a_lo, w0_hi, w0_lo);
      }
      mma_commit(smem_u32(&bar_uv1));
    }
    __syncwarp();
  } else {
    // -------------------------------------------------------------- row threads
    const int r = tid;  // tile row = tensor-memory lane
    const int m = m0 + r;
    const bool live = m < M;
    float x[kR];
    // b = LN0(cand_proj row)
    if (live) {
      const float4 *src = reinterpret_cast<const float4 *>(cand_proj + (int64_t)m * kR);
#pragma unroll
      for (int q = 0; q < kR / 4; ++q) {
        const float4 v = __ldg(src + q);
        x[4 * q] = v.x; x[4 * q + 1] = v.y; x[4 * q + 2] = v.z; x[4 * q + 3] = v.w;
      }
      ln0_inplace(x, eps);
    } else {
#pragma unroll
      for (int k = 0; k < kR; ++k) x[k] = 0.f;
    }
    store_split_row(smem + kOffA, smem + kOffA + kMat, r, x);
    fence_proxy_async();
    mbar_arrive(smem_u32(&bar_a));

    // z = gamma * LN0(y + Gf[slot]) + beta
    bool ok = mbar_wait(smem_u32(&bar_fuse), 0, &s_abort, err) && !s_abort;
    ok = __all_sync(DC_FULL_MASK, ok);
    tc_fence_after();
    if (ok) {
      const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        float v[32];
        tmem_ld32(lane_base + cc * 32, v);
#pragma unroll
        for (int k = 0; k < 32; ++k) x[cc * 32 + k] = v[k];
      }
      if (live) {
        const float4 *gf = reinterpret_cast<const float4 *>(Gf + (int64_t)(m / K) * kR);
#pragma unroll
        for (int q = 0; q < kR / 4; ++q) {
          const float4 g = __ldg(gf + q);
          x[4 * q] += g.x; x[4 * q + 1] += g.y; x[4 * q + 2] += g.z; x[4 * q + 3] += g.w;
        }
        ln0_inplace(x, eps);
#pragma unroll
        for (int k = 0; k < kR; ++k) x[k] = fmaf(__ldg(gamma + k), x[k], __ldg(beta + k));
      } else {
#pragma unroll
        for (int k = 0; k < kR; ++k) x[k] = 0.f;
      }
      store_split_row(smem + kOffA, smem + kOffA + kMat, r, x);
    }
    fence_proxy_async();
    mbar_arrive(smem_u32(&bar_a2));

    // U (or V) = W1 z + w_l l
    const float *wl = half == 0 ? w_la : w_lb;
    float *dst = (half == 0 ? U : Vout) + (int64_t)m * kH;
    const float lv = live ? __ldg(topk_val + m) : 0.f;
#pragma unroll 1
    for (int ch = 0; ch < 2; ++ch) {
      bool ok2 = mbar_wait(smem_u32(ch == 0 ? &bar_uv0 : &bar_uv1), 0, &s_abort, err) && !s_abort;
      ok2 = __all_sync(DC_FULL_MASK, ok2);
      tc_fence_after();
      if (!ok2) break;
      const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16) + 128u * (1 + ch);
#pragma unroll 1
      for (int cc = 0; cc < 4; ++cc) {
        float v[32];
        tmem_ld32(lane_base + cc * 32, v);
        if (live) {
          const int j0 = ch * 128 + cc * 32;
          float4 *d4 = reinterpret_cast<float4 *>(dst + j0);
#pragma unroll
          for (int q = 0; q < 8; ++q)
            d4[q] = make_float4(fmaf(__ldg(wl + j0 + 4 * q), lv, v[4 * q]),
                                fmaf(__ldg(wl + j0 + 4 * q + 1), lv, v[4 * q + 1]),
                                fmaf(__ldg(wl + j0 + 4 * q + 2), lv, v[4 * q + 2]),
                                fmaf(__ldg(wl + j0 + 4 * q + 3), lv, v[4 * q + 3]));
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (s_abort && warp == 4 && lane == 0) {
    // a wait expired: let the copies and MMAs already issued land first
    mbar_drain(smem_u32(&bar_w0), 0);
    mbar_drain(smem_u32(&bar_w1), 0);
    if (w2_issued) mbar_drain(smem_u32(&bar_w2), 0);
    mbar_drain(smem_u32(&bar_uv1), 0);
  }
  __syncthreads();
  if (warp == 4) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

cudaError_t launch_cand_mlp_tc(const CandMlpMaps &maps, const float *cand_proj, const float *Gf,
                               const float *topk_val, const MlpWeightsDev &w, int K, int M, float eps,
                               float *U, float *V, int *err, cudaStream_t st) {
  if (M == 0) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(k_cand_mlp_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kSmemBytes);
  if (e != cudaSuccess) return e;
  dim3 grid(2, (M + kRows - 1) / kRows);
  k_cand_mlp_tc<<<grid, kThreads, kSmemBytes, st>>>(maps.fb_hi, maps.fb_lo, maps.w1_hi, maps.w1_lo,
                                                    cand_proj, Gf, topk_val, w.gamma, w.beta, w.w_la,
                                                    w.w_lb, K, M, eps, U, V, err);
  return cudaGetLastError();
}

}  // namespace dc
