// proj_tc.cu -- row-gathered projections C = A W^T on the 5th-generation
// tensor cores (tcgen05.mma, accumulator in tensor memory).
//
// DCOCO page ("Contextual Correction of Parallel Drafts for Speculative
// Decoding"), Method step details (2)-(3): the embedding rows E[c] of the
// candidates (gathered by token id) and the draft-slot hidden states h_i are
// projected by bias-free maps (W_cand; W_ctx and the two halves of W_pair).
//
// Precision: A (bf16) is exact; each fp32 weight is split into bf16 hi + lo
// (w = hi + lo to ~2^-17 relative), and both products accumulate into the same
// fp32 accumulator: C = A hi^T + A lo^T.
//
// Tile: 128 rows x 128 outputs, k-blocks of 64 (one 128-byte swizzle atom),
// a 4-stage ring in 128B-swizzled K-major shared memory.  Each operand takes
// the path that suits it: warps 0-3 gather the A rows with 16-byte cp.async
// (many small independent rows), one thread of warp 4 brings the hi and lo
// weight blocks as two 2D TMA tiles (large blocks, the same for every CTA);
// a stage is full when the 128 gatherers have arrived and the TMA bytes have
// landed.  One thread of warp 5 (which also owns the tensor-memory
// allocation) issues the MMAs; warps 0-3 then drain the accumulator with
// tcgen05.ld.  Split-K over gridDim.z: every split writes an fp32
// partial tile and the tile's last CTA (atomic counter) adds the partials in
// split order, so the result does not depend on which CTA finished last.
// Every wait is bounded in time; on expiry the kernel records kErrTimeout in
// the device status word and leaves without touching the output.
#include <cuda.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace dc {
namespace {

constexpr int kStages = 4;
constexpr int kTileM = 128, kTileN = 128, kTileK = 64;
constexpr int kTileBytes = kTileM * kTileK * 2;        // 16 KB (A, hi or lo)
constexpr int kStageBytes = 3 * kTileBytes;             // A + hi + lo
constexpr int kGatherThreads = 128;  // warps 0-3: A gather, then epilogue
constexpr int kThreads = 192;        // + warp 4 (weight TMA) + warp 5 (MMA)
constexpr uint32_t kStageTx = 2u * kTileBytes;  // weight bytes per stage
constexpr uint32_t kTmemCols = 128;
constexpr int kMaxSplits = 8;

constexpr uint32_t kIdesc = tc::idesc_bf16(kTileM, kTileN);

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}


using namespace tc;

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1)
k_proj_tc(const uint16_t *__restrict__ table, const __grid_constant__ CUtensorMap map_hi,
          const __grid_constant__ CUtensorMap map_lo, const int32_t *__restrict__ ids, int slots,
          int B, int M, int d, int V, int No, int kb_per_split, float *__restrict__ C,
          float *__restrict__ part, unsigned *__restrict__ tile_count, int *err) {
  extern __shared__ uint8_t smem_raw[];
  // the swizzle atoms need 1024-byte alignment in the shared window
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  __shared__ __align__(8) unsigned long long bar_full[kStages], bar_empty[kStages], bar_done;
  __shared__ int s_rows[kTileM];  // table row of each tile row (A operand)
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ int s_last;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n0 = blockIdx.x * kTileN, m0 = blockIdx.y * kTileM, split = blockIdx.z;
  const int nkb_total = d / kTileK;
  const int kb0 = split * kb_per_split;
  const int nkb = min(kb_per_split, nkb_total - kb0);
  const uint32_t sbase = smem_u32(smem);

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&bar_full[s]), kGatherThreads + 1);
      mbar_init(smem_u32(&bar_empty[s]), 1);
    }
    mbar_init(smem_u32(&bar_done), 1);
    s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (tid < kTileM) {
    const int m = m0 + tid;
    int row = 0;  // rows past M load table row 0; their results are never stored
    if (m < M) {
      if (MODE == 0) {
        row = ids[m];
        if (row < 0 || row >= V) {
          atomicOr(err, kErrBadCandidateId);
          row = 0;
        }
      } else {
        const int n = m / B, i = m - n * B;
        row = n * slots + i + 1;
      }
    }
    s_rows[tid] = row;
  }
  if (warp == 5) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&s_tmem)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;

  int issued = 0;  // stages whose weight TMA this thread issued
  if (warp < 4) {
    // ------------------------------------------------------------ A gather (cp.async)
    const int t = tid;
    const int c = t & 7;              // 16-byte chunk of the 128-byte k-row
    const int rq = (t >> 3) & 7;      // row within an 8-row swizzle group
    const uint32_t off0 = (uint32_t)((t >> 6) * 1024 + rq * 128 + ((c ^ rq) * 16));
    const uint16_t *arow[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) arow[j] = table + (int64_t)s_rows[(t >> 3) + 16 * j] * d + c * 8;
    int it = 0;
    for (; it < nkb; ++it) {
      const int s = it % kStages;
      if (it >= kStages &&
          !mbar_wait(smem_u32(&bar_empty[s]), ((it / kStages) - 1) & 1, &s_abort, err))
        break;
      const int kel = (kb0 + it) * kTileK;
      const uint32_t sa = sbase + s * kStageBytes + off0;
#pragma unroll
      for (int j = 0; j < 8; ++j) cp_async16(sa + j * 2048, arow[j] + kel);
      cp_async_commit();
      if (it >= kStages - 1) {
        cp_async_wait<kStages - 1>();
        fence_proxy_async();
        mbar_arrive(smem_u32(&bar_full[(it - (kStages - 1)) % kStages]));
      }
    }
    cp_async_wait<0>();
    fence_proxy_async();
    for (int r = max(0, it - (kStages - 1)); r < it; ++r) mbar_arrive(smem_u32(&bar_full[r % kStages]));
  } else if (warp == 4) {
    if (lane == 0) {
      // ------------------------------------------------------------ weight TMA
      for (int it = 0; it < nkb; ++it, ++issued) {
        const int s = it % kStages;
        if (it >= kStages &&
            !mbar_wait(smem_u32(&bar_empty[s]), ((it / kStages) - 1) & 1, &s_abort, err))
          break;
        const uint32_t full = smem_u32(&bar_full[s]);
        const uint32_t sa = sbase + s * kStageBytes;
        const int kx = (kb0 + it) * kTileK;
        mbar_arrive_expect_tx(full, kStageTx);
        tma_load_2d(sa + kTileBytes, &map_hi, kx, n0, full);
        tma_load_2d(sa + 2 * kTileBytes, &map_lo, kx, n0, full);
      }
    }
  } else if (warp == 5 && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    for (int it = 0; it < nkb; ++it) {
      const int s = it % kStages;
      if (!mbar_wait(smem_u32(&bar_full[s]), (it / kStages) & 1, &s_abort, err)) break;
      tc_fence_after();
      const uint32_t sa = sbase + s * kStageBytes;
#pragma unroll
      for (int k = 0; k < kTileK / 16; ++k) {
        const uint64_t ad = sw128_desc(sa + k * 32);
        mma_bf16(tmem, ad, sw128_desc(sa + kTileBytes + k * 32), kIdesc, (it > 0 || k > 0) ? 1u : 0u);
        mma_bf16(tmem, ad, sw128_desc(sa + 2 * kTileBytes + k * 32), kIdesc, 1u);
      }
      mma_commit(smem_u32(&bar_empty[s]));
    }
    mma_commit(smem_u32(&bar_done));
  }
  __syncwarp();

  // ---------------------------------------------------------------- epilogue
  const bool split_k = gridDim.z > 1;
  if (warp < 4) {
    bool ok = mbar_wait(smem_u32(&bar_done), 0, &s_abort, err) && !s_abort;
    ok = __all_sync(DC_FULL_MASK, ok);  // tcgen05.ld below is warp-collective
    tc_fence_after();
    if (ok) {
      const int row = m0 + warp * 32 + lane;
      float *dst = split_k ? part + ((int64_t)split * gridDim.y * kTileM + row) * No + n0
                           : C + (int64_t)row * No + n0;
#pragma unroll 1
      for (int cc = 0; cc < kTileN / 32; ++cc) {
        float v[32];
        tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(cc * 32), v);
        if (row < M || split_k) {
          float4 *d4 = reinterpret_cast<float4 *>(dst + cc * 32);
#pragma unroll
          for (int q = 0; q < 8; ++q) d4[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (s_abort) {
    // a wait expired: let everything already issued land before leaving
    if (warp == 4 && lane == 0)
      for (int s = 0; s < kStages && s < issued; ++s) {
        const int last = s + kStages * ((issued - 1 - s) / kStages);
        mbar_drain(smem_u32(&bar_full[s]), (last / kStages) & 1);
      }
    if (warp == 5 && lane == 0) mbar_drain(smem_u32(&bar_done), 0);
    __syncthreads();
  }
  if (warp == 5) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols)
                 : "memory");
  }
  if (!split_k || s_abort) return;

  // ---------------------------------------------------------------- split-K reduction
  __threadfence();
  __syncthreads();
  const int tile = blockIdx.y * gridDim.x + blockIdx.x;
  if (tid == 0) s_last = (atomicAdd(&tile_count[tile], 1u) == gridDim.z - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const int rows = min(kTileM, M - m0);
  const int64_t pstride = (int64_t)gridDim.y * kTileM * No;
  const int nz = (int)gridDim.z;  // <= kMaxSplits
  for (int e = tid; e < rows * (kTileN / 4); e += kThreads) {
    const int r = e / (kTileN / 4), q = e - r * (kTileN / 4);
    const int64_t off = (int64_t)(m0 + r) * No + n0 + q * 4;
    float4 p[kMaxSplits];
#pragma unroll
    for (int z = 0; z < kMaxSplits; ++z)  // every partial load in flight at once
      if (z < nz) p[z] = __ldcg(reinterpret_cast<const float4 *>(part + z * pstride + off));
    float4 acc = p[0];
#pragma unroll
    for (int z = 1; z < kMaxSplits; ++z)
      if (z < nz) {
        acc.x += p[z].x; acc.y += p[z].y; acc.z += p[z].z; acc.w += p[z].w;
      }
    *reinterpret_cast<float4 *>(C + off) = acc;
  }
  if (tid == 0) tile_count[tile] = 0u;
}

}  // namespace

size_t proj_tc_smem_bytes() { return (size_t)kStages * kStageBytes + 1024; }

int proj_tc_splits(int d, int requested) {
  const int nkb = d / kTileK;
  int s = std::max(1, std::min(std::min(requested, kMaxSplits), nkb));
  const int per = (nkb + s - 1) / s;
  return (nkb + per - 1) / per;  // no empty split
}

namespace {
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
    else
      cudaGetLastError();
  }
  return fn;
}
}  // namespace

bool encode_bf16_rows_map(CUtensorMap *map, const void *base, int rows, int d, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || rows <= 0 || d % kTileK != 0 || (reinterpret_cast<uintptr_t>(base) & 15u)) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)d * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kTileK, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_f32_rows_map(CUtensorMap *map, const void *base, int rows, int cols, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || rows <= 0 || cols % 32 != 0 || (reinterpret_cast<uintptr_t>(base) & 15u)) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * 4};
  const cuuint32_t box[2] = {32, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void *>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_proj_tc(int mode, const uint16_t *table, const CUtensorMap &map_hi,
                           const CUtensorMap &map_lo, const int32_t *ids, int slots, int B, int M, int d,
                           int V, int No, int splits, float *C, float *part, unsigned *tile_count,
                           int *err, cudaStream_t st) {
  if (M == 0) return cudaSuccess;
  if (No % kTileN != 0 || d % kTileK != 0 || splits < 1 || splits > kMaxSplits) return cudaErrorInvalidValue;
  const int nkb = d / kTileK;
  const int per = (nkb + splits - 1) / splits;
  dim3 grid(No / kTileN, (M + kTileM - 1) / kTileM, splits);
  const size_t smem = proj_tc_smem_bytes();
  cudaError_t e;
  if (mode == 0) {
    e = cudaFuncSetAttribute(k_proj_tc<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    k_proj_tc<0><<<grid, kThreads, smem, st>>>(table, map_hi, map_lo, ids, slots, B, M, d, V, No, per, C,
                                              part, tile_count, err);
  } else {
    e = cudaFuncSetAttribute(k_proj_tc<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    k_proj_tc<1><<<grid, kThreads, smem, st>>>(table, map_hi, map_lo, ids, slots, B, M, d, V, No, per, C,
                                              part, tile_count, err);
  }
  return cudaGetLastError();
}

}  // namespace dc
