// proj_tc.cu -- row-gathered projections C = A W^T on the 5th-generation
// tensor cores (tcgen05.mma, accumulator in tensor memory).
//
// DCOCO page ("Contextual Correction of Parallel Drafts for Speculative
// Decoding"), Method step details (2)-(3): the embedding rows E[c] of the
// candidates (gathered by token id) and the draft-slot hidden states h_i are
// projected by bias-free maps (W_cand; W_ctx and the two halves of W_pair).
//
// Precision: A (bf16) is exact; each fp32 weight is split into bf16 hi + lo
// (w = hi + lo to ~2^-17 relative).  The hi and lo blocks of a k-block sit
// one after the other in shared memory, so one N = 256 MMA takes both: its
// accumulator holds A hi^T in columns [0, 128) and A lo^T in [128, 256), and
// the epilogue adds the two (fp32).  One N = 256 instruction reads the A
// block once for both halves.  A job may instead run in fp16 (the candidate
// rows: each gathered bf16 row is converted in shared memory, exactly inside
// the fp16 range, and the weights are rounded to fp16 once, 2^-11 relative):
// one N = 128 MMA per k-step, half the tensor work and weight bytes, within
// the score tolerance (the LayerNorm after the product keeps the error
// relative).
//
// Tile: 256 rows (two 128-row accumulators) x 128 outputs, k-blocks of 64
// (one 128-byte swizzle atom) in 128B-swizzled K-major shared memory.  Each
// operand takes the path that suits it: warps 0-7 gather the A rows with
// 16-byte cp.async into a 4-deep ring (many small independent rows from HBM:
// the depth keeps enough bytes in flight), one thread of warp 8 brings the hi
// and lo weight blocks as two 2D TMA tiles into a 3-deep ring (the same
// blocks for every CTA, served from L2).  One thread of warp 9 (which also
// owns the tensor-memory allocation) issues the MMAs once both rings hold the
// k-block; warps 0-7 then drain the accumulators with tcgen05.ld into shared
// memory.
// Split-K over gridDim.z: the splits of a tile form one thread-block
// cluster and add their partial tiles through distributed shared memory in
// split order, so the result does not depend on timing.
// One launch serves up to two products ("jobs": the candidate rows and the
// draft-slot rows), their tiles listed one after the other along gridDim.y,
// so that both fill the device in a single wave.  Draft-slot tiles depend on
// nothing the previous kernel writes and start without waiting for it.
// A job may ask for its rows LayerNormed instead (non-affine, the step (2)
// normalisation of the candidate representation): the reduction holds each
// finished 128-wide row in one warp, normalises it there and stores it as
// bf16 hi + lo, the operand format of the next map's tensor-core product.
// Every wait is bounded in time; on expiry the kernel records kErrTimeout in
// the device status word and does not store its rows.
#include <cuda.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"
#include "launch.h"

namespace dc {
namespace {

constexpr int kTileN = 128, kTileK = 64;
constexpr int kSubM = 128;                             // rows per accumulator (MMA M)
constexpr int kSubBytes = kSubM * kTileK * 2;          // 16 KB: 128 rows x 64 k of bf16
constexpr uint32_t kStageTx = 2u * kSubBytes;          // weight bytes per k-block (hi + lo)
constexpr int kMaxSplits = 8;       // a cluster of at most 8 CTAs (portable size)
constexpr int kBoxBytes = kSubM * 128;  // one 32-column fp32 box of a 128-row output tile
constexpr uint32_t kIdesc = tc::idesc_bf16(kSubM, 2 * kTileN);  // hi and lo blocks stacked
constexpr uint32_t kIdescF16 = tc::idesc_f16(kSubM, kTileN);     // one fp16 weight block

// A CTA owns MT x 128 rows (MT accumulators of 128 x 128 in tensor memory)
// so that every weight k-block it brings in feeds MT MMAs.  Two rings: the
// gathered A rows come from HBM (long latency: a deep ring keeps enough bytes
// in flight), the weights from L2 (a shorter ring suffices).
template <int MT>
struct ProjGeom {
  static constexpr int kTileM = MT * kSubM;
  static constexpr int kGather = MT * 128;               // gather threads (warps 0 .. 4 MT - 1)
  static constexpr int kThreads = kGather + 64;          // + weight-TMA warp + MMA warp
  static constexpr int kWarpTma = 4 * MT, kWarpMma = 4 * MT + 1;
  static constexpr int kStageA = MT * kSubBytes;
  static constexpr int kStagesA = MT == 1 ? 8 : 4, kStagesW = 3;
  static constexpr int kRingA = kStagesA * kStageA;      // A ring, then the W ring
  static constexpr int kSmemUsed = kRingA + kStagesW * 2 * kSubBytes;
  static constexpr uint32_t kTmemCols = MT * 256;  // per accumulator: hi products, then lo
  static_assert(kSmemUsed + 1024 <= 227 * 1024 - 1024, "shared memory");
  static_assert(MT * 4 * kBoxBytes <= kSmemUsed, "the output tile is staged in the (idle) rings");
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}


using namespace tc;

// The 16-byte chunks this thread gathered into one A stage (rows 16 j
// apart), bf16 -> fp16 in place (round to nearest; every bf16 value within
// the fp16 range below 65504 is exact down to 2^-14 and rounded to 2^-24
// below).
__device__ __forceinline__ void convert_chunks_f16(uint32_t addr0) {
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint32_t a = addr0 + j * 2048;
    uint32_t w[4];
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]) : "r"(a));
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float lo = __uint_as_float(w[q] << 16), hi = __uint_as_float(w[q] & 0xFFFF0000u);
      asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(w[q]) : "f"(hi), "f"(lo));
    }
    asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(a), "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3])
                 : "memory");
  }
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Address of the same shared-memory location in cluster CTA `rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t saddr, int rank) {
  uint32_t d;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(d) : "r"(saddr), "r"(rank));
  return d;
}
__device__ __forceinline__ float4 ld_dsmem_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

template <int MT>
__global__ void __launch_bounds__(ProjGeom<MT>::kThreads, 1)
k_proj_tc(ProjJob job0, ProjJob job1, const __grid_constant__ CUtensorMap map0_hi,
          const __grid_constant__ CUtensorMap map0_lo, const __grid_constant__ CUtensorMap map1_hi,
          const __grid_constant__ CUtensorMap map1_lo, int slots, int B, int d, int V, int kb_per_split,
          int *err) {
  using G = ProjGeom<MT>;
  constexpr int kTileM = G::kTileM, kStagesA = G::kStagesA, kStagesW = G::kStagesW;
  extern __shared__ uint8_t smem_raw[];
  // the swizzle atoms need 1024-byte alignment in the shared window
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  __shared__ __align__(8) unsigned long long full_a[kStagesA], empty_a[kStagesA], full_w[kStagesW],
      empty_w[kStagesW], bar_done;
  __shared__ int s_rows[kTileM];  // table row of each tile row (A operand)
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // this CTA's job and tile: job 0's tiles come first along y
  const bool second = (int)blockIdx.y >= job0.tiles;
  const ProjJob &job = second ? job1 : job0;
  const CUtensorMap *map_hi = second ? &map1_hi : &map0_hi;
  const CUtensorMap *map_lo = second ? &map1_lo : &map0_lo;
  const int tile = (int)blockIdx.y - (second ? job0.tiles : 0);
  const int ntn = job.No / kTileN;
  const int n0 = (tile % ntn) * kTileN, m0 = (tile / ntn) * kTileM, split = blockIdx.z;
  const int M = job.M, No = job.No;
  const uint16_t *__restrict__ table = job.table;
  const int32_t *__restrict__ ids = job.ids;
  float *__restrict__ C = job.C;
  uint16_t *__restrict__ ln_hi = job.ln_hi;
  uint16_t *__restrict__ ln_lo = job.ln_lo;
  const float ln_eps = job.ln_eps;
  const bool f16 = job.f16;
  // candidate rows [m0, m0 + kTileM) come from draft-slot rows row_first..row_last
  const int row_first = job.row_ready ? m0 / job.cands_per_row : 0;
  const int row_last = job.row_ready ? (min(m0 + kTileM, M) - 1) / job.cands_per_row : -1;
  const int nkb_total = d / kTileK;
  const int kb0 = split * kb_per_split;
  const int nkb = min(kb_per_split, nkb_total - kb0);
  const uint32_t sbase = smem_u32(smem);
  pdl_trigger();

  if (tid == 0) {
    for (int s = 0; s < kStagesA; ++s) {
      mbar_init(smem_u32(&full_a[s]), G::kGather);
      mbar_init(smem_u32(&empty_a[s]), 1);
    }
    for (int s = 0; s < kStagesW; ++s) {
      mbar_init(smem_u32(&full_w[s]), 1);
      mbar_init(smem_u32(&empty_w[s]), 1);
    }
    mbar_init(smem_u32(&bar_done), 1);
    s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == G::kWarpMma) tmem_alloc(smem_u32(&s_tmem), G::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;

  int issued = 0;  // stages whose weight TMA this thread issued
  if (warp < 4 * MT) {
    // ------------------------------------------------------------ A gather (cp.async)
    // The row table first.  A gathered job's row ids come from the previous
    // kernel; a draft-slot job reads only the call's inputs and writes a
    // buffer no earlier kernel of the call touches, so it need not wait.  (The
    // weight stream below starts at once either way.)
    static_assert(G::kGather == kTileM, "one gather thread per tile row");
    if (ids && job.row_ready) {
      // the tile's draft-slot rows, one waiting thread each: the streaming
      // top-K releases each row's flag once its ids are stored
      if (tid <= row_last - row_first &&
          !wait_flag(job.row_ready + row_first + tid, &s_abort, err))
        s_abort = 1;
      asm volatile("bar.sync 1, %0;" ::"n"(G::kGather) : "memory");
    } else if (ids) {
      pdl_wait();
    }
    {
      const int m = m0 + tid;
      int row = 0;  // rows past M load table row 0; their results are never stored
      if (m < M) {
        if (ids) {
          row = __ldcg(ids + m);  // the previous kernel's output: via L2
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
    asm volatile("bar.sync 1, %0;" ::"n"(G::kGather) : "memory");  // the gather threads only
    // thread t: 16-byte chunk c of the 128-byte k-row, rows (t >> 3) + 16 j of
    // its 128-row sub-tile t >> 7
    const int t = tid & 127, sub = tid >> 7;
    const int c = t & 7;              // 16-byte chunk of the 128-byte k-row
    const int rq = (t >> 3) & 7;      // row within an 8-row swizzle group
    const uint32_t off0 = (uint32_t)(sub * kSubBytes + (t >> 6) * 1024 + rq * 128 + ((c ^ rq) * 16));
    const uint16_t *arow[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) arow[j] = table + (int64_t)s_rows[sub * 128 + (t >> 3) + 16 * j] * d + c * 8;
    int it = 0;
    for (; it < nkb; ++it) {
      const int s = it % kStagesA;
      if (it >= kStagesA &&
          !mbar_wait(smem_u32(&empty_a[s]), ((it / kStagesA) - 1) & 1, &s_abort, err))
        break;
      const int kel = (kb0 + it) * kTileK;
      const uint32_t sa = sbase + s * G::kStageA + off0;
#pragma unroll
      for (int j = 0; j < 8; ++j) cp_async16(sa + j * 2048, arow[j] + kel);
      cp_async_commit();
      if (it >= kStagesA - 1) {
        cp_async_wait<kStagesA - 1>();
        const int r = it - (kStagesA - 1);
        if (f16) convert_chunks_f16(sbase + (r % kStagesA) * G::kStageA + off0);
        fence_proxy_async();
        mbar_arrive(smem_u32(&full_a[r % kStagesA]));
      }
    }
    cp_async_wait<0>();
    for (int r = max(0, it - (kStagesA - 1)); r < it; ++r) {
      if (f16) convert_chunks_f16(sbase + (r % kStagesA) * G::kStageA + off0);
      fence_proxy_async();
      mbar_arrive(smem_u32(&full_a[r % kStagesA]));
    }
  } else if (warp == G::kWarpTma) {
    if (lane == 0) {
      // ------------------------------------------------------------ weight TMA
      for (int it = 0; it < nkb; ++it, ++issued) {
        const int s = it % kStagesW;
        if (it >= kStagesW &&
            !mbar_wait(smem_u32(&empty_w[s]), ((it / kStagesW) - 1) & 1, &s_abort, err))
          break;
        const uint32_t full = smem_u32(&full_w[s]);
        const uint32_t sw = sbase + G::kRingA + s * 2 * kSubBytes;
        const int kx = (kb0 + it) * kTileK;
        mbar_arrive_expect_tx(full, f16 ? (uint32_t)kSubBytes : kStageTx);
        tma_load_2d(sw, map_hi, kx, n0, full);
        if (!f16) tma_load_2d(sw + kSubBytes, map_lo, kx, n0, full);
      }
    }
  } else if (warp == G::kWarpMma && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    for (int it = 0; it < nkb; ++it) {
      const int s = it % kStagesA, t = it % kStagesW;
      if (!mbar_wait(smem_u32(&full_a[s]), (it / kStagesA) & 1, &s_abort, err) ||
          !mbar_wait(smem_u32(&full_w[t]), (it / kStagesW) & 1, &s_abort, err))
        break;
      tc_fence_after();
      const uint32_t sa = sbase + s * G::kStageA, sw = sbase + G::kRingA + t * 2 * kSubBytes;
#pragma unroll
      for (int k = 0; k < kTileK / 16; ++k) {
        // bf16: B = 256 rows, the hi block's 128, then the lo block's (16 KB
        // further, the next 8-row groups at the descriptor's 1024-byte
        // stride); fp16: the one weight block, N = 128
        const uint64_t bd = sw128_desc(sw + k * 32);
#pragma unroll
        for (int h = 0; h < MT; ++h) {
          const uint64_t ad = sw128_desc(sa + h * kSubBytes + k * 32);
          mma_bf16(tmem + h * 256, ad, bd, f16 ? kIdescF16 : kIdesc, (it > 0 || k > 0) ? 1u : 0u);
        }
      }
      mma_commit(smem_u32(&empty_a[s]));
      mma_commit(smem_u32(&empty_w[t]));
    }
    mma_commit(smem_u32(&bar_done));
  }
  __syncwarp();

  // ---------------------------------------------------------------- epilogue
  // The accumulators go to shared memory (the A ring is idle once bar_done
  // fired), each as four 32-column fp32 boxes, 128-byte swizzled so that the
  // row threads' 16-byte stores and the reducers' reads are conflict-free.
  if (warp < 4 * MT) {
    bool ok = mbar_wait(smem_u32(&bar_done), 0, &s_abort, err) && !s_abort;
    ok = __all_sync(DC_FULL_MASK, ok);  // tcgen05.ld below is warp-collective
    tc_fence_after();
    if (ok) {
      const int sub = warp >> 2, q4 = warp & 3;  // accumulator, lane quadrant
      const int r = q4 * 32 + lane;              // row within the accumulator
#pragma unroll 1
      for (int cc = 0; cc < kTileN / 32; ++cc) {
        float v[32], vl[32];
        const uint32_t t0 = tmem + ((uint32_t)(q4 * 32) << 16) + (uint32_t)(sub * 256 + cc * 32);
        tmem_ld32(t0, v);
        if (!f16) {
          tmem_ld32(t0 + 128, vl);
#pragma unroll
          for (int k = 0; k < 32; ++k) v[k] += vl[k];
        }
        if (nkb <= 0)  // an empty split holds no products
#pragma unroll
          for (int k = 0; k < 32; ++k) v[k] = 0.f;
        uint8_t *box = smem + (sub * 4 + cc) * kBoxBytes + r * 128;
#pragma unroll
        for (int q = 0; q < 8; ++q)
          *reinterpret_cast<float4 *>(box + ((q ^ (r & 7)) * 16)) =
              make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (s_abort) {
    // a wait expired: let everything already issued land before leaving
    if (warp == G::kWarpTma && lane == 0)
      for (int s = 0; s < kStagesW && s < issued; ++s) {
        const int last = s + kStagesW * ((issued - 1 - s) / kStagesW);
        mbar_drain(smem_u32(&full_w[s]), (last / kStagesW) & 1);
      }
    if (warp == G::kWarpMma && lane == 0) mbar_drain(smem_u32(&bar_done), 0);
    __syncthreads();
  }
  if (warp == G::kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, G::kTmemCols);
  }

  // ---------------------------------------------------------------- split-K reduction
  // The splits of a tile form one cluster.  After the cluster barrier every
  // partial tile is visible through distributed shared memory; CTA z adds
  // rows [z R/S, (z+1) R/S) of all S partials in split order (so the result
  // does not depend on timing) and stores them, 512 contiguous bytes per
  // row.  Every CTA passes both cluster barriers on every path; the second
  // keeps each partial alive until its readers are done.
  cluster_sync();
  const int S = (int)gridDim.z;
  const int z = (int)cluster_ctarank();
  const int rows_per = kTileM / S;  // S divides 128
  const int r0 = z * rows_per;
  const uint32_t own = smem_u32(smem);
  uint32_t peer[kMaxSplits];
#pragma unroll
  for (int q = 0; q < kMaxSplits; ++q) peer[q] = q < S ? mapa_shared(own, q) : 0u;
  const int nchunks = rows_per * (kTileN / 4);
  for (int e0 = tid; e0 < nchunks; e0 += G::kThreads * 2) {
    float4 acc[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int e = e0 + u * G::kThreads;
      acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (e < nchunks) {
        const int r = r0 + e / (kTileN / 4), c = e % (kTileN / 4), rr = r & 127;
        const uint32_t off =
            (uint32_t)(((r >> 7) * 4 + (c >> 3)) * kBoxBytes + rr * 128 + (((c & 7) ^ (rr & 7)) * 16));
        float4 p[kMaxSplits];
#pragma unroll
        for (int q = 0; q < kMaxSplits; ++q)  // every partial read in flight at once
          if (q < S) p[q] = ld_dsmem_f4(peer[q] + off);
        acc[u] = p[0];
#pragma unroll
        for (int q = 1; q < kMaxSplits; ++q)
          if (q < S) {
            acc[u].x += p[q].x; acc[u].y += p[q].y; acc[u].z += p[q].z; acc[u].w += p[q].w;
          }
      }
    }
    // e < nchunks and s_abort are warp-uniform: a warp's 32 chunks are one
    // whole row (nchunks and the thread count are multiples of 32)
    if (s_abort) continue;
    const int c = tid & 31;  // = e % (kTileN / 4) for both rows
    if (ln_hi) {
      // LN0 of the two finished rows (lane c holds columns 4c .. 4c + 3 of
      // each): the mean, then the population variance of the deviations; the
      // two rows' warp sums interleave
      float4 v[2];
      float sm[2], sq[2];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        v[u] = acc[u];
        sm[u] = (v[u].x + v[u].y) + (v[u].z + v[u].w);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1)
#pragma unroll
        for (int u = 0; u < 2; ++u) sm[u] += __shfl_xor_sync(DC_FULL_MASK, sm[u], o);
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const float mean = sm[u] * (1.0f / kTileN);
        v[u].x -= mean; v[u].y -= mean; v[u].z -= mean; v[u].w -= mean;
        sq[u] = (v[u].x * v[u].x + v[u].y * v[u].y) + (v[u].z * v[u].z + v[u].w * v[u].w);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1)
#pragma unroll
        for (int u = 0; u < 2; ++u) sq[u] += __shfl_xor_sync(DC_FULL_MASK, sq[u], o);
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int e = e0 + u * G::kThreads;
        const int r = r0 + e / (kTileN / 4);
        if (e >= nchunks || m0 + r >= M) continue;
        const float inv = rsqrtf(sq[u] * (1.0f / kTileN) + ln_eps);
        const float x[4] = {v[u].x * inv, v[u].y * inv, v[u].z * inv, v[u].w * inv};
        uint32_t h[4], l[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          h[k] = bf16_rn_bits(x[k]);
          l[k] = bf16_rn_bits(x[k] - bf16_bits_to_float(h[k]));
        }
        const int64_t o = (int64_t)(m0 + r) * kTileN + c * 4;
        *reinterpret_cast<uint2 *>(ln_hi + o) = make_uint2(h[0] | (h[1] << 16), h[2] | (h[3] << 16));
        *reinterpret_cast<uint2 *>(ln_lo + o) = make_uint2(l[0] | (l[1] << 16), l[2] | (l[3] << 16));
      }
    } else {
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int e = e0 + u * G::kThreads;
        const int r = r0 + e / (kTileN / 4);
        if (e < nchunks && m0 + r < M)
          *reinterpret_cast<float4 *>(C + (int64_t)(m0 + r) * No + n0 + c * 4) = acc[u];
      }
    }
  }
  cluster_sync();
  // every CTA of the cluster is past its flag wait: clear the flags for the
  // next call
  if (job.row_ready && cluster_ctarank() == 0 && tid <= row_last - row_first) job.row_ready[row_first + tid] = 0u;
}

}  // namespace


int proj_tc_splits(int d, int requested) {
  // the largest power of two (it must divide the 128 tile rows that the
  // cluster shares out) up to the request that leaves no split empty
  const int nkb = d / kTileK;
  int s = 1;
  while (s * 2 <= std::min(requested, kMaxSplits)) s *= 2;
  for (; s > 1; s /= 2) {
    const int per = (nkb + s - 1) / s;
    if ((nkb + per - 1) / per == s) break;
  }
  return s;
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

namespace {
bool encode_16bit_rows_map(CUtensorMap *map, CUtensorMapDataType type, const void *base, int rows, int d,
                           int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || rows <= 0 || d % kTileK != 0 || (reinterpret_cast<uintptr_t>(base) & 15u)) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)d * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kTileK, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, type, 2, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
}  // namespace

bool encode_bf16_rows_map(CUtensorMap *map, const void *base, int rows, int d, int box_rows) {
  return encode_16bit_rows_map(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, rows, d, box_rows);
}

bool encode_f16_rows_map(CUtensorMap *map, const void *base, int rows, int d, int box_rows) {
  return encode_16bit_rows_map(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, base, rows, d, box_rows);
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

cudaError_t launch_proj_tc(const ProjJob &a, const CUtensorMap &a_hi, const CUtensorMap &a_lo,
                           const ProjJob *b, const CUtensorMap *b_hi, const CUtensorMap *b_lo, int slots,
                           int B, int d, int V, int splits, int *err, cudaStream_t st, bool pdl) {
  constexpr int MT = 2;
  using G = ProjGeom<MT>;
  auto bad = [&](const ProjJob &j) {
    return j.No % kTileN != 0 || j.M < 0 || !j.table || (!j.C && !j.ln_hi) ||
           (j.ln_hi && (j.No != kTileN || !j.ln_lo)) || (j.row_ready && (!j.ids || j.cands_per_row < 1)) ||
           j.tiles != ((j.M + G::kTileM - 1) / G::kTileM) * (j.No / kTileN);
  };
  if (d % kTileK != 0 || splits < 1 || splits > kMaxSplits || (kSubM % splits) != 0 || bad(a) ||
      (b && (bad(*b) || !b_hi || !b_lo)))
    return cudaErrorInvalidValue;
  const ProjJob none{};
  const ProjJob &j1 = b ? *b : none;
  const int tiles = a.tiles + j1.tiles;
  if (tiles == 0) return cudaSuccess;
  const int nkb = d / kTileK;
  const int per = (nkb + splits - 1) / splits;
  const dim3 grid(1, tiles, splits);
  const size_t smem = (size_t)G::kSmemUsed + 1024;
  cudaError_t e = cudaFuncSetAttribute(k_proj_tc<MT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  // the splits of one tile form a cluster
  e = launch_ex(k_proj_tc<MT>, grid, dim3(G::kThreads), smem, st, pdl, grid.z, a, j1, a_hi, a_lo,
                b ? *b_hi : a_hi, b ? *b_lo : a_lo, slots, B, d, V, per, err);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

int proj_tc_tiles(int M, int No) { return ((M + 2 * kSubM - 1) / (2 * kSubM)) * (No / kTileN); }

}  // namespace dc
