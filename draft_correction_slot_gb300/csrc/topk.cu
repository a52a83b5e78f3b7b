// topk.cu -- step 1: per-slot top-K of bf16 logits.
//
// DCOCO page ("Contextual Correction of Parallel Drafts for Speculative
// Decoding"), Method step details (1): each draft slot keeps the top-K
// candidates of its draft logits.  Order: value descending, then token id
// ascending; -0 == +0.
//
// Design (HBM-bound, one pass over the logits, no barrier while streaming):
//   * A row (request n, draft slot i) is cut into `nseg` segments, one
//     256-thread CTA each; the CTA's 8 warps each stream a contiguous slice of
//     the segment, 4 coalesced 16-byte vectors per lane per iteration, with the
//     next iteration's loads in flight while the current one is examined.
//   * Each warp keeps its running top-K sorted in registers (lane k holds the
//     k-th best as a 64-bit key  order16(value) << 32 | 0xFFFFFFFF - id, so one
//     unsigned compare orders by value, then by lower id).
//   * First iteration: the K-th largest of the 32 lane maxima (radix select
//     with ballots) is a lower bound of the slice's K-th value -- K lanes each
//     hold an element at least that large -- so only elements >= it are
//     inserted.  Later iterations: a vector is examined only if its packed
//     bf16x2 maximum beats the running K-th value strictly (an equal value
//     cannot enter: its id is larger than every id already kept).
//   * Each element must also reach a lower bound of the row's K-th value: the
//     best K-th key published so far by any warp of the CTA (shared memory) or
//     by an earlier segment of the row (global memory; segments are launched
//     segment-major, so most CTAs start with a high bound).
//   * Survivors are extracted divergently into a per-warp shared buffer, then
//     inserted warp-cooperatively (shuffle-shift insert), so the cost follows
//     the number of candidates.  The 8 warp lists are merged in shared memory by rank
//     (own position + binary-search counts in the other lists); with several
//     segments, each CTA publishes its list and the last CTA of the row
//     (atomic counter, reset after use) merges them the same way.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace dc {

namespace {

constexpr int kThreads = kTopkThreads;
constexpr int kWarps = kThreads / 32;
constexpr int kU = 4;                 // vectors per lane per iteration
constexpr int kStep = 32 * kU;        // vectors per warp iteration
constexpr uint32_t kNegInf2 = 0xFF80FF80u;

typedef unsigned long long u64;

__device__ __forceinline__ u64 make_key(uint32_t bits16, uint32_t id) {
  return ((u64)bf16_order_key(bits16) << 32) | (u64)(0xFFFFFFFFu - id);
}

__device__ __forceinline__ u64 shfl_u64(u64 v, int src) {
  uint32_t lo = __shfl_sync(DC_FULL_MASK, (uint32_t)v, src);
  uint32_t hi = __shfl_sync(DC_FULL_MASK, (uint32_t)(v >> 32), src);
  return ((u64)hi << 32) | lo;
}

__device__ __forceinline__ u64 shfl_up_u64(u64 v) {
  uint32_t lo = __shfl_up_sync(DC_FULL_MASK, (uint32_t)v, 1);
  uint32_t hi = __shfl_up_sync(DC_FULL_MASK, (uint32_t)(v >> 32), 1);
  return ((u64)hi << 32) | lo;
}

// Insert `key` (warp-uniform, unique) into the descending register list.
template <int K>
__device__ __forceinline__ void warp_insert(u64 &list, u64 &kth, u64 key, int lane) {
  const u64 prev = shfl_up_u64(list);
  u64 nl = (list > key) ? list : ((lane == 0 || prev > key) ? key : prev);
  list = lane < K ? nl : 0ull;
  kth = shfl_u64(list, K - 1);
}

__device__ __forceinline__ u64 shfl_xor_u64(u64 v, int m) {
  uint32_t lo = __shfl_xor_sync(DC_FULL_MASK, (uint32_t)v, m);
  uint32_t hi = __shfl_xor_sync(DC_FULL_MASK, (uint32_t)(v >> 32), m);
  return ((u64)hi << 32) | lo;
}

// Bitonic sort of one key per lane, descending over the 32 lanes.
__device__ __forceinline__ u64 warp_sort32_desc(u64 x, int lane) {
#pragma unroll
  for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      const u64 o = shfl_xor_u64(x, j);
      const bool keep_max = (((lane & j) == 0) == ((lane & k) == 0));
      x = keep_max ? (o > x ? o : x) : (o < x ? o : x);
    }
  }
  return x;
}

// Top K of two descending lists held in lanes (a: lanes < K, b: 32 lanes,
// zero padded): max(a_i, b_{K-1-i}) is the top-K set as a bitonic sequence;
// a half-cleaner network sorts it.
template <int K>
__device__ __forceinline__ u64 warp_merge_topk(u64 a, u64 b, int lane) {
  const u64 br = shfl_u64(b, (K - 1 - lane) & 31);
  u64 x = (lane < K) ? (a > br ? a : br) : 0ull;
#pragma unroll
  for (int j = K >> 1; j > 0; j >>= 1) {
    const u64 o = shfl_xor_u64(x, j);
    const bool lower = (lane & j) == 0;
    x = lower ? (o > x ? o : x) : (o < x ? o : x);
  }
  return lane < K ? x : 0ull;
}

// bf16 bits with order key one below / above `key` (saturating).
__device__ __forceinline__ uint32_t bf16_from_key(uint32_t key) {
  return (key & 0x8000u) ? (key & 0x7FFFu) : (~key & 0xFFFFu);
}

__device__ __forceinline__ void load_vecs(uint4 (&v)[kU], const uint16_t *rowp, int base, int end,
                                          int lane) {
#pragma unroll
  for (int u = 0; u < kU; ++u) {
    const int j = base + lane + 32 * u;
    if (j < end) v[u] = ld_stream_v4(rowp + (int64_t)j * 8);
    else v[u] = make_uint4(kNegInf2, kNegInf2, kNegInf2, kNegInf2);
  }
}

template <int K>
__global__ void __launch_bounds__(kThreads, 4)
k_topk(const uint16_t *__restrict__ logits, int64_t stride, int slots, int B, int V, int nseg,
       int vecs_per_warp, u64 *__restrict__ part, unsigned *__restrict__ row_count,
       u64 *__restrict__ row_bound, int32_t *__restrict__ out_ids, float *__restrict__ out_val) {
  // s_buf: one iteration's candidates per warp (streaming phase)
  __shared__ __align__(16) uint32_t s_buf[kWarps][kStep * 8];
  __shared__ int s_bcnt[kWarps];
  __shared__ u64 s_lists[kWarps * K];
  __shared__ u64 s_top[K];
  __shared__ u64 s_cta_bound;
  __shared__ int s_flag;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int row = blockIdx.x, seg = blockIdx.y;  // segment-major launch order
  const int n = row / B, i = row - n * B;
  const uint16_t *rowp = logits + ((int64_t)n * slots + i + 1) * stride;
  const int nvec = V >> 3, tail = V & 7;
  const int gw = seg * kWarps + warp;
  const int w0 = min(gw * vecs_per_warp, nvec);
  const int w1 = min(w0 + vecs_per_warp, nvec);
  if (lane == 0) s_bcnt[warp] = 0;
  if (tid == 0) s_cta_bound = __ldcg(row_bound + row);  // K-th key of an earlier segment, or 0
  __syncthreads();

  u64 list = 0ull, kth = 0ull;
  uint4 cur[kU], nxt[kU];
  if (w0 < w1) load_vecs(cur, rowp, w0, w1, lane);
  for (int base = w0; base < w1; base += kStep) {
    if (base + kStep < w1) load_vecs(nxt, rowp, base + kStep, w1, lane);
    uint32_t vm2[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u)
      vm2[u] = bf16x2_max(bf16x2_max(cur[u].x, cur[u].y), bf16x2_max(cur[u].z, cur[u].w));
    const uint32_t lm2 = bf16x2_max(bf16x2_max(vm2[0], vm2[1]), bf16x2_max(vm2[2], vm2[3]));
    // An element can reach the row's top-K only if
    //   key >= bound: bound = the K-th key of some slice of this row (another
    //     warp's, an earlier segment's, or -- first iteration -- the K-th
    //     largest lane maximum, since K lanes each hold an element that large);
    //   and, once this warp holds K elements, value > its own K-th value (an
    //     equal value arriving later has a larger id and cannot displace it).
    // Both fold into one order-key threshold tkey: value key >= tkey.
    const u64 sb = *(volatile u64 *)&s_cta_bound;
    uint32_t tkey = sb ? (uint32_t)(sb >> 32) : 0u;
    if (base == w0 && sb == 0ull) {
      const float lm = fmaxf(bf16_bits_to_float(lm2 & 0xFFFFu), bf16_bits_to_float(lm2 >> 16));
      const uint32_t key = bf16_order_key(__float_as_uint(lm) >> 16);
      uint32_t pre = 0;
#pragma unroll
      for (int bit = 15; bit >= 0; --bit) {
        const uint32_t trial = pre | (1u << bit);
        if (__popc(__ballot_sync(DC_FULL_MASK, key >= trial)) >= K) pre = trial;
      }
      tkey = max(tkey, pre);
    }
    if (base != w0 && kth != 0ull) tkey = max(tkey, min((uint32_t)(kth >> 32) + 1u, 0xFFFFu));
    // packed skip test: every element of the lane is below tkey iff
    // max(lane max, below) == below, with below = the value just under tkey
    bool lane_hit = true;
    uint32_t below2 = 0u;
    if (tkey > 0x007Fu) {  // tkey above -inf: some elements can be skipped
      // key 0x7FFF would decode to -0, and max(+0, -0) may return -0: step
      // one further down there (skipping less is always safe)
      const uint32_t b = bf16_from_key(tkey - 1u == 0x7FFFu ? 0x7FFEu : tkey - 1u);
      below2 = b | (b << 16);
      lane_hit = bf16x2_max(lm2, below2) != below2;
    }
    if (__any_sync(DC_FULL_MASK, lane_hit)) {
      if (lane_hit) {
        const float thr = order_key_to_float(tkey);  // value >= thr <=> key >= tkey
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          const int j = base + lane + 32 * u;
          if (j >= w1) continue;
          if (below2 != 0u && bf16x2_max(vm2[u], below2) == below2) continue;
          const uint32_t wd[4] = {cur[u].x, cur[u].y, cur[u].z, cur[u].w};
          const uint32_t off = (uint32_t)(lane + 32 * u) * 8u;
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const uint32_t bits = (q & 1) ? (wd[q >> 1] >> 16) : (wd[q >> 1] & 0xFFFFu);
            if (bf16_bits_to_float(bits) >= thr || tkey <= 0x007Fu) {
              const int pos = atomicAdd(&s_bcnt[warp], 1);
              s_buf[warp][pos] = (bf16_order_key(bits) << 16) | (0xFFFFu - (off + (uint32_t)q));
            }
          }
        }
      }
      __syncwarp();
      const int cnt = s_bcnt[warp];
      const uint32_t id0 = (uint32_t)base * 8u;
      if (cnt <= 4) {
        for (int e = 0; e < cnt; ++e) {
          const uint32_t k32 = s_buf[warp][e];
          const u64 key = ((u64)(k32 >> 16) << 32) | (u64)(0xFFFFFFFFu - (id0 + 0xFFFFu - (k32 & 0xFFFFu)));
          if (key > kth) warp_insert<K>(list, kth, key, lane);
        }
      } else {
        for (int e0 = 0; e0 < cnt; e0 += 32) {
          u64 key = 0ull;
          if (e0 + lane < cnt) {
            const uint32_t k32 = s_buf[warp][e0 + lane];
            key = ((u64)(k32 >> 16) << 32) | (u64)(0xFFFFFFFFu - (id0 + 0xFFFFu - (k32 & 0xFFFFu)));
          }
          list = warp_merge_topk<K>(list, warp_sort32_desc(key, lane), lane);
        }
        kth = shfl_u64(list, K - 1);
      }
      __syncwarp();
      if (lane == 0) {
        s_bcnt[warp] = 0;
        if (kth) atomicMax(&s_cta_bound, kth);
      }
      __syncwarp();
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) cur[u] = nxt[u];
  }
  // the scalar tail (V % 8 elements) belongs to the row's last warp
  if (tail && seg == nseg - 1 && warp == kWarps - 1) {
    uint32_t bits = 0u;
    if (lane < tail) bits = rowp[(int64_t)nvec * 8 + lane];
    unsigned m = __ballot_sync(DC_FULL_MASK, lane < tail);
    const u64 mykey = make_key(bits, (uint32_t)(nvec * 8 + lane));
    while (m) {
      const int src = __ffs(m) - 1;
      m &= m - 1;
      const u64 key = shfl_u64(mykey, src);
      if (key > kth) warp_insert<K>(list, kth, key, lane);
    }
  }
  if (lane < K) s_lists[warp * K + lane] = list;
  __syncthreads();
  if (warp == 0) {  // merge the 8 warp lists
    u64 acc = lane < K ? s_lists[lane] : 0ull;
    for (int w = 1; w < kWarps; ++w)
      acc = warp_merge_topk<K>(acc, lane < K ? s_lists[w * K + lane] : 0ull, lane);
    if (lane < K) s_top[lane] = acc;
  }
  __syncthreads();

  if (nseg > 1) {
    u64 *my = part + ((int64_t)row * nseg + seg) * K;
    if (tid < K) {
      my[tid] = s_top[tid];
      __threadfence();
    }
    __syncthreads();
    if (tid == 0) {
      if (s_top[K - 1]) atomicMax(row_bound + row, s_top[K - 1]);  // for later segments
      const unsigned prev = atomicAdd(&row_count[row], 1u);
      s_flag = (prev == (unsigned)(nseg - 1));
    }
    __syncthreads();
    if (!s_flag) return;
    // last CTA of the row: merge the nseg segment lists
    __threadfence();
    if (warp == 0) {
      const u64 *rp = part + (int64_t)row * nseg * K;
      u64 acc = lane < K ? __ldcg(rp + lane) : 0ull;
      for (int sg = 1; sg < nseg; ++sg)
        acc = warp_merge_topk<K>(acc, lane < K ? __ldcg(rp + sg * K + lane) : 0ull, lane);
      if (lane < K) s_top[lane] = acc;
      if (lane == 0) {  // ready for the next call
        row_count[row] = 0u;
        row_bound[row] = 0ull;
      }
    }
    __syncthreads();
  }
  if (tid < K) {
    const u64 x = s_top[tid];
    out_ids[(int64_t)row * K + tid] = (int32_t)(0xFFFFFFFFu - (uint32_t)(x & 0xFFFFFFFFull));
    out_val[(int64_t)row * K + tid] = order_key_to_float((uint32_t)(x >> 32));
  }
}

}  // namespace

TopkPlan topk_plan(int V, int rows, int slots_per_wave) {
  const int nvec = V >> 3;
  TopkPlan p;
  // every warp streams at least two iterations; at most kTopkMaxChunks segments
  const int max_seg = std::max(1, std::min(kTopkMaxChunks, nvec / (kWarps * 2 * kStep)));
  p.nchunks = 1;
  if (rows > 0 && slots_per_wave > 0) {
    double best = -1.0;
    for (int s = 1; s <= max_seg; ++s) {
      const long long total = (long long)rows * s;
      const long long waves = (total + slots_per_wave - 1) / slots_per_wave;
      const double eff = (double)total / (double)(waves * slots_per_wave);
      if (eff > best + 1e-9) {
        best = eff;
        p.nchunks = s;
      }
    }
  }
  p.chunk_vecs = (nvec + p.nchunks * kWarps - 1) / (p.nchunks * kWarps);  // vectors per warp
  return p;
}

int topk_max_segments(int V) {
  const int nvec = V >> 3;
  return std::max(1, std::min(kTopkMaxChunks, nvec / (kWarps * 2 * kStep)));
}

template <int K>
static int topk_occupancy_k() {
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k_topk<K>, kThreads, 0) != cudaSuccess) {
    cudaGetLastError();
    return 1;
  }
  return occ > 0 ? occ : 1;
}

int topk_occupancy(int K) {
  switch (K) {
    case 8: return topk_occupancy_k<8>();
    case 16: return topk_occupancy_k<16>();
    case 32: return topk_occupancy_k<32>();
    default: return 1;
  }
}

cudaError_t launch_topk(int K, const uint16_t *logits, int64_t stride, int slots, int N, int V,
                        const TopkPlan &plan, unsigned long long *part, unsigned *row_count,
                        unsigned long long *row_bound, int32_t *ids, float *vals, cudaStream_t st) {
  const int B = slots - 1;
  if (N == 0) return cudaSuccess;
  dim3 grid(N * B, plan.nchunks);
  switch (K) {
    case 8:
      k_topk<8><<<grid, kThreads, 0, st>>>(logits, stride, slots, B, V, plan.nchunks, plan.chunk_vecs,
                                           part, row_count, row_bound, ids, vals);
      break;
    case 16:
      k_topk<16><<<grid, kThreads, 0, st>>>(logits, stride, slots, B, V, plan.nchunks, plan.chunk_vecs,
                                            part, row_count, row_bound, ids, vals);
      break;
    case 32:
      k_topk<32><<<grid, kThreads, 0, st>>>(logits, stride, slots, B, V, plan.nchunks, plan.chunk_vecs,
                                            part, row_count, row_bound, ids, vals);
      break;
    default:
      return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace dc
