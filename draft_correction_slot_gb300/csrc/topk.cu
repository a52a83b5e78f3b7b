// topk.cu -- step 1: per-slot top-K of bf16 logits.
//
// DCOCO page ("Contextual Correction of Parallel Drafts for Speculative
// Decoding"), Method step details (1): each draft slot keeps the top-K
// candidates of its draft logits.  Order: value descending, then token id
// ascending; -0 == +0.
//
// Design (HBM-bound; one pass over the logits):
//   * Each row (request n, draft slot i) is cut into chunks of <= 2048
//     16-byte vectors (16384 logits).  One 256-thread CTA per (row, chunk);
//     every thread issues its 8 streaming 16-byte loads up front.
//   * Threshold: a thread's maximum over its (up to) 64 logits is computed
//     with packed bf16x2 max.  In each warp, the K-th largest of the 32 lane
//     maxima T_w (radix select over 16-bit order keys with ballots) is a
//     lower bound of the chunk's K-th largest value, because K different
//     lanes each hold an element >= T_w.  The CTA takes max_w T_w.
//   * Only lanes whose maximum reaches the threshold rescan their vectors;
//     survivors go to a shared list as unique 32-bit keys
//     (order key << 16 | 0xFFFF - local index) and are ranked exactly.
//     If the list overflows (e.g. many equal values), an exact 4-pass 8-bit
//     radix select over the chunk's keys finds the K-th key instead.
//   * The chunk's best K go to `part` as 64-bit keys
//     (order key << 32 | 0xFFFFFFFF - token id); the last CTA of the row
//     (atomic counter) merges the chunk lists, each already sorted, by
//     rank = own position + binary-search counts in the other lists.
#include "common.cuh"
#include "kernels.h"

namespace dc {

namespace {

constexpr int kThreads = kTopkThreads;
constexpr int kVpt = kTopkVecPerThread;
constexpr int kWarps = kThreads / 32;
constexpr int kListCap = 1024;
constexpr uint32_t kNegInf2 = 0xFF80FF80u;

__device__ __forceinline__ uint32_t chunk_key(uint32_t bits16, uint32_t local) {
  return (bf16_order_key(bits16) << 16) | (0xFFFFu - local);
}

// Number of entries of the descending list l[0..n) strictly greater than x.
__device__ __forceinline__ int count_greater(const unsigned long long *l, int n,
                                             unsigned long long x) {
  int lo = 0, hi = n;  // answer in [lo, hi]
  while (lo < hi) {
    int mid = (lo + hi) >> 1;
    if (l[mid] > x) lo = mid + 1; else hi = mid;
  }
  return lo;
}

template <int K>
__global__ void __launch_bounds__(kThreads, 3)
k_topk(const uint16_t *__restrict__ logits, int64_t stride, int slots, int B, int V, int nchunks,
       int chunk_vecs, unsigned long long *__restrict__ part, unsigned *__restrict__ row_count,
       int32_t *__restrict__ out_ids, float *__restrict__ out_val) {
  __shared__ uint32_t s_list[kListCap];
  __shared__ unsigned long long s_merge[kTopkMaxChunks * K];
  __shared__ uint32_t s_thr[kWarps];
  __shared__ uint32_t s_top[K];
  __shared__ unsigned s_hist[256];
  __shared__ int s_cnt;
  __shared__ int s_flag;
  __shared__ unsigned s_sel, s_krem;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int c = blockIdx.x;          // chunk
  const int row = blockIdx.y;        // n * B + i
  const int n = row / B, i = row - n * B;
  const uint16_t *rowp = logits + ((int64_t)n * slots + i + 1) * stride;

  const int nvec = V >> 3, tail = V & 7;
  const int v0 = c * chunk_vecs;
  const int v1 = min(v0 + chunk_vecs, nvec);
  const bool last_chunk = (c == nchunks - 1);

  if (tid == 0) s_cnt = 0;
  if (tid < K) s_top[tid] = 0u;

  // ---- stream the chunk into registers
  uint4 v[kVpt];
#pragma unroll
  for (int k = 0; k < kVpt; ++k) {
    const int j = v0 + tid + k * kThreads;
    if (j < v1) v[k] = ld_stream_v4(rowp + (int64_t)j * 8);
    else v[k] = make_uint4(kNegInf2, kNegInf2, kNegInf2, kNegInf2);
  }
  const bool has_tail = last_chunk && tid < tail;
  uint32_t tail_bits = 0xFF80u;
  if (has_tail) tail_bits = rowp[(int64_t)nvec * 8 + tid];

  // ---- per-vector and per-thread maxima (packed bf16x2)
  uint32_t vmax2[kVpt];
  uint32_t tmax2 = kNegInf2;
#pragma unroll
  for (int k = 0; k < kVpt; ++k) {
    vmax2[k] = bf16x2_max(bf16x2_max(v[k].x, v[k].y), bf16x2_max(v[k].z, v[k].w));
    tmax2 = bf16x2_max(tmax2, vmax2[k]);
  }
  float tmax = fmaxf(bf16_bits_to_float(tmax2 & 0xFFFFu), bf16_bits_to_float(tmax2 >> 16));
  if (has_tail) tmax = fmaxf(tmax, bf16_bits_to_float(tail_bits));

  // ---- warp radix select of the K-th largest lane maximum
  const uint32_t tkey = bf16_order_key(__float_as_uint(tmax) >> 16);
  uint32_t prefix = 0;
#pragma unroll
  for (int bit = 15; bit >= 0; --bit) {
    const uint32_t trial = prefix | (1u << bit);
    const int cnt = __popc(__ballot_sync(DC_FULL_MASK, tkey >= trial));
    if (cnt >= K) prefix = trial;
  }
  if (lane == 0) s_thr[warp] = prefix;
  __syncthreads();
  uint32_t thr_key = s_thr[0];
#pragma unroll
  for (int w = 1; w < kWarps; ++w) thr_key = max(thr_key, s_thr[w]);
  const float thr = order_key_to_float(thr_key);

  // ---- collect survivors (value >= threshold)
  if (tmax >= thr) {
#pragma unroll
    for (int k = 0; k < kVpt; ++k) {
      const int j = v0 + tid + k * kThreads;
      if (j < v1) {
        const float vm = fmaxf(bf16_bits_to_float(vmax2[k] & 0xFFFFu),
                               bf16_bits_to_float(vmax2[k] >> 16));
        if (vm >= thr) {
          const uint32_t w4[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const uint32_t bits = (q & 1) ? (w4[q >> 1] >> 16) : (w4[q >> 1] & 0xFFFFu);
            if (bf16_bits_to_float(bits) >= thr) {
              const int pos = atomicAdd(&s_cnt, 1);
              if (pos < kListCap) s_list[pos] = chunk_key(bits, (uint32_t)((j - v0) * 8 + q));
            }
          }
        }
      }
    }
    if (has_tail && bf16_bits_to_float(tail_bits) >= thr) {
      const int pos = atomicAdd(&s_cnt, 1);
      if (pos < kListCap) s_list[pos] = chunk_key(tail_bits, (uint32_t)((v1 - v0) * 8 + tid));
    }
  }
  __syncthreads();
  int nlist = s_cnt;

  if (nlist > kListCap) {
    // ---- overflow: exact radix select of the K-th largest chunk key
    const int chunk_n = (v1 - v0) * 8 + (last_chunk ? tail : 0);
    uint32_t pre = 0, msk = 0;
    unsigned krem = (unsigned)min(K, chunk_n);
    for (int pass = 0; pass < 4; ++pass) {
      const int shift = 24 - 8 * pass;
      s_hist[tid] = 0u;  // kThreads == 256 bins
      __syncthreads();
#pragma unroll
      for (int k = 0; k < kVpt; ++k) {
        const int j = v0 + tid + k * kThreads;
        if (j < v1) {
          const uint32_t w4[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const uint32_t bits = (q & 1) ? (w4[q >> 1] >> 16) : (w4[q >> 1] & 0xFFFFu);
            const uint32_t key = chunk_key(bits, (uint32_t)((j - v0) * 8 + q));
            if ((key & msk) == pre) atomicAdd(&s_hist[(key >> shift) & 0xFFu], 1u);
          }
        }
      }
      if (has_tail) {
        const uint32_t key = chunk_key(tail_bits, (uint32_t)((v1 - v0) * 8 + tid));
        if ((key & msk) == pre) atomicAdd(&s_hist[(key >> shift) & 0xFFu], 1u);
      }
      __syncthreads();
      if (tid == 0) {
        unsigned acc = 0;
        int dsel = 0;
        for (int dg = 255; dg >= 0; --dg) {
          const unsigned h = s_hist[dg];
          if (acc + h >= krem) { dsel = dg; break; }
          acc += h;
        }
        s_sel = (unsigned)dsel;
        s_krem = krem - acc;
      }
      __syncthreads();
      pre |= s_sel << shift;
      msk |= 0xFFu << shift;
      krem = s_krem;
      __syncthreads();
    }
    // exactly min(K, chunk_n) keys are >= pre
    if (tid == 0) s_cnt = 0;
    __syncthreads();
#pragma unroll
    for (int k = 0; k < kVpt; ++k) {
      const int j = v0 + tid + k * kThreads;
      if (j < v1) {
        const uint32_t w4[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const uint32_t bits = (q & 1) ? (w4[q >> 1] >> 16) : (w4[q >> 1] & 0xFFFFu);
          const uint32_t key = chunk_key(bits, (uint32_t)((j - v0) * 8 + q));
          if (key >= pre) {
            const int pos = atomicAdd(&s_cnt, 1);
            if (pos < K) s_list[pos] = key;
          }
        }
      }
    }
    if (has_tail) {
      const uint32_t key = chunk_key(tail_bits, (uint32_t)((v1 - v0) * 8 + tid));
      if (key >= pre) {
        const int pos = atomicAdd(&s_cnt, 1);
        if (pos < K) s_list[pos] = key;
      }
    }
    __syncthreads();
    nlist = min(s_cnt, K);
  }

  // ---- exact ranks among the survivors (keys are unique)
  for (int e = tid; e < nlist; e += kThreads) {
    const uint32_t x = s_list[e];
    int rank = 0;
    for (int m = 0; m < nlist; ++m) rank += (s_list[m] > x);
    if (rank < K) s_top[rank] = x;
  }
  __syncthreads();

  // ---- publish the chunk's sorted best K
  unsigned long long *my = part + ((int64_t)row * nchunks + c) * K;
  if (tid < K) {
    const uint32_t x = s_top[tid];
    unsigned long long o = 0ull;  // empty slot sorts below every real key
    if (x != 0u) {
      const uint32_t id = (uint32_t)(v0 * 8) + (0xFFFFu - (x & 0xFFFFu));
      o = ((unsigned long long)(x >> 16) << 32) | (unsigned long long)(0xFFFFFFFFu - id);
    }
    my[tid] = o;
    __threadfence();
  }
  __syncthreads();
  if (tid == 0) {
    const unsigned prev = atomicAdd(&row_count[row], 1u);
    s_flag = (prev == (unsigned)(nchunks - 1));
  }
  __syncthreads();
  if (!s_flag) return;

  // ---- last CTA of the row: merge the nchunks sorted lists
  __threadfence();
  const int total = nchunks * K;
  const unsigned long long *rp = part + (int64_t)row * nchunks * K;
  for (int e = tid; e < total; e += kThreads) s_merge[e] = __ldcg(rp + e);
  __syncthreads();
  for (int e = tid; e < total; e += kThreads) {
    const unsigned long long x = s_merge[e];
    if (x == 0ull) continue;
    const int ce = e / K;
    int rank = e - ce * K;
    for (int c2 = 0; c2 < nchunks && rank < K; ++c2)
      if (c2 != ce) rank += count_greater(s_merge + c2 * K, K, x);
    if (rank < K) {
      out_ids[(int64_t)row * K + rank] = (int32_t)(0xFFFFFFFFu - (uint32_t)(x & 0xFFFFFFFFull));
      out_val[(int64_t)row * K + rank] = order_key_to_float((uint32_t)(x >> 32));
    }
  }
  if (tid == 0) row_count[row] = 0u;  // ready for the next call
}

}  // namespace

TopkPlan topk_plan(int V) {
  const int nvec = V >> 3;
  const int cap = kThreads * kVpt;
  TopkPlan p;
  p.nchunks = nvec > 0 ? (nvec + cap - 1) / cap : 1;
  p.chunk_vecs = nvec > 0 ? (nvec + p.nchunks - 1) / p.nchunks : 0;
  return p;
}

cudaError_t launch_topk(int K, const uint16_t *logits, int64_t stride, int slots, int N, int V,
                        const TopkPlan &plan, unsigned long long *part, unsigned *row_count,
                        int32_t *ids, float *vals, cudaStream_t st) {
  const int B = slots - 1;
  dim3 grid(plan.nchunks, N * B);
  if (N == 0) return cudaSuccess;
  switch (K) {
    case 8:
      k_topk<8><<<grid, kThreads, 0, st>>>(logits, stride, slots, B, V, plan.nchunks, plan.chunk_vecs,
                                           part, row_count, ids, vals);
      break;
    case 16:
      k_topk<16><<<grid, kThreads, 0, st>>>(logits, stride, slots, B, V, plan.nchunks, plan.chunk_vecs,
                                            part, row_count, ids, vals);
      break;
    case 32:
      k_topk<32><<<grid, kThreads, 0, st>>>(logits, stride, slots, B, V, plan.nchunks, plan.chunk_vecs,
                                            part, row_count, ids, vals);
      break;
    default:
      return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace dc
