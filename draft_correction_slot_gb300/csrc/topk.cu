// topk.cu -- step 1: per-slot top-K of bf16 logits.
//
// DCOCO page ("Contextual Correction of Parallel Drafts for Speculative
// Decoding"), Method step details (1): each draft slot keeps the top-K
// candidates of its draft logits.  Order: value descending, then token id
// ascending; -0 == +0.
//
// Design (HBM-bound; every logit is read from HBM exactly once):
//   * A row (request n, draft slot i) is cut into `nseg` segments of at most
//     20480 16-byte vectors, one 256-thread CTA each (usually one per row).
//   * Pass 1 -- stream: each warp reads a contiguous slice of the segment,
//     4 coalesced 16-byte vectors per lane per iteration with the next ones in
//     flight, and stores each vector's maximum (packed bf16x2 max) in shared
//     memory.  Nothing else happens while streaming, except that with the
//     candidate features each lane also keeps a running log-sum-exp
//     (exp(x - m) as 2^(fma(x, log2 e, -m log2 e)), two partial sums).
//   * Pass 2 -- bound: T = the K-th largest maximum of the groups of 64
//     vectors.  K groups each hold an element >= T, so the segment's K-th
//     value is >= T: every element of the segment's top-K lies in a vector
//     whose maximum reaches T.  Those vectors (typically about K of them) are
//     listed in order.
//   * Pass 3 -- select: the listed vectors are read again (L2) and their
//     elements >= T ranked exactly, as 64-bit keys
//     order16(value) << 32 | 0xFFFFFFFF - id (one unsigned compare orders by
//     value, then by lower id), with bitonic warp merges.
//   * Degenerate segments (many ties at the bound, -inf masks) list too many
//     vectors; they are streamed again with per-warp running lists instead:
//     each warp keeps its top-K in registers and only elements above the
//     running bounds are inserted.
//   * With several segments, each CTA publishes its list and the last CTA of
//     the row (atomic counter, reset after use) merges them.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "launch.h"
#include "topk_warp.cuh"

namespace dc {

namespace {

constexpr int kThreads = kTopkThreads;
constexpr int kWarps = kThreads / 32;
constexpr int kU = 4;                 // vectors per lane per iteration
constexpr int kStep = 32 * kU;        // vectors per warp iteration
constexpr int kSerialMax = 8;         // up to this many candidates: serial inserts
constexpr int kPrefetchAhead = 4;     // L2 prefetch distance, in iterations (fallback)
constexpr int kGroup = 64;            // vectors per group in the bound of pass 2
constexpr int kMaxSegVecs = 20480;    // vectors per segment (16-bit maxima in shared memory)
constexpr int kRawWords = (kWarps * kStep * 8 > kMaxSegVecs / 2) ? kWarps * kStep * 8 : kMaxSegVecs / 2;
constexpr int kMaxGroups = kMaxSegVecs / kGroup;
constexpr int kCandGroups = 64;       // groups reaching the bound beyond this: degenerate path
constexpr int kMaxHitsPerLane = 4;    // hit vectors a lane re-loads (more: degenerate path)
constexpr int kCandElems = 8 * kWarps * 32 * kMaxHitsPerLane / 4;  // key buffer (fits s_raw)
constexpr uint32_t kNegInf2 = 0xFF80FF80u;

using namespace topk_warp;

// Logits are read once by the stream and again, for the few vectors that
// reach the bound, right after it: normal L2 priority keeps those re-reads
// in L2; L1 is bypassed.
__device__ __forceinline__ uint4 ld_stream(const void *ptr) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(ptr));
  return v;
}

__device__ __forceinline__ void load_vecs(uint4 (&v)[kU], const uint16_t *rowp, int base, int end,
                                          int lane) {
#pragma unroll
  for (int u = 0; u < kU; ++u) {
    const int j = base + lane + 32 * u;
    if (j < end) v[u] = ld_stream(rowp + (int64_t)j * 8);
    else v[u] = make_uint4(kNegInf2, kNegInf2, kNegInf2, kNegInf2);
  }
}

// Fallback for degenerate segments: each warp streams [w0, w1) again and
// keeps its own top-K, inserting only elements whose key reaches the running
// bound (the CTA-shared bound, never below `floor_key`, or its own K-th).
template <int K>
__device__ __forceinline__ u64 stream_fallback(const uint16_t *rowp, int w0, int w1, uint32_t floor_key,
                                               u64 *s_cta_bound, uint32_t *s_bufw, int lane) {
  u64 list = 0ull, kth = 0ull;
  uint4 cur[kU], nxt[kU];
  if (w0 < w1) load_vecs(cur, rowp, w0, w1, lane);
  // one iteration: kU vectors per lane, starting at vector `base`
  auto process = [&](const uint4 (&v)[kU], int base) {
      uint32_t vm2[kU];
  #pragma unroll
      for (int u = 0; u < kU; ++u)
        vm2[u] = bf16x2_max(bf16x2_max(v[u].x, v[u].y), bf16x2_max(v[u].z, v[u].w));
      const uint32_t lm2 = bf16x2_max(bf16x2_max(vm2[0], vm2[1]), bf16x2_max(vm2[2], vm2[3]));
      // An element can reach the row's top-K only if
      //   key >= bound: bound = the K-th key of some slice of this row (another
      //     warp's, an earlier segment's, or -- first iteration -- the K-th
      //     largest lane maximum, since K lanes each hold an element that large);
      //   and, once this warp holds K elements, value > its own K-th value (an
      //     equal value arriving later has a larger id and cannot displace it).
      // Both fold into one order-key threshold tkey: value key >= tkey.
      const u64 sb = *(volatile u64 *)s_cta_bound;
      uint32_t tkey = max(floor_key, sb ? (uint32_t)(sb >> 32) : 0u);
      if (base == w0 && tkey == 0u) {
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
        // this lane's candidate mask, bit 8u+q = element q of vector u: the
        // packed test max(x, below) != below marks x above `below` (ties to
        // +-0 may add false positives, which the exact key compare of the
        // insert rejects or which cannot displace a real top-K member)
        uint32_t emask = 0u;
        if (lane_hit) {
#pragma unroll
          for (int u = 0; u < kU; ++u) {
            const int j = base + lane + 32 * u;
            if (j >= w1) continue;
            if (below2 == 0u) {
              emask |= 0xFFu << (8 * u);
              continue;
            }
            const uint32_t wd[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              const uint32_t dif = bf16x2_max(wd[h], below2) ^ below2;
              emask |= (((dif & 0xFFFFu) != 0u ? 1u : 0u) | ((dif >> 16) != 0u ? 2u : 0u)) << (8 * u + 2 * h);
            }
          }
        }
        // warp-exclusive scan of the candidate counts gives each lane its slots
        const int c = __popc(emask);
        int incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int t = __shfl_up_sync(DC_FULL_MASK, incl, o);
          if (lane >= o) incl += t;
        }
        const int cnt = __shfl_sync(DC_FULL_MASK, incl, 31);
        int pos = incl - c;
        while (emask) {
          const int e = __ffs(emask) - 1;
          emask &= emask - 1;
          const int u = e >> 3, q = e & 7;
          const uint4 vv = u == 0 ? v[0] : (u == 1 ? v[1] : (u == 2 ? v[2] : v[3]));
          const uint32_t wd = (q >> 1) == 0 ? vv.x : ((q >> 1) == 1 ? vv.y : ((q >> 1) == 2 ? vv.z : vv.w));
          const uint32_t bits = (q & 1) ? (wd >> 16) : (wd & 0xFFFFu);
          const uint32_t off = (uint32_t)(lane + 32 * u) * 8u + (uint32_t)q;
          s_bufw[pos++] = (bf16_order_key(bits) << 16) | (0xFFFFu - off);
        }
        __syncwarp();
        const uint32_t id0 = (uint32_t)base * 8u;
        if (cnt <= kSerialMax) {
          for (int e = 0; e < cnt; ++e) {
            const uint32_t k32 = s_bufw[e];
            const u64 key = ((u64)(k32 >> 16) << 32) | (u64)(0xFFFFFFFFu - (id0 + 0xFFFFu - (k32 & 0xFFFFu)));
            if (key > kth) warp_insert<K>(list, kth, key, lane);
          }
        } else {
          for (int e0 = 0; e0 < cnt; e0 += 32) {
            u64 key = 0ull;
            if (e0 + lane < cnt) {
              const uint32_t k32 = s_bufw[e0 + lane];
              key = ((u64)(k32 >> 16) << 32) | (u64)(0xFFFFFFFFu - (id0 + 0xFFFFu - (k32 & 0xFFFFu)));
            }
            list = warp_merge_topk<K>(list, warp_sort32_desc(key, lane), lane);
          }
          kth = shfl_u64(list, K - 1);
        }
        if (lane == 0 && kth > sb) atomicMax(s_cta_bound, kth);
        __syncwarp();  // s_buf is rewritten by the next iteration
      }
  };
  // L2 prefetch kPrefetchAhead iterations ahead of the register loads, so
  // DRAM keeps streaming while the warp examines its current vectors
  auto prefetch = [&](int b) {
    if (lane == 0 && b < w1)
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(rowp + (int64_t)b * 8),
                   "r"((uint32_t)min(kStep, w1 - b) * 16u)
                   : "memory");
  };
#pragma unroll
  for (int a = 1; a <= kPrefetchAhead; ++a) prefetch(w0 + a * kStep);
  // ping-pong between two register buffers; the next loads are always in flight
  for (int base = w0; base < w1; base += 2 * kStep) {
    prefetch(base + (kPrefetchAhead + 1) * kStep);
    if (base + kStep < w1) load_vecs(nxt, rowp, base + kStep, w1, lane);
    process(cur, base);
    if (base + kStep >= w1) break;
    prefetch(base + (kPrefetchAhead + 2) * kStep);
    if (base + 2 * kStep < w1) load_vecs(cur, rowp, base + 2 * kStep, w1, lane);
    process(nxt, base + kStep);
  }
  return list;
}

// One warp: the digit d of a 256-bin histogram (bins scanned from 255 down)
// whose bin holds the rank-th largest key (rank >= 1), and the count of keys
// in the bins above it.  *digit = -1 when the histogram holds fewer than rank
// keys.  Lane l owns bins 255 - 8l ... 248 - 8l.
__device__ __forceinline__ void radix_digit(const int *hist, int rank, int lane, int *digit, int *above) {
  int c[8], sum = 0;
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    c[q] = hist[255 - 8 * lane - q];
    sum += c[q];
  }
  int incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(DC_FULL_MASK, incl, o);
    if (lane >= o) incl += y;
  }
  const int excl = incl - sum;  // keys in the bins above this lane's
  int d = -1, ab = 0;
  if (excl < rank && rank <= incl) {
    int acc = excl;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      if (d < 0 && acc + c[q] >= rank) {
        d = 255 - 8 * lane - q;
        ab = acc;
      }
      acc += c[q];
    }
  }
  const unsigned m = __ballot_sync(DC_FULL_MASK, d >= 0);
  if (m) {
    const int src = __ffs(m) - 1;
    d = __shfl_sync(DC_FULL_MASK, d, src);
    ab = __shfl_sync(DC_FULL_MASK, ab, src);
  }
  if (lane == 0) {
    *digit = m ? d : -1;
    *above = ab;
  }
}

// Merge (m, s) pairs, s a sum of exp(x - m) (m = -inf: empty).
constexpr float kLog2e = 1.44269504088896340736f;
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void lse_merge(float &m, float &s, float m2, float s2) {
  const float mm = fmaxf(m, m2);
  if (mm == -INFINITY) return;
  s = (m == -INFINITY ? 0.f : s * __expf(m - mm)) + (m2 == -INFINITY ? 0.f : s2 * __expf(m2 - mm));
  m = mm;
}

// kLse: the stream also accumulates the row's log-sum-exp (each lane a running
// maximum and sum of exp(x - maximum) over the vectors it reads), and the
// publishing block writes the candidates' vocabulary-normalised features
// (LiLiCorr page, App. A: top-K fused with the normalisation, in one pass
// over the logits): per candidate k, [log p, p, l_0 - l_k, k / K, k == 0],
// p the softmax over the whole vocabulary.  With several segments each block
// leaves its (maximum, sum) in part_lse and the merging block combines them.
template <int K, bool kLse>
__global__ void __launch_bounds__(kThreads, 4)
k_topk(const uint16_t *__restrict__ logits, int64_t stride, int slots, int B, int V, int nseg,
       int seg_vecs, u64 *__restrict__ part, unsigned *__restrict__ row_count,
       int32_t *__restrict__ out_ids, float *__restrict__ out_val, float2 *__restrict__ part_lse,
       float *__restrict__ out_feat, TopkHandoff hand) {
  // s_vmax (pass 1-2: per-vector maxima, bf16 bits), s_keys (pass 3:
  // candidate elements) and the fallback's per-warp candidate buffers share
  // storage; each use ends at a barrier before the next begins
  static_assert(kCandElems * 8 <= kRawWords * 4, "alias");
  __shared__ __align__(16) uint32_t s_raw[kRawWords];
  uint16_t *s_vmax = reinterpret_cast<uint16_t *>(s_raw);
  u64 *s_keys = reinterpret_cast<u64 *>(s_raw);
  __shared__ uint16_t s_gkey[kMaxGroups];   // order key of each group's maximum
  __shared__ int s_cand[kCandGroups];       // candidate groups
  __shared__ u64 s_lists[kWarps * K];
  __shared__ int s_hist[2][256];  // radix-select histograms of the group keys
  __shared__ int s_digit, s_above;
  __shared__ u64 s_top[K];
  __shared__ u64 s_cta_bound;
  __shared__ int s_ncand, s_nkeys, s_flag;
  __shared__ uint32_t s_tkey;
  __shared__ float s_lm[kWarps], s_ls[kWarps];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // with the handoff the grid is one-dimensional, segments of a row adjacent
  // (blocks are dispatched in index order, so rows finish from the first on)
  const int row = hand.row_ready ? (int)blockIdx.x / nseg : (int)blockIdx.x;
  const int seg = hand.row_ready ? (int)blockIdx.x - row * nseg : (int)blockIdx.y;
  const int n = row / B, i = row - n * B;
  const uint16_t *rowp = logits + ((int64_t)n * slots + i + 1) * stride;
  const int nvec = V >> 3, tail = V & 7;
  const int v0 = min(seg * seg_vecs, nvec), v1 = min(v0 + seg_vecs, nvec);
  const int nv = min(v1 - v0, kMaxSegVecs);           // vectors of this segment
  const bool has_tail = tail && seg == nseg - 1;
  // warp ranges are whole 64-vector groups, so each 128-vector step of a warp
  // covers exactly two groups and their maxima come from two warp reductions
  const int per_warp = ((nv + kWarps - 1) / kWarps + kGroup - 1) / kGroup * kGroup;
  const int ng = (nv + kGroup - 1) / kGroup;
  const int w0 = v0 + min(warp * per_warp, nv), w1 = v0 + min((warp + 1) * per_warp, nv);
  pdl_trigger();
  if (tid < K) s_top[tid] = 0ull;
  for (int e = tid; e < 2 * 256; e += kThreads) (&s_hist[0][0])[e] = 0;
  if (tid == 0) {
    s_ncand = 0;
    s_nkeys = 0;
    s_flag = 0;
    s_cta_bound = 0ull;
  }

  // ---------------------------------------------------------------- pass 1: stream
  // kLse: this lane's running maximum and its sum of exp(x - lm), kept as two
  // partial sums; nb = -lm log2 e, so exp(x - lm) = 2^(fma(x, log2 e, nb))
  float lm = -INFINITY, ls = 0.f, ls2 = 0.f, nb = 0.f;
  {
    uint4 a[kU], b[kU];
    static_assert(kStep == 2 * kGroup && kU == 4, "one step = two groups of 64 vectors");
    auto store = [&](const uint4 (&v)[kU], int base) {
      uint32_t gk[2] = {0u, 0u};  // order keys of the two groups' maxima (0: empty)
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int j = base + lane + 32 * u;
        if (j < w1 && j - v0 < kMaxSegVecs) {  // the plan keeps segments within the buffer
          const uint32_t m2 = bf16x2_max(bf16x2_max(v[u].x, v[u].y), bf16x2_max(v[u].z, v[u].w));
          const uint32_t m = bf16x2_max(m2, m2 >> 16) & 0xFFFFu;
          s_vmax[j - v0] = (uint16_t)m;
          gk[u >> 1] = max(gk[u >> 1], bf16_order_key(m));
          if (kLse) {
            const float vm = bf16_bits_to_float(m);
            if (vm > lm) {
              const float f = lm == -INFINITY ? 0.f : __expf(lm - vm);
              ls *= f;
              ls2 *= f;
              lm = vm;
              nb = -vm * kLog2e;
            }
            if (lm != -INFINITY) {
              const uint32_t wd[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
              for (int h = 0; h < 4; ++h) {
                ls += ex2_approx(fmaf(bf16_bits_to_float(wd[h] & 0xFFFFu), kLog2e, nb));
                ls2 += ex2_approx(fmaf(bf16_bits_to_float(wd[h] >> 16), kLog2e, nb));
              }
            }
          }
        }
      }
      const int g = (base - v0) / kGroup;
      const uint32_t k0 = __reduce_max_sync(DC_FULL_MASK, gk[0]);
      const uint32_t k1 = __reduce_max_sync(DC_FULL_MASK, gk[1]);
      if (lane == 0) {  // the second group may start the next warp's range
        if (g < ng) s_gkey[g] = (uint16_t)k0;
        if (g + 1 < ng && base + kGroup < w1) s_gkey[g + 1] = (uint16_t)k1;
      }
    };
    if (w0 < w1) load_vecs(a, rowp, w0, w1, lane);
    for (int base = w0; base < w1; base += 2 * kStep) {
      if (base + kStep < w1) load_vecs(b, rowp, base + kStep, w1, lane);
      store(a, base);
      if (base + kStep >= w1) break;
      if (base + 2 * kStep < w1) load_vecs(a, rowp, base + 2 * kStep, w1, lane);
      store(b, base + kStep);
    }
  }
  if (kLse) {
    ls += ls2;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float om = __shfl_xor_sync(DC_FULL_MASK, lm, off), os = __shfl_xor_sync(DC_FULL_MASK, ls, off);
      lse_merge(lm, ls, om, os);
    }
    if (lane == 0) {
      s_lm[warp] = lm;
      s_ls[warp] = ls;
    }
  }
  __syncthreads();
  if (kLse && tid == 0) {
    float m = s_lm[0], sum = s_ls[0];
    for (int w = 1; w < kWarps; ++w) lse_merge(m, sum, s_lm[w], s_ls[w]);
    if (has_tail)  // the last V % 8 tokens, outside the vector stream
      for (int t = nvec * 8; t < V; ++t) lse_merge(m, sum, bf16_bits_to_float(rowp[t]), 1.f);
    s_lm[0] = m;
    s_ls[0] = sum;
  }

  // ---------------------------------------------------------------- pass 2: bound
  // The bound is the K-th largest group key, found by a two-digit radix
  // select over the (16-bit) group keys: a histogram of the high bytes, the
  // bin holding the K-th largest, then a histogram of the low bytes within
  // it.  Fewer than K groups (a tiny segment) leave the bound at 0: every
  // vector is listed.
  for (int g = tid; g < ng; g += kThreads) atomicAdd(&s_hist[0][s_gkey[g] >> 8], 1);
  __syncthreads();
  if (warp == 0) radix_digit(s_hist[0], K, lane, &s_digit, &s_above);
  __syncthreads();
  const int hb = s_digit;
  if (hb >= 0)
    for (int g = tid; g < ng; g += kThreads)
      if ((s_gkey[g] >> 8) == hb) atomicAdd(&s_hist[1][s_gkey[g] & 0xFF], 1);
  __syncthreads();
  if (warp == 0) {
    int lb = -1, dummy = 0;
    if (hb >= 0) radix_digit(s_hist[1], K - s_above, lane, &lb, &dummy);
    if (lane == 0) s_tkey = (hb >= 0 && lb >= 0) ? ((uint32_t)hb << 8) | (uint32_t)lb : 0u;
  }
  __syncthreads();
  const uint32_t tkey = s_tkey;
  // candidate groups (maximum >= bound), in any order
  for (int g = tid; g < ng; g += kThreads)
    if (s_gkey[g] >= tkey) {
      const int pos = atomicAdd(&s_ncand, 1);
      if (pos < kCandGroups) s_cand[pos] = g;
    }
  __syncthreads();
  const int ncg = s_ncand;
  // each warp takes candidate groups; lane l checks maxima l and l+32 of each.
  // A lane holding more hit vectors than its registers take sends the
  // segment down the degenerate path.
  int nhit = 0;
  if (ncg <= kCandGroups) {
    for (int c = warp; c < ncg; c += kWarps) {
      const int g = s_cand[c];
#pragma unroll
      for (int h = 0; h < kGroup / 32; ++h) {
        const int e = g * kGroup + h * 32 + lane;
        nhit += (e < nv && bf16_order_key(s_vmax[e]) >= tkey);
      }
    }
    if (nhit > kMaxHitsPerLane) atomicMax(&s_flag, 1);
  }
  __syncthreads();
  bool fallback = ncg > kCandGroups || s_flag != 0;

  if (!fallback) {
    // ------------------------------------------------------------ pass 3: select
    // re-load every hit vector of the warp's groups at once, then keep the
    // elements >= bound as exact keys
    nhit = 0;
    int hj[kMaxHitsPerLane];
    for (int c = warp; c < ncg; c += kWarps) {
      const int g = s_cand[c];
#pragma unroll
      for (int h = 0; h < kGroup / 32; ++h) {
        const int e = g * kGroup + h * 32 + lane;
        if (e < nv && bf16_order_key(s_vmax[e]) >= tkey) {
#pragma unroll
          for (int t = 0; t < kMaxHitsPerLane; ++t)  // hj[nhit] with a constant index
            if (t == nhit) hj[t] = v0 + e;
          ++nhit;
        }
      }
    }
    uint4 q[kMaxHitsPerLane];
#pragma unroll
    for (int h = 0; h < kMaxHitsPerLane; ++h)
      if (h < nhit) q[h] = ld_stream(rowp + (int64_t)hj[h] * 8);
    __syncthreads();  // s_vmax is overwritten by the keys below
#pragma unroll
    for (int h = 0; h < kMaxHitsPerLane; ++h) {
      if (h >= nhit) continue;
      const uint32_t wd[4] = {q[h].x, q[h].y, q[h].z, q[h].w};
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const uint32_t bits = (e & 1) ? (wd[e >> 1] >> 16) : (wd[e >> 1] & 0xFFFFu);
        if (bf16_order_key(bits) >= tkey) {
          const int pos = atomicAdd(&s_nkeys, 1);
          if (pos < kCandElems) s_keys[pos] = make_key(bits, (uint32_t)hj[h] * 8u + (uint32_t)e);
        }
      }
    }
    if (has_tail && tid < tail) {
      const uint32_t bits = rowp[(int64_t)nvec * 8 + tid];
      if (bf16_order_key(bits) >= tkey) {
        const int pos = atomicAdd(&s_nkeys, 1);
        if (pos < kCandElems) s_keys[pos] = make_key(bits, (uint32_t)(nvec * 8 + tid));
      }
    }
    __syncthreads();
    const int nkeys = s_nkeys;
    fallback = nkeys > kCandElems;  // too many elements at the bound: degenerate path
    if (!fallback) {
      // exact ranks (keys are unique)
      for (int e = tid; e < nkeys; e += kThreads) {
        const u64 x = s_keys[e];
        int rank = 0;
        for (int j = 0; j < nkeys; ++j) rank += s_keys[j] > x;
        if (rank < K) s_top[rank] = x;
      }
    }
    __syncthreads();
  }
  if (fallback) {
    // ------------------------------------------------------------ degenerate segment
    __syncthreads();  // s_vmax is reused as the candidate buffers below
    const uint32_t floor_key = tkey;
    u64 list = stream_fallback<K>(rowp, w0, w1, floor_key, &s_cta_bound,
                                  s_raw + warp * (kStep * 8), lane);
    // the scalar tail (V % 8 elements) belongs to the last warp
    if (has_tail && warp == kWarps - 1) {
      u64 kth = shfl_u64(list, K - 1);
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
  }

  // everything above only reads the logits; the previous kernel in the stream
  // may still read the buffers written below -- except with the handoff, where
  // the previous kernel is the projection, which waits for this one's rows
  if (!hand.row_ready) pdl_wait();
  if (nseg > 1) {
    u64 *my = part + ((int64_t)row * nseg + seg) * K;
    if (tid < K) {
      my[tid] = s_top[tid];
      __threadfence();
    }
    if (kLse && tid == 0) {
      part_lse[(int64_t)row * nseg + seg] = make_float2(s_lm[0], s_ls[0]);
      __threadfence();
    }
    __syncthreads();
    if (tid == 0) {
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
      if (lane == 0) row_count[row] = 0u;  // ready for the next call
      if (kLse && lane == 0) {
        float m = -INFINITY, sum = 0.f;
        for (int sg = 0; sg < nseg; ++sg) {
          const float2 ms = __ldcg(part_lse + (int64_t)row * nseg + sg);
          lse_merge(m, sum, ms.x, ms.y);
        }
        s_lm[0] = m;
        s_ls[0] = sum;
      }
    }
    __syncthreads();
  }
  if (tid < K) {
    const u64 x = s_top[tid];
    const uint32_t id = 0xFFFFFFFFu - (uint32_t)(x & 0xFFFFFFFFull);
    const float val = order_key_to_float((uint32_t)(x >> 32));
    out_ids[(int64_t)row * K + tid] = (int32_t)id;
    out_val[(int64_t)row * K + tid] = val;
    if (kLse) {
      const float m = s_lm[0];
      const float lse = m == -INFINITY ? -INFINITY : m + __logf(s_ls[0]);
      const float top = order_key_to_float((uint32_t)(s_top[0] >> 32));
      const float logp = val == -INFINITY ? -INFINITY : val - lse;
      float *f = out_feat + ((int64_t)row * K + tid) * 5;
      f[0] = logp;
      f[1] = val == -INFINITY ? 0.f : __expf(logp);
      f[2] = top - val;
      f[3] = (float)tid / (float)K;
      f[4] = tid == 0 ? 1.f : 0.f;
    }
  }
  if (hand.row_ready && warp == 0) {
    // hand the row to the projection: release its flag once its ids and
    // values are stored, and bring its candidates' embedding rows to L2
    __syncwarp();
    if (lane == 0) {
      __threadfence();
      asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(hand.row_ready + row), "r"(1u) : "memory");
    }
    if (hand.E && lane < K) {
      const uint32_t id = 0xFFFFFFFFu - (uint32_t)(s_top[lane] & 0xFFFFFFFFull);
      if (id < (uint32_t)V)
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(hand.E + (int64_t)id * hand.d),
                     "r"((uint32_t)hand.d * 2u)
                     : "memory");
    }
  }
}

}  // namespace

TopkPlan topk_plan(int V, int rows, int slots_per_wave) {
  const int nvec = std::max(1, V >> 3);
  const int s_min = (nvec + kMaxSegVecs - 1) / kMaxSegVecs;
  const int s_max = std::max(s_min, std::min(kTopkMaxChunks, nvec / 2048));
  // cost of a launch: waves x (vectors per segment + a fixed per-CTA cost
  // worth ~3000 vectors: the bound, the listing and the selection)
  TopkPlan p;
  p.nchunks = s_min;
  double best = -1.0;
  for (int s = s_min; s <= s_max; ++s) {
    const long long total = (long long)std::max(rows, 1) * s;
    const long long waves = (total + std::max(slots_per_wave, 1) - 1) / std::max(slots_per_wave, 1);
    const double cost = (double)waves * ((nvec + s - 1) / s + 3000);
    if (best < 0 || cost < best - 1e-9) {
      best = cost;
      p.nchunks = s;
    }
  }
  p.chunk_vecs = (nvec + p.nchunks - 1) / p.nchunks;  // vectors per segment
  return p;
}

int topk_max_segment_vecs() { return kMaxSegVecs; }

int topk_min_segments(int V) {
  const int nvec = std::max(1, V >> 3);
  return (nvec + kMaxSegVecs - 1) / kMaxSegVecs;
}

int topk_max_segments(int V) {
  const int nvec = std::max(1, V >> 3);
  const int s_min = (nvec + kMaxSegVecs - 1) / kMaxSegVecs;
  return std::max(s_min, std::min(kTopkMaxChunks, nvec / 2048));
}

template <int K>
static int topk_occupancy_k() {
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k_topk<K, false>, kThreads, 0) != cudaSuccess) {
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

template <int K>
static cudaError_t launch_topk_k(const dim3 &grid, const dim3 &block, cudaStream_t st, bool pdl,
                                 const uint16_t *logits, int64_t stride, int slots, int B, int V, const TopkPlan &plan,
                                 unsigned long long *part, unsigned *row_count, int32_t *ids, float *vals,
                                 float2 *part_lse, float *feat, const TopkHandoff &hand) {
  if (feat)
    return launch_ex(k_topk<K, true>, grid, block, 0, st, pdl, 0, logits, stride, slots, B, V, plan.nchunks,
                     plan.chunk_vecs, part, row_count, ids, vals, part_lse, feat, hand);
  return launch_ex(k_topk<K, false>, grid, block, 0, st, pdl, 0, logits, stride, slots, B, V, plan.nchunks,
                   plan.chunk_vecs, part, row_count, ids, vals, part_lse, feat, hand);
}

cudaError_t launch_topk(int K, const uint16_t *logits, int64_t stride, int slots, int N, int V,
                        const TopkPlan &plan, unsigned long long *part, unsigned *row_count,
                        int32_t *ids, float *vals, cudaStream_t st, bool pdl, float2 *part_lse, float *feat,
                        const TopkHandoff &hand) {
  const int B = slots - 1;
  if (N == 0) return cudaSuccess;
  if (feat && plan.nchunks > 1 && !part_lse) return cudaErrorInvalidValue;
  if (hand.row_ready && feat) return cudaErrorInvalidValue;
  const dim3 grid = hand.row_ready ? dim3(N * B * plan.nchunks, 1) : dim3(N * B, plan.nchunks);
  const dim3 block(kThreads);
  cudaError_t e;
  switch (K) {
    case 8:
      e = launch_topk_k<8>(grid, block, st, pdl, logits, stride, slots, B, V, plan, part, row_count, ids, vals,
                           part_lse, feat, hand);
      break;
    case 16:
      e = launch_topk_k<16>(grid, block, st, pdl, logits, stride, slots, B, V, plan, part, row_count, ids, vals,
                            part_lse, feat, hand);
      break;
    case 32:
      e = launch_topk_k<32>(grid, block, st, pdl, logits, stride, slots, B, V, plan, part, row_count, ids, vals,
                            part_lse, feat, hand);
      break;
    default:
      return cudaErrorInvalidValue;
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace dc
