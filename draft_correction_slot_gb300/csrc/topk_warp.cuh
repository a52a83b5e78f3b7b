// topk_warp.cuh -- warp-level pieces of the top-K kernels: 64-bit
// (value, id) keys and warp-held descending lists of the K best keys.
//
// A key packs order16(value) << 32 | (2^32 - 1 - id), so one unsigned
// compare orders by value descending, then by token id ascending (the
// top-K order of the DCOCO page's step (1) with the lowest-index tie rule).
#pragma once

#include <stdint.h>

#include "common.cuh"

namespace dc {
namespace topk_warp {

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

__device__ __forceinline__ u64 shfl_xor_key(u64 v, int m) {
  uint32_t lo = __shfl_xor_sync(DC_FULL_MASK, (uint32_t)v, m);
  uint32_t hi = __shfl_xor_sync(DC_FULL_MASK, (uint32_t)(v >> 32), m);
  return ((u64)hi << 32) | lo;
}
__device__ __forceinline__ u64 shfl_key(u64 v, int src) { return shfl_u64(v, src); }

// Bitonic sort of one key per lane, descending over the 32 lanes.
template <class T>
__device__ __forceinline__ T warp_sort32_desc(T x, int lane) {
#pragma unroll
  for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      const T o = shfl_xor_key(x, j);
      const bool keep_max = (((lane & j) == 0) == ((lane & k) == 0));
      x = keep_max ? (o > x ? o : x) : (o < x ? o : x);
    }
  }
  return x;
}

// Top K of two descending lists held in lanes (a: lanes < K, b: 32 lanes,
// zero padded): max(a_i, b_{K-1-i}) is the top-K set as a bitonic sequence;
// a half-cleaner network sorts it.
template <int K, class T>
__device__ __forceinline__ T warp_merge_topk(T a, T b, int lane) {
  const T br = shfl_key(b, (K - 1 - lane) & 31);
  T x = (lane < K) ? (a > br ? a : br) : T(0);
#pragma unroll
  for (int j = K >> 1; j > 0; j >>= 1) {
    const T o = shfl_xor_key(x, j);
    const bool lower = (lane & j) == 0;
    x = lower ? (o > x ? o : x) : (o < x ? o : x);
  }
  return lane < K ? x : T(0);
}

// bf16 bits with order key one below / above `key` (saturating).
__device__ __forceinline__ uint32_t bf16_from_key(uint32_t key) {
  return (key & 0x8000u) ? (key & 0x7FFFu) : (~key & 0xFFFFu);
}


// One warp: the digit d of a 256-bin histogram (bins scanned from 255 down)
// whose bin holds the rank-th largest key (rank >= 1), and the number of keys
// in the bins above it, returned to every lane.  digit = -1 when the
// histogram holds fewer than rank keys.  Lane l reads bins 255 - 8l ... 248 - 8l.
__device__ __forceinline__ void warp_radix_digit(const int *hist, int rank, int lane, int &digit, int &above) {
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
  const int excl = incl - sum;
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
  digit = -1;
  above = 0;
  if (m) {
    const int src = __ffs(m) - 1;
    digit = __shfl_sync(DC_FULL_MASK, d, src);
    above = __shfl_sync(DC_FULL_MASK, ab, src);
  }
}

}  // namespace topk_warp
}  // namespace dc
