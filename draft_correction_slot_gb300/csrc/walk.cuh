// walk.cuh -- step 5 for one request: prefix-first greedy walk and greedy
// verify, as a block-wide device function (256 threads).
//
// DCOCO page, Method step details (5) and Core method; LiLiCorr Sec. 3.5
// Eq. (8): the first draft slot takes the draft argmax (candidate 0 of its
// value-sorted pool); then k_{p+1} = argmax_b S_p(k_p, b), ties to the lowest
// b.  "Faster Decoding", greedy-verification contract: accept the longest
// prefix of the proposal that equals the target's greedy tokens.
//
// Every thread first takes (pair p, predecessor a) rows and finds the best
// successor (lowest index on ties) and its gap to the second best, reading
// the scores through L2 (they may have been written by other blocks of the
// same launch); one thread then follows the walk through that table,
// B-1 dependent shared-memory reads.
#pragma once

#include <stdint.h>

#include "common.cuh"

namespace dc {

constexpr int kWalkMaxRows = 31 * 32;  // (B-1) * K, B <= 31, K <= 32

// scores: [(B-1)][K][K] of this request; ids: [B][K]; target: [B] or null.
// s_best / s_gap: kWalkMaxRows entries; s_choice: 32.  Called by every thread
// of the block, which must have 256 threads.
template <int K>
__device__ __forceinline__ void walk_verify_request(const float *scores, const int32_t *ids,
                                                    const int32_t *target, int B, int32_t *tokens,
                                                    int32_t *choice, float *margin, int32_t *accept_len,
                                                    int *s_best, float *s_gap, int *s_choice) {
  const int tid = threadIdx.x;
  const int P = B - 1, rows = P * K;
  for (int r = tid; r < rows; r += 256) {
    float row[K];
    const float4 *src = reinterpret_cast<const float4 *>(scores + (int64_t)r * K);
#pragma unroll
    for (int q = 0; q < K / 4; ++q) {
      const float4 v = __ldcg(src + q);
      row[4 * q] = v.x; row[4 * q + 1] = v.y; row[4 * q + 2] = v.z; row[4 * q + 3] = v.w;
    }
    int best = 0;
    float bv = row[0];
#pragma unroll
    for (int b = 1; b < K; ++b)
      if (row[b] > bv) {
        bv = row[b];
        best = b;
      }
    float second = -INFINITY;
#pragma unroll
    for (int b = 0; b < K; ++b)
      if (b != best) second = fmaxf(second, row[b]);
    s_best[r] = best;
    s_gap[r] = bv - second;
  }
  __syncthreads();
  if (tid == 0) {
    int k = 0;
    s_choice[0] = 0;
    for (int p = 0; p < P; ++p) {
      k = s_best[p * K + k];
      s_choice[p + 1] = k;
    }
  }
  __syncthreads();
  if (tid < 32) {
    int tok = 0;
    if (tid < B) {
      const int k = s_choice[tid];
      tok = ids[tid * K + k];
      tokens[tid] = tok;
      if (choice) choice[tid] = k;
      if (margin && tid < P) margin[tid] = s_gap[tid * K + k];
    }
    if (target) {
      const bool mismatch = tid < B && tok != target[tid];
      const unsigned mm = __ballot_sync(DC_FULL_MASK, mismatch);
      if (tid == 0) *accept_len = mm ? (__ffs(mm) - 1) : B;
    }
  }
}

}  // namespace dc
