// walk.cu -- step 5: prefix-first greedy walk and greedy verify.
//
// DCOCO page, Method step details (5) and Core method; LiLiCorr Sec. 3.5
// Eq. (8): the first draft slot takes the draft argmax (candidate 0 of its
// value-sorted pool); then k_{p+1} = argmax_b S_p(k_p, b), ties to the lowest
// b.  The walk is O(B K) and touches no weights.
// "Faster Decoding", greedy-verification contract: accept the longest prefix
// of the proposal that equals the target's greedy tokens.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace dc {
namespace {

// One CTA per request.  The request's (B-1) K x K scores are staged in
// shared memory (rows padded to K+1 floats: conflict-free row scans); every
// thread then finds, for one (pair p, predecessor a) row, the best successor
// (lowest index on ties) and the gap to the second best; finally one thread
// follows the walk through that table, B-1 dependent shared-memory reads.
constexpr int kMaxRows = 31 * 32;  // (B-1) * K, B <= 31, K <= 32

template <int K>
__global__ void __launch_bounds__(256)
k_walk_verify(const float *__restrict__ scores, const int32_t *__restrict__ topk_ids,
              const int32_t *__restrict__ target, int N, int B, int32_t *__restrict__ tokens,
              int32_t *__restrict__ choice, float *__restrict__ margin,
              int32_t *__restrict__ accept_len) {
  extern __shared__ float sc[];  // [(B-1) K][K+1]
  __shared__ int s_best[kMaxRows];
  __shared__ float s_gap[kMaxRows];
  __shared__ int s_choice[32];
  const int n = blockIdx.x, tid = threadIdx.x;
  const int P = B - 1, rows = P * K;
  const float *src = scores + (int64_t)n * rows * K;
  for (int e0 = 0; e0 < rows * K; e0 += 256 * 8) {
    float v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int e = e0 + tid + 256 * u;
      if (e < rows * K) v[u] = __ldg(src + e);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int e = e0 + tid + 256 * u;
      if (e < rows * K) sc[(e / K) * (K + 1) + (e % K)] = v[u];
    }
  }
  __syncthreads();
  for (int r = tid; r < rows; r += 256) {
    const float *row = sc + r * (K + 1);
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
  const int64_t slot0 = (int64_t)n * B;
  if (tid < 32) {
    int tok = 0;
    if (tid < B) {
      const int k = s_choice[tid];
      tok = topk_ids[(slot0 + tid) * K + k];
      tokens[slot0 + tid] = tok;
      if (choice) choice[slot0 + tid] = k;
      if (margin && tid < P) margin[(int64_t)n * P + tid] = s_gap[tid * K + k];
    }
    if (target) {
      const bool mismatch = tid < B && tok != target[slot0 + tid];
      const unsigned mm = __ballot_sync(DC_FULL_MASK, mismatch);
      if (tid == 0) accept_len[n] = mm ? (__ffs(mm) - 1) : B;
    }
  }
}

}  // namespace

template <int K>
static cudaError_t walk_k(const float *scores, const int32_t *topk_ids, const int32_t *target, int N,
                          int B, int32_t *tokens, int32_t *choice, float *margin, int32_t *accept_len,
                          cudaStream_t st) {
  const size_t smem = (size_t)(B - 1) * K * (K + 1) * sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(k_walk_verify<K>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  k_walk_verify<K><<<N, 256, smem, st>>>(scores, topk_ids, target, N, B, tokens, choice, margin,
                                         accept_len);
  return cudaGetLastError();
}

cudaError_t launch_walk_verify(int K, const float *scores, const int32_t *topk_ids,
                               const int32_t *target, int N, int B, int32_t *tokens,
                               int32_t *choice, float *margin, int32_t *accept_len,
                               cudaStream_t st) {
  if (N == 0) return cudaSuccess;
  switch (K) {
    case 8: return walk_k<8>(scores, topk_ids, target, N, B, tokens, choice, margin, accept_len, st);
    case 16: return walk_k<16>(scores, topk_ids, target, N, B, tokens, choice, margin, accept_len, st);
    case 32: return walk_k<32>(scores, topk_ids, target, N, B, tokens, choice, margin, accept_len, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace dc
