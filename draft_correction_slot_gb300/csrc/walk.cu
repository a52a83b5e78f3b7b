// walk.cu -- step 5: prefix-first greedy walk and greedy verify.
//
// DCOCO page, Method step details (5) and Core method; LiLiCorr Sec. 3.5
// Eq. (8): the first draft slot takes the draft argmax (candidate 0 of its
// value-sorted pool); then k_{p+1} = argmax_b S_p(k_p, b), ties to the lowest
// b.  The walk is O(B K) and touches no weights.
// "Faster Decoding", greedy-verification contract: accept the longest prefix
// of the proposal that equals the target's greedy tokens.
//
// One warp per request; lane b holds S_p(k_p, b).
#include "common.cuh"
#include "kernels.h"

namespace dc {
namespace {

template <int K>
__global__ void __launch_bounds__(256)
k_walk_verify(const float *__restrict__ scores, const int32_t *__restrict__ topk_ids,
              const int32_t *__restrict__ target, int N, int B, int32_t *__restrict__ tokens,
              int32_t *__restrict__ choice, float *__restrict__ margin,
              int32_t *__restrict__ accept_len) {
  const int lane = threadIdx.x & 31;
  const int n = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (n >= N) return;
  const int64_t slot0 = (int64_t)n * B;
  int k = 0;
  int my_token = 0;  // lane i keeps the token of slot i (B <= 31)
  if (lane == 0) my_token = topk_ids[slot0 * K];
  if (lane == 0 && choice) choice[slot0] = 0;

  for (int p = 0; p < B - 1; ++p) {
    const float *row = scores + (((int64_t)n * (B - 1) + p) * K + k) * K;
    const float v = lane < K ? row[lane] : -INFINITY;
    float bv = v;
    int bi = lane < K ? lane : 0x7fffffff;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(DC_FULL_MASK, bv, o);
      const int oi = __shfl_xor_sync(DC_FULL_MASK, bi, o);
      if (ov > bv || (ov == bv && oi < bi)) {
        bv = ov;
        bi = oi;
      }
    }
    const float second = warp_max(lane == bi ? -INFINITY : v);
    k = bi;
    const int32_t tok = topk_ids[(slot0 + p + 1) * K + k];
    if (lane == p + 1) my_token = tok;
    if (lane == 0) {
      if (choice) choice[slot0 + p + 1] = k;
      if (margin) margin[(int64_t)n * (B - 1) + p] = bv - second;
    }
  }
  if (lane < B) tokens[slot0 + lane] = my_token;
  if (target) {
    const bool mismatch = lane < B && my_token != target[slot0 + lane];
    const unsigned mm = __ballot_sync(DC_FULL_MASK, mismatch);
    if (lane == 0) accept_len[n] = mm ? (__ffs(mm) - 1) : B;
  }
}

}  // namespace

cudaError_t launch_walk_verify(int K, const float *scores, const int32_t *topk_ids,
                               const int32_t *target, int N, int B, int32_t *tokens,
                               int32_t *choice, float *margin, int32_t *accept_len,
                               cudaStream_t st) {
  if (N == 0) return cudaSuccess;
  const int grid = (N + 7) / 8;
  switch (K) {
    case 8: k_walk_verify<8><<<grid, 256, 0, st>>>(scores, topk_ids, target, N, B, tokens, choice, margin, accept_len); break;
    case 16: k_walk_verify<16><<<grid, 256, 0, st>>>(scores, topk_ids, target, N, B, tokens, choice, margin, accept_len); break;
    case 32: k_walk_verify<32><<<grid, 256, 0, st>>>(scores, topk_ids, target, N, B, tokens, choice, margin, accept_len); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace dc
