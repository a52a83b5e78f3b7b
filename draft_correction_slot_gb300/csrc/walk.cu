// walk.cu -- step 5 as its own launch (the cosine variant; the MLP variant
// runs it in the last block of each request's pair scores): one block per
// request, see walk.cuh.  path_rule 0: greedy walk, 1: highest-scoring path,
// 2: beam walk.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "walk.cuh"

namespace dc {
namespace {

template <int K>
__global__ void __launch_bounds__(256)
k_walk_verify(const float *__restrict__ scores, const int32_t *__restrict__ topk_ids,
              const int32_t *__restrict__ target, int N, int B, int32_t *__restrict__ tokens,
              int32_t *__restrict__ choice, float *__restrict__ margin,
              int32_t *__restrict__ accept_len, int path_rule, int beam_width, int beam_topm) {
  __shared__ int s_best[kWalkMaxRows];
  __shared__ float s_gap[kWalkMaxRows];
  __shared__ int s_choice[32];
  const int n = blockIdx.x, P = B - 1;
  const int64_t slot0 = (int64_t)n * B;
  const float *sc = scores + (int64_t)n * P * K * K;
  const int32_t *tg = target ? target + slot0 : nullptr;
  int32_t *ch = choice ? choice + slot0 : nullptr, *al = accept_len ? accept_len + n : nullptr;
  float *mg = margin ? margin + (int64_t)n * P : nullptr;
  extern __shared__ float4 s_dyn[];  // the request's scores, when the launch gave room for them
  const bool fits = (size_t)P * K * K * sizeof(float) <= dynamic_smem_bytes();
  if (path_rule == 1)
    viterbi_verify_request<K>(sc, topk_ids + slot0 * K, tg, B, tokens + slot0, ch, mg, al, s_best, s_gap, s_choice,
                              fits ? reinterpret_cast<float *>(s_dyn) : nullptr);
  else if (path_rule == 2)
    beam_verify_request<K>(sc, topk_ids + slot0 * K, tg, B, tokens + slot0, ch, mg, al, beam_width, beam_topm, s_best,
                           s_gap, s_choice, fits ? reinterpret_cast<float *>(s_dyn) : nullptr);
  else
    walk_verify_request<K>(sc, topk_ids + slot0 * K, tg, B, tokens + slot0, ch, mg, al, s_best, s_gap, s_choice);
}

}  // namespace

template <int K>
static cudaError_t walk_k(const float *scores, const int32_t *topk_ids, const int32_t *target, int N,
                          int B, int32_t *tokens, int32_t *choice, float *margin, int32_t *accept_len,
                          int path_rule, int beam_width, int beam_topm, cudaStream_t st) {
  // the highest-scoring path and the beam walk read the request's scores from shared memory
  // when they fit the default 48 KB window
  const size_t sc_bytes = (size_t)(B - 1) * K * K * sizeof(float);
  const size_t dyn = path_rule != 0 && sc_bytes <= 48 * 1024 ? sc_bytes : 0;
  k_walk_verify<K><<<N, 256, dyn, st>>>(scores, topk_ids, target, N, B, tokens, choice, margin,
                                           accept_len, path_rule, beam_width, beam_topm);
  return cudaGetLastError();
}

cudaError_t launch_walk_verify(int K, const float *scores, const int32_t *topk_ids,
                               const int32_t *target, int N, int B, int32_t *tokens,
                               int32_t *choice, float *margin, int32_t *accept_len,
                               int path_rule, int beam_width, int beam_topm, cudaStream_t st) {
  if (N == 0) return cudaSuccess;
  switch (K) {
    case 8:
      return walk_k<8>(scores, topk_ids, target, N, B, tokens, choice, margin, accept_len, path_rule, beam_width,
                       beam_topm, st);
    case 16:
      return walk_k<16>(scores, topk_ids, target, N, B, tokens, choice, margin, accept_len, path_rule, beam_width,
                        beam_topm, st);
    case 32:
      return walk_k<32>(scores, topk_ids, target, N, B, tokens, choice, margin, accept_len, path_rule, beam_width,
                        beam_topm, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace dc
