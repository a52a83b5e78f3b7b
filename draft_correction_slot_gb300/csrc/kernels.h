// kernels.h -- internal launchers of the library's CUDA kernels.
// Every launcher enqueues on `st` and returns the cudaGetLastError() of its
// launch; none allocates or synchronises.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace dc {

// ---------------------------------------------------------------- top-K
// Split-vocabulary top-K: logits row size V is cut into `nchunks` chunks of
// `chunk_vecs` 16-byte vectors; one CTA per (row, chunk) keeps its chunk's
// best K in `part` (rows*nchunks*K packed keys), and the last CTA of each row
// (counted in `row_count`, rows entries, zero between calls) merges them.
struct TopkPlan {
  int nchunks;
  int chunk_vecs;
};
constexpr int kTopkThreads = 256;
constexpr int kTopkVecPerThread = 8;
constexpr int kTopkMaxChunks = 64;
TopkPlan topk_plan(int V);
cudaError_t launch_topk(int K, const uint16_t *logits, int64_t stride, int slots, int N, int V,
                        const TopkPlan &plan, unsigned long long *part, unsigned *row_count,
                        int32_t *ids, float *vals, cudaStream_t st);

// ---------------------------------------------------------------- projections
// C[m][o] = sum_k A_m[k] * W[o][k] with A_m a bf16 row of length d and W fp32
// [No][d].  Row addressing: mode 0 gathers A_m = base[ids[m]] (ids < V, else
// the device error word gets kErrBadCandidateId and row 0 is used); mode 1
// takes A_m = base[(m / B) * slots + (m % B) + 1] (the draft-slot rows of a
// [N][slots][d] tensor).
cudaError_t launch_rows_gemm(int mode, const uint16_t *base, const int32_t *ids, int slots, int B,
                             int M, int d, int V, const float *W, int No, float *C, int *err,
                             cudaStream_t st);

// ---------------------------------------------------------------- representations
struct MlpWeightsDev {
  const float *wfb_t;   // [r][r]  W_fuse[:, :r] transposed ([in][out])
  const float *wfg_t;   // [r][r]  W_fuse[:, r:] transposed
  const float *gamma;   // [r]
  const float *beta;    // [r]
  const float *w1s_t;   // [r][H]  W1[:, 0:r] transposed
  const float *w1a_t;   // [r][H]  W1[:, r:2r] transposed
  const float *w1b_t;   // [r][H]  W1[:, 2r:3r] transposed
  const float *w_la;    // [H]     W1[:, 3r]
  const float *w_lb;    // [H]     W1[:, 3r+1]
  const float *b1;      // [H]
  const float *w2;      // [H]
  const float *b2;      // [1]
};

// Per draft slot: g = LN0(ctx), Gf = W_fuse[:, r:] g; per pair:
// s_p = Hp_p + Hq_{p+1}, P_p = W1_s s_p + b1.  slot_proj is [N*B][3r] =
// (W_ctx h | W_pair[:, :d] h | W_pair[:, d:] h).
cudaError_t launch_slot_post(const float *slot_proj, int N, int B, float eps, const MlpWeightsDev &w,
                             float *Gf, float *P, cudaStream_t st);

// Per candidate: b = LN0(cand_proj), z = gamma*LN0(W_fuse[:, :r] b + Gf) + beta,
// U = W1_a z + w_la l, V = W1_b z + w_lb l.
cudaError_t launch_cand_post(int K, const float *cand_proj, const float *topk_val, const float *Gf,
                             int N, int B, float eps, const MlpWeightsDev &w, float *U, float *V,
                             cudaStream_t st);

// S[n,p,a,b] = l_{p+1}(b) + b2 + sum_j w2_j GELU(P_pj + U_{p,a,j} + V_{p+1,b,j}).
cudaError_t launch_pair_score(int K, const float *U, const float *V, const float *P,
                              const float *topk_val, const float *w2, const float *b2, int N, int B,
                              float *scores, cudaStream_t st);

// ---------------------------------------------------------------- cosine variant
// y = cand_io[m] + slot_io[slot(m)]; out/in halves L2-normalised -> O, I [M][r].
cudaError_t launch_cos_post(int K, const float *cand_io, const float *slot_io, int N, int B,
                            float *O, float *I, cudaStream_t st);
cudaError_t launch_cos_score(int K, const float *O, const float *I, const float *topk_val,
                             float sigma, int N, int B, float *scores, cudaStream_t st);

// ---------------------------------------------------------------- walk + verify
cudaError_t launch_walk_verify(int K, const float *scores, const int32_t *topk_ids,
                               const int32_t *target, int N, int B, int32_t *tokens,
                               int32_t *choice, float *margin, int32_t *accept_len,
                               cudaStream_t st);

}  // namespace dc
