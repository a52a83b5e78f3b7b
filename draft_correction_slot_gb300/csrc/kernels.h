// kernels.h -- internal launchers of the library's CUDA kernels.
// Every launcher enqueues on `st` and returns the cudaGetLastError() of its
// launch; none allocates or synchronises.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace dc {

// ---------------------------------------------------------------- top-K
// Segmented top-K: each logits row is cut into `nchunks` segments of
// `chunk_vecs` 16-byte vectors, one CTA per (row, segment).  With several
// segments, every CTA publishes its best K to `part` (rows * nchunks * K
// packed keys) and the last CTA of the row, counted in `row_count` (rows
// entries, zero between calls), merges them.  With `pdl` the launch may
// overlap the end of the previous kernel in the stream (the kernel waits for
// it before its first global write).
struct TopkPlan {
  int nchunks;     // segments per row
  int chunk_vecs;  // 16-byte vectors per segment
};
constexpr int kTopkThreads = 256;
constexpr int kTopkMaxChunks = 64;
// Segment count that gives the shortest launch for `rows` rows on a device
// holding `slots_per_wave` resident top-K CTAs.
TopkPlan topk_plan(int V, int rows, int slots_per_wave);
int topk_min_segments(int V);  // fewest segments whose per-vector maxima fit a CTA
int topk_max_segment_vecs();   // 16-byte vectors a segment may hold
int topk_max_segments(int V);
int topk_occupancy(int K);  // resident top-K CTAs per SM
// With `feat` (fp32 [rows][K][5]) the same pass also accumulates each row's
// log-sum-exp and writes the candidates' vocabulary-normalised features
// [log p, p, l_0 - l_k, k / K, k == 0]; part_lse (float2 [rows][nchunks]) is
// then needed when nchunks > 1.
// Handoff to a projection already running beside the top-K (launched
// before it): the grid is one-dimensional with a row's segments adjacent, so
// rows finish in order; each finished row releases row_ready[row] = 1 (the
// projection clears it) and its candidates' embedding rows E[id] (d bf16
// each) are prefetched into L2.  The kernel then does not wait for the
// previous kernel in the stream (it is the projection, which waits for it).
struct TopkHandoff {
  unsigned *row_ready = nullptr;
  const uint16_t *E = nullptr;
  int d = 0;
};
cudaError_t launch_topk(int K, const uint16_t *logits, int64_t stride, int slots, int N, int V,
                        const TopkPlan &plan, unsigned long long *part, unsigned *row_count,
                        int32_t *ids, float *vals, cudaStream_t st, bool pdl, float2 *part_lse = nullptr,
                        float *feat = nullptr, const TopkHandoff &hand = TopkHandoff());

// ---------------------------------------------------------------- projections
// C[m][o] = sum_k A_m[k] * W[o][k] with A_m a bf16 row of length d, on the
// tensor cores.  A job with `ids` gathers A_m = table[ids[m]] (ids < V, else
// the device status word gets kErrBadCandidateId and row 0 is used); a job
// without takes A_m = table[(m / B) * slots + (m % B) + 1] (the draft-slot
// rows of a [N][slots][d] tensor).  W comes as bf16 hi and lo halves ([No][d]
// each, No % 128 == 0, d % 64 == 0) through two TMA maps (box 64 x 128).
// A CTA owns 256 rows x 128 outputs of one job; `splits` (a power of two
// <= 8, from proj_tc_splits) splits the k range over the CTAs of one
// cluster, which add their partial tiles through distributed shared memory.
// One launch runs one or two jobs, the second one's tiles after the first's.
// With `pdl` the launch may overlap the end of the previous kernel in the
// stream (a gathering job waits for it before it reads the row ids; a
// draft-slot job does not wait).
struct ProjJob {
  const uint16_t *table;  // bf16 [rows][d]
  const int32_t *ids;     // [M] table rows, or null for draft-slot rows
  float *C;               // fp32 [M][No]
  int M, No;
  int tiles;              // proj_tc_tiles(M, No)
  // With ln_hi set (No == 128), each output row leaves as LN0(row) (non-
  // affine, eps ln_eps) split into bf16 hi ([M][128], ln_hi) and lo (the
  // rounding remainder, ln_lo) instead of fp32 in C.
  uint16_t *ln_hi = nullptr, *ln_lo = nullptr;
  float ln_eps = 0.f;
  // With row_ready set (a gathering job launched before the top-K that
  // fills it, see TopkHandoff), a tile waits for the flags of its draft-slot
  // rows (candidate m belongs to row m / cands_per_row) instead of for the
  // previous kernel, and clears them when done.
  unsigned *row_ready = nullptr;
  int cands_per_row = 0;
  // fp16 instead of bf16 hi + lo: A is converted in shared memory (its values
  // must lie within the fp16 range, |a| < 65504) and W comes as one fp16
  // matrix through the `hi` map (the `lo` map is not read).
  bool f16 = false;
};
int proj_tc_splits(int d, int requested);
int proj_tc_tiles(int M, int No);
// 2D bf16 [rows][d] tensor map, 128B swizzle, box 64 x box_rows.
bool encode_bf16_rows_map(CUtensorMap *map, const void *base, int rows, int d, int box_rows);
// The same for fp16 elements.
bool encode_f16_rows_map(CUtensorMap *map, const void *base, int rows, int d, int box_rows);
// 2D fp32 [rows][cols] tensor map, 128B swizzle, box 32 x box_rows
// (cols % 32 == 0).
bool encode_f32_rows_map(CUtensorMap *map, const void *base, int rows, int cols, int box_rows);
cudaError_t launch_proj_tc(const ProjJob &a, const CUtensorMap &a_hi, const CUtensorMap &a_lo,
                           const ProjJob *b, const CUtensorMap *b_hi, const CUtensorMap *b_lo, int slots,
                           int B, int d, int V, int splits, int *err, cudaStream_t st, bool pdl);

// ---------------------------------------------------------------- representations
struct MlpWeightsDev {
  const float *w_la;    // [H]     W1[:, 3r]
  const float *w_lb;    // [H]     W1[:, 3r+1]
  const float *b1;      // [H]  b1 + W1[:, r:2r] beta + W1[:, 2r:3r] beta
  const float *w2;      // [H]
  const float *b2;      // [1]
  const float *w_fg;    // [r][r]  W_fuse[:, r:], in the candidate maps' register order
};

// Tensor-core forms of the per-slot and per-candidate steps.  The maps
// address bf16 hi / lo halves (box 64 x 128, 128B swizzle) of W_fuse[:, :r]
// and W_fuse[:, r:] ([r][r] each), [W1[:, r:2r] ; W1[:, 2r:3r]] diag(gamma)
// ([2H][r]) and W1[:, :r] ([H][r]).
struct MlpMaps {
  CUtensorMap fb_hi, fb_lo, w1_hi, w1_lo, fg_hi, fg_lo, w1s_hi, w1s_lo;
};
// The per-slot and per-candidate maps, in one launch (no block waits for
// another).  Per draft slot i (used for i < B-1):
// P_i = W1[:, :r] (W_pair[:, :d] h_i + W_pair[:, d:] h_{i+1}) + b1' ([rows][H]),
// b1' = b1 + W1[:, r:2r] beta + W1[:, 2r:3r] beta.
// slot_proj is [N*B][3r] = (W_ctx h | W_pair[:, :d] h | W_pair[:, d:] h).
// Per candidate: b = LN0(W_cand E[c]) (from the projection, as bf16 hi and
// lo), g = LN0(W_ctx h) of its slot,
// z = gamma*LN0(W_fuse[:, :r] b + W_fuse[:, r:] g) + beta,
// U = W1_a z + w_la l, V = W1_b z + w_lb l, computed as U = (W1_a diag(gamma))
// n + w_la l with n = LN0(...) (beta's share W1_a beta + W1_b beta is in P,
// so P + U + V is unchanged).  M = N * B * K candidates
// (8 <= K, K divides 128), candidate m belongs to draft slot m / K.
// Tiles move by TMA: `slot.sp` reads slot_proj, `slot.p` writes P,
// `cand.u` / `cand.v` write U and V ([rows][H]) -- fp32 maps with box
// 32 x 128 -- and `cand.bh` / `cand.bl` read b's hi and lo halves (bf16
// [rows][r], box 64 x 128), all over at least the call's rows (rows of the
// last tile past the call's count receive the outputs of stale or all-zero
// input rows).  The launch may overlap the end of the previous kernel
// (programmatic serialization).
struct SlotIoMaps {
  CUtensorMap sp, p;
};
struct CandIoMaps {
  CUtensorMap bh, bl, u, v;
};
cudaError_t launch_maps_tc(const MlpMaps &maps, const SlotIoMaps &slot, const CandIoMaps &cand,
                           const float *slot_proj, const float *topk_val, const MlpWeightsDev &w, int N, int B,
                           int K, float eps, int *err, cudaStream_t st);

// Step 5 outputs and state for a launch that ends with the walk: per-request
// arrays (tokens, choice, accept_len [N][B] / [N]; margin [N][B-1]; target or
// null) and req_count (N entries, zero between calls) counting each
// request's finished pairs.  path_rule 0: prefix-first greedy walk; 1:
// highest-scoring path (Viterbi); 2: beam walk (beam_width 1..4, beam_topm
// 1..K).
struct WalkArgs {
  const int32_t *topk_ids;
  const int32_t *target;  // or null
  int32_t *tokens, *choice, *accept_len;
  float *margin;
  unsigned *req_count;
  int path_rule;    // 0: prefix-first greedy walk, 1: highest-scoring path, 2: beam walk
  int beam_width;   // path rule 2: partial paths kept, 1..4
  int beam_topm;    // path rule 2: successors per predecessor, 1..K
};

// S[n,p,a,b] = l_{p+1}(b) + b2 + sum_j w2_j GELU(P_pj + U_{p,a,j} + V_{p+1,b,j}),
// with P indexed by draft slot ([N*B][H]),
// then, in the last block of each request, its path selection and verify.
cudaError_t launch_pair_score_walk(int K, const float *U, const float *V, const float *P,
                                   const float *topk_val, const float *w2, const float *b2, int N, int B,
                                   float *scores, const WalkArgs &wk, cudaStream_t st);

// ---------------------------------------------------------------- cosine variant
// y = cand_io[m] + slot_io[slot(m)] ([M][2r] and [N*B][2r]), the out half
// (columns 0..r-1) and the in half L2-normalised (x / max(|x|, 1e-12));
// S[n,p,a,b] = sigma <o_{p,a}, i_{p+1,b}> + l_{p+1}(b); then, in the last
// block of each request, its path selection and verify.
cudaError_t launch_cos_pair_walk(int K, const float *cand_io, const float *slot_io, const float *topk_val,
                                 float sigma, int N, int B, float *scores, const WalkArgs &wk, cudaStream_t st);

// ---------------------------------------------------------------- stochastic verify
// Point-mass proposal `tokens` [N][B] against target logits [N][B+1][stride]
// (bf16; row B of a request is the bonus position), temperature 1: slot j is
// accepted iff u_acc[n][j] < q_j(y_j); at the first rejection the corrected
// token is drawn from q_j without y_j, after B acceptances from row B; a draw
// takes the smallest token whose cumulative weight (vocabulary order)
// exceeds u_draw[n] times the total.  Scratch: chunk_m / chunk_s
// [N*(B+1)][verify_chunks(V)], row_lse [N*(B+1)], req_count [N] (zero
// between calls).  q_acc [N][B] receives q_j(y_j).
int verify_chunks(int V);
cudaError_t launch_verify_stochastic(const uint16_t *target, int64_t stride, int V, int N, int B,
                                     const int32_t *tokens, const float *u_acc, const float *u_draw,
                                     float *chunk_m, float *chunk_s, float *row_lse, float *q_acc,
                                     unsigned *req_count, int32_t *accept_len, int32_t *next_token,
                                     cudaStream_t st);

// One CTA waits (tc::mbar_wait, limit_ns) on an mbarrier nothing completes:
// the wait expires and ORs kErrTimeout into *err.
cudaError_t launch_wait_timeout(unsigned long long limit_ns, int *err, cudaStream_t st);

}  // namespace dc
