/*
 * oracle.h -- plain CPU reference of the DCOCO draft-correction path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code with
 * the CUDA library: no headers, helpers, tables or constants.
 *
 * Sources (pages, by title):
 *   [DCOCO]    "Contextual Correction of Parallel Drafts for Speculative
 *              Decoding" (paper summary page): "Core method" section and
 *              "Method step details" items (1)-(5).
 *   [LiLiCorr] "LiLiCorr: Lightweight Likelihood Correlation of Parallel
 *              Drafts for Speculative Decoding": Sec. 3.2 Eq. (1) (cosine
 *              matching), Sec. 3.5 Eq. (8) (greedy walk), App. E Eq. (12)
 *              (highest-scoring path, Viterbi), App. A (top-K fused with
 *              the vocabulary normalisation of the candidate features).
 *   The [DCOCO] page's reproduction assessment, weaknesses (2)-(3): the beam
 *              walk with top-m successors; its "Core method": stochastic
 *              verification of a point-mass proposal.
 *   [FD]       "Faster Decoding" (textbook chapter): the expected-yield
 *              identity E[Y] = 1 + sum_k s_k and the greedy-verification
 *              contract.
 *
 * Arithmetic: bf16 inputs are widened exactly; fp32 weights are used as given;
 * every sum is accumulated in double.  Layouts are row-major, Linear weights
 * are [out][in].
 *
 * Parity status: every function here is pinned by a CPU test against a value
 * the pages print, a closed form, a library routine or brute force, except
 * the learned-score VALUES of a trained corrector, which the pages never print
 * (there are no trained weights): for those, parity rests on the structural
 * pins (zero output layer, single-feature probes, parameter count).
 */
#ifndef DCOCO_ORACLE_H
#define DCOCO_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
  int V;        /* vocabulary size */
  int d;        /* hidden / embedding width */
  int slots;    /* block positions, anchor included (16) -> B = slots-1 draft slots */
  int K;        /* candidates per draft slot */
  int r;        /* representation width (128) */
  int H;        /* MLP hidden width (256) */
  double ln_eps;
  int beam_width; /* path rule 2: partial paths kept (>= 1)      */
  int beam_topm;  /* path rule 2: successors per beam (0 = all K) */
} orc_dims;

typedef struct {            /* fp32, row-major, [out][in] */
  const float *w_cand;      /* [r][d]           */
  const float *w_ctx;       /* [r][d]           */
  const float *w_fuse;      /* [r][2r]          */
  const float *ln_gamma;    /* [r]              */
  const float *ln_beta;     /* [r]              */
  const float *w_pair;      /* [r][2d]          */
  const float *w1;          /* [H][3r+2]        */
  const float *b1;          /* [H]              */
  const float *w2;          /* [H]              */
  const float *b2;          /* [1]              */
  const float *w_io;        /* [2r][2d], cosine variant only */
} orc_weights;

typedef struct {            /* optional per-request intermediates (NULL = skip) */
  double *b;                /* [B][K][r]  LN0(W_cand E[c])            */
  double *g;                /* [B][r]     LN0(W_ctx h_i)              */
  double *z;                /* [B][K][r]  affine-LN fused candidate   */
  double *s;                /* [B-1][r]   slot-pair state             */
  double *o;                /* [B][K][r]  cosine variant out vectors  */
  double *in;               /* [B][K][r]  cosine variant in vectors   */
} orc_intermediates;

double orc_bf16_to_double(uint16_t bits);

/* Step 1: top-K of one logit row, value descending then id ascending. */
void orc_topk_row(const uint16_t *row, int V, int K, int32_t *ids, float *vals);

/* Non-affine LayerNorm: (x - mean) / sqrt(var_pop + eps). */
void orc_ln0(const double *x, int n, double eps, double *y);

/* y = W x with W fp32 [out][in]. */
void orc_matvec(const float *W, int out, int in, const double *x, double *y);

/* GELU, exact erf form. */
double orc_gelu(double x);

/* Step 2: g = LN0(W_ctx h). */
void orc_context(const orc_dims *dm, const orc_weights *w, const uint16_t *h, double *g);

/* Step 2: b = LN0(W_cand e), z = gamma * LN0(W_fuse [b; g]) + beta. */
void orc_candidate(const orc_dims *dm, const orc_weights *w, const uint16_t *e,
                   const double *g, double *b, double *z);

/* Step 3: s_p = W_pair [h_p; h_{p+1}]. */
void orc_pair_state(const orc_dims *dm, const orc_weights *w, const uint16_t *h_p,
                    const uint16_t *h_q, double *s);

/* Step 4: S = l_b + b2 + w2 . GELU(W1 [s; z_a; z_b; l_a; l_b] + b1). */
double orc_transition(const orc_dims *dm, const orc_weights *w, const double *s,
                      const double *z_a, const double *z_b, double l_a, double l_b);

/* Cosine variant: [o; in] = W_io [e; h], each L2-normalised. */
void orc_cosine_vectors(const orc_dims *dm, const orc_weights *w, const uint16_t *e,
                        const uint16_t *h, double *o, double *in);
double orc_cosine_transition(int r, double sigma, const double *o_a, const double *in_b, double l_b);

/* Step 5: prefix-first greedy walk over scores [B-1][K][K]. choice[0] = 0. */
void orc_walk(const double *scores, int B, int K, int32_t *choice, double *margin);

/* Highest-scoring path over scores [B-1][K][K] by dynamic programming
 * (Viterbi), choice[0] = 0, ties to the lowest index; margin[p] = gap between
 * the best and second-best predecessor of the chosen candidate at p+1. */
void orc_viterbi(const double *scores, int B, int K, int32_t *choice, double *margin);
/* The same program with single-precision totals (t = total + score rounded to
 * float at every step), to compare decisions with a single-precision kernel. */
void orc_viterbi_f32(const float *scores, int B, int K, int32_t *choice, float *margin);

/* Beam walk over scores [B-1][K][K]: the W partial paths of highest
 * cumulative score, each extended to its m best successors (m <= 0 or > K:
 * all); choice[0] = 0; margin[p] = the chosen successor's score minus the best
 * other successor score along the answer.  _f32: the same with float totals. */
void orc_beam(const double *scores, int B, int K, int W, int m, int32_t *choice, double *margin);
void orc_beam_f32(const float *scores, int B, int K, int W, int m, int32_t *choice, float *margin);

/* Greedy verify: number of leading slots whose token equals the target. */
int orc_verify(const int32_t *tokens, const int32_t *target, int B);

/* Candidate features of one row: for its K best tokens (orc_topk_row order),
 * feat [K][5] = [log p, p, l_0 - l_k, k/K, k == 0], p = softmax over V. */
void orc_topk_features(const uint16_t *row, int V, int K, double *feat);

/* Stochastic verification of the point-mass proposal `tokens` [B] against
 * target logits [B+1][stride] (temperature 1): slot j accepted iff
 * u_acc[j] < q_j(tokens[j]); at the first rejection j, next_token is drawn
 * from q_j without tokens[j]; after B acceptances from q_B (the bonus
 * position).  A draw takes the smallest v whose cumulative weight (vocabulary
 * order) exceeds u_draw times the total.  q_acc [B] may be NULL. */
void orc_verify_stochastic(const uint16_t *target, int64_t stride, int V, int B, const int32_t *tokens,
                           const float *u_acc, float u_draw, int32_t *accept_len, int32_t *next_token,
                           double *q_acc);

/* E[Y] = 1 + sum_k prod_{j<=k} cond[j]; survival[k] receives the products. */
double orc_expected_yield(const double *cond, int n, double *survival);

/* Number of corrector parameters implied by the shapes the oracle reads. */
long long orc_param_count(int d, int r, int H);

/* Whole path for one request.
 * variant 0 = MLP transition (DCOCO), 1 = cosine matching (LiLiCorr-style);
 * path_rule 0 = prefix-first greedy walk, 1 = highest-scoring path (Viterbi),
 * 2 = beam walk (dm->beam_width, dm->beam_topm).
 * logits [slots][stride] bf16, hidden [slots][d] bf16, E [V][d] bf16,
 * target [B] or NULL.  Outputs: topk_ids/topk_val [B][K], scores [B-1][K][K],
 * choice/tokens [B], margin [B-1], accept_len [1] (when target != NULL).
 * Returns 0, or -1 on bad arguments / allocation failure. */
int orc_correct_request(const orc_dims *dm, const orc_weights *w, int variant, double sigma, int path_rule,
                        const uint16_t *logits, int64_t stride, const uint16_t *hidden,
                        const uint16_t *E, const int32_t *target,
                        int32_t *topk_ids, float *topk_val, double *scores,
                        int32_t *choice, int32_t *tokens, double *margin, int32_t *accept_len,
                        orc_intermediates *inter);

#ifdef __cplusplus
}
#endif
#endif
