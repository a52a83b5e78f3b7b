/*
 * dcoco.h -- C ABI of the GB300 draft-correction library (DCOCO hot path).
 *
 * The method (pages by title):
 *   [DCOCO]    "Contextual Correction of Parallel Drafts for Speculative
 *              Decoding": Core method; Method step details (1)-(5).
 *   [LiLiCorr] "LiLiCorr: Lightweight Likelihood Correlation of Parallel
 *              Drafts for Speculative Decoding": Sec. 3.2 Eq. (1) (cosine
 *              in/out matching), Sec. 3.5 Eq. (8) (greedy walk), App. E
 *              Eq. (12) (highest-scoring path).
 *   [FD]       "Faster Decoding": greedy-verification contract.
 *
 * One DFlash-style drafter forward pass gives, per request, a block of
 * `slots` positions: slot 0 is the anchor (the last committed token) and
 * slots 1..B (B = slots-1) are draft slots, each with full-vocabulary logits
 * l_i and a hidden state h_i.  dcoco_correct runs, on the caller's stream:
 *
 *   1. top-K: the K best tokens of every draft slot's logits
 *      (value descending, token id ascending; -0 == +0)    [DCOCO] step (1)
 *   2. candidate representations, width r = 128:
 *        b = LN(W_cand E[c]),  g_i = LN(W_ctx h_i)          (no affine)
 *        z = LN_{gamma,beta}(W_fuse [b; g_i])               [DCOCO] step (2)
 *      and slot-pair states s_p = W_pair [h_p; h_{p+1}]     [DCOCO] step (3)
 *   3. transition scores for p = 1..B-1, a, b < K:
 *        S_p(a,b) = l_{p+1}(b) + Delta([s_p; z_p^a; z_{p+1}^b; l_p(a); l_{p+1}(b)])
 *      Delta = 386 -> 256 -> 1 MLP with (erf) GELU          [DCOCO] step (4)
 *      (variant 1: S_p(a,b) = sigma cos(o_p^a, in_{p+1}^b) + l_{p+1}(b),
 *       [o; in] = W_io [E[c]; h_i]                          [LiLiCorr] Eq. (1))
 *   4. path selection, k_1 = 0 (draft argmax) in both rules:
 *      path_rule 0, prefix-first greedy walk:
 *        k_{p+1} = argmax_b S_p(k_p, b), ties to the lowest b
 *                                                [DCOCO] step (5); [LiLiCorr] Eq. (8)
 *      path_rule 1, highest-scoring path: the k maximizing sum_p S_p(k_p, k_{p+1})
 *        (dynamic program, fp32 totals, ties to the lowest index) [LiLiCorr] App. E Eq. (12)
 *      path_rule 2, beam walk: the beam_width partial paths of highest
 *        cumulative score, each extended to its beam_topm best successors;
 *        the best complete path       [DCOCO] reproduction assessment (2)-(3)
 *   5. greedy verify: accept_len = length of the longest prefix of the chosen
 *      tokens equal to the target tokens                    [FD]
 *
 * Conventions for every call:
 *   - Status: 0 = OK, negative = error (DCOCO_E*).  Argument errors are
 *     reported before anything is launched.
 *   - Streams are passed as `void *` and mean cudaStream_t (NULL = legacy
 *     default stream).  All work is stream-ordered and asynchronous: no call
 *     except dcoco_get_device_status, the *_host entry and the create/destroy
 *     calls synchronises with the host.
 *   - Ownership: the caller owns every input and output buffer; the library
 *     owns its handle workspace and its packed weights.  Only dcoco_create
 *     and dcoco_weights_create allocate device memory; dcoco_correct and
 *     dcoco_topk never allocate.
 *   - Layouts are row-major and dense unless a stride is given.  bf16 means
 *     IEEE bfloat16 bit patterns (uint16).  Logits must be finite or -inf
 *     (NaN is not supported).
 *   - A handle is not thread-safe and its workspace is shared by every call:
 *     calls on one handle must be ordered (same stream, or synchronised).
 *   - Outputs are bitwise deterministic for identical inputs and do not depend
 *     on the batch size (each request is computed independently).
 */
#ifndef DCOCO_H
#define DCOCO_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DCOCO_OK 0
#define DCOCO_EINVAL (-1)       /* null pointer, bad size/stride/alignment    */
#define DCOCO_EUNSUPPORTED (-2) /* K not in {8,16,32}, r != 128, H != 256 ... */
#define DCOCO_EBATCH (-3)       /* batch < 0 or > max_batch                   */
#define DCOCO_ECUDA (-4)        /* a CUDA runtime call failed                 */
#define DCOCO_ENOMEM (-5)       /* device or host allocation failed           */
#define DCOCO_EDEVICE (-6)      /* a kernel flagged bad data (see status)     */

typedef struct dcoco_handle dcoco_handle;   /* config + device workspace        */
typedef struct dcoco_weights dcoco_weights; /* packed device copy of the weights */

typedef struct {
  int vocab;        /* V >= K, V <= 1,048,576                                  */
  int hidden;       /* d, a positive multiple of 64                           */
  int slots;        /* block positions including the anchor, 3..32 (16)       */
  int topk;         /* K in {8, 16, 32}                                        */
  int rank;         /* r, must be 128                                          */
  int mlp_hidden;   /* H, must be 256                                          */
  int max_batch;    /* largest batch any call on this handle will pass, >= 1  */
  int variant;      /* 0 = MLP transition (DCOCO), 1 = cosine matching        */
  float sigma;      /* cosine scale (variant 1)                               */
  float ln_eps;     /* LayerNorm epsilon (1e-5)                                */
  int host_staging; /* nonzero: also allocate device staging buffers so that
                       dcoco_correct_host can be used                        */
  int path_rule;    /* 0 = prefix-first greedy walk, 1 = highest-scoring path,
                       2 = beam walk                                          */
  int beam_width;   /* path_rule 2: partial paths kept, 1..4                  */
  int beam_topm;    /* path_rule 2: successors per predecessor, 1..K (0 = K)  */
} dcoco_config;

/* Corrector weights, fp32, PyTorch Linear layout [out][in], row-major.
 * Variant 0 needs w_cand..b2; variant 1 needs w_io only. */
typedef struct {
  const float *w_cand;   /* [r][d]     */
  const float *w_ctx;    /* [r][d]     */
  const float *w_fuse;   /* [r][2r]    */
  const float *ln_gamma; /* [r]        */
  const float *ln_beta;  /* [r]        */
  const float *w_pair;   /* [r][2d]    */
  const float *w1;       /* [H][3r+2]  */
  const float *b1;       /* [H]        */
  const float *w2;       /* [H]        */
  const float *b2;       /* [1]        */
  const float *w_io;     /* [2r][2d]   */
  int on_device;         /* 1: pointers are device memory, 0: host memory */
} dcoco_weight_ptrs;

/* Per-call inputs (device pointers). */
typedef struct {
  const void *logits;          /* bf16 [N][slots][stride]; 16-byte aligned   */
  int64_t logits_slot_stride;  /* elements between slot rows; >= V, % 8 == 0 */
  const void *hidden;          /* bf16 [N][slots][d]; 16-byte aligned        */
  const void *cand_embed;      /* bf16 [V][d] frozen token-embedding table;
                                  entries below 65504 in magnitude (the
                                  candidate projection runs in fp16)        */
  const int32_t *target_tokens;/* int32 [N][B] target greedy tokens, or NULL */
} dcoco_inputs;

/* Per-call outputs (device pointers; NULL = not wanted unless stated). */
typedef struct {
  int32_t *tokens;     /* [N][B] chosen token ids -- required               */
  int32_t *choice;     /* [N][B] chosen candidate index per slot            */
  float *scores;       /* [N][B-1][K][K] transition scores S_p(a,b)         */
  int32_t *accept_len; /* [N] accepted prefix length in [0,B]; required iff
                          target_tokens != NULL                             */
  int32_t *topk_ids;   /* [N][B][K] candidate token ids, best first         */
  float *topk_val;     /* [N][B][K] candidate logits (exact bf16 values)    */
  float *margin;       /* [N][B-1] path_rule 0 and 2: the chosen successor's
                          score minus the best other successor score
                          (for rule 0, best minus second best); path_rule 1:
                          best minus
                          second-best predecessor total of the chosen
                          candidate at slot p+1 (+inf when only one
                          predecessor is possible)                         */
  float *cand_feat;    /* [N][B][K][5] vocabulary-normalised candidate
                          features, or NULL (then not computed): per
                          candidate k of a slot, [log p, p, l_0 - l_k, k/K,
                          1 if k == 0], p = softmax of the slot's logits over
                          the whole vocabulary.  The top-K pass then also
                          accumulates each row's log-sum-exp ([LiLiCorr]
                          App. A: top-K fused with the normalisation); the
                          path itself still uses the raw logits.  Device
                          entry only (dcoco_correct_host: EINVAL).         */
} dcoco_outputs;

/* Library version, major*10000 + minor*100 + patch. */
int dcoco_version(void);

/* Human-readable text for a status code (static storage). */
const char *dcoco_status_string(int status);

/* Validate `cfg` and allocate the workspace for max_batch requests on the
 * current CUDA device.  *out is set only on success.  Errors: EINVAL (null
 * pointer, bad sizes), EUNSUPPORTED (K, r, H outside the supported set),
 * ENOMEM, ECUDA.  Validation happens before any CUDA call. */
int dcoco_create(const dcoco_config *cfg, dcoco_handle **out);

/* Copy and pack the corrector weights to the device (fp32 transposes and
 * bf16 hi/lo splits for the tensor-core projections).  Synchronises
 * `stream` before returning.  The caller's buffers may be freed afterwards.
 * Errors: EINVAL (null handle/out/pointer needed by the variant), ENOMEM,
 * ECUDA. */
int dcoco_weights_create(dcoco_handle *h, const dcoco_weight_ptrs *w, void *stream,
                         dcoco_weights **out);

/* The whole correction path (steps 1-5 above) for `batch` requests, launched
 * on `stream`.  Never allocates; never synchronises.  batch == 0 is a no-op.
 * Errors: EINVAL (null/misaligned pointers, stride < V or % 8 != 0, tokens
 * NULL, accept_len NULL while target_tokens is set, weights from another
 * handle), EBATCH (batch < 0 or > max_batch), ECUDA (launch failure). */
int dcoco_correct(dcoco_handle *h, const dcoco_weights *w, int batch,
                  const dcoco_inputs *in, const dcoco_outputs *out, void *stream);

/* Same path with HOST buffers: copies hidden (and target tokens) from host
 * memory into the handle's staging buffers; logits in page-locked host memory
 * the device can address (e.g. cudaHostAlloc) are read in place by the top-K
 * over the host link, provided the driver reports one page-locked range
 * that holds every byte the call reads ((batch * slots - 1) * stride + vocab
 * elements from `logits`); other logits are copied to staging first.  Runs
 * dcoco_correct, copies the requested outputs back to the host pointers in
 * `out`, and synchronises `stream`.  The host buffers must stay unchanged
 * until the call returns.  `in->cand_embed` stays a DEVICE pointer (the
 * frozen table is resident).  Requires host_staging at create.
 * Errors: as dcoco_correct, plus EINVAL if the handle has no staging. */
int dcoco_correct_host(dcoco_handle *h, const dcoco_weights *w, int batch,
                       const dcoco_inputs *in, const dcoco_outputs *out, void *stream);

/* The test dcoco_correct_host applies before it reads host logits in
 * place: 1 if [ptr, ptr + bytes) lies inside [range_start, range_start +
 * range_size) (the page-locked range the driver reports for ptr), else 0.
 * Pure arithmetic: no CUDA call. */
int dcoco_host_range_covers(uint64_t range_start, uint64_t range_size, uint64_t ptr, uint64_t bytes);

/* Stochastic verification (temperature 1) of a point-mass proposal, the
 * alternative to the greedy verify of step 5 for sampling targets.
 *   [DCOCO] Core method: the proposal y_j is accepted with probability
 *   q_j(y_j); on rejection the corrected token is resampled from
 *   q_j(v) 1[v != y_j] / (1 - q_j(y_j)).  [FD] Modified rejection sampling:
 *   left to right, stop at the first rejection; after all B acceptances one
 *   bonus token from the target at the next position.
 * target_logits: bf16 [batch][B+1][target_stride] (B = slots - 1), the
 *   target's logits at draft slots 1..B (rows 0..B-1) and at the bonus
 *   position (row B); q_j is the softmax of row j.  target_stride >= vocab,
 *   multiple of 8; 16-byte aligned base.
 * tokens: int32 [batch][B], the proposal (e.g. dcoco_correct's tokens).
 * u_accept: fp32 [batch][B], u_draw: fp32 [batch]: uniforms in [0, 1) that
 *   the caller draws; slot j is accepted iff u_accept[n][j] < q_j(y_j), and a
 *   draw takes the smallest token whose cumulative weight in vocabulary order
 *   exceeds u_draw[n] times the total weight.
 * Outputs (device): accept_len int32 [batch] (accepted draft tokens, 0..B),
 *   next_token int32 [batch] (the corrected token, or the bonus token),
 *   q_accept fp32 [batch][B] (q_j(y_j); NULL = not wanted).
 * fp32 arithmetic: decisions within ~1e-6 of a threshold may differ from an
 * exact computation.  One launch; uses the handle's workspace, never
 * allocates.  Errors: EINVAL (null pointer, bad stride or alignment), EBATCH,
 * ECUDA. */
int dcoco_verify_stochastic(dcoco_handle *h, int batch, const void *target_logits, int64_t target_stride,
                            const int32_t *tokens, const float *u_accept, const float *u_draw, int32_t *accept_len,
                            int32_t *next_token, float *q_accept, void *stream);

/* Step 1 alone: top-K ids and values of every draft slot, written to
 * topk_ids / topk_val ([N][B][K], device).  Uses the handle's workspace,
 * never allocates.  Errors as dcoco_correct. */
int dcoco_topk(dcoco_handle *h, int batch, const void *logits, int64_t logits_slot_stride,
               int32_t *topk_ids, float *topk_val, void *stream);

/* Step 1 alone WITHOUT a handle and without allocating anything.  The page
 * has no counterpart: this entry exists for callers that cannot allocate
 * device memory (dcoco_create calls cudaMalloc) -- e.g. a plugin inside a
 * serving engine that reserved all device memory for its own pool, or code on
 * a latency-critical path where cudaMalloc, which can synchronise the device,
 * is not acceptable.  Its scratch is a fixed 4 MiB array that every GPU
 * loading the library holds until the process exits.
 *   batch, slots, vocab, topk: as dcoco_config / dcoco_topk.  Two limits,
 *     both checked before any CUDA call, reject a call with DCOCO_EBATCH:
 *     (1) batch * (slots - 1) <= DCOCO_TOPK_NOALLOC_MAX_ROWS (4096 draft-slot
 *     rows, i.e. 273 requests of 16 slots);
 *     (2) the per-segment candidate lists must fit the array's list area of
 *     (4 MiB - 16 KiB) / 8 = 522,240 entries at the fewest segments the
 *     vocabulary allows: rows * topk * ceil((vocab / 8) / 20480) <= 522,240
 *     (rows = batch * (slots - 1)).  At vocab 151,936 that is always met; at
 *     vocab 2^20 and topk 32 it allows at most 2331 rows.
 *     Within limit (2), a call whose plan wants more segments than the area
 *     holds runs with fewer, longer segments (same results, slower).
 *   logits, logits_slot_stride, topk_ids, topk_val, stream: as dcoco_topk
 *     (device pointers, outputs [batch][slots-1][topk]).
 * Results are identical to dcoco_topk's.  No cudaMalloc / cudaFree or other
 * allocating routine is called.  The first call on a device (with that
 * device current) looks up the scratch address and the device's SM count;
 * make that first call before any stream capture.  Every call shares the one
 * array per device, so calls whose work overlaps on the GPU (other streams,
 * other host threads) race and corrupt each other: order them.  Errors:
 * EUNSUPPORTED, EINVAL, EBATCH (sizes above), ECUDA. */
#define DCOCO_TOPK_NOALLOC_MAX_ROWS 4096
int dcoco_topk_noalloc(int batch, int slots, int vocab, int topk, const void *logits,
                       int64_t logits_slot_stride, int32_t *topk_ids, float *topk_val,
                       void *stream);

/* Planning query for dcoco_topk_noalloc on the current device (no kernel
 * launch, no allocation): *segments receives the number of segments per row
 * the call would use and *planned_segments the number the handle-based
 * dcoco_topk would use for the same rows; they differ when the fixed list
 * area holds fewer.  The first query on a device performs the same one-time
 * set-up as the first dcoco_topk_noalloc call.  Errors: EINVAL (NULL
 * outputs), EUNSUPPORTED / EINVAL / EBATCH as dcoco_topk_noalloc, ECUDA. */
int dcoco_topk_noalloc_plan(int batch, int slots, int vocab, int topk, int *segments,
                            int *planned_segments);

/* Synchronise the handle's last stream and return DCOCO_OK, or DCOCO_EDEVICE
 * if a kernel recorded bad data (e.g. a candidate id outside [0,V)) or a
 * bounded wait that expired (the kernel then skips its stores and returns)
 * since the last call to this function (the flag is then cleared), or ECUDA. */
int dcoco_get_device_status(dcoco_handle *h);

/* Self-test of the failure path shared by every bounded wait in the kernels:
 * launches, on `stream`, one block that waits (with the kernels' own wait
 * routine) on an mbarrier that nothing completes, giving up after limit_ns
 * nanoseconds (1e3 .. 1e9).  The handle's device status word then records
 * the timeout: dcoco_get_device_status returns DCOCO_EDEVICE once, and the
 * context stays usable.  No fault, no trap, no hang.  Errors: EINVAL (NULL
 * handle, limit out of range), ECUDA (launch). */
int dcoco_selftest_wait_timeout(dcoco_handle *h, long long limit_ns, void *stream);

/* Tracing: number of kernels this handle has launched since it was created
 * (every launch of dcoco_correct / dcoco_correct_host / dcoco_topk counts).
 * Returns -1 for a NULL handle. */
long long dcoco_kernel_launches(const dcoco_handle *h);

/* Tracing: when enabled (nonzero), dcoco_correct records a CUDA event on its
 * stream before the first kernel and after every kernel, for up to 1024
 * calls; dcoco_stage_read then reports the per-kernel time.  Enabling costs
 * one event record per kernel.  Returns DCOCO_OK or EINVAL (NULL handle). */
int dcoco_stage_timing(dcoco_handle *h, int enable);

/* Tracing: synchronise the recorded events and write, for each kernel stage
 * s < min(max_stages, *n_stages), the summed duration in milliseconds over
 * the recorded calls to ms[s]; *calls receives the number of calls summed and
 * *n_stages the number of stages of the handle's variant.  The record is then
 * cleared.  Errors: EINVAL (NULL arguments), ECUDA. */
int dcoco_stage_read(dcoco_handle *h, int max_stages, float *ms, int *calls, int *n_stages);

/* Tracing: name of kernel stage `s` of the handle's variant ("topk",
 * "proj", ...), or NULL if out of range. */
const char *dcoco_stage_name(const dcoco_handle *h, int s);

/* Release packed weights / the handle.  NULL is allowed.  Synchronises the
 * device before freeing. */
void dcoco_weights_destroy(dcoco_weights *w);
void dcoco_destroy(dcoco_handle *h);

#ifdef __cplusplus
}
#endif
#endif /* DCOCO_H */
