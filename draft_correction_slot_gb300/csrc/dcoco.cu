// dcoco.cu -- C ABI: argument validation, workspace, weight packing and the
// launch sequence of the correction path (declared in include/dcoco.h).
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <new>
#include <vector>

#include "../../include/dcoco.h"
#include "kernels.h"

namespace {

constexpr int kR = 128;
constexpr int kH = 256;

struct Workspace {
  unsigned long long *part = nullptr;
  float2 *part_lse = nullptr;  // per (row, segment) (maximum, sum of exp) for the candidate features
  unsigned *row_count = nullptr;
  unsigned *row_ready = nullptr;  // per draft-slot row: top-K stored (1), cleared by the projection
  int32_t *ids = nullptr;
  float *vals = nullptr;
  float *slot_proj = nullptr;  // [N*B][3r]  (variant 1: [N*B][2r])
  float *cand_proj = nullptr;  // variant 1: [N*B*K][2r]
  uint16_t *b_hi = nullptr, *b_lo = nullptr;  // variant 0: LN0(W_cand E[c]) as bf16 hi, lo [N*B*K][r]
  float *P = nullptr;          // [N*B][H] (rows of the last slot unused)
  float *U = nullptr;          // [N*B*K][H]  (variant 0)
  float *V = nullptr;          // [N*B*K][H]  (variant 0)
  float *scores = nullptr;     // [N*(B-1)][K][K]
  int32_t *choice = nullptr;   // [N*B]
  float *margin = nullptr;     // [N*(B-1)]
  int *err = nullptr;          // device status word
  unsigned *req_count = nullptr;  // finished pairs per request (zero between calls)
  // stochastic verify: per target row chunk statistics, log-sum-exp, q_j(y_j), counters
  float *v_chunk_m = nullptr, *v_chunk_s = nullptr, *v_lse = nullptr, *v_q = nullptr;
  unsigned *v_count = nullptr;
  // host staging (dcoco_correct_host)
  uint16_t *st_logits = nullptr;  // [N][slots][st_stride]
  int64_t st_stride = 0;
  uint16_t *st_hidden = nullptr;  // [N][slots][d]
  int32_t *st_target = nullptr;   // [N*B]
  int32_t *st_tokens = nullptr;   // [N*B]
  int32_t *st_accept = nullptr;   // [N]
};

}  // namespace

namespace {
constexpr int kMaxStages = 8;
constexpr int kMaxTimedCalls = 1024;
// Stage lists of the launch orders: 0 the MLP variant, 1 the cosine variant.
constexpr int kStageKinds = 2;
const char *const kStageNames[kStageKinds][kMaxStages] = {
    {"topk", "proj", "maps", "pair_walk", nullptr, nullptr, nullptr, nullptr},
    {"topk", "proj", "cos_pair_walk", nullptr, nullptr, nullptr, nullptr, nullptr}};
int stage_count(int kind) {
  int n = 0;
  while (n < kMaxStages && kStageNames[kind][n]) ++n;
  return n;
}
}  // namespace

struct dcoco_handle {
  dcoco_config cfg;
  int device = 0;
  int B = 0;
  int topk_segments_max = 1;  // partial-list capacity per row
  int topk_wave = 1;          // resident top-K CTAs on the device (SMs x occupancy)
  int splits = 1;             // split-K of the projections (fixed per handle, so
                              // results do not depend on the batch size)
  void *block = nullptr;  // one device allocation holding the workspace
  Workspace ws;
  dc::CandIoMaps cand_io;  // TMA maps of b (hi, lo), U, V (variant 0)
  dc::SlotIoMaps slot_io;  // TMA maps of slot_proj, P (variant 0)
  cudaStream_t last_stream = nullptr;
  long long launches = 0;            // kernels launched so far
  bool timing = false;               // record per-stage events
  int timed_calls = 0;               // calls recorded since the last read
  int timed_kind[1024] = {};          // stage list of each recorded call
  int read_kind = -1;                 // stage list of the last dcoco_stage_read
  std::vector<cudaEvent_t> events;   // kMaxTimedCalls x (stages + 1), created on demand
};

struct dcoco_weights {
  const dcoco_handle *owner = nullptr;
  int device = 0;
  void *block = nullptr;
  // projection weights as bf16 hi / lo halves, [rows][d] each
  uint16_t *cand_f16 = nullptr;                     // W_cand [r][d] as fp16 (variant 1: W_io[:, :d], [2r][d])
  uint16_t *slot_hi = nullptr, *slot_lo = nullptr;  // [W_ctx ; W_pair[:, :d] ; W_pair[:, d:]] [3r][d]
                                                    // (variant 1: W_io[:, d:], [2r][d])
  CUtensorMap map_cand_f16, map_slot_hi, map_slot_lo;  // TMA maps
  // the 128-deep maps of the MLP as bf16 hi / lo (variant 0): W_fuse[:, :r],
  // W_fuse[:, r:] ([r][r]), [W1[:, r:2r] ; W1[:, 2r:3r]] ([2H][r]), W1[:, :r] ([H][r])
  uint16_t *fb_hi = nullptr, *fb_lo = nullptr, *fg_hi = nullptr, *fg_lo = nullptr;
  uint16_t *w1ab_hi = nullptr, *w1ab_lo = nullptr, *w1s_hi = nullptr, *w1s_lo = nullptr;
  dc::MlpMaps mlp_maps;
  dc::MlpWeightsDev mlp{};
};

namespace {

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// fp32 -> bf16, round to nearest even (NaN -> quiet NaN)
inline uint16_t f32_to_bf16(float f) {
  uint32_t u;
  std::memcpy(&u, &f, sizeof u);
  if ((u & 0x7FFFFFFFu) > 0x7F800000u) return 0x7FC0u;
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}
// fp32 -> fp16 bits, round to nearest even (subnormals kept; beyond the
// fp16 range: infinity; NaN -> quiet NaN).
inline uint16_t f32_to_f16(float f) {
  uint32_t x;
  std::memcpy(&x, &f, sizeof x);
  const uint32_t sign = (x >> 16) & 0x8000u, ax = x & 0x7FFFFFFFu;
  if (ax >= 0x7F800000u) return (uint16_t)(sign | (ax > 0x7F800000u ? 0x7E00u : 0x7C00u));
  if (ax >= 0x477FF000u) return (uint16_t)(sign | 0x7C00u);  // rounds to 65536 or more
  if (ax < 0x33000000u) return (uint16_t)sign;                // below 2^-25: rounds to 0
  const int e = (int)(ax >> 23) - 127;
  const uint32_t mant = (ax & 0x7FFFFFu) | 0x800000u;         // value = mant 2^(e - 23)
  uint32_t h, rem, half;
  if (e >= -14) {  // normal: 10 mantissa bits, 13 dropped
    h = ((uint32_t)(e + 15) << 10) + ((mant >> 13) & 0x3FFu);
    rem = mant & 0x1FFFu;
    half = 0x1000u;
  } else {         // subnormal: units of 2^-24
    const int sh = -(e + 1);
    h = mant >> sh;
    rem = mant & ((1u << sh) - 1u);
    half = 1u << (sh - 1);
  }
  if (rem > half || (rem == half && (h & 1u))) ++h;  // a carry moves into the exponent correctly
  return (uint16_t)(sign | h);
}

inline float bf16_to_f32(uint16_t b) {
  const uint32_t u = (uint32_t)b << 16;
  float f;
  std::memcpy(&f, &u, sizeof f);
  return f;
}

struct Carver {  // sub-allocates a byte range, 256-byte aligned pieces
  size_t off = 0;
  char *base = nullptr;
  template <class T>
  T *take(size_t n) {
    off = (off + 255) & ~size_t(255);
    T *p = base ? reinterpret_cast<T *>(base + off) : nullptr;
    off += n * sizeof(T);
    return p;
  }
};

void carve_workspace(Carver &c, const dcoco_config &cfg, int B, int topk_segments_max, Workspace &ws) {
  const size_t N = (size_t)cfg.max_batch, K = (size_t)cfg.topk, d = (size_t)cfg.hidden;
  const size_t rows = N * B, cands = rows * K;
  ws.part = c.take<unsigned long long>(rows * (size_t)topk_segments_max * K);
  ws.part_lse = c.take<float2>(rows * (size_t)topk_segments_max);
  ws.row_count = c.take<unsigned>(rows);
  ws.row_ready = c.take<unsigned>(rows);
  ws.ids = c.take<int32_t>(cands);
  ws.vals = c.take<float>(cands);
  ws.slot_proj = c.take<float>(rows * 3 * kR);
  // the candidate rows: LN0'd bf16 hi/lo (MLP variant) or fp32 [2r] (cosine)
  ws.cand_proj = c.take<float>(cfg.variant == 0 ? 0 : cands * 2 * kR);
  ws.b_hi = c.take<uint16_t>(cfg.variant == 0 ? cands * kR : 0);
  ws.b_lo = c.take<uint16_t>(cfg.variant == 0 ? cands * kR : 0);
  ws.P = c.take<float>(N * B * kH);
  ws.U = c.take<float>(cfg.variant == 0 ? cands * kH : 0);
  ws.V = c.take<float>(cfg.variant == 0 ? cands * kH : 0);
  ws.scores = c.take<float>(N * (B - 1) * K * K);
  ws.choice = c.take<int32_t>(rows);
  ws.margin = c.take<float>(N * (B - 1));
  ws.err = c.take<int>(1);
  ws.req_count = c.take<unsigned>(N);
  const size_t vrows = N * (size_t)cfg.slots, vch = (size_t)dc::verify_chunks(cfg.vocab);
  ws.v_chunk_m = c.take<float>(vrows * vch);
  ws.v_chunk_s = c.take<float>(vrows * vch);
  ws.v_lse = c.take<float>(vrows);
  ws.v_q = c.take<float>(rows);
  ws.v_count = c.take<unsigned>(N);
  if (cfg.host_staging) {
    ws.st_stride = ((int64_t)cfg.vocab + 7) & ~int64_t(7);
    ws.st_logits = c.take<uint16_t>(N * cfg.slots * (size_t)ws.st_stride);
    ws.st_hidden = c.take<uint16_t>(N * cfg.slots * d);
    ws.st_target = c.take<int32_t>(rows);
    ws.st_tokens = c.take<int32_t>(rows);
    ws.st_accept = c.take<int32_t>(N);
  }
}

int validate_config(const dcoco_config *cfg) {
  if (!cfg) return DCOCO_EINVAL;
  if (cfg->rank != kR || cfg->mlp_hidden != kH) return DCOCO_EUNSUPPORTED;
  if (cfg->topk != 8 && cfg->topk != 16 && cfg->topk != 32) return DCOCO_EUNSUPPORTED;
  if (cfg->variant != 0 && cfg->variant != 1) return DCOCO_EUNSUPPORTED;
  if (cfg->path_rule < 0 || cfg->path_rule > 2) return DCOCO_EUNSUPPORTED;
  if (cfg->path_rule == 2 && (cfg->beam_width < 1 || cfg->beam_width > 4 || cfg->beam_topm < 0 ||
                              cfg->beam_topm > cfg->topk))
    return DCOCO_EUNSUPPORTED;
  if (cfg->slots < 3 || cfg->slots > 32) return DCOCO_EUNSUPPORTED;
  if (cfg->vocab < cfg->topk || cfg->vocab > (1 << 20)) return DCOCO_EINVAL;
  if (cfg->hidden <= 0 || cfg->hidden % 64 != 0) return DCOCO_EINVAL;
  if (cfg->max_batch < 1 || cfg->max_batch > (1 << 16)) return DCOCO_EINVAL;
  if (!(cfg->ln_eps > 0.f)) return DCOCO_EINVAL;
  return DCOCO_OK;
}

int validate_call(const dcoco_handle *h, const dcoco_weights *w, int batch, const dcoco_inputs *in,
                  const dcoco_outputs *out, bool device_ptrs) {
  if (!h || !w || !in || !out) return DCOCO_EINVAL;
  if (w->owner != h) return DCOCO_EINVAL;
  if (batch < 0 || batch > h->cfg.max_batch) return DCOCO_EBATCH;
  if (batch == 0) return DCOCO_OK;
  if (!in->logits || !in->hidden || !in->cand_embed || !out->tokens) return DCOCO_EINVAL;
  if (in->target_tokens && !out->accept_len) return DCOCO_EINVAL;
  if (in->logits_slot_stride < h->cfg.vocab) return DCOCO_EINVAL;
  if (device_ptrs) {
    if (in->logits_slot_stride % 8 != 0) return DCOCO_EINVAL;
    if (!aligned16(in->logits) || !aligned16(in->hidden) || !aligned16(in->cand_embed))
      return DCOCO_EINVAL;
  } else if (!aligned16(in->cand_embed) || out->cand_feat) {  // features: device entry only
    return DCOCO_EINVAL;
  }
  return DCOCO_OK;
}

inline int cuda_status(cudaError_t e) { return e == cudaSuccess ? DCOCO_OK : DCOCO_ECUDA; }

// The base address and size of the allocation (or registered range) that
// holds `p`, from the driver's pointer attributes.  False when the driver
// does not know the pointer.
bool host_range_of(const void *p, uint64_t *start, uint64_t *size) {
  typedef CUresult (*PtrAttrFn)(void *, CUpointer_attribute, CUdeviceptr);
  static PtrAttrFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuPointerGetAttribute", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PtrAttrFn>(f);
    else
      cudaGetLastError();
  }
  if (!fn) return false;
  CUdeviceptr base = 0;
  size_t n = 0;
  const CUdeviceptr dp = (CUdeviceptr) reinterpret_cast<uintptr_t>(p);
  if (fn(&base, CU_POINTER_ATTRIBUTE_RANGE_START_ADDR, dp) != CUDA_SUCCESS ||
      fn(&n, CU_POINTER_ATTRIBUTE_RANGE_SIZE, dp) != CUDA_SUCCESS)
    return false;
  *start = (uint64_t)base;
  *size = (uint64_t)n;
  return true;
}

// Successors each beam keeps (0 in the config means all K).
inline int beam_topm(const dcoco_config &cfg) { return cfg.beam_topm > 0 ? cfg.beam_topm : cfg.topk; }

#define DC_TRY(expr)                       \
  do {                                     \
    cudaError_t e_ = (expr);               \
    if (e_ != cudaSuccess) return DCOCO_ECUDA; \
  } while (0)

// Records the stage boundaries of one call (when timing is on) and counts
// the launches.
struct StageClock {
  dcoco_handle *h;
  cudaStream_t st;
  cudaEvent_t *ev = nullptr;  // kMaxStages + 1 events of this call, or null
  int s = 0;
  StageClock(dcoco_handle *h_, cudaStream_t st_, int kind) : h(h_), st(st_) {
    if (h->timing && h->timed_calls < kMaxTimedCalls) {
      ev = h->events.data() + (size_t)h->timed_calls * (kMaxStages + 1);
      h->timed_kind[h->timed_calls] = kind;
      ++h->timed_calls;
      cudaEventRecord(ev[0], st);
    }
  }
  // a launch that ends a stage
  cudaError_t done(cudaError_t e) {
    ++h->launches;
    ++s;
    if (e == cudaSuccess && ev) e = cudaEventRecord(ev[s], st);
    return e;
  }
};

// The launch sequence; all pointers are device pointers and validated.
// logits_in_host_memory: the logits are page-locked host memory read in
// place (dcoco_correct_host); the top-K then reads them with ordinary loads
// (the one-pass kernel) rather than bulk asynchronous copies.
int run_path(dcoco_handle *h, const dcoco_weights *w, int N, const dcoco_inputs *in,
             const dcoco_outputs *out, cudaStream_t st, bool logits_in_host_memory = false) {
  const dcoco_config &cfg = h->cfg;
  const Workspace &ws = h->ws;
  const int B = h->B, K = cfg.topk, d = cfg.hidden, V = cfg.vocab;
  const uint16_t *logits = static_cast<const uint16_t *>(in->logits);
  const uint16_t *hidden = static_cast<const uint16_t *>(in->hidden);
  const uint16_t *E = static_cast<const uint16_t *>(in->cand_embed);
  int32_t *ids = out->topk_ids ? out->topk_ids : ws.ids;
  float *vals = out->topk_val ? out->topk_val : ws.vals;
  float *scores = out->scores ? out->scores : ws.scores;
  int32_t *choice = out->choice ? out->choice : ws.choice;
  float *margin = out->margin ? out->margin : ws.margin;
  h->last_stream = st;
  // the top-K hands its rows to the projection one by one (flags), except
  // with the candidate features (the features' top-K accumulates the
  // log-sum-exp) or logits in host memory (read by ordinary loads)
  const bool handoff = out->cand_feat == nullptr && !logits_in_host_memory;
  StageClock clk(h, st, cfg.variant);

  const int rows = N * B, cands = rows * K;
  const int r_out = cfg.variant == 0 ? kR : 2 * kR;          // candidate outputs
  const int s_out = cfg.variant == 0 ? 3 * kR : 2 * kR;      // draft-slot outputs
  dc::ProjJob cj{E, ids, ws.cand_proj, cands, r_out, dc::proj_tc_tiles(cands, r_out)};
  cj.f16 = true;  // the candidate rows in fp16: one MMA per k-step
  if (cfg.variant == 0) {
    // the reduction leaves b = LN0(W_cand E[c]) ready for the fuse product
    cj.C = nullptr;
    cj.ln_hi = ws.b_hi;
    cj.ln_lo = ws.b_lo;
    cj.ln_eps = cfg.ln_eps;
  }
  const dc::ProjJob sj{hidden, nullptr, ws.slot_proj, rows, s_out, dc::proj_tc_tiles(rows, s_out)};
  // step 1: candidate pools.  Without the candidate features each finished
  // row releases a flag (features or logits in host memory: no handoff).
  // (Prefetching the rows' candidate embeddings into L2 from here was
  // measured: the top-K 4 us slower, the projection no faster.)
  const dc::TopkPlan plan = dc::topk_plan(V, N * B, h->topk_wave);
  dc::TopkHandoff hand;
  if (handoff) {
    hand.row_ready = ws.row_ready;
    cj.row_ready = ws.row_ready;
    cj.cands_per_row = K;
  }
  DC_TRY(clk.done(dc::launch_topk(K, logits, in->logits_slot_stride, cfg.slots, N, V, plan, ws.part, ws.row_count,
                                  ids, vals, st, false, ws.part_lse, out->cand_feat, hand)));
  // step 2 (and the slot-pair state): the candidate rows and the draft-slot
  // rows go through one projection launch, which fills the device in one
  // wave.  It overlaps the top-K's tail: its blocks take SMs as the top-K's
  // leave, the draft-slot tiles start at once and each candidate tile waits
  // for its own rows' flags (or, without the handoff, for the whole top-K).
  DC_TRY(clk.done(dc::launch_proj_tc(cj, w->map_cand_f16, w->map_cand_f16, &sj, &w->map_slot_hi, &w->map_slot_lo,
                                     cfg.slots, B, d, V, h->splits, ws.err, st, true)));
  if (cfg.variant == 0) {
    // steps 2-3: per-slot / per-pair terms, z and the layer-1 partials U, V
    DC_TRY(clk.done(dc::launch_maps_tc(w->mlp_maps, h->slot_io, h->cand_io, ws.slot_proj, vals, w->mlp, N, B,
                                       K, cfg.ln_eps, ws.err, st)));
    // steps 4-5: all (B-1) K^2 transition scores, then each request's walk
    // and verify in its last block
    const dc::WalkArgs wk{ids, in->target_tokens, out->tokens, choice,
                          in->target_tokens ? out->accept_len : nullptr, margin, ws.req_count,
                          cfg.path_rule, cfg.beam_width, beam_topm(cfg)};
    DC_TRY(clk.done(dc::launch_pair_score_walk(K, ws.U, ws.V, ws.P, vals, w->mlp.w2, w->mlp.b2, N, B,
                                               scores, wk, st)));
    return DCOCO_OK;
  }
  // steps 4-5: normalised in/out vectors, all (B-1) K^2 cosine scores, then
  // each request's walk and verify in its last block
  const dc::WalkArgs wk{ids, in->target_tokens, out->tokens, choice,
                        in->target_tokens ? out->accept_len : nullptr, margin, ws.req_count,
                        cfg.path_rule, cfg.beam_width, beam_topm(cfg)};
  DC_TRY(clk.done(dc::launch_cos_pair_walk(K, ws.cand_proj, ws.slot_proj, vals, cfg.sigma, N, B, scores, wk, st)));
  return DCOCO_OK;
}

// Host-side packing of the fp32 vectors of the MLP (the 128-deep maps go to
// the device as bf16 hi / lo halves, see dcoco_weights_create).
void pack_mlp(const dcoco_weight_ptrs &w, std::vector<float> &buf, size_t off[8]) {
  const int r = kR, H = kH, in = 3 * kR + 2;
  size_t o = 0;
  auto take = [&](size_t n) { size_t at = (o + 63) & ~size_t(63); o = at + n; return at; };
  off[0] = take(0);      // (unused)
  off[1] = take(0);      // (unused)
  off[2] = take(H);      // w_la = W1[:, 3r]
  off[3] = take(H);      // w_lb = W1[:, 3r+1]
  off[4] = take(H);      // b1' = b1 + W1[:, r:2r] beta + W1[:, 2r:3r] beta (beta of z, moved into P)
  off[5] = take(H);      // w2
  off[6] = take(1);      // b2
  off[7] = take((size_t)r * r);  // W_fuse[:, r:], in the candidate maps' register order
  buf.assign(o, 0.f);
  for (int j = 0; j < H; ++j) {
    buf[off[2] + j] = w.w1[(size_t)j * in + 3 * r];
    buf[off[3] + j] = w.w1[(size_t)j * in + 3 * r + 1];
    double bj = w.b1[j];
    for (int k = 0; k < r; ++k)
      bj += ((double)w.w1[(size_t)j * in + r + k] + (double)w.w1[(size_t)j * in + 2 * r + k]) * w.ln_beta[k];
    buf[off[4] + j] = (float)bj;
    buf[off[5] + j] = w.w2[j];
  }
  buf[off[6]] = w.b2[0];
  // Thread `lane` of warp `wp` holds W_fuse[o][r + 32 g + e], o = 32 (wp / 4)
  // + lane, g = wp % 4, e < 32, and loads it as 8 float4 steps; step i of the
  // warp reads 512 contiguous bytes: element ((wp * 8 + i) * 32 + lane) * 4 + j
  // is e = 4 i + j.
  for (int wp = 0; wp < r / 8; ++wp)
    for (int i = 0; i < 8; ++i)
      for (int lane = 0; lane < 32; ++lane)
        for (int j = 0; j < 4; ++j) {
          const int o2 = 32 * (wp / 4) + lane, k = 32 * (wp % 4) + 4 * i + j;
          buf[off[7] + ((size_t)(wp * 8 + i) * 32 + lane) * 4 + j] = w.w_fuse[(size_t)o2 * 2 * r + r + k];
        }
}

}  // namespace

extern "C" {

int dcoco_version(void) { return 100; }

int dcoco_host_range_covers(uint64_t range_start, uint64_t range_size, uint64_t ptr, uint64_t bytes) {
  if (range_size == 0 || ptr < range_start) return 0;
  const uint64_t off = ptr - range_start;
  return off <= range_size && bytes <= range_size - off ? 1 : 0;
}

const char *dcoco_status_string(int s) {
  switch (s) {
    case DCOCO_OK: return "ok";
    case DCOCO_EINVAL: return "invalid argument";
    case DCOCO_EUNSUPPORTED: return "unsupported configuration";
    case DCOCO_EBATCH: return "batch outside [0, max_batch]";
    case DCOCO_ECUDA: return "CUDA runtime error";
    case DCOCO_ENOMEM: return "out of memory";
    case DCOCO_EDEVICE: return "a kernel flagged bad input data";
    default: return "unknown status";
  }
}

int dcoco_create(const dcoco_config *cfg, dcoco_handle **out) {
  if (!out) return DCOCO_EINVAL;
  int rc = validate_config(cfg);
  if (rc != DCOCO_OK) return rc;
  dcoco_handle *h = new (std::nothrow) dcoco_handle();
  if (!h) return DCOCO_ENOMEM;
  h->cfg = *cfg;
  h->B = cfg->slots - 1;
  h->topk_segments_max = dc::topk_max_segments(cfg->vocab);
  int sms = 0;
  if (cudaGetDevice(&h->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, h->device) != cudaSuccess) {
    delete h;
    return DCOCO_ECUDA;
  }
  h->topk_wave = sms * dc::topk_occupancy(cfg->topk);
  {
    // split-K of the projection: up to eight CTAs per tile (a portable
    // cluster), as many as keep the largest call (max_batch) in one wave of
    // one CTA per SM (a second wave repeats the fill, drain and reduction);
    // fixed per handle, so results do not depend on the batch
    const int rows_cap = cfg->max_batch * h->B, cands_cap = rows_cap * cfg->topk;
    const int r_out = cfg->variant == 0 ? kR : 2 * kR, s_out = cfg->variant == 0 ? 3 * kR : 2 * kR;
    const int tiles = dc::proj_tc_tiles(cands_cap, r_out) + dc::proj_tc_tiles(rows_cap, s_out);
    int want = 8;
    while (want > 1 && (long long)tiles * want > sms) want /= 2;
    h->splits = dc::proj_tc_splits(cfg->hidden, want);
  }
  Carver sizer;
  carve_workspace(sizer, h->cfg, h->B, h->topk_segments_max, h->ws);
  const size_t bytes = sizer.off + 256;
  if (cudaMalloc(&h->block, bytes) != cudaSuccess) {
    cudaGetLastError();
    delete h;
    return DCOCO_ENOMEM;
  }
  Carver c;
  c.base = static_cast<char *>(h->block);
  carve_workspace(c, h->cfg, h->B, h->topk_segments_max, h->ws);
  const int rows_cap = cfg->max_batch * h->B, cands_cap = rows_cap * cfg->topk;
  const bool maps_ok =
      cfg->variant != 0 ||
      (dc::encode_bf16_rows_map(&h->cand_io.bh, h->ws.b_hi, cands_cap, kR, 128) &&
       dc::encode_bf16_rows_map(&h->cand_io.bl, h->ws.b_lo, cands_cap, kR, 128) &&
       dc::encode_f32_rows_map(&h->cand_io.u, h->ws.U, cands_cap, kH, 128) &&
       dc::encode_f32_rows_map(&h->cand_io.v, h->ws.V, cands_cap, kH, 128) &&
       dc::encode_f32_rows_map(&h->slot_io.sp, h->ws.slot_proj, rows_cap, 3 * kR, 128) &&
       dc::encode_f32_rows_map(&h->slot_io.p, h->ws.P, rows_cap, kH, 128));
  if (!maps_ok || cudaMemset(h->block, 0, bytes) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) {
    cudaGetLastError();
    cudaFree(h->block);
    delete h;
    return DCOCO_ECUDA;
  }
  *out = h;
  return DCOCO_OK;
}

int dcoco_weights_create(dcoco_handle *h, const dcoco_weight_ptrs *wp, void *stream,
                         dcoco_weights **out) {
  if (!h || !wp || !out) return DCOCO_EINVAL;
  const dcoco_config &cfg = h->cfg;
  const int r = kR, d = cfg.hidden;
  if (cfg.variant == 0) {
    if (!wp->w_cand || !wp->w_ctx || !wp->w_fuse || !wp->ln_gamma || !wp->ln_beta || !wp->w_pair ||
        !wp->w1 || !wp->b1 || !wp->w2 || !wp->b2)
      return DCOCO_EINVAL;
  } else if (!wp->w_io) {
    return DCOCO_EINVAL;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);

  // Bring the fp32 weights to the host (if needed).
  auto fetch = [&](const float *p, size_t n, std::vector<float> &dst) -> int {
    dst.resize(n);
    if (wp->on_device) {
      if (cudaMemcpy(dst.data(), p, n * sizeof(float), cudaMemcpyDeviceToHost) != cudaSuccess)
        return DCOCO_ECUDA;
    } else {
      std::memcpy(dst.data(), p, n * sizeof(float));
    }
    return DCOCO_OK;
  };
  std::vector<float> w_cand, w_ctx, w_fuse, gam, bet, w_pair, w1, b1, w2, b2, w_io;
  int rc = DCOCO_OK;
  if (cfg.variant == 0) {
    if ((rc = fetch(wp->w_cand, (size_t)r * d, w_cand)) || (rc = fetch(wp->w_ctx, (size_t)r * d, w_ctx)) ||
        (rc = fetch(wp->w_fuse, (size_t)r * 2 * r, w_fuse)) || (rc = fetch(wp->ln_gamma, r, gam)) ||
        (rc = fetch(wp->ln_beta, r, bet)) || (rc = fetch(wp->w_pair, (size_t)r * 2 * d, w_pair)) ||
        (rc = fetch(wp->w1, (size_t)kH * (3 * r + 2), w1)) || (rc = fetch(wp->b1, kH, b1)) ||
        (rc = fetch(wp->w2, kH, w2)) || (rc = fetch(wp->b2, 1, b2)))
      return rc;
  } else if ((rc = fetch(wp->w_io, (size_t)2 * r * 2 * d, w_io))) {
    return rc;
  }

  // Projection weights: rows of the stacked matrices, split into bf16 hi/lo.
  const int cand_rows = cfg.variant == 0 ? r : 2 * r;
  const int slot_rows = cfg.variant == 0 ? 3 * r : 2 * r;
  std::vector<uint16_t> proj((size_t)(cand_rows + 2 * slot_rows) * d);
  uint16_t *c_f16 = proj.data();
  uint16_t *s_hi = c_f16 + (size_t)cand_rows * d, *s_lo = s_hi + (size_t)slot_rows * d;
  auto f16_row = [&](const float *src, uint16_t *dst) {
    for (int k = 0; k < d; ++k) dst[k] = f32_to_f16(src[k]);
  };
  auto split_row = [&](const float *src, uint16_t *hi, uint16_t *lo) {
    for (int k = 0; k < d; ++k) {
      const uint16_t hb = f32_to_bf16(src[k]);
      hi[k] = hb;
      lo[k] = f32_to_bf16(src[k] - bf16_to_f32(hb));
    }
  };
  if (cfg.variant == 0) {
    for (int o = 0; o < r; ++o) {
      f16_row(w_cand.data() + (size_t)o * d, c_f16 + (size_t)o * d);
      split_row(w_ctx.data() + (size_t)o * d, s_hi + (size_t)o * d, s_lo + (size_t)o * d);
      split_row(w_pair.data() + (size_t)o * 2 * d, s_hi + (size_t)(r + o) * d, s_lo + (size_t)(r + o) * d);
      split_row(w_pair.data() + (size_t)o * 2 * d + d, s_hi + (size_t)(2 * r + o) * d,
                s_lo + (size_t)(2 * r + o) * d);
    }
  } else {
    for (int o = 0; o < 2 * r; ++o) {
      f16_row(w_io.data() + (size_t)o * 2 * d, c_f16 + (size_t)o * d);
      split_row(w_io.data() + (size_t)o * 2 * d + d, s_hi + (size_t)o * d, s_lo + (size_t)o * d);
    }
  }
  // The 128-deep MLP maps (variant 0), split the same way, in the order
  // fb, fg, w1ab, w1s, each as hi then lo.
  const size_t n_rr = (size_t)kR * kR, n_w1ab = (size_t)2 * kH * kR, n_w1s = (size_t)kH * kR;
  if (cfg.variant == 0) {
    std::vector<uint16_t> cm(2 * (2 * n_rr + n_w1ab + n_w1s));
    uint16_t *fbh = cm.data(), *fbl = fbh + n_rr, *fgh = fbl + n_rr, *fgl = fgh + n_rr;
    uint16_t *w1h = fgl + n_rr, *w1l = w1h + n_w1ab, *wsh = w1l + n_w1ab, *wsl = wsh + n_w1s;
    auto split_vec = [&](const float *src, uint16_t *hi, uint16_t *lo) {
      for (int k = 0; k < kR; ++k) {
        const uint16_t hb = f32_to_bf16(src[k]);
        hi[k] = hb;
        lo[k] = f32_to_bf16(src[k] - bf16_to_f32(hb));
      }
    };
    for (int o = 0; o < kR; ++o) {
      split_vec(w_fuse.data() + (size_t)o * 2 * kR, fbh + (size_t)o * kR, fbl + (size_t)o * kR);
      split_vec(w_fuse.data() + (size_t)o * 2 * kR + kR, fgh + (size_t)o * kR, fgl + (size_t)o * kR);
    }
    const size_t in1 = 3 * kR + 2;
    // the candidate parts of layer 1 take z's gamma: W1[:, r:2r] diag(gamma), W1[:, 2r:3r] diag(gamma)
    std::vector<float> wa(kR), wb(kR);
    for (int j = 0; j < kH; ++j) {
      for (int k = 0; k < kR; ++k) {
        wa[k] = (float)((double)w1[j * in1 + kR + k] * gam[k]);
        wb[k] = (float)((double)w1[j * in1 + 2 * kR + k] * gam[k]);
      }
      split_vec(wa.data(), w1h + (size_t)j * kR, w1l + (size_t)j * kR);
      split_vec(wb.data(), w1h + (size_t)(kH + j) * kR, w1l + (size_t)(kH + j) * kR);
      split_vec(w1.data() + j * in1, wsh + (size_t)j * kR, wsl + (size_t)j * kR);
    }
    proj.insert(proj.end(), cm.begin(), cm.end());
  }
  const size_t n_proj = proj.size();
  std::vector<float> mlp;
  size_t off[8] = {};
  if (cfg.variant == 0) {
    dcoco_weight_ptrs hw = *wp;
    hw.w_fuse = w_fuse.data(); hw.ln_gamma = gam.data(); hw.ln_beta = bet.data();
    hw.w1 = w1.data(); hw.b1 = b1.data(); hw.w2 = w2.data(); hw.b2 = b2.data();
    pack_mlp(hw, mlp, off);
  }
  const size_t proj_bytes = ((n_proj * sizeof(uint16_t)) + 255) & ~size_t(255);
  const size_t total = proj_bytes + mlp.size() * sizeof(float) + 256;

  dcoco_weights *w = new (std::nothrow) dcoco_weights();
  if (!w) return DCOCO_ENOMEM;
  w->owner = h;
  w->device = h->device;
  if (cudaMalloc(&w->block, total) != cudaSuccess) {
    cudaGetLastError();
    delete w;
    return DCOCO_ENOMEM;
  }
  char *base = static_cast<char *>(w->block);
  uint16_t *dproj = reinterpret_cast<uint16_t *>(base);
  float *dmlp = reinterpret_cast<float *>(base + proj_bytes);
  bool ok = cudaMemcpyAsync(dproj, proj.data(), n_proj * sizeof(uint16_t), cudaMemcpyHostToDevice,
                            st) == cudaSuccess;
  if (ok && !mlp.empty())
    ok = cudaMemcpyAsync(dmlp, mlp.data(), mlp.size() * sizeof(float), cudaMemcpyHostToDevice, st) ==
         cudaSuccess;
  ok = ok && cudaStreamSynchronize(st) == cudaSuccess;
  if (!ok) {
    cudaFree(w->block);
    delete w;
    return DCOCO_ECUDA;
  }
  w->cand_f16 = dproj;
  w->slot_hi = w->cand_f16 + (size_t)cand_rows * d;
  w->slot_lo = w->slot_hi + (size_t)slot_rows * d;
  if (cfg.variant == 0) {
    w->fb_hi = w->slot_lo + (size_t)slot_rows * d;
    w->fb_lo = w->fb_hi + n_rr;
    w->fg_hi = w->fb_lo + n_rr;
    w->fg_lo = w->fg_hi + n_rr;
    w->w1ab_hi = w->fg_lo + n_rr;
    w->w1ab_lo = w->w1ab_hi + n_w1ab;
    w->w1s_hi = w->w1ab_lo + n_w1ab;
    w->w1s_lo = w->w1s_hi + n_w1s;
  }
  if (!dc::encode_f16_rows_map(&w->map_cand_f16, w->cand_f16, cand_rows, d, 128) ||
      !dc::encode_bf16_rows_map(&w->map_slot_hi, w->slot_hi, slot_rows, d, 128) ||
      !dc::encode_bf16_rows_map(&w->map_slot_lo, w->slot_lo, slot_rows, d, 128) ||
      (cfg.variant == 0 &&
       (!dc::encode_bf16_rows_map(&w->mlp_maps.fb_hi, w->fb_hi, kR, kR, 128) ||
        !dc::encode_bf16_rows_map(&w->mlp_maps.fb_lo, w->fb_lo, kR, kR, 128) ||
        !dc::encode_bf16_rows_map(&w->mlp_maps.fg_hi, w->fg_hi, kR, kR, 128) ||
        !dc::encode_bf16_rows_map(&w->mlp_maps.fg_lo, w->fg_lo, kR, kR, 128) ||
        !dc::encode_bf16_rows_map(&w->mlp_maps.w1_hi, w->w1ab_hi, 2 * kH, kR, 128) ||
        !dc::encode_bf16_rows_map(&w->mlp_maps.w1_lo, w->w1ab_lo, 2 * kH, kR, 128) ||
        !dc::encode_bf16_rows_map(&w->mlp_maps.w1s_hi, w->w1s_hi, kH, kR, 128) ||
        !dc::encode_bf16_rows_map(&w->mlp_maps.w1s_lo, w->w1s_lo, kH, kR, 128)))) {
    cudaFree(w->block);
    delete w;
    return DCOCO_ECUDA;
  }
  if (cfg.variant == 0) {
    dc::MlpWeightsDev &m = w->mlp;
    m.w_la = dmlp + off[2]; m.w_lb = dmlp + off[3];
    m.b1 = dmlp + off[4]; m.w2 = dmlp + off[5]; m.b2 = dmlp + off[6]; m.w_fg = dmlp + off[7];
  }
  *out = w;
  return DCOCO_OK;
}

int dcoco_correct(dcoco_handle *h, const dcoco_weights *w, int batch, const dcoco_inputs *in,
                  const dcoco_outputs *out, void *stream) {
  int rc = validate_call(h, w, batch, in, out, true);
  if (rc != DCOCO_OK || batch == 0) return rc;
  return run_path(h, w, batch, in, out, static_cast<cudaStream_t>(stream));
}

int dcoco_correct_host(dcoco_handle *h, const dcoco_weights *w, int batch, const dcoco_inputs *in,
                       const dcoco_outputs *out, void *stream) {
  int rc = validate_call(h, w, batch, in, out, false);
  if (rc != DCOCO_OK || batch == 0) return rc;
  if (!h->cfg.host_staging) return DCOCO_EINVAL;
  const dcoco_config &cfg = h->cfg;
  const Workspace &ws = h->ws;
  const int B = h->B, K = cfg.topk;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t rows = (size_t)batch * cfg.slots;
  // inputs.  Logits in page-locked host memory that the device can address
  // are read in place by the top-K (over the host link, at the rate a copy
  // would get, without the copy's serial step before the kernel); otherwise
  // their rows are copied to the dense staging buffer first.  Hidden states
  // and targets (small) are copied.
  const void *logits_dev = nullptr;
  {
    // In place only if the whole extent the top-K reads lies inside one
    // page-locked range (a caller may have registered part of a buffer).
    const uint64_t extent = (uint64_t)((rows - 1) * in->logits_slot_stride + cfg.vocab) * sizeof(uint16_t);
    cudaPointerAttributes pa;
    uint64_t r0 = 0, rsize = 0;
    if (cudaPointerGetAttributes(&pa, in->logits) == cudaSuccess && pa.type == cudaMemoryTypeHost &&
        pa.devicePointer && aligned16(pa.devicePointer) && in->logits_slot_stride % 8 == 0 &&
        host_range_of(in->logits, &r0, &rsize) &&
        dcoco_host_range_covers(r0, rsize, reinterpret_cast<uintptr_t>(in->logits), extent))
      logits_dev = pa.devicePointer;
    cudaGetLastError();  // an unregistered pointer is not an error here
  }
  if (!logits_dev)
    DC_TRY(cudaMemcpy2DAsync(ws.st_logits, ws.st_stride * sizeof(uint16_t), in->logits,
                             in->logits_slot_stride * sizeof(uint16_t), cfg.vocab * sizeof(uint16_t),
                             rows, cudaMemcpyHostToDevice, st));
  DC_TRY(cudaMemcpyAsync(ws.st_hidden, in->hidden, rows * cfg.hidden * sizeof(uint16_t),
                         cudaMemcpyHostToDevice, st));
  if (in->target_tokens)
    DC_TRY(cudaMemcpyAsync(ws.st_target, in->target_tokens, (size_t)batch * B * sizeof(int32_t),
                           cudaMemcpyHostToDevice, st));
  dcoco_inputs din = *in;
  din.logits = logits_dev ? logits_dev : ws.st_logits;
  din.logits_slot_stride = logits_dev ? in->logits_slot_stride : ws.st_stride;
  din.hidden = ws.st_hidden;
  din.target_tokens = in->target_tokens ? ws.st_target : nullptr;
  dcoco_outputs dout = {};
  dout.tokens = ws.st_tokens;
  dout.accept_len = in->target_tokens ? ws.st_accept : nullptr;
  rc = run_path(h, w, batch, &din, &dout, st, logits_dev != nullptr);
  if (rc != DCOCO_OK) return rc;
  // outputs: tokens, accept_len (+ optional extras from the workspace)
  DC_TRY(cudaMemcpyAsync(out->tokens, ws.st_tokens, (size_t)batch * B * sizeof(int32_t),
                         cudaMemcpyDeviceToHost, st));
  if (in->target_tokens)
    DC_TRY(cudaMemcpyAsync(out->accept_len, ws.st_accept, (size_t)batch * sizeof(int32_t),
                           cudaMemcpyDeviceToHost, st));
  if (out->topk_ids)
    DC_TRY(cudaMemcpyAsync(out->topk_ids, ws.ids, (size_t)batch * B * K * sizeof(int32_t),
                           cudaMemcpyDeviceToHost, st));
  if (out->topk_val)
    DC_TRY(cudaMemcpyAsync(out->topk_val, ws.vals, (size_t)batch * B * K * sizeof(float),
                           cudaMemcpyDeviceToHost, st));
  if (out->scores)
    DC_TRY(cudaMemcpyAsync(out->scores, ws.scores, (size_t)batch * (B - 1) * K * K * sizeof(float),
                           cudaMemcpyDeviceToHost, st));
  if (out->choice)
    DC_TRY(cudaMemcpyAsync(out->choice, ws.choice, (size_t)batch * B * sizeof(int32_t),
                           cudaMemcpyDeviceToHost, st));
  if (out->margin)
    DC_TRY(cudaMemcpyAsync(out->margin, ws.margin, (size_t)batch * (B - 1) * sizeof(float),
                           cudaMemcpyDeviceToHost, st));
  return cuda_status(cudaStreamSynchronize(st));
}

int dcoco_topk(dcoco_handle *h, int batch, const void *logits, int64_t stride, int32_t *topk_ids,
               float *topk_val, void *stream) {
  if (!h) return DCOCO_EINVAL;
  if (batch < 0 || batch > h->cfg.max_batch) return DCOCO_EBATCH;
  if (batch == 0) return DCOCO_OK;
  if (!logits || !topk_ids || !topk_val) return DCOCO_EINVAL;
  if (stride < h->cfg.vocab || stride % 8 != 0 || !aligned16(logits)) return DCOCO_EINVAL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  h->last_stream = st;
  ++h->launches;
  const dc::TopkPlan plan = dc::topk_plan(h->cfg.vocab, batch * h->B, h->topk_wave);
  // Launched without programmatic overlap: the kernel streams the logits
  // before its dependency wait, so it must not start while the caller's
  // previous kernel on the stream may still be writing them.
  return cuda_status(dc::launch_topk(h->cfg.topk, static_cast<const uint16_t *>(logits), stride,
                                     h->cfg.slots, batch, h->cfg.vocab, plan, h->ws.part,
                                     h->ws.row_count, topk_ids, topk_val, st, false));
}

int dcoco_verify_stochastic(dcoco_handle *h, int batch, const void *target_logits, int64_t target_stride,
                            const int32_t *tokens, const float *u_accept, const float *u_draw, int32_t *accept_len,
                            int32_t *next_token, float *q_accept, void *stream) {
  if (!h) return DCOCO_EINVAL;
  if (batch < 0 || batch > h->cfg.max_batch) return DCOCO_EBATCH;
  if (batch == 0) return DCOCO_OK;
  if (!target_logits || !tokens || !u_accept || !u_draw || !accept_len || !next_token) return DCOCO_EINVAL;
  if (target_stride < h->cfg.vocab || target_stride % 8 != 0 || !aligned16(target_logits)) return DCOCO_EINVAL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  h->last_stream = st;
  ++h->launches;
  const Workspace &ws = h->ws;
  return cuda_status(dc::launch_verify_stochastic(
      static_cast<const uint16_t *>(target_logits), target_stride, h->cfg.vocab, batch, h->B, tokens, u_accept,
      u_draw, ws.v_chunk_m, ws.v_chunk_s, ws.v_lse, q_accept ? q_accept : ws.v_q, ws.v_count, accept_len,
      next_token, st));
}

int dcoco_selftest_wait_timeout(dcoco_handle *h, long long limit_ns, void *stream) {
  if (!h || limit_ns < 1000 || limit_ns > 1000000000LL) return DCOCO_EINVAL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  h->last_stream = st;
  ++h->launches;
  return cuda_status(dc::launch_wait_timeout((unsigned long long)limit_ns, h->ws.err, st));
}

int dcoco_get_device_status(dcoco_handle *h) {
  if (!h) return DCOCO_EINVAL;
  if (cudaStreamSynchronize(h->last_stream) != cudaSuccess) return DCOCO_ECUDA;
  int flag = 0;
  if (cudaMemcpy(&flag, h->ws.err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return DCOCO_ECUDA;
  if (flag != 0) {
    if (cudaMemset(h->ws.err, 0, sizeof(int)) != cudaSuccess) return DCOCO_ECUDA;
    return DCOCO_EDEVICE;
  }
  return DCOCO_OK;
}

void dcoco_weights_destroy(dcoco_weights *w) {
  if (!w) return;
  cudaDeviceSynchronize();
  cudaFree(w->block);
  delete w;
}

void dcoco_destroy(dcoco_handle *h) {
  if (!h) return;
  cudaDeviceSynchronize();
  for (cudaEvent_t e : h->events) cudaEventDestroy(e);
  cudaFree(h->block);
  delete h;
}

long long dcoco_kernel_launches(const dcoco_handle *h) { return h ? h->launches : -1; }

int dcoco_stage_timing(dcoco_handle *h, int enable) {
  if (!h) return DCOCO_EINVAL;
  if (enable && h->events.empty()) {
    const size_t n = (size_t)kMaxTimedCalls * (kMaxStages + 1);
    h->events.resize(n, nullptr);
    for (size_t i = 0; i < n; ++i)
      if (cudaEventCreate(&h->events[i]) != cudaSuccess) {
        for (size_t j = 0; j < i; ++j) cudaEventDestroy(h->events[j]);
        h->events.clear();
        return DCOCO_ECUDA;
      }
  }
  h->timing = enable != 0;
  return DCOCO_OK;
}

int dcoco_stage_read(dcoco_handle *h, int max_stages, float *ms, int *calls, int *n_stages) {
  if (!h || !ms || !calls || !n_stages || max_stages < 0) return DCOCO_EINVAL;
  // the stage list of the first recorded call; calls with another list are skipped
  const int kind = h->timed_calls > 0 ? h->timed_kind[0] : h->cfg.variant;
  const int ns = stage_count(kind);
  h->read_kind = kind;
  *n_stages = ns;
  *calls = 0;
  for (int s = 0; s < max_stages && s < ns; ++s) ms[s] = 0.f;
  for (int c = 0; c < h->timed_calls; ++c) {
    if (h->timed_kind[c] != kind) continue;
    cudaEvent_t *ev = h->events.data() + (size_t)c * (kMaxStages + 1);
    if (cudaEventSynchronize(ev[ns]) != cudaSuccess) return DCOCO_ECUDA;
    for (int s = 0; s < max_stages && s < ns; ++s) {
      float t = 0.f;
      if (cudaEventElapsedTime(&t, ev[s], ev[s + 1]) != cudaSuccess) return DCOCO_ECUDA;
      ms[s] += t;
    }
    ++*calls;
  }
  h->timed_calls = 0;
  return DCOCO_OK;
}

const char *dcoco_stage_name(const dcoco_handle *h, int s) {
  if (!h) return nullptr;
  const int kind = h->read_kind >= 0 ? h->read_kind : h->cfg.variant;
  if (s < 0 || s >= stage_count(kind)) return nullptr;
  return kStageNames[kind][s];
}

}  // extern "C"
