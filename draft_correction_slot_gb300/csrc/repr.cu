// repr.cu -- step 4, the K x K transition scores of every slot pair (with
// step 5 in the last block of each request), for the MLP and the cosine
// variants.
//
// DCOCO page ("Contextual Correction of Parallel Drafts for Speculative
// Decoding"), Method step details (4):
//   S_p(a,b) = l_{p+1}(b) + Delta([s_p; z_p^a; z_{p+1}^b; l_p(a); l_{p+1}(b)]),
//   Delta = 386 -> 256 -> 1 MLP with GELU, weights shared by all slots.
// Layer 1 of Delta is linear in its concatenated input, so it splits into a
// per-pair part P_p = W1_s s_p + b1, a predecessor part U = W1_a z^a + w_la l(a)
// and a successor part V = W1_b z^b + w_lb l(b) (computed in mlp_tc.cu).  Each
// of the (B-1) K^2 pairs then costs one add, one GELU and one 256-long dot
// with w2.  All arithmetic is fp32.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "walk.cuh"
#include "launch.h"

namespace dc {
namespace {

constexpr int R = 128;  // representation width
constexpr int H = 256;  // MLP hidden width


// ---------------------------------------------------------------- step 5
// The last block of request n to finish its pair (counted in req_count,
// zero between calls) selects the request's path (greedy walk, highest-
// scoring path or beam walk) and verifies it.  Called by every thread of a
// 256-thread block after the block's scores are stored; `sm` is the block's
// dynamic shared memory (the walk's tables, and the request's scores for
// path rules 1 and 2 when they fit).
template <int K>
__device__ __forceinline__ void request_tail(float *sm, int n, int B, const float *scores, const WalkArgs &wk) {
  const int tid = threadIdx.x;
  __shared__ int s_last;
  __shared__ int s_choice[32];
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(&wk.req_count[n], 1u) == (unsigned)(B - 2);
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  int *s_best = reinterpret_cast<int *>(sm);
  float *s_gap = sm + kWalkMaxRows;
  const int64_t slot0 = (int64_t)n * B;
  const float *sc = scores + (int64_t)n * (B - 1) * K * K;
  const int32_t *tg = wk.target ? wk.target + slot0 : nullptr;
  int32_t *ch = wk.choice ? wk.choice + slot0 : nullptr, *al = wk.accept_len ? wk.accept_len + n : nullptr;
  float *mg = wk.margin ? wk.margin + (int64_t)n * (B - 1) : nullptr;
  if (wk.path_rule != 0) {
    // the request's scores go to shared memory past the walk's tables when they fit
    float *s_sc = sm + 2 * kWalkMaxRows;
    const bool fits = (2 * kWalkMaxRows + (size_t)(B - 1) * K * K) * sizeof(float) <= dynamic_smem_bytes();
    if (wk.path_rule == 1)
      viterbi_verify_request<K>(sc, wk.topk_ids + slot0 * K, tg, B, wk.tokens + slot0, ch, mg, al, s_best, s_gap,
                                s_choice, fits ? s_sc : nullptr);
    else
      beam_verify_request<K>(sc, wk.topk_ids + slot0 * K, tg, B, wk.tokens + slot0, ch, mg, al, wk.beam_width,
                             wk.beam_topm, s_best, s_gap, s_choice, fits ? s_sc : nullptr);
  } else {
    walk_verify_request<K>(sc, wk.topk_ids + slot0 * K, tg, B, wk.tokens + slot0, ch, mg, al, s_best, s_gap,
                           s_choice, reinterpret_cast<int *>(sm + 2 * kWalkMaxRows));
  }
  if (tid == 0) wk.req_count[n] = 0u;  // ready for the next call
}

// ---------------------------------------------------------------- pair scores
// With x = (P_p + U_{p,a} + V_{p+1,b}) / sqrt(2) and w' = w2 / sqrt(2),
//   w2_j GELU(sqrt(2) x_j) = w'_j x_j (1 + erf(x_j)) = w'_j x_j + w'_j |x_j| erf(|x_j|).
// The first term is separable, sum_j w'_j x_j = d_a + d_b with
// d_a = sum_j w'_j (P_p + U_{p,a})_j / sqrt(2) and d_b = sum_j w'_j V_{p+1,b,j} / sqrt(2),
// so the K^2 x H inner loop only evaluates w' |x| erf(|x|).
//
// erfc on x >= 0 is evaluated as 2^p(x), p a degree-5 polynomial fitted to
// log2 erfc(x) on [0, 5] (weighted least squares, iterated towards the
// smallest maximum of |x (erfc(x) - 2^p(x))|, the error that reaches the
// scores; the fit script is fit_erfc.py beside this package): in fp32 that
// error stays below 7e-7 for every x in [0, 12], and beyond, p falls like
// -x^5, so 2^p underflows to 0 as erfc does.  Per element: five FMAs and one
// hardware base-2 exponential (the special-function unit's fastest
// operation), then w' |x| (1 - erfc(|x|)) as |x| (w' - w' erfc(|x|)), one
// FMA for the bracket and one into the accumulator -- eight FMA-pipe lane
// operations.
constexpr float kErfc0 = -3.75319205e-05f, kErfc1 = -1.62746069f, kErfc2 = -0.919982363f;
constexpr float kErfc3 = -0.146592411f, kErfc4 = 0.028338989f, kErfc5 = -0.00267746694f;

// Two fp32 lanes in one 64-bit register, for the packed f32x2 arithmetic.
typedef unsigned long long f2_t;
__device__ __forceinline__ f2_t f2_pack(float lo, float hi) {
  f2_t d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
  return d;
}
__device__ __forceinline__ void f2_unpack(f2_t v, float &lo, float &hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ f2_t f2_fma(f2_t a, f2_t b, f2_t c) {
  f2_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ f2_t f2_add(f2_t a, f2_t b) {
  f2_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f2_t f2_abs(f2_t a) { return a & 0x7FFFFFFF7FFFFFFFull; }
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// One CTA per slot pair (n, p).  Shared memory holds the K rows
// (P_p + U_{p,a}) / sqrt(2) and the K rows V_{p+1,b} / sqrt(2); each thread
// takes a 4 x 4 block of (a, b) over a strided slice of hidden-unit pairs
// (j, j+1) = 2s, 2s + 2 NS, ... (NS slices), the pair in the two lanes of
// the packed arithmetic, so every loaded value feeds four evaluations.  The
// slices' partial sums meet in shared memory and are added in slice order,
// so the result does not depend on scheduling.
template <int K>
struct PairGeom {
  static constexpr int T = 4;                      // (a, b) block per thread
  static constexpr int NT = (K / T) * (K / T);     // blocks
  static constexpr int NS = 256 / NT;              // slices of hidden-unit pairs
  static constexpr int JP = H / 2 / NS;            // pairs per slice
  // row stride (floats, even): the 64-bit reads of a half-warp hit distinct banks
  static constexpr int LD = K == 32 ? H + 2 : H + 4;
  static constexpr int RED = K * K + 1;            // partial-sum row stride
  // the partial sums reuse the staged rows once the main loop is done
  static_assert((size_t)NS * RED <= 2 * (size_t)K * LD, "partial sums fit the staged rows");
  static constexpr size_t pair_floats = 2 * (size_t)K * LD + H + 2 * K;
  // the walk reuses the first 3 kWalkMaxRows words (best, gap, the request's ids)
  static constexpr size_t smem_floats = pair_floats > 3 * (size_t)kWalkMaxRows ? pair_floats : 3 * (size_t)kWalkMaxRows;
};

// Three blocks per SM (the launch's residency cap): up to 85 registers a
// thread, enough for the compiler to interleave several of a thread's 16
// independent evaluations (64 serialised them and left the FMA pipe idle).
template <int K>
__global__ void __launch_bounds__(256, 3)
k_pair_score(const float *__restrict__ U, const float *__restrict__ V,
             const float *__restrict__ P, const float *__restrict__ topk_val,
             const float *__restrict__ w2, const float *__restrict__ b2, int B,
             float *__restrict__ scores, WalkArgs wk) {
  using G = PairGeom<K>;
  constexpr float kInvSqrt2 = 0.70710678118654752440f;
  extern __shared__ float sm[];
  float *pu = sm;                   // [K][LD]  (P_p + U_{p,a}) / sqrt(2)
  float *vs = pu + K * G::LD;       // [K][LD]  V_{p+1,b} / sqrt(2)
  float *w2s = vs + K * G::LD;      // [H]      w2 / sqrt(2)
  float *dab = w2s + H;             // [2K]     d_a, then d_b
  float *red = sm;                  // [NS][RED] partial sums, over pu and vs after the main loop
  const int np = blockIdx.x;        // n * (B-1) + p
  const int n = np / (B - 1), p = np - n * (B - 1);
  const int tid = threadIdx.x;
  pdl_trigger();
  pdl_wait();  // U, V (and this call's outputs) belong to the previous kernel until here
  const int64_t ca = ((int64_t)n * B + p) * K;      // first candidate of slot p
  const int64_t cb = ca + K;                         // first candidate of slot p+1
  const float *Pp = P + ((int64_t)n * B + p) * H;  // P is indexed by draft slot
  // Everything this call's earlier kernels wrote is read through L2 (ld.cg),
  // never the non-coherent path: with the programmatic launch this kernel is
  // already alive while they write it.
  __shared__ float s_tv[32];  // l_{p+1}(b), read at the end; loaded now
  const float bias = __ldg(b2);
  if (tid < K) s_tv[tid] = __ldcg(topk_val + cb + tid);

  // K * H / 4 is a multiple of 256: every thread has K / 4 chunks, all loads in flight together
  static_assert((K * H / 4) % 256 == 0, "whole staging rounds");
#pragma unroll
  for (int e4 = tid; e4 < K * H / 4; e4 += 256) {
    const int c = e4 / (H / 4), j = (e4 - c * (H / 4)) * 4;
    const float4 u = __ldcg(reinterpret_cast<const float4 *>(U + (ca + c) * H + j));
    const float4 pp = __ldcg(reinterpret_cast<const float4 *>(Pp + j));
    const float4 v = __ldcg(reinterpret_cast<const float4 *>(V + (cb + c) * H + j));
    float *x = pu + c * G::LD + j, *y = vs + c * G::LD + j;
    x[0] = (u.x + pp.x) * kInvSqrt2; x[1] = (u.y + pp.y) * kInvSqrt2;
    x[2] = (u.z + pp.z) * kInvSqrt2; x[3] = (u.w + pp.w) * kInvSqrt2;
    y[0] = v.x * kInvSqrt2; y[1] = v.y * kInvSqrt2; y[2] = v.z * kInvSqrt2; y[3] = v.w * kInvSqrt2;
  }
  w2s[tid] = w2[tid] * kInvSqrt2;
  __syncthreads();

  // separable part: 256 / 2K threads per row, each the hidden-unit pairs
  // part, part + TPR, ... (neighbouring lanes read neighbouring pairs), the
  // partial sums met by shuffles in a fixed order
  {
    constexpr int TPR = 256 / (2 * K);
    static_assert(TPR * 2 * K == 256 && TPR <= 32, "whole rows per warp");
    const int row = tid / TPR, part = tid - row * TPR;
    const float *xr = row < K ? pu + row * G::LD : vs + (row - K) * G::LD;
    float d0 = 0.f, d1 = 0.f;
#pragma unroll
    for (int i = 0; i < H / (2 * TPR); ++i) {
      const int j = 2 * (part + TPR * i);
      const float2 x = *reinterpret_cast<const float2 *>(xr + j);
      const float2 wv = *reinterpret_cast<const float2 *>(w2s + j);
      d0 = fmaf(wv.x, x.x, d0);
      d1 = fmaf(wv.y, x.y, d1);
    }
    float d = d0 + d1;
#pragma unroll
    for (int o = TPR / 2; o > 0; o >>= 1) d += __shfl_xor_sync(DC_FULL_MASK, d, o);
    if (part == 0) dab[row] = d;
  }

  const int blk = tid / G::NS, sl = tid - blk * G::NS;
  const int a0 = (blk / (K / G::T)) * G::T, b0 = (blk % (K / G::T)) * G::T;
  const f2_t c0 = f2_pack(kErfc0, kErfc0), c1 = f2_pack(kErfc1, kErfc1), c2 = f2_pack(kErfc2, kErfc2);
  const f2_t c3 = f2_pack(kErfc3, kErfc3), c4 = f2_pack(kErfc4, kErfc4), c5 = f2_pack(kErfc5, kErfc5);
  f2_t acc[G::T][G::T];
#pragma unroll
  for (int i = 0; i < G::T; ++i)
#pragma unroll
    for (int k = 0; k < G::T; ++k) acc[i][k] = 0ull;
#pragma unroll 4
  for (int jj = 0; jj < G::JP; ++jj) {
    const int j = 2 * (sl + jj * G::NS);
    const float2 wv = *reinterpret_cast<const float2 *>(w2s + j);
    const f2_t w = f2_pack(wv.x, wv.y), nw = f2_pack(-wv.x, -wv.y);
    f2_t xa[G::T], yb[G::T];
#pragma unroll
    for (int i = 0; i < G::T; ++i) {
      const float2 xv = *reinterpret_cast<const float2 *>(pu + (a0 + i) * G::LD + j);
      const float2 yv = *reinterpret_cast<const float2 *>(vs + (b0 + i) * G::LD + j);
      xa[i] = f2_pack(xv.x, xv.y);
      yb[i] = f2_pack(yv.x, yv.y);
    }
#pragma unroll
    for (int i = 0; i < G::T; ++i)
#pragma unroll
      for (int k = 0; k < G::T; ++k) {
        const f2_t ax = f2_abs(f2_add(xa[i], yb[k]));
        f2_t q = f2_fma(c5, ax, c4);
        q = f2_fma(q, ax, c3);
        q = f2_fma(q, ax, c2);
        q = f2_fma(q, ax, c1);
        q = f2_fma(q, ax, c0);  // log2 erfc(|x|)
        float q0, q1;
        f2_unpack(q, q0, q1);
        const f2_t rr = f2_pack(ex2_approx(q0), ex2_approx(q1));  // erfc(|x|)
        // w' |x| (1 - erfc) = |x| (w' - w' erfc): two operations
        acc[i][k] = f2_fma(ax, f2_fma(nw, rr, w), acc[i][k]);
      }
  }
  __syncthreads();  // every thread is done with pu and vs, which the partial sums overwrite
  float *rs = red + sl * G::RED;
#pragma unroll
  for (int i = 0; i < G::T; ++i)
#pragma unroll
    for (int k = 0; k < G::T; ++k) {
      float lo, hi;
      f2_unpack(acc[i][k], lo, hi);
      rs[(a0 + i) * K + b0 + k] = lo + hi;
    }
  __syncthreads();

  for (int e = tid; e < K * K; e += 256) {
    float sum = 0.f;
#pragma unroll 8
    for (int s2 = 0; s2 < G::NS; ++s2) sum += red[s2 * G::RED + e];
    const int aa = e / K, bb = e - aa * K;
    scores[(int64_t)np * K * K + e] = s_tv[bb] + bias + (dab[aa] + dab[K + bb]) + sum;
  }

  request_tail<K>(sm, n, B, scores, wk);
}

// ---------------------------------------------------------------- cosine variant
// One block per slot pair (n, p), the cosine variant's steps 4-5 in one
// launch: the out-vectors of slot p's candidates and the in-vectors of slot
// p+1's are summed from their candidate and draft-slot parts and
// normalised (x / max(|x|, 1e-12), one warp per vector) into shared memory,
// then S_p(a, b) = sigma <o_a, i_b> + l_{p+1}(b), then the request tail.
// (Each slot's vectors are normalised by the two blocks that read them.)
template <int K>
struct CosGeom {
  static constexpr size_t vec_floats = 2 * (size_t)K * (R + 1);
  static constexpr size_t min_floats = vec_floats > 3 * (size_t)kWalkMaxRows ? vec_floats : 3 * (size_t)kWalkMaxRows;
};

template <int K>
__global__ void __launch_bounds__(256)
k_cos_pair(const float *__restrict__ cand_io, const float *__restrict__ slot_io,
           const float *__restrict__ topk_val, float sigma, int B, float *__restrict__ scores, WalkArgs wk) {
  extern __shared__ float sm[];
  float(*os)[R + 1] = reinterpret_cast<float(*)[R + 1]>(sm);
  float(*is)[R + 1] = reinterpret_cast<float(*)[R + 1]>(sm + K * (R + 1));
  const int np = blockIdx.x;
  const int n = np / (B - 1), p = np - n * (B - 1);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  pdl_trigger();
  pdl_wait();  // cand_io, slot_io (and this call's outputs) belong to the previous kernels until here
  const int64_t sa = (int64_t)n * B + p, sb = sa + 1;  // draft-slot rows of slots p and p+1
  // everything this call's earlier kernels wrote is read through L2 (ld.cg);
  // a warp's 2K / 8 vectors load together, then sum, normalise and store
  constexpr int RW = 2 * K / 8;  // vectors per warp
  float x[RW][4];
#pragma unroll
  for (int i = 0; i < RW; ++i) {
    const int row = warp + 8 * i;
    const bool out = row < K;
    const int c = out ? row : row - K;
    const float *cv = cand_io + ((out ? sa : sb) * K + c) * 2 * R + (out ? 0 : R);
    const float *sv = slot_io + (out ? sa : sb) * 2 * R + (out ? 0 : R);
#pragma unroll
    for (int u = 0; u < 4; ++u) x[i][u] = __ldcg(cv + lane + 32 * u) + __ldcg(sv + lane + 32 * u);
  }
  const float tv = tid < K ? __ldcg(topk_val + sb * K + tid) : 0.f;  // l_{p+1}(b)
#pragma unroll
  for (int i = 0; i < RW; ++i) {
    const int row = warp + 8 * i;
    const bool out = row < K;
    const int c = out ? row : row - K;
    const float ss = warp_sum(x[i][0] * x[i][0] + x[i][1] * x[i][1] + x[i][2] * x[i][2] + x[i][3] * x[i][3]);
    const float scale = 1.0f / fmaxf(sqrtf(ss), 1e-12f);
    float *dst = out ? os[c] : is[c];
#pragma unroll
    for (int u = 0; u < 4; ++u) dst[lane + 32 * u] = x[i][u] * scale;
  }
  __shared__ float s_tv[32];
  if (tid < K) s_tv[tid] = tv;
  __syncthreads();
  // each dot product as four interleaved partial sums (k mod 4), added as
  // (p0 + p1) + (p2 + p3)
  for (int e = tid; e < K * K; e += 256) {
    const int a = e / K, bb = e - a * K;
    float p0 = 0.f, p1 = 0.f, p2 = 0.f, p3 = 0.f;
#pragma unroll 8
    for (int k = 0; k < R; k += 4) {
      p0 = fmaf(os[a][k], is[bb][k], p0);
      p1 = fmaf(os[a][k + 1], is[bb][k + 1], p1);
      p2 = fmaf(os[a][k + 2], is[bb][k + 2], p2);
      p3 = fmaf(os[a][k + 3], is[bb][k + 3], p3);
    }
    scores[(int64_t)np * K * K + e] = fmaf(sigma, (p0 + p1) + (p2 + p3), s_tv[bb]);
  }
  __syncthreads();  // the request tail reuses the vectors' shared memory
  request_tail<K>(sm, n, B, scores, wk);
}

}  // namespace

template <int K>
static cudaError_t pair_score_k(const float *U, const float *V, const float *P, const float *tv,
                                const float *w2, const float *b2, int N, int B, float *scores,
                                const WalkArgs &wk, cudaStream_t st) {
  // The blocks are launched early (programmatic overlap) onto whatever SMs
  // the previous kernel frees first; more than the even share per SM would
  // leave those SMs finishing last.  The shared-memory request caps the
  // resident blocks per SM at ceil(blocks / SMs).
  const int blocks = N * (B - 1);
  int dev = 0, sms = 1, sm_smem = 0, reserved = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sm_smem, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev);
  if (e != cudaSuccess) return e;
  size_t smem = PairGeom<K>::smem_floats * sizeof(float);
  const int per_sm = (blocks + sms - 1) / sms;
  if (per_sm < 8) {
    // one block more than per_sm must not fit: (per_sm + 1) (smem + reserved) > sm_smem
    const size_t cap = (size_t)(sm_smem / (per_sm + 1) - reserved + 16) & ~size_t(15);
    if (cap > smem && (size_t)per_sm * (cap + reserved) <= (size_t)sm_smem) smem = cap;
  }
  e = cudaFuncSetAttribute(k_pair_score<K>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  e = launch_ex(k_pair_score<K>, dim3(blocks), dim3(256), smem, st, true, 0, U, V, P, tv, w2, b2, B, scores,
                wk);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_pair_score_walk(int K, const float *U, const float *V, const float *P,
                                   const float *topk_val, const float *w2, const float *b2, int N, int B,
                                   float *scores, const WalkArgs &wk, cudaStream_t st) {
  if (N == 0) return cudaSuccess;
  switch (K) {
    case 8: return pair_score_k<8>(U, V, P, topk_val, w2, b2, N, B, scores, wk, st);
    case 16: return pair_score_k<16>(U, V, P, topk_val, w2, b2, N, B, scores, wk, st);
    case 32: return pair_score_k<32>(U, V, P, topk_val, w2, b2, N, B, scores, wk, st);
    default: return cudaErrorInvalidValue;
  }
}


template <int K>
static cudaError_t cos_pair_k(const float *cand_io, const float *slot_io, const float *tv, float sigma, int N,
                              int B, float *scores, const WalkArgs &wk, cudaStream_t st) {
  // path rules 1 and 2 stage the request's scores in shared memory when the
  // device allows it (up to 227 KB a block)
  size_t floats = CosGeom<K>::min_floats;
  const size_t with_scores = 2 * (size_t)kWalkMaxRows + (size_t)(B - 1) * K * K;
  if (wk.path_rule != 0 && with_scores * sizeof(float) <= 200 * 1024 && with_scores > floats) floats = with_scores;
  const size_t smem = floats * sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(k_cos_pair<K>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  e = launch_ex(k_cos_pair<K>, dim3(N * (B - 1)), dim3(256), smem, st, true, 0, cand_io, slot_io, tv, sigma, B,
                scores, wk);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_cos_pair_walk(int K, const float *cand_io, const float *slot_io, const float *topk_val,
                                 float sigma, int N, int B, float *scores, const WalkArgs &wk, cudaStream_t st) {
  if (N == 0) return cudaSuccess;
  switch (K) {
    case 8: return cos_pair_k<8>(cand_io, slot_io, topk_val, sigma, N, B, scores, wk, st);
    case 16: return cos_pair_k<16>(cand_io, slot_io, topk_val, sigma, N, B, scores, wk, st);
    case 32: return cos_pair_k<32>(cand_io, slot_io, topk_val, sigma, N, B, scores, wk, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace dc
