// verify.cu -- stochastic verification of a point-mass proposal
// (temperature 1), as its own launch after dcoco_correct.
//
// DCOCO page ("Contextual Correction of Parallel Drafts for Speculative
// Decoding"), Core method: a drafter that emits one token deterministically
// proposes the point mass p_j(v) = 1[v = y_j]; speculative sampling then
// accepts y_j with probability q_j(y_j) and, on rejection, resamples from
// r_j(v) = q_j(v) 1[v != y_j] / (1 - q_j(y_j)).  "Faster Decoding", Modified
// rejection sampling preserves the target distribution: left to right, stop
// at the first rejection with the corrected token; after full acceptance one
// bonus token from the target at the next position.
//
// One block per target row (request n, position j <= B) streams the row once:
// each warp takes 1024-token chunks and records the chunk's maximum and sum of
// exp(x - max); the row's log-sum-exp follows, and for j < B the acceptance
// probability q_j(y_j).  The last block of a request (a per-request counter)
// then finds the first rejection (u_j >= q_j(y_j)), and draws the corrected or
// bonus token by inverse transform in vocabulary order: a scan over the row's
// chunk weights picks the chunk, a scan inside the chunk picks the token.
// fp32 throughout: the row pass takes exp(x - m) as 2^(x log2 e - m log2 e)
// (one fma and the hardware ex2 per token, four partial sums, the next
// chunk's loads in flight); the rest uses CUDA's __expf / __logf.
#include <cstdint>

#include "common.cuh"
#include "kernels.h"

namespace dc {
namespace {

constexpr int kThreads = 256, kWarps = kThreads / 32;
constexpr int kChunk = 1024;  // tokens per chunk statistic (128 vectors of 8)

constexpr float kLog2e = 1.44269504088896340736f;
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Merge (m, s) pairs: s is a sum of exp(x - m).
__device__ __forceinline__ void lse_merge(float &m, float &s, float m2, float s2) {
  const float mm = fmaxf(m, m2);
  if (mm == -INFINITY) return;  // both empty
  s = (m == -INFINITY ? 0.f : s * __expf(m - mm)) + (m2 == -INFINITY ? 0.f : s2 * __expf(m2 - mm));
  m = mm;
}

// Inclusive block scan of one float per thread (256 threads); returns the
// thread's inclusive prefix and, in *total, the block sum.
__device__ __forceinline__ float block_scan(float v, float *s_warp, float *total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const float y = __shfl_up_sync(DC_FULL_MASK, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  float before = 0.f, all = 0.f;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    const float t = s_warp[w];
    before += w < warp ? t : 0.f;
    all += t;
  }
  __syncthreads();
  *total = all;
  return before + x;
}

// The row pass: one fma, one ex2 and a few ALU operations per token; the
// next chunk's loads are issued before the current chunk's arithmetic.
__global__ void __launch_bounds__(kThreads)
k_verify_stochastic(const uint16_t *__restrict__ target, int64_t stride, int V, int B,
                    const int32_t *__restrict__ tokens, const float *__restrict__ u_acc,
                    const float *__restrict__ u_draw, int nchunks, float *__restrict__ chunk_m,
                    float *__restrict__ chunk_s, float *__restrict__ row_lse, float *__restrict__ q_acc,
                    unsigned *__restrict__ req_count, int32_t *__restrict__ accept_len,
                    int32_t *__restrict__ next_token) {
  __shared__ float s_m[kWarps], s_s[kWarps], s_warp[kWarps];
  __shared__ unsigned s_bal[kWarps];  // per-warp ballots of the chunk search
  __shared__ int s_last, s_row, s_excl, s_tok;
  __shared__ float s_t, s_base;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int row = blockIdx.x, n = row / (B + 1), j = row - n * (B + 1);
  const uint16_t *x = target + (int64_t)row * stride;

  // ---------------------------------------------------------------- row statistics
  float wm = -INFINITY, ws = 0.f;  // this warp's running (max, sum)
  auto load_chunk = [&](int c, uint32_t (&wr)[16]) {
    const int v0 = c * kChunk;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int t0 = v0 + (q * 32 + lane) * 8;  // first token of this lane's vector
      uint4 w4 = make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u);  // -inf
      if (t0 + 8 <= V) {
        w4 = __ldcs(reinterpret_cast<const uint4 *>(x + t0));
      } else if (t0 < V) {
        uint16_t e[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) e[k] = t0 + k < V ? x[t0 + k] : (uint16_t)0xFF80u;
        w4 = make_uint4(e[0] | (uint32_t)e[1] << 16, e[2] | (uint32_t)e[3] << 16, e[4] | (uint32_t)e[5] << 16,
                        e[6] | (uint32_t)e[7] << 16);
      }
      wr[4 * q] = w4.x; wr[4 * q + 1] = w4.y; wr[4 * q + 2] = w4.z; wr[4 * q + 3] = w4.w;
    }
  };
  uint32_t wnext[16];
  if (warp < nchunks) load_chunk(warp, wnext);
  for (int c = warp; c < nchunks; c += kWarps) {
    uint32_t wr[16];  // this lane's 32 tokens as packed bf16 pairs, in token order
#pragma unroll
    for (int k = 0; k < 16; ++k) wr[k] = wnext[k];
    if (c + kWarps < nchunks) load_chunk(c + kWarps, wnext);  // in flight during this chunk's arithmetic
    // the chunk maximum on the packed pairs (exact), then over the warp
    uint32_t mx = bf16x2_max(wr[0], wr[1]);
#pragma unroll
    for (int k = 2; k < 16; ++k) mx = bf16x2_max(mx, wr[k]);
    float m = warp_max(fmaxf(bf16_lo(mx), bf16_hi(mx)));
    float s = 0.f;
    if (m != -INFINITY) {
      // exp(x - m) = 2^(x log2 e - m log2 e): one fma and one ex2 per token,
      // four partial sums
      const float mb = -m * kLog2e;
      float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        s4[(2 * k) & 3] += ex2_approx(fmaf(bf16_lo(wr[k]), kLog2e, mb));
        s4[(2 * k + 1) & 3] += ex2_approx(fmaf(bf16_hi(wr[k]), kLog2e, mb));
      }
      s = (s4[0] + s4[1]) + (s4[2] + s4[3]);
    }
    s = warp_sum(s);
    if (lane == 0) {
      chunk_m[(int64_t)row * nchunks + c] = m;
      chunk_s[(int64_t)row * nchunks + c] = s;
    }
    lse_merge(wm, ws, m, s);
  }
  if (lane == 0) {
    s_m[warp] = wm;
    s_s[warp] = ws;
  }
  __syncthreads();
  if (tid == 0) {
    float m = s_m[0], s = s_s[0];
    for (int w = 1; w < kWarps; ++w) lse_merge(m, s, s_m[w], s_s[w]);
    const float lse = m == -INFINITY ? -INFINITY : m + __logf(s);
    row_lse[row] = lse;
    if (j < B) {
      const int y = tokens[n * B + j];
      const float xy = (y >= 0 && y < V) ? __uint_as_float((uint32_t)x[y] << 16) : -INFINITY;
      q_acc[n * B + j] = xy == -INFINITY ? 0.f : __expf(xy - lse);
    }
  }

  // ---------------------------------------------------------------- the request's draw
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(&req_count[n], 1u) == (unsigned)B;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  if (tid == 0) {
    int a = 0;
    while (a < B && __ldcg(u_acc + n * B + a) < __ldcg(q_acc + n * B + a)) ++a;
    accept_len[n] = a;
    const int r = n * (B + 1) + a;  // a < B: the rejected slot's row; a == B: the bonus row
    s_row = r;
    s_excl = a < B ? tokens[n * B + a] : -1;
    s_tok = -1;
  }
  __syncthreads();
  const int r = s_row, excl = s_excl;
  const uint16_t *xr = target + (int64_t)r * stride;
  const float lse = __ldcg(row_lse + r);
  const float wex = (excl >= 0 && excl < V) ? __expf(__uint_as_float((uint32_t)xr[excl] << 16) - lse) : 0.f;
  // chunk weights (the excluded token's weight removed from its chunk), and the threshold
  float total = 0.f;
  for (int c0 = 0; c0 < nchunks; c0 += kThreads) {
    const int c = c0 + tid;
    float w = 0.f;
    if (c < nchunks) {
      const float m = __ldcg(chunk_m + (int64_t)r * nchunks + c);
      w = m == -INFINITY ? 0.f : __ldcg(chunk_s + (int64_t)r * nchunks + c) * __expf(m - lse);
      if (excl >= 0 && excl / kChunk == c) w = fmaxf(w - wex, 0.f);
    }
    float tot;
    block_scan(w, s_warp, &tot);
    total += tot;
  }
  if (tid == 0) s_t = __ldcg(u_draw + n) * total;
  __syncthreads();
  const float t = s_t;
  // the chunk whose inclusive cumulative weight first exceeds t
  float base = 0.f;
  int chunk = -1;
  for (int c0 = 0; c0 < nchunks && chunk < 0; c0 += kThreads) {
    const int c = c0 + tid;
    float w = 0.f;
    if (c < nchunks) {
      const float m = __ldcg(chunk_m + (int64_t)r * nchunks + c);
      w = m == -INFINITY ? 0.f : __ldcg(chunk_s + (int64_t)r * nchunks + c) * __expf(m - lse);
      if (excl >= 0 && excl / kChunk == c) w = fmaxf(w - wex, 0.f);
    }
    float tot;
    const float inc = base + block_scan(w, s_warp, &tot);
    const bool hit = (c < nchunks) & (w > 0.f) & (inc > t);
    const unsigned bal = __ballot_sync(DC_FULL_MASK, hit);
    if (lane == 0) s_bal[warp] = bal;
    __syncthreads();
    // first hit in this batch (threads in order)
    int f = -1;
#pragma unroll
    for (int k = kWarps - 1; k >= 0; --k) {
      const unsigned b = s_bal[k];
      f = b ? k * 32 + __ffs(b) - 1 : f;
    }
    if (f >= 0) {
      chunk = c0 + f;
      if (tid == f) s_base = inc - w;  // cumulative weight before the chunk
    }
    base += tot;
    __syncthreads();
  }
  if (tid == 0) s_tok = -1;
  __syncthreads();
  if (chunk >= 0) {
    // inside the chunk: 4 consecutive tokens per thread
    const float cb = s_base;
    const int v0 = chunk * kChunk + tid * 4;
    float w4[4], sum = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int v = v0 + k;
      w4[k] = (v < V && v != excl) ? __expf(__uint_as_float((uint32_t)xr[v] << 16) - lse) : 0.f;
      sum += w4[k];
    }
    float tot;
    float c = cb + block_scan(sum, s_warp, &tot) - sum;  // before this thread's tokens
    int found = -1;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      c += w4[k];
      if (found < 0 && w4[k] > 0.f && c > t) found = v0 + k;
    }
    if (found >= 0) atomicMin(reinterpret_cast<unsigned *>(&s_tok), (unsigned)found);
    __syncthreads();
  }
  if (tid == 0) {
    int tok = s_tok;
    if (tok < 0) {
      // rounding past the end of the cumulative sum: the last token with weight
      for (int v = V - 1; v >= 0; --v)
        if (v != excl && __uint_as_float((uint32_t)xr[v] << 16) != -INFINITY) {
          tok = v;
          break;
        }
    }
    next_token[n] = tok;
    req_count[n] = 0u;  // ready for the next call
  }
}

}  // namespace

int verify_chunks(int V) { return (V + kChunk - 1) / kChunk; }

cudaError_t launch_verify_stochastic(const uint16_t *target, int64_t stride, int V, int N, int B,
                                     const int32_t *tokens, const float *u_acc, const float *u_draw,
                                     float *chunk_m, float *chunk_s, float *row_lse, float *q_acc,
                                     unsigned *req_count, int32_t *accept_len, int32_t *next_token,
                                     cudaStream_t st) {
  if (N == 0) return cudaSuccess;
  k_verify_stochastic<<<N * (B + 1), kThreads, 0, st>>>(target, stride, V, B, tokens, u_acc, u_draw,
                                                        verify_chunks(V), chunk_m, chunk_s, row_lse, q_acc,
                                                        req_count, accept_len, next_token);
  return cudaGetLastError();
}

}  // namespace dc
