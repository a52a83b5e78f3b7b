// mlp_tc.cu -- the 128-deep maps of the representation and transition steps
// on the tensor cores: per draft slot, the context half of the fuse map and
// the pair part of layer 1; per candidate, the LayerNorms, the fuse map and
// the candidate parts of layer 1.
//
// DCOCO page ("Contextual Correction of Parallel Drafts for Speculative
// Decoding"), Method step details (2)-(4):
//   g_i = LN(W_ctx h_i),  b = LN(W_cand E[c])          (non-affine)
//   z = gamma * LN(W_fuse[:, :r] b + W_fuse[:, r:] g_i) + beta
//   s_p = W_pair [h_p; h_{p+1}]
// and layer 1 of the transition MLP, which is linear in its concatenated
// input [s_p; z^a; z^b; l(a); l(b)], split by input block:
//   P_p = W1[:, :r] s_p + b1                        (per slot pair)
//   U = W1[:, r:2r] z + W1[:, 3r] l(c),  V = W1[:, 2r:3r] z + W1[:, 3r+1] l(c)
// (U feeds the candidate's transitions as predecessor, V as successor.)
//
// Every map here is a dense 128-deep contraction over 128-row tiles: A (the
// LayerNormed or summed rows) is split in registers into bf16 hi + lo and
// stored 128B-swizzled, the weights come pre-split through TMA, and three MMA
// passes (hi.hi + hi.lo + lo.hi) accumulate in fp32 tensor memory, which
// keeps fp32-level accuracy.  Sixteen row warps hold the tile: row r (a
// tensor-memory lane) is shared by four threads, one per 32-column quarter,
// which meet in shared memory for the LayerNorm sums; one thread of warp 16
// issues the TMA copies and MMAs.  Every wait is bounded in time
// (kErrTimeout in the status word).
#include <cuda_bf16.h>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"
#include "launch.h"

namespace dc {
namespace {

using namespace tc;

constexpr int kR = 128, kH = 256;
constexpr int kRows = 128;                 // tile rows (MMA M)
constexpr int kKBlk = 128 * 64 * 2;        // 128 rows x 64 k of bf16: 16 KB
constexpr int kMat = 2 * kKBlk;            // 128 rows x 128 k: 32 KB
// shared memory: A (hi, lo) | W0 (hi, lo) | ...
constexpr int kOffA = 0, kOffW0 = 2 * kMat;
constexpr int kRowWarps = 16;
constexpr int kRowThreads = kRowWarps * 32;  // 4 threads per tile row
constexpr int kThreads = kRowThreads + 32;   // + the control warp
constexpr int kQ = 32;                       // columns per row thread
constexpr uint32_t kIdesc = idesc_bf16(128, 128);
constexpr uint32_t kWTx = 2 * kMat;          // one matrix pair (hi + lo): 64 KB

// Everything one launch of k_maps_tc needs (a __grid_constant__ parameter, so
// the tensor maps stay in parameter space for the TMA instructions).
struct MapsParams {
  MlpMaps maps;
  SlotIoMaps slot;
  CandIoMaps cand;
  const float *slot_proj;  // [N*B][3r]
  const float *w_fg;       // W_fuse[:, r:], fp32 [r][r]
  const float *topk_val, *w_la, *w_lb, *b1;
  int NB;                  // draft slots in the call
  int slot_ctas;           // 2 per 128-slot tile (the two halves of P)
  int K, M;                // candidates per slot, candidates in the call
  float eps;
  int *err;
};

// Barrier over the row threads only (the control warp keeps issuing).
__device__ __forceinline__ void rows_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kRowThreads) : "memory");
}
// The same barrier, returning whether `v` holds in every row thread.
__device__ __forceinline__ bool rows_all(bool v) {
  uint32_t out;
  asm volatile(
      "{\n.reg .pred p, q;\n"
      "setp.ne.u32 q, %1, 0;\n"
      "bar.red.and.pred p, 1, %2, q;\n"
      "selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(out)
      : "r"((uint32_t)v), "n"(kRowThreads)
      : "memory");
  return out != 0;
}

// Row r's columns [32 q, 32 q + 32) as bf16 hi and lo into the 128B-swizzled
// K-major A tiles (two 64-wide k-blocks each).
__device__ __forceinline__ void store_split_part(uint8_t *a_hi, uint8_t *a_lo, int r, int q,
                                                 const float (&x)[kQ]) {
  const int kb = q >> 1;
#pragma unroll
  for (int cc = 0; cc < 4; ++cc) {
    const int c = (q & 1) * 4 + cc;  // 16-byte chunk within the 128-byte row
    uint32_t hw[4], lw[4];
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      const float v0 = x[cc * 8 + 2 * p], v1 = x[cc * 8 + 2 * p + 1];
      const uint32_t h0 = bf16_rn_bits(v0), h1 = bf16_rn_bits(v1);
      const uint32_t l0 = bf16_rn_bits(v0 - __uint_as_float(h0 << 16));
      const uint32_t l1 = bf16_rn_bits(v1 - __uint_as_float(h1 << 16));
      hw[p] = h0 | (h1 << 16);
      lw[p] = l0 | (l1 << 16);
    }
    const int off = kb * kKBlk + (r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) * 16);
    *reinterpret_cast<uint4 *>(a_hi + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
    *reinterpret_cast<uint4 *>(a_lo + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
  }
}

// Sum over a row's four quarter-threads, in quarter order (the same value in
// all four).  `red` is [4][kRows] shared floats.
__device__ __forceinline__ float row_sum(float v, float *red, int r, int q) {
  red[q * kRows + r] = v;
  rows_sync();
  return (red[r] + red[kRows + r]) + (red[2 * kRows + r] + red[3 * kRows + r]);
}

__device__ __forceinline__ float sum32(const float (&x)[kQ]) {
  float a0 = x[0], a1 = x[1], a2 = x[2], a3 = x[3];
#pragma unroll
  for (int k = 4; k < kQ; k += 4) {
    a0 += x[k];
    a1 += x[k + 1];
    a2 += x[k + 2];
    a3 += x[k + 3];
  }
  return (a0 + a1) + (a2 + a3);
}

// Barrier over half of the row threads (group 0: warps 0-7, group 1: warps
// 8-15), returning whether `v` holds in all of them.
__device__ __forceinline__ bool half_rows_all(int grp, bool v) {
  uint32_t out;
  asm volatile(
      "{\n.reg .pred p, q;\n"
      "setp.ne.u32 q, %1, 0;\n"
      "bar.red.and.pred p, %2, %3, q;\n"
      "selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(out)
      : "r"((uint32_t)v), "r"(2 + grp), "n"(kRowThreads / 2)
      : "memory");
  return out != 0;
}

// Non-affine LayerNorm of a 128-wide row held as four 32-column quarters:
// population variance, eps inside the square root.  Every row thread calls
// it (it holds two row barriers); red0 / red1 are two distinct [4][kRows]
// buffers.
__device__ __forceinline__ void ln0_part(float (&x)[kQ], float eps, float *red0, float *red1, int r, int q) {
  const float mean = row_sum(sum32(x), red0, r, q) * (1.0f / kR);
  float sq[kQ];
#pragma unroll
  for (int k = 0; k < kQ; ++k) {
    x[k] -= mean;
    sq[k] = x[k] * x[k];
  }
  const float var = row_sum(sum32(sq), red1, r, q) * (1.0f / kR);
  const float inv = rsqrtf(var + eps);
#pragma unroll
  for (int k = 0; k < kQ; ++k) x[k] *= inv;
}

__device__ __forceinline__ void load32(float (&x)[kQ], const float *src) {
  const float4 *s4 = reinterpret_cast<const float4 *>(src);
#pragma unroll
  for (int i = 0; i < kQ / 4; ++i) {
    const float4 v = __ldg(s4 + i);
    x[4 * i] = v.x; x[4 * i + 1] = v.y; x[4 * i + 2] = v.z; x[4 * i + 3] = v.w;
  }
}

constexpr int kBox = 128 * 128;  // one fp32 box: 128 rows x 32 columns, 16 KB

// 16-byte chunk c of row r in a swizzled 128-byte-row box at `box`.
__device__ __forceinline__ uint8_t *box_chunk(uint8_t *box, int r, int c) {
  return box + r * 128 + ((c ^ (r & 7)) * 16);
}

// 3-pass split product of one 128-deep contraction into tensor memory at `tmem`.
__device__ __forceinline__ void mma_split(uint32_t tmem, uint32_t a_hi, uint32_t a_lo, uint32_t w_hi,
                                          uint32_t w_lo) {
#pragma unroll
  for (int kb = 0; kb < 2; ++kb)
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t o = kb * kKBlk + k * 32;
      const uint64_t ah = sw128_desc(a_hi + o), al = sw128_desc(a_lo + o);
      mma_bf16(tmem, ah, sw128_desc(w_hi + o), kIdesc, (kb | k) ? 1u : 0u);
      mma_bf16(tmem, ah, sw128_desc(w_lo + o), kIdesc, 1u);
      mma_bf16(tmem, al, sw128_desc(w_hi + o), kIdesc, 1u);
    }
}

__device__ __forceinline__ void load_pair(uint32_t w_hi, uint32_t w_lo, const CUtensorMap *mh,
                                          const CUtensorMap *ml, int row, uint32_t bar) {
  mbar_arrive_expect_tx(bar, kWTx);
  for (int kb = 0; kb < 2; ++kb) {
    tma_load_2d(w_hi + kb * kKBlk, mh, kb * 64, row, bar);
    tma_load_2d(w_lo + kb * kKBlk, ml, kb * 64, row, bar);
  }
}

// ---------------------------------------------------------------- per draft slot
// One CTA per (128-slot tile, output chunk): chunks 1 and 2 write the two
// 128-wide halves of P_i = W1[:, :r] s_i + b1,
// s_i = W_pair[:, :d] h_i + W_pair[:, d:] h_{i+1}, indexed by draft slot (rows
// of the last slot of a request are not used).  (Chunk 0, Gf = W_fuse[:, r:] g,
// is computed by the candidate blocks themselves.)
// slot_proj rows are (W_ctx h | W_pair[:, :d] h | W_pair[:, d:] h).
// The input tiles arrive by TMA (fp32 boxes of 128 rows x 32 columns,
// 128-byte swizzled), so every row thread's 16-byte shared-memory access is
// conflict-free and the global traffic is whole lines; P leaves by TMA.
// Shared memory: X (64 KB): the first input tile, then the A operand (hi, lo);
// Y (64 KB): the second input tile (chunks 1, 2), then the output tile;
// W (64 KB): the weight pair.
constexpr int kSlotOffX = 0, kSlotOffY = 2 * kMat, kSlotOffW = 4 * kMat;
constexpr int kSlotSmemBytes = 6 * kMat + 1024;

__device__ __forceinline__ void slot_role(const MapsParams &mp, int chunk, int tile, float eps, int *err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  __shared__ __align__(8) unsigned long long bar_w, bar_in, bar_a, bar_mma;
  __shared__ float s_red[2][4 * kRows];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int m0 = tile * kRows;
  const uint32_t sb = smem_u32(smem);
  const uint32_t a_hi = sb + kSlotOffX, a_lo = sb + kSlotOffX + kMat;
  const uint32_t w_hi = sb + kSlotOffW, w_lo = sb + kSlotOffW + kMat;

  if (tid == 0) {
    mbar_init(smem_u32(&bar_w), 1);
    mbar_init(smem_u32(&bar_in), 1);
    mbar_init(smem_u32(&bar_a), kRowThreads);
    mbar_init(smem_u32(&bar_mma), 1);
    s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kRowWarps) tmem_alloc(smem_u32(&s_tmem), 128);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;

  if (warp == kRowWarps) {
    if (lane == 0) {
      // ------------------------------------------------------------ control thread
      if (chunk == 0)
        load_pair(w_hi, w_lo, &mp.maps.fg_hi, &mp.maps.fg_lo, 0, smem_u32(&bar_w));
      else
        load_pair(w_hi, w_lo, &mp.maps.w1s_hi, &mp.maps.w1s_lo, (chunk - 1) * 128, smem_u32(&bar_w));
      pdl_wait();  // slot_proj comes from the previous kernels
      // chunk 0: W_ctx h of the tile's slots; chunks 1, 2: W_pair[:, :d] h of
      // the tile's slots and W_pair[:, d:] h of the slots one row further on
      const uint32_t in = smem_u32(&bar_in);
      mbar_arrive_expect_tx(in, (chunk == 0 ? 4 : 8) * kBox);
      if (chunk == 0) {
        for (int bx = 0; bx < 4; ++bx) tma_load_2d(sb + kSlotOffX + bx * kBox, &mp.slot.sp, bx * 32, m0, in);
      } else {
        for (int bx = 0; bx < 4; ++bx) {
          tma_load_2d(sb + kSlotOffX + bx * kBox, &mp.slot.sp, kR + bx * 32, m0, in);
          tma_load_2d(sb + kSlotOffY + bx * kBox, &mp.slot.sp, 2 * kR + bx * 32, m0 + 1, in);
        }
      }
      if (mbar_wait(smem_u32(&bar_w), 0, &s_abort, err) && mbar_wait(smem_u32(&bar_a), 0, &s_abort, err)) {
        tc_fence_after();
        mma_split(tmem, a_hi, a_lo, w_hi, w_lo);
      }
      mma_commit(smem_u32(&bar_mma));
    }
    __syncwarp();
  } else {
    // -------------------------------------------------------------- row threads
    const int qd = warp & 3, q = warp >> 2;  // lane quadrant, column quarter
    const int r = qd * 32 + lane;           // tile row = tensor-memory lane
    float x[kQ];
    const bool ok0 = rows_all(mbar_wait(smem_u32(&bar_in), 0, &s_abort, err) && !s_abort);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (ok0) {
        v = *reinterpret_cast<const float4 *>(box_chunk(smem + kSlotOffX + q * kBox, r, c));
        if (chunk != 0) {
          const float4 y = *reinterpret_cast<const float4 *>(box_chunk(smem + kSlotOffY + q * kBox, r, c));
          v.x += y.x; v.y += y.y; v.z += y.z; v.w += y.w;
        }
      }
      x[4 * c] = v.x; x[4 * c + 1] = v.y; x[4 * c + 2] = v.z; x[4 * c + 3] = v.w;
    }
    if (chunk == 0)
      ln0_part(x, eps, s_red[0], s_red[1], r, q);  // holds row barriers
    else
      rows_sync();  // every row thread has read X before it becomes the A operand
    store_split_part(smem + kSlotOffX, smem + kSlotOffX + kMat, r, q, x);
    fence_proxy_async();
    mbar_arrive(smem_u32(&bar_a));

    bool ok = mbar_wait(smem_u32(&bar_mma), 0, &s_abort, err) && !s_abort;
    ok = __all_sync(DC_FULL_MASK, ok);
    tc_fence_after();
    if (ok) {
      float v[kQ];
      tmem_ld32(tmem + ((uint32_t)(qd * 32) << 16) + q * kQ, v);
      if (chunk != 0) {
        float bb[kQ];
        load32(bb, mp.b1 + (chunk - 1) * 128 + q * kQ);
#pragma unroll
        for (int k = 0; k < kQ; ++k) v[k] += bb[k];
      }
      // the output tile: quarter q is box q of Y (free since the row barrier above)
#pragma unroll
      for (int c = 0; c < 8; ++c)
        *reinterpret_cast<float4 *>(box_chunk(smem + kSlotOffY + q * kBox, r, c)) =
            make_float4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
    }
    fence_proxy_async();
    if (rows_all(ok) && tid == 0) {
      for (int bx = 0; bx < 4; ++bx)
        tma_store_2d(&mp.slot.p, sb + kSlotOffY + bx * kBox, (chunk - 1) * 128 + bx * 32, m0);
      bulk_commit();
      bulk_wait_all();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (s_abort && warp == kRowWarps && lane == 0) {
    mbar_drain(smem_u32(&bar_w), 0);
    mbar_drain(smem_u32(&bar_in), 0);
    mbar_drain(smem_u32(&bar_mma), 0);
  }
  __syncthreads();
  if (warp == kRowWarps) {
    tc_fence_after();
    tmem_dealloc(tmem, 128);
  }
}

// ---------------------------------------------------------------- per candidate
// One CTA per (128-candidate tile, half): half 0 writes U, half 1 writes V;
// both recompute z (a 128x128 map, cheap) and the context term
// Gf = W_fuse[:, r:] LN0(W_ctx h) of the tile's draft slots (128 / K of them):
// fp32 dot products, each thread holding a 32-long slice of one W_fuse row
// (loaded while the block waits for the previous kernel), partial sums met
// by warp shuffles.  b = LN0(W_cand E[c]) arrives ready as bf16 hi and lo
// (the projection's reduction normalises and splits each row), straight
// into the fuse product's A operand.  Tensor memory: [0,128) the fuse
// product, [128,384) the 256 layer-1 outputs of this half.  Shared memory
// (three 64 KB regions), by phase:
//   A:  b (hi, lo), then z (hi, lo);                  then outputs 128..255
//   W0: W_fuse[:, :r] (hi, lo), then layer-1 rows 128..255 of this half
//   S:  layer-1 rows 0..127 of this half;             then outputs 0..127
// All tiles move by TMA; the fp32 output boxes use the same 128-byte swizzle
// as the bf16 operands, so the row threads' 16-byte accesses are
// conflict-free.
constexpr int kOffS = 4 * kMat;
constexpr int kCandSmemBytes = 6 * kMat + 1024;
constexpr int kMapsSmemBytes = kCandSmemBytes > kSlotSmemBytes ? kCandSmemBytes : kSlotSmemBytes;
constexpr uint32_t kCandTmemCols = 512;
constexpr int kMaxSlots = kRows / 8;  // draft slots in a candidate tile, K >= 8
constexpr int kGSeg = 36;             // s_g row: four 32-float segments padded to 36 (bank spread)
constexpr int kGLd = 4 * kGSeg;

__device__ __forceinline__ void cand_role(const MapsParams &mp, int half, int tile, int K, int M, float eps,
                                          int *err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  __shared__ __align__(8) unsigned long long bar_w0, bar_b, bar_w1, bar_w2, bar_fuse, bar_a2, bar_uv0, bar_uv1;
  __shared__ float s_red[2][4 * kRows];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ float s_wl[kH];                               // this half's w_l
  __shared__ __align__(16) float s_g[kMaxSlots][kGLd];     // LN0(W_ctx h) of the tile's slots
  __shared__ __align__(16) float s_gf[kMaxSlots][kR];      // Gf of the tile's slots
  __shared__ float s_gq[2][4][kR];                         // Gf quarter partials, two slots in flight

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int m0 = tile * kRows;
  const int slot0 = m0 / K, nslots = kRows / K;  // the tile's draft slots (K divides 128)
  const uint32_t sb = smem_u32(smem);
  const uint32_t a_hi = sb + kOffA, a_lo = sb + kOffA + kMat;
  const uint32_t w0_hi = sb + kOffW0, w0_lo = sb + kOffW0 + kMat;
  const uint32_t s_hi = sb + kOffS, s_lo = sb + kOffS + kMat;

  if (tid == 0) {
    mbar_init(smem_u32(&bar_w0), 1);
    mbar_init(smem_u32(&bar_b), 1);
    mbar_init(smem_u32(&bar_w1), 1);
    mbar_init(smem_u32(&bar_w2), 1);
    mbar_init(smem_u32(&bar_fuse), 1);
    mbar_init(smem_u32(&bar_a2), kRowThreads);
    mbar_init(smem_u32(&bar_uv0), 1);
    mbar_init(smem_u32(&bar_uv1), 1);
    s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kRowWarps) tmem_alloc(smem_u32(&s_tmem), kCandTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  const int wrow0 = half * kH;  // first row of this half's block in [W1_a ; W1_b]
  bool w2_issued = false;

  if (warp == kRowWarps) {
    if (lane == 0) {
      // ------------------------------------------------------------ control thread
      // the weights first: W_fuse[:, :r] to W0, layer-1 rows 0..127 to S
      load_pair(w0_hi, w0_lo, &mp.maps.fb_hi, &mp.maps.fb_lo, 0, smem_u32(&bar_w0));
      load_pair(s_hi, s_lo, &mp.maps.w1_hi, &mp.maps.w1_lo, wrow0, smem_u32(&bar_w1));
      pdl_wait();  // b comes from the previous kernel
      load_pair(a_hi, a_lo, &mp.cand.bh, &mp.cand.bl, m0, smem_u32(&bar_b));
      // y = W_fuse[:, :r] b
      if (mbar_wait(smem_u32(&bar_w0), 0, &s_abort, err) && mbar_wait(smem_u32(&bar_b), 0, &s_abort, err)) {
        tc_fence_after();
        mma_split(tmem, a_hi, a_lo, w0_hi, w0_lo);
      }
      mma_commit(smem_u32(&bar_fuse));
      // once the fuse MMAs have read W0, it takes layer-1 rows 128..255
      if (mbar_wait(smem_u32(&bar_fuse), 0, &s_abort, err)) {
        load_pair(w0_hi, w0_lo, &mp.maps.w1_hi, &mp.maps.w1_lo, wrow0 + 128, smem_u32(&bar_w2));
        w2_issued = true;
      }
      if (mbar_wait(smem_u32(&bar_a2), 0, &s_abort, err) && mbar_wait(smem_u32(&bar_w1), 0, &s_abort, err)) {
        tc_fence_after();
        mma_split(tmem + 128, a_hi, a_lo, s_hi, s_lo);
      }
      mma_commit(smem_u32(&bar_uv0));
      if (w2_issued && mbar_wait(smem_u32(&bar_w2), 0, &s_abort, err)) {
        tc_fence_after();
        mma_split(tmem + 256, a_hi, a_lo, w0_hi, w0_lo);
      }
      mma_commit(smem_u32(&bar_uv1));
    }
    __syncwarp();
  } else {
    // -------------------------------------------------------------- row threads
    const int qd = warp & 3, q = warp >> 2;  // lane quadrant, column quarter
    const int r = qd * 32 + lane;           // tile row = tensor-memory lane
    const int m = m0 + r;
    const bool live = m < M;
    const uint32_t lane_base = tmem + ((uint32_t)(qd * 32) << 16);
    // Weights first (they do not depend on the previous kernel), all loads in
    // flight before any use: this thread's slice of W_fuse[:, r:] (output go,
    // inputs [32 gk, 32 gk + 32)) to registers; w_l reaches shared memory
    // after the dependency wait (the output phase reads it, behind several
    // row barriers).  The input quarter gk is the same for the whole warp, so
    // every read of g below is a broadcast.
    const int gk = warp & 3, go = (warp >> 2) * 32 + lane;
    float wfg[32];
    {
      // packed so that each step of the warp reads 512 contiguous bytes
      const float4 *src = reinterpret_cast<const float4 *>(mp.w_fg) + warp * 8 * 32 + lane;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float4 v = __ldg(src + i * 32);
        wfg[4 * i] = v.x; wfg[4 * i + 1] = v.y; wfg[4 * i + 2] = v.z; wfg[4 * i + 3] = v.w;
      }
    }
    const float wlv = tid < kH ? __ldg((half == 0 ? mp.w_la : mp.w_lb) + tid) : 0.f;
    float x[kQ];
    // W_ctx h of the tile's slots (slot_proj, from the previous kernel); one
    // warp per slot, four columns per lane
    pdl_wait();
    if (tid < kH) s_wl[tid] = wlv;
    const int gs = slot0 + warp;
    float4 gx = make_float4(0.f, 0.f, 0.f, 0.f);
    if (warp < nslots && gs < mp.NB)
      gx = __ldcg(reinterpret_cast<const float4 *>(mp.slot_proj + (int64_t)gs * 3 * kR) + lane);

    // g = LN0(W_ctx h) of each slot (warp-wide sums), then
    // Gf[s][o] = sum_k W_fuse[o][r + k] g[s][k]: thread (go, gk) adds its
    // 32-long slice for every slot; the four quarter sums meet in shared
    // memory (two slots' buffers alternate, one row barrier per slot) and
    // are added as (q0 + q1) + (q2 + q3).  This runs while the tensor cores
    // compute the fuse product.
    if (warp < nslots) {
      const float mean = warp_sum((gx.x + gx.y) + (gx.z + gx.w)) * (1.0f / kR);
      const float4 dv = make_float4(gx.x - mean, gx.y - mean, gx.z - mean, gx.w - mean);
      const float var = warp_sum((dv.x * dv.x + dv.y * dv.y) + (dv.z * dv.z + dv.w * dv.w)) * (1.0f / kR);
      const float inv = rsqrtf(var + eps);
      const int k0 = lane * 4;
      *reinterpret_cast<float4 *>(&s_g[warp][(k0 >> 5) * kGSeg + (k0 & 31)]) =
          make_float4(dv.x * inv, dv.y * inv, dv.z * inv, dv.w * inv);
    }
    rows_sync();
    for (int sl = 0; sl < nslots; ++sl) {
      const float4 *gv = reinterpret_cast<const float4 *>(&s_g[sl][gk * kGSeg]);
      float a0 = 0.f, a1 = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float4 g4 = gv[i];
        a0 = fmaf(wfg[4 * i], g4.x, a0);
        a1 = fmaf(wfg[4 * i + 1], g4.y, a1);
        a0 = fmaf(wfg[4 * i + 2], g4.z, a0);
        a1 = fmaf(wfg[4 * i + 3], g4.w, a1);
      }
      float(&gq)[4][kR] = s_gq[sl & 1];
      gq[gk][go] = a0 + a1;
      rows_sync();  // also orders the previous use of this buffer before the next write to it
      if (gk == 0) s_gf[sl][go] = (gq[0][go] + gq[1][go]) + (gq[2][go] + gq[3][go]);
    }

    // z = gamma * LN0(y + Gf[slot]) + beta, with gamma folded into the
    // layer-1 weights and beta into P's bias when the weights are packed:
    // the A operand of layer 1 is LN0(y + Gf[slot]) itself (every row thread
    // takes part: the LayerNorm holds row barriers)
    // (the row barrier also publishes s_gf)
    const bool ok = rows_all(mbar_wait(smem_u32(&bar_fuse), 0, &s_abort, err) && !s_abort);
    tc_fence_after();
    if (ok) {
      tmem_ld32(lane_base + q * kQ, x);
      if (live) {
        const float4 *g4 = reinterpret_cast<const float4 *>(&s_gf[r / K][q * kQ]);
#pragma unroll
        for (int i = 0; i < kQ / 4; ++i) {
          const float4 v = g4[i];
          x[4 * i] += v.x; x[4 * i + 1] += v.y; x[4 * i + 2] += v.z; x[4 * i + 3] += v.w;
        }
      } else {
#pragma unroll
        for (int k = 0; k < kQ; ++k) x[k] = 0.f;
      }
      ln0_part(x, eps, s_red[0], s_red[1], r, q);
      store_split_part(smem + kOffA, smem + kOffA + kMat, r, q, x);
    }
    fence_proxy_async();
    mbar_arrive(smem_u32(&bar_a2));

    // U (or V) = W1 z + w_l l: quarter q takes outputs [64 q, 64 q + 64),
    // staged as fp32 boxes 2q, 2q+1 (outputs 0..127 in S, 128..255 in A)
    const float *wl = s_wl + q * 64;
    const float lv = live ? __ldcg(mp.topk_val + m) : 0.f;  // the top-K's output: via L2
    bool ok2 = mbar_wait(smem_u32(q < 2 ? &bar_uv0 : &bar_uv1), 0, &s_abort, err) && !s_abort;
    ok2 = __all_sync(DC_FULL_MASK, ok2);
    tc_fence_after();
    if (ok2) {
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {
        float v[kQ];
        tmem_ld32(lane_base + 128 + q * 64 + h * kQ, v);
        const float *wv = wl + h * kQ;
        const int bx = 2 * q + h;
        uint8_t *box = smem + (bx < 4 ? kOffS + bx * kBox : kOffA + (bx - 4) * kBox);
#pragma unroll
        for (int c = 0; c < 8; ++c)
          *reinterpret_cast<float4 *>(box_chunk(box, r, c)) =
              make_float4(fmaf(wv[4 * c], lv, v[4 * c]), fmaf(wv[4 * c + 1], lv, v[4 * c + 1]),
                          fmaf(wv[4 * c + 2], lv, v[4 * c + 2]), fmaf(wv[4 * c + 3], lv, v[4 * c + 3]));
      }
    }
    // Each output half leaves as soon as its quarters are staged: warps of
    // quarters 0-1 (outputs 0..127, boxes 0-3) and of quarters 2-3 (outputs
    // 128..255, boxes 4-7) meet at their own barrier and their first thread
    // issues the group's four stores.
    fence_proxy_async();
    const int grp = q >> 1;
    if (half_rows_all(grp, ok2) && (tid & 255) == 0) {
      const CUtensorMap *map = half == 0 ? &mp.cand.u : &mp.cand.v;
      for (int bx = 4 * grp; bx < 4 * grp + 4; ++bx)
        tma_store_2d(map, sb + (bx < 4 ? kOffS + bx * kBox : kOffA + (bx - 4) * kBox), bx * 32, m0);
      bulk_commit();
      bulk_wait_read();  // the block may leave once the tile is read; the writes land before the grid ends
    }
  }

  tc_fence_before();
  __syncthreads();
  if (s_abort && warp == kRowWarps && lane == 0) {
    // a wait expired: let the copies and MMAs already issued land first
    mbar_drain(smem_u32(&bar_w0), 0);
    mbar_drain(smem_u32(&bar_b), 0);
    mbar_drain(smem_u32(&bar_w1), 0);
    if (w2_issued) mbar_drain(smem_u32(&bar_w2), 0);
    mbar_drain(smem_u32(&bar_uv1), 0);
  }
  __syncthreads();
  if (warp == kRowWarps) {
    tc_fence_after();
    tmem_dealloc(tmem, kCandTmemCols);
  }
}

// ---------------------------------------------------------------- the launch
// One launch runs both: blocks [0, slot_ctas) are the per-slot blocks
// (P half, slot tile), the rest the per-candidate blocks (half, candidate
// tile).  No block waits for another.
__global__ void __launch_bounds__(kThreads, 1)
k_maps_tc(const __grid_constant__ MapsParams mp) {
  pdl_trigger();
  const int b = (int)blockIdx.x;
  if (b < mp.slot_ctas)
    slot_role(mp, 1 + (b & 1), b >> 1, mp.eps, mp.err);
  else
    cand_role(mp, (b - mp.slot_ctas) & 1, (b - mp.slot_ctas) >> 1, mp.K, mp.M, mp.eps, mp.err);
}

}  // namespace

cudaError_t launch_maps_tc(const MlpMaps &maps, const SlotIoMaps &slot, const CandIoMaps &cand,
                           const float *slot_proj, const float *topk_val, const MlpWeightsDev &w, int N, int B,
                           int K, float eps, int *err, cudaStream_t st) {
  const int NB = N * B, M = NB * K;
  if (NB == 0) return cudaSuccess;
  if (K < 8 || kRows % K != 0) return cudaErrorInvalidValue;
  MapsParams mp;
  mp.maps = maps;
  mp.slot = slot;
  mp.cand = cand;
  mp.slot_proj = slot_proj;
  mp.w_fg = w.w_fg;
  mp.topk_val = topk_val;
  mp.w_la = w.w_la;
  mp.w_lb = w.w_lb;
  mp.b1 = w.b1;
  mp.NB = NB;
  mp.slot_ctas = 2 * ((NB + kRows - 1) / kRows);
  mp.K = K;
  mp.M = M;
  mp.eps = eps;
  mp.err = err;
  const int blocks = mp.slot_ctas + 2 * ((M + kRows - 1) / kRows);
  cudaError_t e = cudaFuncSetAttribute(k_maps_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, kMapsSmemBytes);
  if (e != cudaSuccess) return e;
  e = launch_ex(k_maps_tc, dim3(blocks), dim3(kThreads), kMapsSmemBytes, st, true, 0, mp);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace dc
