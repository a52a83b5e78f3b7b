// proj_simt.cu -- row-gathered projection C = A W^T on CUDA cores (fp32).
//
// DCOCO page, Method step details (2)-(3): the candidate embedding rows
// E[c] (gathered by token id) and the slot hidden states h_i are projected by
// bias-free linear maps (W_cand; W_ctx and the two halves of W_pair).
// A is bf16 (exact in fp32), W is fp32, accumulation is fp32.
//
// Tiles of 64 rows x 64 outputs x 32 k; 256 threads, 4x4 outputs each.
#include "common.cuh"
#include "kernels.h"

namespace dc {
namespace {

constexpr int BM = 64, BN = 64, BK = 32;

template <int MODE>
__global__ void __launch_bounds__(256)
k_rows_gemm(const uint16_t *__restrict__ base, const int32_t *__restrict__ ids, int slots, int B,
            int M, int d, int V, const float *__restrict__ W, int No, float *__restrict__ C,
            int *err) {
  __shared__ float As[BK][BM + 4];
  __shared__ float Ws[BK][BN + 4];
  const int tid = threadIdx.x;
  const int tx = tid & 15, ty = tid >> 4;
  const int m0 = blockIdx.y * BM, o0 = blockIdx.x * BN;

  // the A row this thread stages (row = tid / 4, 8 k-values at (tid % 4) * 8)
  const int lr = tid >> 2, lk = (tid & 3) * 8;
  const int m = m0 + lr;
  const uint16_t *arow = nullptr;
  if (m < M) {
    if (MODE == 0) {
      int id = ids[m];
      if (id < 0 || id >= V) {
        atomicOr(err, kErrBadCandidateId);
        id = 0;
      }
      arow = base + (int64_t)id * d;
    } else {
      const int n = m / B, i = m - n * B;
      arow = base + ((int64_t)n * slots + i + 1) * d;
    }
  }
  const int o = o0 + lr;  // the W row this thread stages
  const float *wrow = (o < No) ? W + (int64_t)o * d : nullptr;

  float acc[4][4] = {};
  for (int k0 = 0; k0 < d; k0 += BK) {
    // stage A (bf16 -> fp32), transposed so the compute loop broadcasts
    uint4 a = make_uint4(0, 0, 0, 0);
    if (arow) a = *reinterpret_cast<const uint4 *>(arow + k0 + lk);
    const uint32_t aw[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
    for (int q = 0; q < 8; ++q)
      As[lk + q][lr] = bf16_bits_to_float((q & 1) ? (aw[q >> 1] >> 16) : (aw[q >> 1] & 0xFFFFu));
    float4 w0 = make_float4(0, 0, 0, 0), w1 = w0;
    if (wrow) {
      w0 = *reinterpret_cast<const float4 *>(wrow + k0 + lk);
      w1 = *reinterpret_cast<const float4 *>(wrow + k0 + lk + 4);
    }
    Ws[lk + 0][lr] = w0.x; Ws[lk + 1][lr] = w0.y; Ws[lk + 2][lr] = w0.z; Ws[lk + 3][lr] = w0.w;
    Ws[lk + 4][lr] = w1.x; Ws[lk + 5][lr] = w1.y; Ws[lk + 6][lr] = w1.z; Ws[lk + 7][lr] = w1.w;
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < BK; ++kk) {
      float av[4], wv[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        av[u] = As[kk][ty * 4 + u];
        wv[u] = Ws[kk][tx * 4 + u];
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int v = 0; v < 4; ++v) acc[u][v] = fmaf(av[u], wv[v], acc[u][v]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int mm = m0 + ty * 4 + u;
    if (mm >= M) continue;
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const int oo = o0 + tx * 4 + v;
      if (oo < No) C[(int64_t)mm * No + oo] = acc[u][v];
    }
  }
}

}  // namespace

cudaError_t launch_rows_gemm(int mode, const uint16_t *base, const int32_t *ids, int slots, int B,
                             int M, int d, int V, const float *W, int No, float *C, int *err,
                             cudaStream_t st) {
  if (M == 0) return cudaSuccess;
  dim3 grid((No + BN - 1) / BN, (M + BM - 1) / BM);
  if (mode == 0)
    k_rows_gemm<0><<<grid, 256, 0, st>>>(base, ids, slots, B, M, d, V, W, No, C, err);
  else
    k_rows_gemm<1><<<grid, 256, 0, st>>>(base, ids, slots, B, M, d, V, W, No, C, err);
  return cudaGetLastError();
}

}  // namespace dc
