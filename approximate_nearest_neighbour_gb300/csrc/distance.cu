// Squared-L2 distance tiles on the CUDA cores (fp32 SIMT), the exact form
// sum_t (q_t - x_t)^2 with no cancellation.
//
// Source: brute-force distance computation of exact search and of the coarse
// quantizer ("Billion-scale similarity search with GPUs", sections 5-6; the
// reading guide "Faiss GPU: k-select that never leaves registers", Step 5:
// the coarse quantizer is a small brute-force search over the centroids).
#include "internal.h"

namespace ivfpq {

namespace {
constexpr int TM = 128, TN = 128, TK = 8, NT = 256;

__global__ void __launch_bounds__(NT)
l2_tile_kernel(const float* __restrict__ Q, int64_t nq, const float* __restrict__ X, int64_t n,
               int d, float* __restrict__ D, int64_t ldd) {
  __shared__ float As[TK][TM + 4];
  __shared__ float Bs[TK][TN + 4];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int64_t row0 = int64_t(blockIdx.y) * TM, col0 = int64_t(blockIdx.x) * TN;
  float acc[8][8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;

  for (int k0 = 0; k0 < d; k0 += TK) {
#pragma unroll
    for (int i = threadIdx.x; i < TM * TK; i += NT) {
      const int r = i / TK, t = i % TK;
      const int gt = k0 + t;
      const int64_t gr = row0 + r, gc = col0 + r;
      As[t][r] = (gr < nq && gt < d) ? __ldg(Q + gr * d + gt) : 0.f;
      Bs[t][r] = (gc < n && gt < d) ? __ldg(X + gc * d + gt) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int t = 0; t < TK; ++t) {
      float a[8], b[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) a[i] = As[t][ty + 16 * i];
#pragma unroll
      for (int j = 0; j < 8; ++j) b[j] = Bs[t][tx + 16 * j];
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float diff = a[i] - b[j];
          acc[i][j] = fmaf(diff, diff, acc[i][j]);
        }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int64_t r = row0 + ty + 16 * i;
    if (r >= nq) continue;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int64_t c = col0 + tx + 16 * j;
      if (c < n) D[r * ldd + c] = acc[i][j];
    }
  }
}
}  // namespace

int l2_distance_tile(const float* Q, int64_t nq, const float* X, int64_t n, int d, float* D,
                     int64_t ldd, cudaStream_t s) {
  if (nq == 0 || n == 0) return IVFPQ_OK;
  dim3 grid{unsigned(ceil_div(n, TN)), unsigned(ceil_div(nq, TM)), 1u};
  l2_tile_kernel<<<grid, NT, 0, s>>>(Q, nq, X, n, d, D, ldd);
  IVFPQ_LAUNCHED();
  return IVFPQ_OK;
}

}  // namespace ivfpq
