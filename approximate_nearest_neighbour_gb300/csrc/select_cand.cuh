// k-selection over the per-row candidate segments of the filtered tensor-core
// distance pass (gemm_tc.cu, l2_tc_filter): WarpSelect over the valid entries
// of each row's segments, one warp per row for k <= 256 and BlockSelect (four
// warps and a shared-memory merge) for longer queues. A row with an overflowed segment (more
// entries found than it holds) is selected instead over exact distances
// sum_t (q_t - x_t)^2 to every column, computed here; the caller re-ranks the
// winners in that exact form anyway.
//
// Source: BlockSelect / WarpSelect ("Billion-scale similarity search with
// GPUs", section 4); exact search by distance tiles (same paper, section 5).
#pragma once

#include "select_inst.cuh"

namespace ivfpq {

constexpr int kCandWarps = 4;

template <int K, int NW>
__global__ void __launch_bounds__(NW * 32)
cand_select_kernel(const uint64_t* __restrict__ cand, const int* __restrict__ scnt, int nseg,
                   int cap_s, const float* __restrict__ Q, const float* __restrict__ X, int64_t n,
                   int d, OutWriter out) {
  constexpr int T = ThreadQ<K>::value;
  extern __shared__ uint32_t sm_cand[];
  const int64_t row = blockIdx.x;
  if (out.o.row_mask && !out.o.row_mask[row]) return;  // the same for the whole block
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int* cnt = scnt + row * nseg;
  int over = 0;
  for (int g = threadIdx.x; g < nseg; g += NW * 32) over |= cnt[g] > cap_s;
  over = __syncthreads_or(over);
  WarpSelect<K, T> ws;
  ws.init(lane);
  if (!over) {
    for (int g = warp; g < nseg; g += NW) {
      const int ns = max(cnt[g], 0);
      const uint64_t* e = cand + (row * nseg + g) * cap_s;
      for (int base = 0; base < ns; base += 32) {
        const int i = base + lane;
        const bool ok = i < ns;
        const uint64_t v = ok ? __ldcs(e + i) : ~uint64_t(0);
        ws.add(uint32_t(v >> 32), uint32_t(v));
      }
    }
  } else {
    const float* qr = Q + row * d;
    const int64_t step = int64_t(NW) * 32;
    for (int64_t base = 0; base < n; base += step) {
      const int64_t c = base + warp * 32 + lane;
      const bool ok = c < n;
      float s = 0.f;
      if (ok) {
        const float* xr = X + c * d;
        for (int t = 0; t < d; ++t) {
          const float df = __ldg(qr + t) - __ldg(xr + t);
          s = fmaf(df, df, s);
        }
      }
      ws.add(ok ? float_to_key(s) : kSentinelKey, ok ? uint32_t(c) : kSentinelIdx);
    }
  }
  ws.finalize();
  block_merge<K, T, NW>(ws, sm_cand, sm_cand + NW * K, warp);
  if (warp == 0) {
#pragma unroll
    for (int r = 0; r < K / 32; ++r) {
      const int i = 32 * r + lane;
      if (i < out.k) out.write(row, 0, i, ws.wk[r], ws.wv[r]);
    }
  }
}

// One warp per row (4 rows per block), for queue lengths up to 256: no
// block-level merge.
template <int K>
__global__ void __launch_bounds__(128)
cand_select_warp_kernel(const uint64_t* __restrict__ cand, const int* __restrict__ scnt,
                        int nseg, int cap_s, int64_t rows, const float* __restrict__ Q,
                        const float* __restrict__ X, int64_t n, int d, OutWriter out) {
  constexpr int T = ThreadQ<K>::value;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = int64_t(blockIdx.x) * 4 + warp;
  if (row >= rows) return;                               // the whole warp
  if (out.o.row_mask && !out.o.row_mask[row]) return;  // the whole warp
  const int* cnt = scnt + row * nseg;
  int over = 0;
  for (int g = lane; g < nseg; g += 32) over |= cnt[g] > cap_s;
  over = __any_sync(kFullMask, over);
  WarpSelect<K, T> ws;
  ws.init(lane);
  if (!over) {
    for (int g = 0; g < nseg; ++g) {
      const int ns = max(cnt[g], 0);
      const uint64_t* e = cand + (row * nseg + g) * cap_s;
      for (int base = 0; base < ns; base += 32) {
        const int i = base + lane;
        const bool ok = i < ns;
        const uint64_t v = ok ? __ldcs(e + i) : ~uint64_t(0);
        ws.add(uint32_t(v >> 32), uint32_t(v));
      }
    }
  } else {
    const float* qr = Q + row * d;
    for (int64_t base = 0; base < n; base += 32) {
      const int64_t c = base + lane;
      const bool ok = c < n;
      float s = 0.f;
      if (ok) {
        const float* xr = X + c * d;
        for (int t = 0; t < d; ++t) {
          const float df = __ldg(qr + t) - __ldg(xr + t);
          s = fmaf(df, df, s);
        }
      }
      ws.add(ok ? float_to_key(s) : kSentinelKey, ok ? uint32_t(c) : kSentinelIdx);
    }
  }
  ws.finalize();
#pragma unroll
  for (int r = 0; r < K / 32; ++r) {
    const int i = 32 * r + lane;
    if (i < out.k) out.write(row, 0, i, ws.wk[r], ws.wv[r]);
  }
}

template <int K>
int launch_cand(const uint64_t* cand, const int* scnt, int nseg, int cap_s, int64_t rows,
                const float* Q, const float* X, int64_t n, int d, const OutWriter& w,
                cudaStream_t s) {
  if constexpr (K <= 256) {
    auto wk = cand_select_warp_kernel<K>;
    wk<<<unsigned(ceil_div(rows, 4)), 128, 0, s>>>(cand, scnt, nseg, cap_s, rows, Q, X, n, d, w);
    IVFPQ_LAUNCHED_K(wk, 0, 128);
    return IVFPQ_OK;
  }
  constexpr int NW = kCandWarps;
  const size_t smem = size_t(NW) * K * 2 * sizeof(uint32_t);
  auto kern = cand_select_kernel<K, NW>;
  if (smem > 48 * 1024) IVFPQ_TRY(set_dynamic_smem(kern, smem));
  kern<<<unsigned(rows), NW * 32, smem, s>>>(cand, scnt, nseg, cap_s, Q, X, n, d, w);
  IVFPQ_LAUNCHED_K(kern, smem, NW * 32);
  return IVFPQ_OK;
}

}  // namespace ivfpq

#define IVFPQ_INST_CAND(K)                                                                   \
  template int ivfpq::launch_cand<K>(const uint64_t*, const int*, int, int, int64_t,         \
                                     const float*, const float*, int64_t, int,               \
                                     const ivfpq::OutWriter&, cudaStream_t);
