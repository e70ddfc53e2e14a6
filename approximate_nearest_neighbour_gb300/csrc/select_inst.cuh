// Row-wise k-selection kernels (BlockSelect = one WarpSelect per warp plus a
// shared-memory merge) and their launchers, instantiated per warp-queue
// length K by the select_k<K>.cu files.
#pragma once

#include "internal.h"
#include "select.cuh"

namespace ivfpq {

struct OutWriter {
  SelectOut o;
  int k;
  int64_t chunks;
  __device__ __forceinline__ void write(int64_t row, int64_t chunk, int i, uint32_t key,
                                        uint32_t v) const {
    switch (o.kind) {
      case OutKind::Float: {
        int64_t p = row * k + i;
        o.vals[p] = key_to_float(key);
        o.idx64[p] = v == kSentinelIdx ? int64_t(-1) : int64_t(v);
        break;
      }
      case OutKind::Dist: {
        int64_t p = row * k + i;
        o.vals[p] = dist_key_to_float(key);
        o.idx64[p] = v == kSentinelIdx ? int64_t(-1) : o.id_map[v];
        break;
      }
      case OutKind::Probes: {
        int64_t p = row * k + i;
        o.idx32[p] = v == kSentinelIdx ? -1 : int32_t(v);
        if (o.vals) o.vals[p] = key_to_float(key);
        break;
      }
      case OutKind::Merge: {
        int64_t p = row * k + i;
        o.vals[p] = key_to_float(key);
        o.idx64[p] = v == kSentinelIdx
                         ? int64_t(-1)
                         : o.id_map[(int64_t(v / o.merge_kin) * o.merge_rows + row) * o.merge_kin +
                                    v % o.merge_kin];
        break;
      }
      case OutKind::Partial: {
        int64_t p = (row * chunks + chunk) * k + i;
        o.pkeys[p] = key;
        o.pidx[p] = v;
        break;
      }
    }
  }
};

__device__ __forceinline__ float4 ld_stream_f4(const float4* p) { return __ldcs(p); }

template <int K, int NW>
__global__ void __launch_bounds__(NW * 32)
select_rows_kernel(const float* __restrict__ vals, int64_t cols, int64_t chunk_len,
                   OutWriter out) {
  constexpr int T = ThreadQ<K>::value;
  extern __shared__ uint32_t sm_sel[];
  const int64_t row = blockIdx.x;
  const int64_t chunk = blockIdx.y;
  if (out.o.row_mask && !out.o.row_mask[row]) return;  // the same for the whole block
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  WarpSelect<K, T> ws;
  ws.init(lane);
  const float* rp = vals + row * cols;
  const int64_t c0 = chunk * chunk_len;
  const int64_t c1 = min(cols, c0 + chunk_len);
  const bool vec = ((cols & 3) == 0) && ((reinterpret_cast<uintptr_t>(vals) & 15) == 0) &&
                   ((c0 & 3) == 0);
  if (vec) {
    const int64_t n4 = (c1 - c0) >> 2;
    const float4* p4 = reinterpret_cast<const float4*>(rp + c0);
    const int64_t step = int64_t(NW) * 32;
    for (int64_t base = 0; base < n4; base += step) {
      const int64_t i4 = base + warp * 32 + lane;
      const bool ok = i4 < n4;
      float4 x = ok ? ld_stream_f4(p4 + i4) : make_float4(0.f, 0.f, 0.f, 0.f);
      const uint32_t c = uint32_t(c0 + i4 * 4);
      ws.add(ok ? float_to_key(x.x) : kSentinelKey, c);
      ws.add(ok ? float_to_key(x.y) : kSentinelKey, c + 1);
      ws.add(ok ? float_to_key(x.z) : kSentinelKey, c + 2);
      ws.add(ok ? float_to_key(x.w) : kSentinelKey, c + 3);
    }
    const int64_t t0 = c0 + n4 * 4;
    if (warp == 0 && t0 < c1) {
      const int64_t c = t0 + lane;
      ws.add(c < c1 ? float_to_key(rp[c]) : kSentinelKey, uint32_t(c));
    }
  } else {
    const int64_t step = int64_t(NW) * 32;
    for (int64_t base = c0; base < c1; base += step) {
      const int64_t c = base + warp * 32 + lane;
      ws.add(c < c1 ? float_to_key(__ldcs(rp + c)) : kSentinelKey, uint32_t(c));
    }
  }
  ws.finalize();
  block_merge<K, T, NW>(ws, sm_sel, sm_sel + NW * K, warp);
  if (warp == 0) {
#pragma unroll
    for (int r = 0; r < K / 32; ++r) {
      const int i = 32 * r + lane;
      if (i < out.k) out.write(row, chunk, i, ws.wk[r], ws.wv[r]);
    }
  }
}

template <int K, int NW>
__global__ void __launch_bounds__(NW * 32)
select_pairs_kernel(const uint32_t* __restrict__ keys, const uint32_t* __restrict__ idx,
                    int64_t len, int64_t chunk_len, OutWriter out) {
  constexpr int T = ThreadQ<K>::value;
  extern __shared__ uint32_t sm_sel[];
  const int64_t row = blockIdx.x;
  const int64_t chunk = blockIdx.y;
  if (out.o.row_mask && !out.o.row_mask[row]) return;  // the same for the whole block
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  WarpSelect<K, T> ws;
  ws.init(lane);
  const uint32_t* kp = keys + row * len;
  const uint32_t* ip = idx + row * len;
  const int64_t c0 = chunk * chunk_len;
  const int64_t c1 = min(len, c0 + chunk_len);
  const int64_t step = int64_t(NW) * 32;
  for (int64_t base = c0; base < c1; base += step) {
    const int64_t c = base + warp * 32 + lane;
    const bool ok = c < c1;
    ws.add(ok ? __ldcs(kp + c) : kSentinelKey, ok ? __ldcs(ip + c) : kSentinelIdx);
  }
  ws.finalize();
  block_merge<K, T, NW>(ws, sm_sel, sm_sel + NW * K, warp);
  if (warp == 0) {
#pragma unroll
    for (int r = 0; r < K / 32; ++r) {
      const int i = 32 * r + lane;
      if (i < out.k) out.write(row, chunk, i, ws.wk[r], ws.wv[r]);
    }
  }
}

template <class Kern>
static int prepare_smem(Kern kern, size_t bytes) {
  return bytes > 48 * 1024 ? set_dynamic_smem(kern, bytes) : IVFPQ_OK;
}

template <int K, int NW>
int launch_rows(const float* vals, int64_t rows, int64_t cols, int64_t chunks,
                       int64_t chunk_len, const OutWriter& w, cudaStream_t s) {
  const size_t smem = NW > 1 ? size_t(NW) * K * 2 * sizeof(uint32_t) : 0;
  auto kern = select_rows_kernel<K, NW>;
  IVFPQ_TRY(prepare_smem(kern, smem));
  dim3 grid{unsigned(rows), unsigned(chunks), 1u};
  kern<<<grid, NW * 32, smem, s>>>(vals, cols, chunk_len, w);
  IVFPQ_LAUNCHED_K(kern, smem, NW * 32);
  return IVFPQ_OK;
}

template <int K, int NW>
int launch_pairs(const uint32_t* keys, const uint32_t* idx, int64_t rows, int64_t len,
                        int64_t chunks, int64_t chunk_len, const OutWriter& w,
                        cudaStream_t s) {
  const size_t smem = NW > 1 ? size_t(NW) * K * 2 * sizeof(uint32_t) : 0;
  auto kern = select_pairs_kernel<K, NW>;
  IVFPQ_TRY(prepare_smem(kern, smem));
  dim3 grid{unsigned(rows), unsigned(chunks), 1u};
  kern<<<grid, NW * 32, smem, s>>>(keys, idx, len, chunk_len, w);
  IVFPQ_LAUNCHED_K(kern, smem, NW * 32);
  return IVFPQ_OK;
}

}  // namespace ivfpq

// Explicit instantiation of launchers, used by the select_*.cu units.
#define IVFPQ_INST_SELECT_ROWS(K, NW)                                                       \
  template int ivfpq::launch_rows<K, NW>(const float*, int64_t, int64_t, int64_t, int64_t,  \
                                         const ivfpq::OutWriter&, cudaStream_t);
#define IVFPQ_INST_SELECT_PAIRS(K, NW)                                                       \
  template int ivfpq::launch_pairs<K, NW>(const uint32_t*, const uint32_t*, int64_t, int64_t, \
                                          int64_t, int64_t, const ivfpq::OutWriter&,         \
                                          cudaStream_t);
