// Exact k-nearest-neighbour search by distance tiles plus k-selection, and
// the flat_knn C entry point.
//
// Source: exact search ("Billion-scale similarity search with GPUs", section
// 5: queries are processed in tiles of t_q rows to bound temporary memory,
// each tile's distances are k-selected; section 4: k-selection).
#include <algorithm>

#include "internal.h"

namespace ivfpq {

namespace {
// Exact squared distances sum_t (q_t - x_t)^2 (fp32, in dimension order) of
// each selected (row, i) pair, as order-preserving keys with the column index,
// for the final re-sort. One warp per (row, i); lane-strided sum.
__global__ void rerank_kernel(const float* __restrict__ Q, const float* __restrict__ X, int d,
                              int64_t rows, int k, const int64_t* __restrict__ idx64,
                              const int32_t* __restrict__ idx32, uint32_t* __restrict__ keys,
                              uint32_t* __restrict__ cols) {
  const int64_t w = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (w >= rows * k) return;
  const int64_t r = w / k;
  const int64_t c = idx64 ? idx64[w] : int64_t(idx32[w]);
  if (c < 0) {
    if (lane == 0) {
      keys[w] = kSentinelKey;
      cols[w] = kSentinelIdx;
    }
    return;
  }
  float s = 0.f;
  for (int t = lane; t < d; t += 32) {
    const float df = Q[r * d + t] - X[c * d + t];
    s = fmaf(df, df, s);
  }
#pragma unroll
  for (int o = 16; o >= 1; o /= 2) s += __shfl_xor_sync(kFullMask, s, o);
  if (lane == 0) {
    keys[w] = float_to_key(s);
    cols[w] = uint32_t(c);
  }
}
}  // namespace

// Bytes of distance workspace per query tile.
static const int64_t kTileBytes = int64_t(2) << 30;

int knn_by_tiles(const float* Q, int64_t nq, const float* X, int64_t n, int d, int k,
                 const SelectOut& out, cudaStream_t s, const TcOperand* xop) {
  if (nq == 0) return IVFPQ_OK;
  int64_t tq = std::max<int64_t>(128, kTileBytes / (4 * std::max<int64_t>(n, 1)) / 128 * 128);
  tq = std::min(std::min(tq, nq), int64_t(65535) * 128);
  Workspace ws(s);
  float* D = nullptr;
  const bool tc = n > 0 && l2_tc_available(d);
  // the re-rank pairs (2 words per selected entry) reuse the distance tile
  const int64_t tile_words = std::max<int64_t>(n, tc ? 2 * int64_t(k) : 1);
  IVFPQ_TRY(ws.alloc(&D, size_t(tq * tile_words)));
  TcOperand qo, xo;
  int* err = nullptr;
  if (tc) {
    const int dpad = tc_dpad(d);
    float *qhi, *qlo, *qn;
    IVFPQ_TRY(ws.alloc(&qhi, size_t(nq) * dpad));
    IVFPQ_TRY(ws.alloc(&qlo, size_t(nq) * dpad));
    IVFPQ_TRY(ws.alloc(&qn, size_t(nq)));
    IVFPQ_TRY(l2_tc_prepare(Q, nq, d, qhi, qlo, qn, s));
    qo.hi = qhi;
    qo.lo = qlo;
    qo.norms = qn;
    if (xop) {
      xo = *xop;
    } else {
      float *xhi, *xlo, *xn;
      IVFPQ_TRY(ws.alloc(&xhi, size_t(n) * dpad));
      IVFPQ_TRY(ws.alloc(&xlo, size_t(n) * dpad));
      IVFPQ_TRY(ws.alloc(&xn, size_t(n)));
      IVFPQ_TRY(l2_tc_prepare(X, n, d, xhi, xlo, xn, s));
      xo.hi = xhi;
      xo.lo = xlo;
      xo.norms = xn;
    }
    IVFPQ_TRY(ws.alloc(&err, 1));
    IVFPQ_CUDA(cudaMemsetAsync(err, 0, sizeof(int), s));
  }
  for (int64_t q0 = 0; q0 < nq; q0 += tq) {
    const int64_t rows = std::min(tq, nq - q0);
    if (tc) {
      const int dpad = tc_dpad(d);
      IVFPQ_TRY(l2_tc_tiles(qo.hi + q0 * dpad, qo.lo + q0 * dpad, qo.norms + q0, rows, xo.hi,
                            xo.lo, xo.norms, n, d, D, n, err, s));
    } else {
      IVFPQ_TRY(l2_distance_tile(Q + q0 * d, rows, X, n, d, D, n, s));
    }
    SelectOut o = out;
    if (o.vals) o.vals += q0 * k;
    if (o.idx64) o.idx64 += q0 * k;
    if (o.idx32) o.idx32 += q0 * k;
    IVFPQ_TRY(kselect_device(D, rows, n, k, o, s));
    if (tc) {
      // The GEMM form loses absolute precision ~eps * (|q|^2 + |x|^2) to
      // cancellation; the winners' distances are recomputed in the direct
      // form and re-sorted.
      uint32_t* rk = reinterpret_cast<uint32_t*>(D);
      uint32_t* rc = rk + rows * k;
      const int64_t warps = rows * k;
      rerank_kernel<<<unsigned(ceil_div(warps * 32, 256)), 256, 0, s>>>(
          Q + q0 * d, X, d, rows, k, o.idx64, o.kind == OutKind::Probes ? o.idx32 : nullptr, rk,
          rc);
      IVFPQ_LAUNCHED();
      IVFPQ_TRY(select_pairs(rk, rc, rows, k, k, 1, k, o, s));
    }
  }
  return IVFPQ_OK;
}

}  // namespace ivfpq

using namespace ivfpq;

extern "C" int flat_knn(const float* db, int64_t n, int d, const float* queries, int64_t nq,
                        int k, float* out_dist, int64_t* out_ids, void* stream) {
  clear_error();
  IVFPQ_REQUIRE(n >= 0 && nq >= 0 && d > 0, "flat_knn: bad sizes (n=%lld nq=%lld d=%d)",
                (long long)n, (long long)nq, d);
  IVFPQ_REQUIRE(k >= 1 && k <= IVFPQ_MAX_K, "flat_knn: k=%d outside [1, %d]", k, IVFPQ_MAX_K);
  IVFPQ_REQUIRE(n < int64_t(0xffffffffLL), "flat_knn: n=%lld too large", (long long)n);
  if (nq == 0) return IVFPQ_OK;
  IVFPQ_REQUIRE(queries && out_dist && out_ids && (db || n == 0), "flat_knn: null pointer");
  SelectOut out;
  out.kind = OutKind::Float;
  out.vals = out_dist;
  out.idx64 = out_ids;
  return knn_by_tiles(queries, nq, db, n, d, k, out, static_cast<cudaStream_t>(stream));
}
