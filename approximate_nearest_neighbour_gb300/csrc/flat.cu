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
// The same with float4 loads (d a multiple of 4, 16-byte aligned rows): 8
// lanes per entry, 4 entries per warp, each lane up to d / 32 float4 of the
// query and of the database row in flight.
__global__ void rerank4_kernel(const float* __restrict__ Q, const float* __restrict__ X, int d,
                               int64_t rows, int k, const int64_t* __restrict__ idx64,
                               const int32_t* __restrict__ idx32, uint32_t* __restrict__ keys,
                               uint32_t* __restrict__ cols) {
  const int64_t e = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 3;
  const int sub = threadIdx.x & 7;
  const bool live = e < rows * k;  // lanes past the end stay for the shuffles
  const int64_t r = live ? e / k : 0;
  const int64_t c = live ? (idx64 ? idx64[e] : int64_t(idx32[e])) : -1;
  float s = 0.f;
  if (c >= 0) {
    const float4* q4 = reinterpret_cast<const float4*>(Q + r * d);
    const float4* x4 = reinterpret_cast<const float4*>(X + c * d);
    for (int j = sub; j < d / 4; j += 8) {
      const float4 a = __ldg(q4 + j), b = __ldg(x4 + j);
      const float dx = a.x - b.x, dy = a.y - b.y, dz = a.z - b.z, dw = a.w - b.w;
      s = fmaf(dx, dx, s);
      s = fmaf(dy, dy, s);
      s = fmaf(dz, dz, s);
      s = fmaf(dw, dw, s);
    }
  }
  s += __shfl_xor_sync(kFullMask, s, 4);
  s += __shfl_xor_sync(kFullMask, s, 2);
  s += __shfl_xor_sync(kFullMask, s, 1);
  if (live && sub == 0) {
    keys[e] = c < 0 ? kSentinelKey : float_to_key(s);
    cols[e] = c < 0 ? kSentinelIdx : uint32_t(c);
  }
}
}  // namespace

// Bytes of distance workspace per query tile.
static const int64_t kTileBytes = int64_t(2) << 30;

namespace {

// Re-ranks the k selected entries of each row of o in the exact direct form
// and re-sorts them (scratch: 2 * rows * k words). The GEMM form loses
// absolute precision ~eps * (|q|^2 + |x|^2) to cancellation.
int rerank(const float* Q, const float* X, int d, int64_t rows, int k, const SelectOut& o,
           uint32_t* scratch, cudaStream_t s) {
  uint32_t* rk = scratch;
  uint32_t* rc = rk + rows * k;
  const int64_t warps = rows * k;
  const bool vec = d % 4 == 0 && (reinterpret_cast<uintptr_t>(Q) & 15) == 0 &&
                   (reinterpret_cast<uintptr_t>(X) & 15) == 0;
  if (vec) {
    rerank4_kernel<<<unsigned(ceil_div(warps * 8, 256)), 256, 0, s>>>(
        Q, X, d, rows, k, o.idx64, o.kind == OutKind::Probes ? o.idx32 : nullptr, rk, rc);
  } else {
    rerank_kernel<<<unsigned(ceil_div(warps * 32, 256)), 256, 0, s>>>(
        Q, X, d, rows, k, o.idx64, o.kind == OutKind::Probes ? o.idx32 : nullptr, rk, rc);
  }
  IVFPQ_LAUNCHED();
  // k > 256: one bitonic sort per row (the pair selection's k-entry queues
  // took 1.8 ms of a 10,000-query flat k = 1024 call)
  if (k > 256) return sort_pairs_rows(rk, rc, rows, k, k, o, s);
  return select_pairs(rk, rc, rows, k, k, 1, k, o, s);
}

// Filtered plan (any k <= IVFPQ_MAX_K, large n). A first tensor-core pass over the
// first ns columns takes, per row, the minimum of u = D - ||q||^2 over each of
// G >= 4k column groups; the k-th smallest of those G minima is an upper
// bound on the row's k-th smallest u over all n columns (it is attained by k
// distinct columns). The full pass then keeps only entries at or below it:
// about k * n / ns of them per row, instead of writing and re-reading the
// whole distance row.
struct FilterPlan {
  int64_t ns = 0;   // columns of the first pass
  int split_a = 0;  // CTAs per query tile in the first pass (G = 128 * split_a)
};

bool filter_plan(int64_t n, int k, FilterPlan* fp) {
  if (k > IVFPQ_MAX_K || n < 2048) return false;
  const int64_t ns = ceil_div(ceil_div(n, 8), 128) * 128;
  const int split_a = int(ceil_div(4 * int64_t(k), 128));
  if (ns / 128 < split_a || 2 * ns > n) return false;
  fp->ns = ns;
  fp->split_a = split_a;
  return true;
}

SelectOut offset_out(const SelectOut& out, int64_t off) {
  SelectOut o = out;
  if (o.vals) o.vals += off;
  if (o.idx64) o.idx64 += off;
  if (o.idx32) o.idx32 += off;
  return o;
}

}  // namespace

int knn_by_tiles(const float* Q, int64_t nq, const float* X, int64_t n, int d, int k,
                 const SelectOut& out, cudaStream_t s, const TcOperand* xop) {
  if (nq == 0) return IVFPQ_OK;
  Workspace ws(s);
  const bool tc = n > 0 && l2_tc_available(d);
  if (!tc) {
    int64_t tq = std::max<int64_t>(128, kTileBytes / (4 * std::max<int64_t>(n, 1)) / 128 * 128);
    tq = std::min(std::min(tq, nq), int64_t(65535) * 128);
    float* D = nullptr;
    IVFPQ_TRY(ws.alloc(&D, size_t(tq * std::max<int64_t>(n, 1))));
    for (int64_t q0 = 0; q0 < nq; q0 += tq) {
      const int64_t rows = std::min(tq, nq - q0);
      if (n > 0) IVFPQ_TRY(l2_distance_tile(Q + q0 * d, rows, X, n, d, D, n, s));
      IVFPQ_TRY(kselect_device(D, rows, n, k, offset_out(out, q0 * k), s));
    }
    return IVFPQ_OK;
  }

  // tensor-core operands
  const int dpad = tc_dpad(d);
  TcOperand qo, xo;
  {
    float *qhi, *qlo, *qn;
    IVFPQ_TRY(ws.alloc(&qhi, size_t(nq) * dpad));
    IVFPQ_TRY(ws.alloc(&qlo, size_t(nq) * dpad));
    IVFPQ_TRY(ws.alloc(&qn, size_t(nq)));
    IVFPQ_TRY(l2_tc_prepare(Q, nq, d, qhi, qlo, qn, s));
    qo.hi = qhi;
    qo.lo = qlo;
    qo.norms = qn;
  }
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
  int* err = nullptr;
  IVFPQ_TRY(device_status_word(&err));

  FilterPlan fp;
  if (filter_plan(n, k, &fp)) {
    const int64_t G0 = 128 * int64_t(fp.split_a);
    // candidate segments: nseg per row from the filter pass's CTA split, each
    // holding 4x its expected share of ~1.5 k n / ns survivors (at least 64)
    auto seg_cap = [&](int nseg) {
      const int64_t expect = ceil_div(3 * int64_t(k) * n, 2 * fp.ns);
      return int(ceil_div(std::max<int64_t>(64, ceil_div(4 * expect, nseg)), 32) * 32);
    };
    int64_t tq = std::min(nq, int64_t(65535) * 128);
    for (;;) {
      const int nseg = 2 * tc_filter_split(tq, n);
      const int64_t row_bytes = 4 * G0 * 4 + 4 + int64_t(nseg) * (seg_cap(nseg) * 8 + 4);
      if (tq <= 128 || tq * row_bytes <= kTileBytes) break;
      tq = std::max<int64_t>(128, (tq / 2) / 128 * 128);
    }
    const int split_b = tc_filter_split(tq, n);
    const int nseg = 2 * split_b;
    const int cap_s = seg_cap(nseg);
    // the first pass's CTAs per query tile: raised from split_a (up to 4x and
    // its column tiles) until the last wave on the SMs is at least 90 % full,
    // which only adds groups (a tighter bound); large coarse stage: 158 CTAs
    // took two waves on 152 SMs
    int split_a = fp.split_a;
    {
      const int64_t qtiles = ceil_div(tq, 128), sms = num_sms();
      for (int64_t sa = fp.split_a; sa <= std::min<int64_t>(4 * fp.split_a, fp.ns / 128); ++sa) {
        const int64_t ctas = qtiles * sa;
        if (10 * ctas >= 9 * ceil_div(ctas, sms) * sms) {
          split_a = int(sa);
          break;
        }
      }
    }
    const int64_t G = 128 * int64_t(split_a);
    float* gmin = nullptr;
    float* bound = nullptr;
    uint64_t* cand = nullptr;
    int* scnt = nullptr;
    IVFPQ_TRY(ws.alloc(&gmin, size_t(tq * G)));
    IVFPQ_TRY(ws.alloc(&bound, size_t(tq)));
    IVFPQ_TRY(ws.alloc(&cand, size_t(tq * nseg) * cap_s));
    IVFPQ_TRY(ws.alloc(&scnt, size_t(tq * nseg)));
    for (int64_t q0 = 0; q0 < nq; q0 += tq) {
      const int64_t rows = std::min(tq, nq - q0);
      IVFPQ_TRY(l2_tc_group_min(qo.hi + q0 * dpad, qo.lo + q0 * dpad, rows, xo.hi, xo.lo,
                                xo.norms, fp.ns, d, split_a, gmin, err, s));
      // a bound of each row's k-th smallest group minimum (radix selection;
      // the k-entry queues of a full selection took 4.7 ms of a 10,000-query
      // flat k = 1024 call)
      IVFPQ_TRY(row_kth_bound(gmin, rows, G, k, bound, s));
      IVFPQ_TRY(l2_tc_filter(qo.hi + q0 * dpad, qo.lo + q0 * dpad, qo.norms + q0, rows, xo.hi,
                             xo.lo, xo.norms, n, d, bound, 1, split_b, cand, scnt, cap_s, err,
                             s));
      const SelectOut o = offset_out(out, q0 * k);
      IVFPQ_TRY(
          select_candidates(cand, scnt, nseg, cap_s, rows, Q + q0 * d, X, n, d, k, o, s));
      // G >= 4k words per row hold the re-rank pairs
      IVFPQ_TRY(rerank(Q + q0 * d, X, d, rows, k, o, reinterpret_cast<uint32_t*>(gmin), s));
    }
    return IVFPQ_OK;
  }

  int64_t tq = std::max<int64_t>(128, kTileBytes / (4 * std::max<int64_t>(n, 1)) / 128 * 128);
  tq = std::min(std::min(tq, nq), int64_t(65535) * 128);
  // the re-rank pairs (2 words per selected entry) reuse the distance tile
  const int64_t tile_words = std::max<int64_t>(n, 2 * int64_t(k));
  float* D = nullptr;
  IVFPQ_TRY(ws.alloc(&D, size_t(tq * tile_words)));
  for (int64_t q0 = 0; q0 < nq; q0 += tq) {
    const int64_t rows = std::min(tq, nq - q0);
    IVFPQ_TRY(l2_tc_tiles(qo.hi + q0 * dpad, qo.lo + q0 * dpad, qo.norms + q0, rows, xo.hi, xo.lo,
                          xo.norms, n, d, D, n, err, s));
    const SelectOut o = offset_out(out, q0 * k);
    IVFPQ_TRY(kselect_device(D, rows, n, k, o, s));
    IVFPQ_TRY(rerank(Q + q0 * d, X, d, rows, k, o, reinterpret_cast<uint32_t*>(D), s));
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
