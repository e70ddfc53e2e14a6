// Exact k-nearest-neighbour search by distance tiles plus k-selection, and
// the flat_knn C entry point.
//
// Source: exact search ("Billion-scale similarity search with GPUs", section
// 5: queries are processed in tiles of t_q rows to bound temporary memory,
// each tile's distances are k-selected; section 4: k-selection).
#include <algorithm>

#include "internal.h"

namespace ivfpq {

// Bytes of distance workspace per query tile.
static const int64_t kTileBytes = int64_t(2) << 30;

int knn_by_tiles(const float* Q, int64_t nq, const float* X, int64_t n, int d, int k,
                 const SelectOut& out, cudaStream_t s) {
  if (nq == 0) return IVFPQ_OK;
  int64_t tq = std::max<int64_t>(128, kTileBytes / (4 * std::max<int64_t>(n, 1)) / 128 * 128);
  tq = std::min(tq, nq);
  Workspace ws(s);
  float* D = nullptr;
  IVFPQ_TRY(ws.alloc(&D, size_t(tq * std::max<int64_t>(n, 1))));
  for (int64_t q0 = 0; q0 < nq; q0 += tq) {
    const int64_t rows = std::min(tq, nq - q0);
    IVFPQ_TRY(l2_distance_tile(Q + q0 * d, rows, X, n, d, D, n, s));
    SelectOut o = out;
    if (o.vals) o.vals += q0 * k;
    if (o.idx64) o.idx64 += q0 * k;
    if (o.idx32) o.idx32 += q0 * k;
    IVFPQ_TRY(kselect_device(D, rows, n, k, o, s));
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
