// Candidate selection entry (see select_cand.cuh); queue lengths above 256
// are instantiated in select_cand_large.cu.
#include <algorithm>

#include "select_cand.cuh"

namespace ivfpq {
extern template int launch_cand<512>(const uint64_t*, const int*, int, int, int64_t,
                                     const float*, const float*, int64_t, int,
                                     const OutWriter&, cudaStream_t);
extern template int launch_cand<1024>(const uint64_t*, const int*, int, int, int64_t,
                                      const float*, const float*, int64_t, int,
                                      const OutWriter&, cudaStream_t);
extern template int launch_cand<2048>(const uint64_t*, const int*, int, int, int64_t,
                                      const float*, const float*, int64_t, int,
                                      const OutWriter&, cudaStream_t);

#define IVFPQ_EXTERN_SHORT(KW)                                                                \
  extern template int launch_cand_short<KW>(const uint64_t*, const int*, int, int, int64_t,    \
                                            uint32_t*, uint32_t*, int*, cudaStream_t);         \
  extern template int launch_cand_check<KW>(const uint32_t*, const uint32_t*, const int*,      \
                                            int64_t, int, int*, cudaStream_t);
IVFPQ_EXTERN_SHORT(64)
IVFPQ_EXTERN_SHORT(128)
IVFPQ_EXTERN_SHORT(256)

namespace {

// k > 256: 16 warps per row with K/8-entry queues, a merge of their 16 x K/8
// entries, and the block kernel with full-length queues again for the rows
// where a short queue may have dropped a result (or a segment overflowed).
// Exact like the block kernel alone; a warp's share of the k best is about
// k / 16, far below K / 8.
template <int K>
int select_long(const uint64_t* cand, const int* scnt, int nseg, int cap_s, int64_t rows,
                const float* Q, const float* X, int64_t n, int d, int k, const SelectOut& out,
                cudaStream_t s) {
  constexpr int KW = K / 8;
  Workspace ws(s);
  uint32_t *pk = nullptr, *pi = nullptr, *tk = nullptr, *ti = nullptr;
  int *over = nullptr, *flags = nullptr;
  IVFPQ_TRY(ws.alloc(&pk, size_t(rows) * 16 * KW));
  IVFPQ_TRY(ws.alloc(&pi, size_t(rows) * 16 * KW));
  IVFPQ_TRY(ws.alloc(&tk, size_t(rows) * k));
  IVFPQ_TRY(ws.alloc(&ti, size_t(rows) * k));
  IVFPQ_TRY(ws.alloc(&over, size_t(rows)));
  IVFPQ_TRY(ws.alloc(&flags, size_t(rows)));
  IVFPQ_TRY(launch_cand_short<KW>(cand, scnt, nseg, cap_s, rows, pk, pi, over, s));
  SelectOut part;
  part.kind = OutKind::Partial;
  part.pkeys = tk;
  part.pidx = ti;
  IVFPQ_TRY(merge_sorted_runs(pk, pi, rows, 16, KW, k, part, s));
  IVFPQ_TRY(launch_cand_check<KW>(pk, tk, over, rows, k, flags, s));
  cand_emit_kernel<<<unsigned(std::min<int64_t>(ceil_div(rows * k, 256), 65535 * 8)), 256, 0,
                     s>>>(tk, ti, rows, k, OutWriter{out, k, 1});
  IVFPQ_LAUNCHED();
  SelectOut ro = out;
  ro.row_mask = flags;
  return launch_cand<K>(cand, scnt, nseg, cap_s, rows, Q, X, n, d, OutWriter{ro, k, 1}, s);
}

}  // namespace

int select_candidates(const uint64_t* cand, const int* scnt, int nseg, int cap_s, int64_t rows,
                      const float* Q, const float* X, int64_t n, int d, int k,
                      const SelectOut& out, cudaStream_t s) {
  if (rows == 0) return IVFPQ_OK;
  OutWriter w{out, k, 1};
  int K = 32;
  while (K < k) K *= 2;
  switch (K) {
    case 512: return select_long<512>(cand, scnt, nseg, cap_s, rows, Q, X, n, d, k, out, s);
    case 1024: return select_long<1024>(cand, scnt, nseg, cap_s, rows, Q, X, n, d, k, out, s);
    case 2048: return select_long<2048>(cand, scnt, nseg, cap_s, rows, Q, X, n, d, k, out, s);
  }
  switch (K) {
    case 32: return launch_cand<32>(cand, scnt, nseg, cap_s, rows, Q, X, n, d, w, s);
    case 64: return launch_cand<64>(cand, scnt, nseg, cap_s, rows, Q, X, n, d, w, s);
    case 128: return launch_cand<128>(cand, scnt, nseg, cap_s, rows, Q, X, n, d, w, s);
    case 256: return launch_cand<256>(cand, scnt, nseg, cap_s, rows, Q, X, n, d, w, s);
    case 512: return launch_cand<512>(cand, scnt, nseg, cap_s, rows, Q, X, n, d, w, s);
    case 1024: return launch_cand<1024>(cand, scnt, nseg, cap_s, rows, Q, X, n, d, w, s);
    case 2048: return launch_cand<2048>(cand, scnt, nseg, cap_s, rows, Q, X, n, d, w, s);
  }
  set_error("candidate selection supports k <= %d (k = %d)", IVFPQ_MAX_K, k);
  return IVFPQ_ERR_UNSUPPORTED;
}

}  // namespace ivfpq
