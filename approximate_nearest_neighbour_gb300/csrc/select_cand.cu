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


namespace {

// k > 32: the radix-bound selection (select_radix.cu), and the WarpSelect
// kernels for the rows it flags (an overflowed segment, or ties around its
// bound). For k > 256, 16 warps with K/8-entry queues, a merge of their
// 16 x K/8 entries and a check took 5.7 of 25.9 ms per 10,000-query flat
// k = 1024 call; for k = 64 / 128 (the coarse quantizer's probes) one warp
// per row took 0.27 / 0.50 ms per 10,000 queries against 65,536 / 262,144
// centroids (coarse stage 1.29 -> 1.21 ms, 3.74 -> 3.49 ms).
template <int K>
int select_long(const uint64_t* cand, const int* scnt, int nseg, int cap_s, int64_t rows,
                const float* Q, const float* X, int64_t n, int d, int k, const SelectOut& out,
                cudaStream_t s) {
  Workspace ws(s);
  int* flags = nullptr;
  IVFPQ_TRY(ws.alloc(&flags, size_t(rows)));
  IVFPQ_TRY(cand_radix_select(cand, scnt, nseg, cap_s, rows, k, out, flags, s));
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
    case 64: return select_long<64>(cand, scnt, nseg, cap_s, rows, Q, X, n, d, k, out, s);
    case 128: return select_long<128>(cand, scnt, nseg, cap_s, rows, Q, X, n, d, k, out, s);
    case 256: return select_long<256>(cand, scnt, nseg, cap_s, rows, Q, X, n, d, k, out, s);
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
