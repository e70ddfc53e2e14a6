// Candidate selection entry (see select_cand.cuh); queue lengths above 256
// are instantiated in select_cand_large.cu.
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

int select_candidates(const uint64_t* cand, const int* scnt, int nseg, int cap_s, int64_t rows,
                      const float* Q, const float* X, int64_t n, int d, int k,
                      const SelectOut& out, cudaStream_t s) {
  if (rows == 0) return IVFPQ_OK;
  OutWriter w{out, k, 1};
  int K = 32;
  while (K < k) K *= 2;
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
