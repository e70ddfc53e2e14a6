// Selection by a radix bound, one block of 512 threads per row: the k-th
// smallest key of a row is located by a 4,096-bin histogram of its top 12 bits
// and then, within that bin, by a histogram of the next 12 bits; the end of
// that 256-key sub-bin is a bound theta with at least k keys <= theta and, on
// spread-out keys, few more. The k smallest are then gathered (keys <= theta)
// into shared memory and sorted with a bitonic network (the helpers are in
// select_radix.cuh). Uses here, where WarpSelect's queues cost most of the
// time:
//  * row_kth_bound: theta alone, an upper bound of each row's k-th smallest
//    value (the filtered tensor-core plan's bound, every k);
//  * candidate selection over the filtered pass's segments for k > 32;
//  * the final sort of the k re-ranked pairs of each row for k > 256.
// (The by-list scan's final selection for k > 256 uses the same helpers, in
// ivfpq_search.cu.)
// A row whose gathered keys do not fit (ties around theta) or whose segment
// overflowed is flagged; the caller redoes it with the full-length kernels.
//
// Source: the k smallest of each row ("Billion-scale similarity search with
// GPUs", section 4, k-selection); the radix bound is this library's own
// choice, exact like the pages' WarpSelect (the result is the k smallest).
#include <algorithm>

#include "select_inst.cuh"
#include "select_radix.cuh"

namespace ivfpq {
namespace {

using radix::bitonic_sort;
using radix::kRBins;
using radix::kRThreads;
using radix::radix_theta;
using radix::RadixShared;

// bound[row] = a float at least the row's k-th smallest value (the float of
// theta; +inf when there is no bound).
__global__ void __launch_bounds__(kRThreads)
row_kth_kernel(const float* __restrict__ vals, int64_t cols, int k, float* __restrict__ bound) {
  __shared__ uint32_t hist[kRBins];
  __shared__ RadixShared sh;
  const int64_t row = blockIdx.x;
  const float* rp = vals + row * cols;
  const uint32_t theta = radix_theta(hist, sh, uint32_t(k), [&](auto f) {
    for (int64_t c = threadIdx.x; c < cols; c += kRThreads) f(float_to_key(__ldg(rp + c)));
  });
  // keys from +inf up (+inf, NaN patterns, the sentinel) bound nothing: +inf
  if (threadIdx.x == 0) bound[row] = theta >= 0xff800000u ? INFINITY : key_to_float(theta);
}

// The k smallest (key, column) entries of each row's candidate segments,
// sorted; rows with an overflowed segment, or more than cap entries <= theta,
// are flagged (flags[row] = 1) and written by the caller's fallback.
__global__ void __launch_bounds__(kRThreads)
cand_radix_kernel(const uint64_t* __restrict__ cand, const int* __restrict__ scnt, int nseg,
                  int cap_s, int k, int cap, OutWriter out, int* __restrict__ flags) {
  extern __shared__ uint32_t sm_radix[];
  uint32_t* hist = sm_radix;
  uint32_t* sk = sm_radix + kRBins;
  uint32_t* sv = sk + cap;
  __shared__ RadixShared sh;
  const int64_t row = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int* cnt = scnt + row * nseg;
  int over = 0;
  for (int g = threadIdx.x; g < nseg; g += kRThreads) over |= cnt[g] > cap_s;
  over = __syncthreads_or(over);
  if (over) {  // block-uniform
    if (threadIdx.x == 0) flags[row] = 1;
    return;
  }
  // warp w takes segments w, w + 16, ...; its lanes stride over the entries
  auto for_each = [&](auto f) {
    for (int g = warp; g < nseg; g += kRThreads / 32) {
      const int ns = max(cnt[g], 0);
      const uint64_t* e = cand + (row * nseg + g) * cap_s;
      for (int i = lane; i < ns; i += 32) f(uint32_t(e[i] >> 32), e[i]);
    }
  };
  const uint32_t theta = radix_theta(hist, sh, uint32_t(k), [&](auto f) {
    for_each([&](uint32_t key, uint64_t) { f(key); });
  });
  if (threadIdx.x == 0) sh.count = 0;
  __syncthreads();
  const uint32_t below = (1u << lane) - 1u;
  for (int g = warp; g < nseg; g += kRThreads / 32) {
    const int ns = max(cnt[g], 0);
    const uint64_t* e = cand + (row * nseg + g) * cap_s;
    for (int base = 0; base < ns; base += 32) {
      const int i = base + lane;
      const uint64_t v = i < ns ? e[i] : ~uint64_t(0);
      const bool pass = i < ns && uint32_t(v >> 32) <= theta;
      const uint32_t bal = __ballot_sync(kFullMask, pass);
      if (bal == 0u) continue;
      uint32_t pos = 0;
      if (lane == 0) pos = atomicAdd(&sh.count, uint32_t(__popc(bal)));
      pos = __shfl_sync(kFullMask, pos, 0) + uint32_t(__popc(bal & below));
      if (pass && pos < uint32_t(cap)) {
        sk[pos] = uint32_t(v >> 32);
        sv[pos] = uint32_t(v);
      }
    }
  }
  __syncthreads();
  const uint32_t n = sh.count;
  if (n > uint32_t(cap)) {  // block-uniform
    if (threadIdx.x == 0) flags[row] = 1;
    return;
  }
  uint32_t P = 32;
  while (P < n) P <<= 1;
  for (uint32_t i = n + threadIdx.x; i < P; i += kRThreads) {
    sk[i] = kSentinelKey;
    sv[i] = kSentinelIdx;
  }
  __syncthreads();
  bitonic_sort(sk, sv, P);
  for (int i = threadIdx.x; i < k; i += kRThreads)
    out.write(row, 0, i, uint32_t(i) < P ? sk[i] : kSentinelKey,
              uint32_t(i) < P ? sv[i] : kSentinelIdx);
  if (threadIdx.x == 0) flags[row] = 0;
}

// Each row's len (key, index) pairs, sorted, the first k written (len <= cap,
// a power of two >= len).
__global__ void __launch_bounds__(kRThreads)
sort_rows_kernel(const uint32_t* __restrict__ keys, const uint32_t* __restrict__ idx, int len,
                 int k, int P, OutWriter out) {
  extern __shared__ uint32_t sm_sort[];
  uint32_t* sk = sm_sort;
  uint32_t* sv = sm_sort + P;
  const int64_t row = blockIdx.x;
  if (out.o.row_mask && !out.o.row_mask[row]) return;  // block-uniform
  for (int i = threadIdx.x; i < P; i += kRThreads) {
    const bool ok = i < len;
    sk[i] = ok ? keys[row * len + i] : kSentinelKey;
    sv[i] = ok ? idx[row * len + i] : kSentinelIdx;
  }
  __syncthreads();
  bitonic_sort(sk, sv, uint32_t(P));
  for (int i = threadIdx.x; i < k; i += kRThreads) out.write(row, 0, i, sk[i], sv[i]);
}

}  // namespace

int row_kth_bound(const float* vals, int64_t rows, int64_t cols, int k, float* bound,
                  cudaStream_t s) {
  if (rows == 0) return IVFPQ_OK;
  IVFPQ_REQUIRE(rows <= 0x7fffffff, "row_kth_bound: %lld rows", (long long)rows);
  row_kth_kernel<<<unsigned(rows), kRThreads, 0, s>>>(vals, cols, k, bound);
  IVFPQ_LAUNCHED();
  return IVFPQ_OK;
}

int cand_radix_select(const uint64_t* cand, const int* scnt, int nseg, int cap_s, int64_t rows,
                      int k, const SelectOut& out, int* flags, cudaStream_t s) {
  if (rows == 0) return IVFPQ_OK;
  IVFPQ_REQUIRE(rows <= 0x7fffffff, "cand_radix_select: %lld rows", (long long)rows);
  int cap = 64;
  while (cap < 2 * k) cap <<= 1;
  const size_t smem = (size_t(kRBins) + 2 * size_t(cap)) * 4;
  IVFPQ_TRY(set_dynamic_smem(cand_radix_kernel, smem));
  cand_radix_kernel<<<unsigned(rows), kRThreads, smem, s>>>(cand, scnt, nseg, cap_s, k, cap,
                                                           OutWriter{out, k, 1}, flags);
  IVFPQ_LAUNCHED_K(cand_radix_kernel, smem, kRThreads);
  return IVFPQ_OK;
}

int sort_pairs_rows(const uint32_t* keys, const uint32_t* idx, int64_t rows, int len, int k,
                    const SelectOut& out, cudaStream_t s) {
  if (rows == 0) return IVFPQ_OK;
  IVFPQ_REQUIRE(rows <= 0x7fffffff && k <= len && len <= 8192,
                "sort_pairs_rows: rows=%lld len=%d k=%d", (long long)rows, len, k);
  int P = 32;
  while (P < len) P <<= 1;
  const size_t smem = size_t(P) * 8;
  IVFPQ_TRY(set_dynamic_smem(sort_rows_kernel, smem));
  sort_rows_kernel<<<unsigned(rows), kRThreads, smem, s>>>(keys, idx, len, k, P,
                                                          OutWriter{out, k, 1});
  IVFPQ_LAUNCHED_K(sort_rows_kernel, smem, kRThreads);
  return IVFPQ_OK;
}

}  // namespace ivfpq
