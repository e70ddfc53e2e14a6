// Dispatch of the row-wise selection kernels by warp-queue length, the
// two-pass selection for few long rows, and the kselect C entry point.
//
// Source: WarpSelect / two-pass k-selection ("Billion-scale similarity search
// with GPUs", section 4 Algorithm 3 and section 5, the paragraph introducing
// the two-pass k-selection with subdivision factor f).
#include <algorithm>
#include <cstring>
#include <mutex>

#include "internal.h"
#include "select_inst.cuh"

namespace ivfpq {

static int queue_len(int k) {
  int K = 32;
  while (K < k) K *= 2;
  return K;
}

#define IVFPQ_EXTERN_SELECT(K, NW)                                                             \
  extern template int launch_rows<K, NW>(const float*, int64_t, int64_t, int64_t, int64_t,     \
                                         const OutWriter&, cudaStream_t);                      \
  extern template int launch_pairs<K, NW>(const uint32_t*, const uint32_t*, int64_t, int64_t,  \
                                          int64_t, int64_t, const OutWriter&, cudaStream_t);
IVFPQ_EXTERN_SELECT(32, 1)
IVFPQ_EXTERN_SELECT(32, 4)
IVFPQ_EXTERN_SELECT(64, 1)
IVFPQ_EXTERN_SELECT(64, 4)
IVFPQ_EXTERN_SELECT(128, 1)
IVFPQ_EXTERN_SELECT(128, 4)
IVFPQ_EXTERN_SELECT(256, 1)
IVFPQ_EXTERN_SELECT(256, 4)
IVFPQ_EXTERN_SELECT(512, 4)
IVFPQ_EXTERN_SELECT(1024, 4)
IVFPQ_EXTERN_SELECT(2048, 4)

// Four warps per block once a chunk holds enough elements to keep them busy
// (always for K >= 512, whose single-warp variants are not built).
static bool use_block(int64_t chunk_len, int K) {
  return K >= 512 || (chunk_len >= 8 * 128 && chunk_len >= 2 * K);
}

template <int K>
static int rows_k(const float* vals, int64_t rows, int64_t cols, int k, int64_t chunks,
                  int64_t chunk_len, const SelectOut& out, cudaStream_t s) {
  OutWriter w{out, k, chunks};
  if constexpr (K >= 512) {
    return launch_rows<K, 4>(vals, rows, cols, chunks, chunk_len, w, s);
  } else {
    if (use_block(chunk_len, K)) return launch_rows<K, 4>(vals, rows, cols, chunks, chunk_len, w, s);
    return launch_rows<K, 1>(vals, rows, cols, chunks, chunk_len, w, s);
  }
}

template <int K>
static int pairs_k(const uint32_t* keys, const uint32_t* idx, int64_t rows, int64_t len, int k,
                   int64_t chunks, int64_t chunk_len, const SelectOut& out, cudaStream_t s) {
  OutWriter w{out, k, chunks};
  if constexpr (K >= 512) {
    return launch_pairs<K, 4>(keys, idx, rows, len, chunks, chunk_len, w, s);
  } else {
    if (use_block(chunk_len, K))
      return launch_pairs<K, 4>(keys, idx, rows, len, chunks, chunk_len, w, s);
    return launch_pairs<K, 1>(keys, idx, rows, len, chunks, chunk_len, w, s);
  }
}

int select_rows(const float* vals, int64_t rows, int64_t cols, int k, int64_t chunks,
                int64_t chunk_len, const SelectOut& out, cudaStream_t s) {
  if (rows == 0) return IVFPQ_OK;
  switch (queue_len(k)) {
    case 32: return rows_k<32>(vals, rows, cols, k, chunks, chunk_len, out, s);
    case 64: return rows_k<64>(vals, rows, cols, k, chunks, chunk_len, out, s);
    case 128: return rows_k<128>(vals, rows, cols, k, chunks, chunk_len, out, s);
    case 256: return rows_k<256>(vals, rows, cols, k, chunks, chunk_len, out, s);
    case 512: return rows_k<512>(vals, rows, cols, k, chunks, chunk_len, out, s);
    case 1024: return rows_k<1024>(vals, rows, cols, k, chunks, chunk_len, out, s);
    case 2048: return rows_k<2048>(vals, rows, cols, k, chunks, chunk_len, out, s);
  }
  set_error("k=%d exceeds the largest supported k (%d)", k, IVFPQ_MAX_K);
  return IVFPQ_ERR_INVALID_ARG;
}

namespace {
// The k smallest of a row's `runs` sorted runs of kw (key, index) pairs
// (ascending, sentinel-padded), by a tree of bitonic merges in shared memory
// (each merge: the mirror comparison of two sorted runs, then half-cleaners):
// one block per row, total = runs * kw rounded up to a power of two.
__global__ void merge_runs_kernel(const uint32_t* __restrict__ pk, const uint32_t* __restrict__ pi,
                                  int runs, int kw, int total, int k, OutWriter out) {
  extern __shared__ uint32_t sm_runs[];
  uint32_t* sk = sm_runs;
  uint32_t* sv = sm_runs + total;
  const int64_t row = blockIdx.x;
  const int len = runs * kw;
  for (int i = threadIdx.x; i < total; i += blockDim.x) {
    const bool ok = i < len;
    sk[i] = ok ? pk[row * len + i] : kSentinelKey;
    sv[i] = ok ? pi[row * len + i] : kSentinelIdx;
  }
  __syncthreads();
  auto cx = [&](int a, int b) {
    const uint32_t ka = sk[a], kb = sk[b];
    if (kb < ka) {
      const uint32_t va = sv[a];
      sk[a] = kb;
      sk[b] = ka;
      sv[a] = sv[b];
      sv[b] = va;
    }
  };
  for (int w = kw; w < total; w *= 2) {
    for (int c = threadIdx.x; c < total / 2; c += blockDim.x) {
      const int pair = c / w, t = c - pair * w;
      cx(pair * 2 * w + t, pair * 2 * w + 2 * w - 1 - t);
    }
    __syncthreads();
    for (int st = w / 2; st >= 1; st /= 2) {
      for (int c = threadIdx.x; c < total / 2; c += blockDim.x) {
        const int blk = c / st;
        const int a = blk * 2 * st + (c - blk * st);
        cx(a, a + st);
      }
      __syncthreads();
    }
  }
  for (int i = threadIdx.x; i < k; i += blockDim.x)
    out.write(row, 0, i, i < total ? sk[i] : kSentinelKey, i < total ? sv[i] : kSentinelIdx);
}

}  // namespace

int merge_sorted_runs(const uint32_t* pk, const uint32_t* pi, int64_t rows, int runs, int kw, int k,
                      const SelectOut& out, cudaStream_t s) {
  if (rows == 0) return IVFPQ_OK;
  const int64_t len = int64_t(runs) * kw;
  int64_t total = kw;
  while (total < len) total *= 2;
  if (total > 8192) return select_pairs(pk, pi, rows, len, k, 1, len, out, s);
  const size_t smem = size_t(total) * 8;
  if (smem > 48 * 1024) IVFPQ_TRY(set_dynamic_smem(merge_runs_kernel, smem));
  merge_runs_kernel<<<unsigned(rows), 256, smem, s>>>(pk, pi, runs, kw, int(total), k,
                                                     OutWriter{out, k, 1});
  IVFPQ_LAUNCHED_K(merge_runs_kernel, smem, 256);
  return IVFPQ_OK;
}

int select_pairs(const uint32_t* keys, const uint32_t* idx, int64_t rows, int64_t len, int k,
                 int64_t chunks, int64_t chunk_len, const SelectOut& out, cudaStream_t s) {
  if (rows == 0) return IVFPQ_OK;
  switch (queue_len(k)) {
    case 32: return pairs_k<32>(keys, idx, rows, len, k, chunks, chunk_len, out, s);
    case 64: return pairs_k<64>(keys, idx, rows, len, k, chunks, chunk_len, out, s);
    case 128: return pairs_k<128>(keys, idx, rows, len, k, chunks, chunk_len, out, s);
    case 256: return pairs_k<256>(keys, idx, rows, len, k, chunks, chunk_len, out, s);
    case 512: return pairs_k<512>(keys, idx, rows, len, k, chunks, chunk_len, out, s);
    case 1024: return pairs_k<1024>(keys, idx, rows, len, k, chunks, chunk_len, out, s);
    case 2048: return pairs_k<2048>(keys, idx, rows, len, k, chunks, chunk_len, out, s);
  }
  set_error("k=%d exceeds the largest supported k (%d)", k, IVFPQ_MAX_K);
  return IVFPQ_ERR_INVALID_ARG;
}

// One pass when there are enough rows to fill the GPU; otherwise each row is
// cut into chunks whose winners (k per chunk) are selected again.
int kselect_device(const float* vals, int64_t rows, int64_t cols, int k, const SelectOut& out,
                   cudaStream_t s) {
  if (rows == 0) return IVFPQ_OK;
  const int64_t target_blocks = 4 * int64_t(num_sms());
  const int64_t min_chunk = std::max<int64_t>(16384, 8 * int64_t(queue_len(k)));
  int64_t chunks = 1;
  if (rows < target_blocks && cols > 2 * min_chunk) {
    chunks = std::min(ceil_div(target_blocks, rows), ceil_div(cols, min_chunk));
  }
  if (chunks <= 1) return select_rows(vals, rows, cols, k, 1, std::max<int64_t>(cols, 1), out, s);
  int64_t chunk_len = ceil_div(ceil_div(cols, chunks), 4) * 4;
  chunks = ceil_div(cols, chunk_len);
  Workspace ws(s);
  uint32_t *pk, *pi;
  IVFPQ_TRY(ws.alloc(&pk, size_t(rows * chunks * k)));
  IVFPQ_TRY(ws.alloc(&pi, size_t(rows * chunks * k)));
  SelectOut part;
  part.kind = OutKind::Partial;
  part.pkeys = pk;
  part.pidx = pi;
  IVFPQ_TRY(select_rows(vals, rows, cols, k, chunks, chunk_len, part, s));
  const int64_t len = chunks * k;
  return select_pairs(pk, pi, rows, len, k, 1, len, out, s);
}

}  // namespace ivfpq

using namespace ivfpq;

extern "C" int kselect(const float* vals, int64_t rows, int64_t cols, int k, float* out_vals,
                       int64_t* out_idx, void* stream) {
  clear_error();
  IVFPQ_REQUIRE(rows >= 0 && cols >= 0, "kselect: negative size (rows=%lld, cols=%lld)",
                (long long)rows, (long long)cols);
  IVFPQ_REQUIRE(k >= 1 && k <= IVFPQ_MAX_K, "kselect: k=%d outside [1, %d]", k, IVFPQ_MAX_K);
  IVFPQ_REQUIRE(cols < int64_t(0xffffffffLL), "kselect: cols=%lld too large", (long long)cols);
  IVFPQ_REQUIRE(rows < (int64_t(1) << 31), "kselect: rows=%lld too large", (long long)rows);
  if (rows == 0) return IVFPQ_OK;
  IVFPQ_REQUIRE(out_vals && out_idx && (vals || cols == 0), "kselect: null pointer");
  SelectOut out;
  out.kind = OutKind::Float;
  out.vals = out_vals;
  out.idx64 = out_idx;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return kselect_device(vals, rows, cols, k, out, s);
}
