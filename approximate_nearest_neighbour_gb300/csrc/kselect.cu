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

namespace {

// Long rows, first level: one block of 16 warps per row.
//  1. A bound: a 4096-bin histogram of the top 12 key bits of the row's first
//     `sample` values (sample >= k). The bin holding the sample's k-th
//     smallest key ends at theta; at least k values of the row are <= theta,
//     so every value of the row's k smallest is <= theta as well.
//  2. Each warp streams its columns (thread t of the block takes float4 t,
//     t + 512, ... when the row is 16-byte aligned, single floats otherwise)
//     into a KW-entry WarpSelect that only sees keys <= theta, and writes its
//     sorted queue to pk/pi[row][warp].
template <int KW>
__global__ void __launch_bounds__(512)
row_short_kernel(const float* __restrict__ vals, int64_t cols, int64_t sample, int k,
                 uint32_t* __restrict__ pk, uint32_t* __restrict__ pi) {
  constexpr int T = ThreadQ<KW>::value;
  constexpr int kBins = 4096, kShift = 20, kPer = kBins / 512;
  __shared__ uint32_t hist[kBins];
  __shared__ uint32_t part[16];
  __shared__ uint32_t theta_s;
  const int64_t row = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float* rp = vals + row * cols;
  for (int b = threadIdx.x; b < kBins; b += 512) hist[b] = 0;
  if (threadIdx.x == 0) theta_s = kSentinelKey;
  __syncthreads();
  for (int64_t c = threadIdx.x; c < sample; c += 512)
    atomicAdd(&hist[float_to_key(__ldg(rp + c)) >> kShift], 1u);
  __syncthreads();
  {
    // the first bin at which the running count reaches k: kPer bins per
    // thread, a warp scan of the thread sums, then the warp totals
    uint32_t h[kPer], sum = 0;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      h[i] = hist[threadIdx.x * kPer + i];
      sum += h[i];
    }
    uint32_t inc = sum;
#pragma unroll
    for (int o = 1; o < 32; o *= 2) {
      const uint32_t v = __shfl_up_sync(kFullMask, inc, o);
      if (lane >= o) inc += v;
    }
    if (lane == 31) part[warp] = inc;
    __syncthreads();
    uint32_t run = inc - sum;
    for (int w = 0; w < warp; ++w) run += part[w];
    if (run < uint32_t(k) && run + sum >= uint32_t(k)) {
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        run += h[i];
        if (run >= uint32_t(k)) {
          const uint32_t b = threadIdx.x * kPer + i;
          theta_s = b == kBins - 1 ? kSentinelKey : ((b + 1) << kShift) - 1;
          break;
        }
      }
    }
  }
  __syncthreads();
  const uint32_t theta = theta_s;
  WarpSelect<KW, T> ws;
  ws.init(lane);
  const bool vec = (cols & 3) == 0 && (reinterpret_cast<uintptr_t>(vals) & 15) == 0;
  if (vec) {
    // Four float4 loads in flight per thread (a rotating buffer), one vote per
    // float4 against theta, and one insert site in the loop so that the
    // inlined queue merge is not copied.
    const float4* p4 = reinterpret_cast<const float4*>(rp);
    const int64_t n4 = cols >> 2;
    auto ld = [&](int64_t i4) {
      return i4 < n4 ? __ldcs(p4 + i4) : make_float4(0.f, 0.f, 0.f, 0.f);
    };
    float4 b0 = ld(threadIdx.x), b1 = ld(threadIdx.x + 512), b2 = ld(threadIdx.x + 1024),
           b3 = ld(threadIdx.x + 1536);
#pragma unroll 1
    for (int64_t i4 = threadIdx.x; i4 - threadIdx.x < n4; i4 += 512) {
      const float4 x = b0;
      b0 = b1;
      b1 = b2;
      b2 = b3;
      b3 = ld(i4 + 2048);
      const bool ok = i4 < n4;
      const uint32_t k0 = ok ? float_to_key(x.x) : kSentinelKey;
      const uint32_t k1 = ok ? float_to_key(x.y) : kSentinelKey;
      const uint32_t k2 = ok ? float_to_key(x.z) : kSentinelKey;
      const uint32_t k3 = ok ? float_to_key(x.w) : kSentinelKey;
      const uint32_t lo = min(min(k0, k1), min(k2, k3));
      if (__any_sync(kFullMask, ok && lo <= theta)) {
#pragma unroll 1
        for (int e = 0; e < 4; ++e) {
          const uint32_t key = e == 0 ? k0 : (e == 1 ? k1 : (e == 2 ? k2 : k3));
          ws.add(ok && key <= theta ? key : kSentinelKey, uint32_t(i4 * 4 + e));
        }
      }
    }
  } else {
#pragma unroll 1
    for (int64_t c = threadIdx.x; c - threadIdx.x < cols; c += 512) {
      const bool ok = c < cols;
      const uint32_t key = ok ? float_to_key(__ldcs(rp + c)) : kSentinelKey;
      if (__any_sync(kFullMask, ok && key <= theta))
        ws.add(ok && key <= theta ? key : kSentinelKey, uint32_t(c));
    }
  }
  ws.finalize();
  const int64_t o = (row * 16 + warp) * KW;
#pragma unroll
  for (int r = 0; r < KW / 32; ++r) {
    pk[o + 32 * r + lane] = ws.wk[r];
    pi[o + 32 * r + lane] = ws.wv[r];
  }
}

// flags[row] = 1 if the merged k best (tk, ascending) may miss an entry that
// a full short queue dropped (its last key not above the k-th).
template <int KW>
__global__ void row_short_check_kernel(const uint32_t* __restrict__ pk,
                                       const uint32_t* __restrict__ tk, int64_t rows, int k,
                                       int* __restrict__ flags) {
  const int64_t r = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (r >= rows) return;
  const uint32_t theta = tk[r * k + k - 1];
  int f = 0;
  for (int w = 0; w < 16; ++w) {
    const uint32_t last = pk[(r * 16 + w) * KW + KW - 1];
    f |= last != kSentinelKey && last <= theta;
  }
  flags[r] = f;
}

// Ascending (key, index) rows [rows][k] through the output writer.
__global__ void row_emit_kernel(const uint32_t* __restrict__ tk, const uint32_t* __restrict__ ti,
                                int64_t rows, int k, OutWriter out) {
  for (int64_t t = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; t < rows * k;
       t += int64_t(gridDim.x) * blockDim.x) {
    const int64_t r = t / k;
    out.write(r, 0, int(t - r * k), tk[t], ti[t]);
  }
}

// Selection over long rows with short queues: the first level above, the
// sorted-run merge of the 16 queues, and the full-length row kernel again for
// the rows a short queue may have cut (a warp's share of the k best is about
// k / 16, far below KW = max(32, K / 8)).
template <int KW>
int select_rows_short(const float* vals, int64_t rows, int64_t cols, int k, const SelectOut& out,
                      cudaStream_t s) {
  Workspace ws(s);
  uint32_t *pk = nullptr, *pi = nullptr, *tk = nullptr, *ti = nullptr;
  int* flags = nullptr;
  IVFPQ_TRY(ws.alloc(&pk, size_t(rows) * 16 * KW));
  IVFPQ_TRY(ws.alloc(&pi, size_t(rows) * 16 * KW));
  IVFPQ_TRY(ws.alloc(&tk, size_t(rows) * k));
  IVFPQ_TRY(ws.alloc(&ti, size_t(rows) * k));
  IVFPQ_TRY(ws.alloc(&flags, size_t(rows)));
  const int64_t sample = std::min<int64_t>(cols, std::max<int64_t>(8192, 16 * int64_t(k)));
  row_short_kernel<KW><<<unsigned(rows), 512, 0, s>>>(vals, cols, sample, k, pk, pi);
  IVFPQ_LAUNCHED();
  SelectOut part;
  part.kind = OutKind::Partial;
  part.pkeys = tk;
  part.pidx = ti;
  IVFPQ_TRY(merge_sorted_runs(pk, pi, rows, 16, KW, k, part, s));
  row_short_check_kernel<KW><<<unsigned(ceil_div(rows, 256)), 256, 0, s>>>(pk, tk, rows, k, flags);
  IVFPQ_LAUNCHED();
  row_emit_kernel<<<unsigned(std::min<int64_t>(ceil_div(rows * k, 256), 65535 * 8)), 256, 0, s>>>(
      tk, ti, rows, k, OutWriter{out, k, 1});
  IVFPQ_LAUNCHED();
  SelectOut ro = out;
  ro.row_mask = flags;
  return select_rows(vals, rows, cols, k, 1, cols, ro, s);
}

}  // namespace

int kselect_device(const float* vals, int64_t rows, int64_t cols, int k, const SelectOut& out,
                   cudaStream_t s) {
  if (rows == 0) return IVFPQ_OK;
  // Many long rows: short warp queues. Otherwise one pass when there are
  // enough rows to fill the GPU, else each row is cut into chunks whose
  // winners (k per chunk) are selected again.
  if (rows >= 4 * int64_t(num_sms()) && cols >= 32768 && cols < (int64_t(1) << 31) &&
      out.kind != OutKind::Partial && !out.row_mask) {
    switch (queue_len(k)) {
      case 32:
      case 64:
      case 128:
      case 256: return select_rows_short<32>(vals, rows, cols, k, out, s);
      case 512: return select_rows_short<64>(vals, rows, cols, k, out, s);
      case 1024: return select_rows_short<128>(vals, rows, cols, k, out, s);
      case 2048: return select_rows_short<256>(vals, rows, cols, k, out, s);
    }
  }
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
