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

// Long rows: one block of 16 warps per row.
//  1. A bound: a 4096-bin histogram of the top 12 key bits of the row's first
//     `sample` values (sample >= k) finds the bin holding the sample's k-th
//     smallest key; a second histogram, of the next 12 bits of the sample
//     keys in that bin, narrows it to a sub-bin of 256 keys, whose end is
//     theta. At least k values of the row are <= theta (the sample's k
//     smallest), so every value of the row's k smallest is <= theta as well,
//     and about k * cols / sample values pass.
//  2. The warps stream the row (thread t of the block takes float4 t, t + 512,
//     ... when the row is 16-byte aligned, single floats otherwise) and append
//     every key <= theta with its column to a shared buffer of `cap` entries
//     (per float4: a warp scan of the lanes' passing counts and one atomic per
//     warp).
//  3. One bitonic sort of the buffer; its first k entries are the result.
// There are at least k candidates (the sample's own). A row with more than
// `cap` writes nothing and sets flags[row] = 1 for the full-queue kernel.
__global__ void __launch_bounds__(512, 3)
row_cand_kernel(const float* __restrict__ vals, int64_t cols, int64_t sample, int k, int cap,
                OutWriter out, int* __restrict__ flags) {
  constexpr int kBins = 4096, kShift = 20, kSub = 8, kPer = kBins / 512;
  extern __shared__ uint32_t sm_cand[];
  uint32_t* hist = sm_cand;
  uint32_t* ck = sm_cand + kBins;
  uint32_t* ci = ck + cap;
  __shared__ uint32_t part[16];
  __shared__ uint32_t theta_s, count_s, bin_s, need_s;
  const int64_t row = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float* rp = vals + row * cols;
  for (int b = threadIdx.x; b < kBins; b += 512) hist[b] = 0;
  if (threadIdx.x == 0) {
    theta_s = kSentinelKey;
    count_s = 0;
    bin_s = kBins - 1;
    need_s = 0;
  }
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
        if (run + h[i] >= uint32_t(k)) {
          bin_s = threadIdx.x * kPer + i;
          need_s = uint32_t(k) - run;  // of the bin's sample keys, in order
          break;
        }
        run += h[i];
      }
    }
  }
  __syncthreads();
  const uint32_t bin = bin_s;
  if (bin == kBins - 1) {  // the top bin (NaN keys and the sentinel's): no bound
    if (threadIdx.x == 0) theta_s = kSentinelKey;
  } else {
    // the next 12 key bits of the sample keys in that bin
    for (int b = threadIdx.x; b < kBins; b += 512) hist[b] = 0;
    __syncthreads();
    for (int64_t c = threadIdx.x; c < sample; c += 512) {
      const uint32_t key = float_to_key(__ldg(rp + c));
      if ((key >> kShift) == bin) atomicAdd(&hist[(key >> kSub) & (kBins - 1)], 1u);
    }
    __syncthreads();
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
    const uint32_t need = need_s;
    if (run < need && run + sum >= need) {
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        run += h[i];
        if (run >= need) {
          const uint32_t sb = threadIdx.x * kPer + i;
          theta_s = (bin << kShift) | (sb << kSub) | ((1u << kSub) - 1u);
          break;
        }
      }
    }
  }
  __syncthreads();
  const uint32_t theta = theta_s;
  const uint32_t below = (1u << lane) - 1u;
  // append the lanes' keys <= theta: the warp's leader reserves the slots
  auto append = [&](bool pass, uint32_t key, uint32_t col) {
    const uint32_t bal = __ballot_sync(kFullMask, pass);
    if (bal == 0u) return;
    const int leader = __ffs(bal) - 1;
    uint32_t base = 0;
    if (lane == leader) base = atomicAdd(&count_s, uint32_t(__popc(bal)));
    base = __shfl_sync(kFullMask, base, leader);
    const uint32_t pos = base + uint32_t(__popc(bal & below));
    if (pass && pos < uint32_t(cap)) {
      ck[pos] = key;
      ci[pos] = col;
    }
  };
  const bool vec = (cols & 3) == 0 && (reinterpret_cast<uintptr_t>(vals) & 15) == 0;
  if (vec) {
    // four float4 loads in flight per thread (a ring of four, unrolled so
    // that no register moves between slots); one vote per float4 skips the
    // appends when no lane holds a key <= theta
    const float4* p4 = reinterpret_cast<const float4*>(rp);
    const int64_t n4 = cols >> 2;
    auto ld = [&](int64_t i4) {
      return i4 < n4 ? __ldcs(p4 + i4) : make_float4(0.f, 0.f, 0.f, 0.f);
    };
    float4 ring[4] = {ld(threadIdx.x), ld(threadIdx.x + 512), ld(threadIdx.x + 1024),
                      ld(threadIdx.x + 1536)};
#pragma unroll 1
    for (int64_t base = threadIdx.x; base - threadIdx.x < n4; base += 2048) {
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int64_t i4 = base + 512 * u;
        const float4 x = ring[u];
        ring[u] = ld(i4 + 2048);
        const bool ok = i4 < n4;
        const uint32_t k0 = float_to_key(x.x), k1 = float_to_key(x.y);
        const uint32_t k2 = float_to_key(x.z), k3 = float_to_key(x.w);
        const uint32_t pm = ok ? uint32_t(k0 <= theta) | (uint32_t(k1 <= theta) << 1) |
                                     (uint32_t(k2 <= theta) << 2) | (uint32_t(k3 <= theta) << 3)
                               : 0u;
        if (__any_sync(kFullMask, pm != 0u)) {
          // this lane's passing keys go to consecutive slots after those of
          // the lanes below it: an inclusive warp scan of the counts, one
          // atomic for the warp's total
          const uint32_t cnt = __popc(pm);
          uint32_t inc = cnt;
#pragma unroll
          for (int o = 1; o < 32; o *= 2) {
            const uint32_t v = __shfl_up_sync(kFullMask, inc, o);
            if (lane >= o) inc += v;
          }
          uint32_t bs = 0;
          if (lane == 31) bs = atomicAdd(&count_s, inc);
          uint32_t pos = __shfl_sync(kFullMask, bs, 31) + inc - cnt;
          const uint32_t c = uint32_t(i4 * 4);
          const uint32_t kk[4] = {k0, k1, k2, k3};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            if ((pm >> j) & 1u) {
              if (pos < uint32_t(cap)) {
                ck[pos] = kk[j];
                ci[pos] = c + j;
              }
              ++pos;
            }
          }
        }
      }
    }
  } else {
#pragma unroll 1
    for (int64_t c = threadIdx.x; c - threadIdx.x < cols; c += 512) {
      const bool ok = c < cols;
      const uint32_t key = ok ? float_to_key(__ldcs(rp + c)) : kSentinelKey;
      append(ok && key <= theta, key, uint32_t(c));
    }
  }
  __syncthreads();
  const uint32_t cnt = count_s;
  if (cnt > uint32_t(cap)) {  // block-uniform
    if (threadIdx.x == 0) flags[row] = 1;
    return;
  }
  if (threadIdx.x == 0) flags[row] = 0;
  uint32_t P = 1;
  while (P < cnt) P <<= 1;
  for (uint32_t i = cnt + threadIdx.x; i < P; i += 512) {
    ck[i] = kSentinelKey;
    ci[i] = kSentinelIdx;
  }
  __syncthreads();
  for (uint32_t size = 2; size <= P; size <<= 1) {
    for (uint32_t stride = size >> 1; stride > 0; stride >>= 1) {
      for (uint32_t t = threadIdx.x; t < P / 2; t += 512) {
        const uint32_t a = 2 * t - (t & (stride - 1));
        const uint32_t b = a + stride;
        const uint32_t ka = ck[a], kb = ck[b];
        if ((ka > kb) == ((a & size) == 0)) {
          const uint32_t va = ci[a];
          ck[a] = kb;
          ck[b] = ka;
          ci[a] = ci[b];
          ci[b] = va;
        }
      }
      __syncthreads();
    }
  }
  for (int i = threadIdx.x; i < k; i += 512)
    out.write(row, 0, i, uint32_t(i) < cnt ? ck[i] : kSentinelKey,
              uint32_t(i) < cnt ? ci[i] : kSentinelIdx);
}

// Selection over many long rows by a bound and a candidate buffer (above);
// the full-length row kernel redoes the rows whose buffer overflowed.
int select_rows_cand(const float* vals, int64_t rows, int64_t cols, int k, const SelectOut& out,
                     cudaStream_t s) {
  constexpr int kMaxCap = 16384;
  const int64_t sample = std::min<int64_t>(cols / 2, std::max<int64_t>(16384, 32 * int64_t(k)));
  const int64_t expect = ceil_div(int64_t(k) * cols, sample);
  int cap = 1024;
  while (cap < 2 * expect + 512 && cap < kMaxCap) cap *= 2;
  const size_t smem = (size_t(4096) + 2 * size_t(cap)) * 4;
  IVFPQ_TRY(set_dynamic_smem(row_cand_kernel, smem));
  Workspace ws(s);
  int* flags = nullptr;
  IVFPQ_TRY(ws.alloc(&flags, size_t(rows)));
  row_cand_kernel<<<unsigned(rows), 512, smem, s>>>(vals, cols, sample, k, cap,
                                                    OutWriter{out, k, 1}, flags);
  IVFPQ_LAUNCHED_K(row_cand_kernel, smem, 512);
  SelectOut ro = out;
  ro.row_mask = flags;
  return select_rows(vals, rows, cols, k, 1, cols, ro, s);
}

}  // namespace

int kselect_device(const float* vals, int64_t rows, int64_t cols, int k, const SelectOut& out,
                   cudaStream_t s) {
  if (rows == 0) return IVFPQ_OK;
  // Many long rows: a bound and a candidate buffer. Otherwise one pass when there are
  // enough rows to fill the GPU, else each row is cut into chunks whose
  // winners (k per chunk) are selected again.
  if (rows >= 4 * int64_t(num_sms()) && cols >= 32768 && cols < (int64_t(1) << 31) &&
      out.kind != OutKind::Partial && !out.row_mask) {
    return select_rows_cand(vals, rows, cols, k, out, s);
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
