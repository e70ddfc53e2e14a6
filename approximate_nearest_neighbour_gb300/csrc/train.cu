// Index preparation on the GPU: Lloyd k-means (coarse quantizer and product
// quantizer training) and the batched IVF-PQ encoder.
//
// Source: "Billion-scale similarity search with GPUs", section 6 (k-means by
// alternating a k = 1 nearest-centroid search and a centroid update; the same
// machinery encodes a database); "Custom 8-bit floating point value format
// ...", index construction steps 1-3 (coarse centroids, residuals, product
// quantizer codebooks of 256 codewords per sub-space, nearest-codeword codes).
//
// Choices: the assignment is the tensor-core k-nearest-neighbour path with
// k = 1 (ties of equal distance go to either centroid); the update sums each
// cluster's members in increasing point order in fp64 (a stable radix sort by
// cluster first), so it is deterministic; an empty cluster keeps its centroid;
// the objective of an assignment pass is the fp64 sum of the exact fp32
// squared distances.
#include <cub/cub.cuh>

#include <algorithm>
#include <vector>

#include "internal.h"

namespace ivfpq {
namespace {

unsigned grid1(int64_t n, int threads) {
  return unsigned(std::max<int64_t>(1, std::min<int64_t>(ceil_div(n, threads), 65535 * 8)));
}

// c[e] = x[init[e]] for e < k (rows of a [n, ldx] matrix, d columns from col0)
__global__ void seed_kernel(const float* __restrict__ x, int64_t ldx, int col0, int d,
                            const int64_t* __restrict__ init, int k, int64_t n,
                            float* __restrict__ c, int* __restrict__ bad) {
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < int64_t(k) * d;
       i += int64_t(gridDim.x) * blockDim.x) {
    const int64_t e = i / d;
    const int t = int(i - e * d);
    const int64_t r = init[e];
    if (r < 0 || r >= n) {
      atomicOr(bad, 1);
      continue;
    }
    c[i] = x[r * ldx + col0 + t];
  }
}

// y[i][t] = x[i][col0 + t] for t < d (a contiguous copy of some columns)
__global__ void columns_kernel(const float* __restrict__ x, int64_t n, int64_t ldx, int col0,
                               int d, float* __restrict__ y) {
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n * d;
       i += int64_t(gridDim.x) * blockDim.x) {
    const int64_t r = i / d;
    y[i] = x[r * ldx + col0 + int(i - r * d)];
  }
}

// assignment index (int64 from the selection) -> int32 key, point index,
// fp64 copy of the distance; a row the selection left without a centroid (-1:
// no finite distance, e.g. a non-finite row) gets key k, past every cluster
__global__ void assign_prep_kernel(const int64_t* __restrict__ idx, const float* __restrict__ dist,
                                   int64_t n, int k, int32_t* __restrict__ key,
                                   int32_t* __restrict__ pt, double* __restrict__ dd) {
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += int64_t(gridDim.x) * blockDim.x) {
    const int64_t c = idx[i];
    key[i] = (c >= 0 && c < k) ? int32_t(c) : k;
    pt[i] = int32_t(i);
    dd[i] = double(dist[i]);
  }
}

// the final assignment: cluster, or -1 where the selection found none
__global__ void assign_out_kernel(const int64_t* __restrict__ idx, int64_t n, int k,
                                  int32_t* __restrict__ out) {
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += int64_t(gridDim.x) * blockDim.x) {
    const int64_t c = idx[i];
    out[i] = (c >= 0 && c < k) ? int32_t(c) : -1;
  }
}

// [start, end) of each cluster in the sorted keys (untouched clusters stay
// at the zero-filled [0, 0); key k, the rows without a centroid, has none)
__global__ void bounds_kernel(const int32_t* __restrict__ sk, int64_t n, int k,
                              int32_t* __restrict__ beg, int32_t* __restrict__ end) {
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += int64_t(gridDim.x) * blockDim.x) {
    const int32_t c = sk[i];
    if (c < 0 || c >= k) continue;
    if (i == 0 || sk[i - 1] != c) beg[c] = int32_t(i);
    if (i == n - 1 || sk[i + 1] != c) end[c] = int32_t(i + 1);
  }
}

// centroid c = mean of its members (fp64 sum in increasing point order);
// empty clusters keep theirs. One block per cluster.
__global__ void update_kernel(const float* __restrict__ x, int64_t ldx, int col0, int d,
                              const int32_t* __restrict__ spt, const int32_t* __restrict__ beg,
                              const int32_t* __restrict__ end, float* __restrict__ cent) {
  const int c = blockIdx.x;
  const int b = beg[c], e = end[c];
  if (e <= b) return;
  for (int t = threadIdx.x; t < d; t += blockDim.x) {
    double s = 0.0;
    for (int i = b; i < e; ++i) s += double(x[int64_t(spt[i]) * ldx + col0 + t]);
    cent[int64_t(c) * d + t] = float(s / double(e - b));
  }
}

// codes[i][j] = argmin_e ||x_i^(j) - c_{l_i}^(j) - y_j(e)||^2 (fp32, direct
// form, lowest e on ties); codebooks_t is [256][m][dsub4]. One thread per (i, j).
__global__ void encode_kernel(const float* __restrict__ x, int64_t n, int d, int m, int dsub,
                              int dsub4, const float* __restrict__ cent, int nlist,
                              const int32_t* __restrict__ lists,
                              const float* __restrict__ cb_t, uint8_t* __restrict__ codes) {
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n * m;
       i += int64_t(gridDim.x) * blockDim.x) {
    const int64_t r = i / m;
    const int j = int(i - r * m);
    const int l = lists[r];
    if (l < 0 || l >= nlist) {  // no centroid (a non-finite row): code 0
      codes[i] = 0;
      continue;
    }
    const float* xr = x + r * d + j * dsub;
    const float* cr = cent + int64_t(l) * d + j * dsub;
    float res[32];
    for (int t = 0; t < dsub; ++t) res[t] = xr[t] - cr[t];
    float best = INFINITY;
    int bi = 0;
    for (int e = 0; e < 256; ++e) {
      const float* y = cb_t + (int64_t(e) * m + j) * dsub4;
      float s = 0.f;
      for (int t = 0; t < dsub; ++t) {
        const float df = res[t] - y[t];
        s = fmaf(df, df, s);
      }
      if (s < best) {
        best = s;
        bi = e;
      }
    }
    codes[i] = uint8_t(bi);
  }
}

// r[i] = x[i] - c[lists[i]] (rows of d floats)
__global__ void residual_kernel(const float* __restrict__ x, int64_t n, int d,
                                const float* __restrict__ cent, int nlist,
                                const int32_t* __restrict__ lists, float* __restrict__ r) {
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n * d;
       i += int64_t(gridDim.x) * blockDim.x) {
    const int64_t row = i / d;
    const int l = lists[row];
    // no centroid (list -1: a non-finite row): NaN residual
    r[i] = (l >= 0 && l < nlist) ? x[i] - cent[int64_t(l) * d + int(i - row * d)] : NAN;
  }
}

// Lower bound of each centroid's squared distance to its nearest other
// centroid, from the two nearest centroids of every centroid (k = 2 search of
// the centroids among themselves; one of the two is the centroid itself).
// The search selects on tensor-core distances whose error is below
// 2^-22 (|c|^2 + |c'|^2) and returns the direct-form fp32 distance of what it
// selected, so the true separation is at least the returned one minus
// 2^-21 (|c|^2 + max |c'|^2) and a relative rounding term; the bound
// subtracts eight times that (2^-18) and 1e-4 relative.
__global__ void separation_kernel(const float* __restrict__ d2, const int64_t* __restrict__ i2,
                                  int nlist, const float* __restrict__ norms,
                                  const float* __restrict__ max_norm, float* __restrict__ sep) {
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= nlist) return;
  const float s2 = i2[2 * int64_t(c)] == c ? d2[2 * int64_t(c) + 1] : d2[2 * int64_t(c)];
  const float margin = 0x1p-18f * (norms[c] + *max_norm);
  sep[c] = fmaxf(0.f, s2 * (1.f - 1e-4f) - margin);
}

// Hint check, one warp per row: the hint h is x's nearest centroid, and the
// only one, if 4 ||x - c_h||^2 < sep[h] (the triangle inequality: for any
// other centroid c, ||x - c|| >= ||c_h - c|| - ||x - c_h|| > ||x - c_h||;
// Elkan, "Using the triangle inequality to accelerate k-means", ICML 2003,
// Lemma 1). Writes the hint as the list of a row that passes and flags the
// others (need[r] = 1) for a full search.
__global__ void hint_check_kernel(const float* __restrict__ x, int64_t n, int d,
                                  const float* __restrict__ cent, int nlist,
                                  const float* __restrict__ sep, const int32_t* __restrict__ hint,
                                  int32_t* __restrict__ lists, int* __restrict__ need) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = int64_t(gridDim.x) * (blockDim.x >> 5);
  for (int64_t r = int64_t(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); r < n;
       r += warps) {
    const int h = hint[r];
    bool pass = false;
    if (h >= 0 && h < nlist) {
      const float* xr = x + r * d;
      const float* cr = cent + int64_t(h) * d;
      float a = 0.f;
      for (int t = lane; t < d; t += 32) {
        const float df = xr[t] - cr[t];
        a = fmaf(df, df, a);
      }
#pragma unroll
      for (int o = 16; o >= 1; o /= 2) a += __shfl_xor_sync(kFullMask, a, o);
      pass = 4.f * a * (1.f + 1e-4f) < sep[h];
    }
    if (lane == 0) {
      lists[r] = pass ? h : -1;
      need[r] = pass ? 0 : 1;
    }
  }
}

// rows[pos[i]] = i for the flagged rows (pos = exclusive prefix sum of need)
__global__ void compact_kernel(const int* __restrict__ need, const int* __restrict__ pos,
                               int64_t n, int32_t* __restrict__ rows) {
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += int64_t(gridDim.x) * blockDim.x)
    if (need[i]) rows[pos[i]] = int32_t(i);
}

// y[i] = x[rows[i]] (rows of d floats)
__global__ void gather_rows_kernel(const float* __restrict__ x, int d,
                                   const int32_t* __restrict__ rows, int64_t cnt,
                                   float* __restrict__ y) {
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < cnt * d;
       i += int64_t(gridDim.x) * blockDim.x) {
    const int64_t r = i / d;
    y[i] = x[int64_t(rows[r]) * d + int(i - r * d)];
  }
}

// lists[rows[i]] = found[i]
__global__ void scatter_lists_kernel(const int32_t* __restrict__ rows,
                                     const int32_t* __restrict__ found, int64_t cnt,
                                     int32_t* __restrict__ lists) {
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < cnt;
       i += int64_t(gridDim.x) * blockDim.x)
    lists[rows[i]] = found[i];
}

}  // namespace

namespace {

// Lloyd iterations on a contiguous [n, d] matrix y: c [k, d] holds the
// initial centroids and receives the trained ones. obj (host, niter + 1, may
// be null) receives the objective of each assignment pass; assign_out (may
// be null) the final assignment.
int lloyd(const float* y, int64_t n, int d, int k, int niter, float* c, int32_t* assign_out,
          double* obj, cudaStream_t s) {
  Workspace ws(s);
  float* dist = nullptr;
  int64_t* idx = nullptr;
  int32_t *key = nullptr, *pt = nullptr, *skey = nullptr, *spt = nullptr;
  int32_t *beg = nullptr, *end = nullptr;
  double *dd = nullptr, *dsum = nullptr;
  IVFPQ_TRY(ws.alloc(&dist, size_t(n)));
  IVFPQ_TRY(ws.alloc(&idx, size_t(n)));
  IVFPQ_TRY(ws.alloc(&key, size_t(n)));
  IVFPQ_TRY(ws.alloc(&pt, size_t(n)));
  IVFPQ_TRY(ws.alloc(&skey, size_t(n)));
  IVFPQ_TRY(ws.alloc(&spt, size_t(n)));
  IVFPQ_TRY(ws.alloc(&beg, size_t(k)));
  IVFPQ_TRY(ws.alloc(&end, size_t(k)));
  IVFPQ_TRY(ws.alloc(&dd, size_t(n)));
  IVFPQ_TRY(ws.alloc(&dsum, 1));
  int end_bit = 1;  // keys 0 .. k (k: no centroid)
  while ((int64_t(1) << end_bit) < int64_t(k) + 1) ++end_bit;
  size_t sort_bytes = 0, red_bytes = 0;
  IVFPQ_CUDA(cub::DeviceRadixSort::SortPairs(nullptr, sort_bytes, key, skey, pt, spt, n, 0,
                                             end_bit, s));
  IVFPQ_CUDA(cub::DeviceReduce::Sum(nullptr, red_bytes, dd, dsum, n, s));
  uint8_t *sort_tmp = nullptr, *red_tmp = nullptr;
  IVFPQ_TRY(ws.alloc(&sort_tmp, sort_bytes));
  IVFPQ_TRY(ws.alloc(&red_tmp, red_bytes));
  SelectOut o;
  o.kind = OutKind::Float;
  o.vals = dist;
  o.idx64 = idx;
  for (int it = 0; it <= niter; ++it) {
    IVFPQ_TRY(knn_by_tiles(y, n, c, k, d, 1, o, s));
    assign_prep_kernel<<<grid1(n, 256), 256, 0, s>>>(idx, dist, n, k, key, pt, dd);
    IVFPQ_LAUNCHED();
    if (obj) {
      IVFPQ_CUDA(cub::DeviceReduce::Sum(red_tmp, red_bytes, dd, dsum, n, s));
      IVFPQ_CUDA(cudaMemcpyAsync(obj + it, dsum, sizeof(double), cudaMemcpyDeviceToHost, s));
      IVFPQ_CUDA(cudaStreamSynchronize(s));
    }
    if (it == niter) {
      if (assign_out) {
        assign_out_kernel<<<grid1(n, 256), 256, 0, s>>>(idx, n, k, assign_out);
        IVFPQ_LAUNCHED();
      }
      break;
    }
    IVFPQ_CUDA(cub::DeviceRadixSort::SortPairs(sort_tmp, sort_bytes, key, skey, pt, spt, n, 0,
                                               end_bit, s));
    IVFPQ_CUDA(cudaMemsetAsync(beg, 0, size_t(k) * sizeof(int32_t), s));
    IVFPQ_CUDA(cudaMemsetAsync(end, 0, size_t(k) * sizeof(int32_t), s));
    bounds_kernel<<<grid1(n, 256), 256, 0, s>>>(skey, n, k, beg, end);
    IVFPQ_LAUNCHED();
    update_kernel<<<unsigned(k), 128, 0, s>>>(y, d, 0, d, spt, beg, end, c);
    IVFPQ_LAUNCHED();
  }
  return IVFPQ_OK;
}

// Seeds rows of c from x[init[e]] (columns col0 .. col0 + d); INVALID_ARG if
// an index is outside [0, n).
int seed(const float* x, int64_t ldx, int col0, int d, const int64_t* init, int k, int64_t n,
         float* c, cudaStream_t s) {
  Workspace ws(s);
  int* bad = nullptr;
  IVFPQ_TRY(ws.alloc(&bad, 1));
  IVFPQ_CUDA(cudaMemsetAsync(bad, 0, sizeof(int), s));
  seed_kernel<<<grid1(int64_t(k) * d, 256), 256, 0, s>>>(x, ldx, col0, d, init, k, n, c, bad);
  IVFPQ_LAUNCHED();
  int h = 0;
  IVFPQ_CUDA(cudaMemcpyAsync(&h, bad, sizeof(int), cudaMemcpyDeviceToHost, s));
  IVFPQ_CUDA(cudaStreamSynchronize(s));
  IVFPQ_REQUIRE(!h, "initial centroid index outside [0, %lld)", (long long)n);
  return IVFPQ_OK;
}

}  // namespace
}  // namespace ivfpq

using namespace ivfpq;

extern "C" int kmeans_lloyd(const float* x, int64_t n, int d, int k, int niter,
                            const int64_t* init, float* centroids, int32_t* assign,
                            double* objective, void* stream) {
  clear_error();
  IVFPQ_REQUIRE(d >= 1 && k >= 1 && niter >= 0, "kmeans_lloyd: bad sizes (d=%d k=%d niter=%d)",
                d, k, niter);
  IVFPQ_REQUIRE(n >= k && n < (int64_t(1) << 31), "kmeans_lloyd: need k <= n < 2^31 (n=%lld)",
                (long long)n);
  IVFPQ_REQUIRE(k <= (1 << 24), "kmeans_lloyd: k=%d above 2^24", k);
  IVFPQ_REQUIRE(x && init && centroids, "kmeans_lloyd: null pointer");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  IVFPQ_TRY(seed(x, d, 0, d, init, k, n, centroids, s));
  return lloyd(x, n, d, k, niter, centroids, assign, objective, s);
}

extern "C" int pq_train(const float* x, int64_t n, int d, int m, int niter, const int64_t* init,
                        float* codebooks, double* objective, void* stream) {
  clear_error();
  IVFPQ_REQUIRE(d >= 1 && m >= 1 && d % m == 0 && niter >= 0,
                "pq_train: bad sizes (d=%d m=%d niter=%d)", d, m, niter);
  IVFPQ_REQUIRE(n >= 256 && n < (int64_t(1) << 31), "pq_train: need 256 <= n < 2^31 (n=%lld)",
                (long long)n);
  IVFPQ_REQUIRE(x && init && codebooks, "pq_train: null pointer");
  const int dsub = d / m;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Workspace ws(s);
  float* y = nullptr;
  IVFPQ_TRY(ws.alloc(&y, size_t(n) * dsub));
  std::vector<double> part(size_t(niter) + 1);
  if (objective)
    for (int i = 0; i <= niter; ++i) objective[i] = 0.0;
  for (int j = 0; j < m; ++j) {
    columns_kernel<<<grid1(n * dsub, 256), 256, 0, s>>>(x, n, d, j * dsub, dsub, y);
    IVFPQ_LAUNCHED();
    float* cj = codebooks + int64_t(j) * 256 * dsub;
    IVFPQ_TRY(seed(x, d, j * dsub, dsub, init, 256, n, cj, s));
    IVFPQ_TRY(lloyd(y, n, dsub, 256, niter, cj, nullptr, objective ? part.data() : nullptr, s));
    if (objective)
      for (int i = 0; i <= niter; ++i) objective[i] += part[i];
  }
  return IVFPQ_OK;
}

extern "C" int ivfpq_encode(const ivfpq_index* ix, const float* x, int64_t n, int32_t* list_ids,
                            uint8_t* codes, void* stream) {
  clear_error();
  IVFPQ_REQUIRE(ix, "ivfpq_encode: null index");
  IVFPQ_REQUIRE(n >= 0 && n < (int64_t(1) << 31), "ivfpq_encode: n=%lld", (long long)n);
  IVFPQ_REQUIRE(ix->dsub <= 32, "ivfpq_encode: d/m=%d above 32", ix->dsub);
  if (n == 0) return IVFPQ_OK;
  IVFPQ_REQUIRE(x && list_ids && codes, "ivfpq_encode: null pointer");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  SelectOut o;
  o.kind = OutKind::Probes;
  o.idx32 = list_ids;
  TcOperand xo;
  xo.hi = ix->cent_hi;
  xo.lo = ix->cent_lo;
  xo.norms = ix->cent_norms;
  IVFPQ_TRY(knn_by_tiles(x, n, ix->centroids, ix->nlist, ix->d, 1, o, s,
                         ix->cent_hi ? &xo : nullptr));
  encode_kernel<<<grid1(n * ix->m, 256), 256, 0, s>>>(x, n, ix->d, ix->m, ix->dsub, ix->dsub4,
                                                      ix->centroids, ix->nlist, list_ids,
                                                      ix->codebooks, codes);
  IVFPQ_LAUNCHED();
  return IVFPQ_OK;
}

namespace ivfpq {
namespace {

// The separation bounds of the index's centroids (computed once).
int centroid_separation(const ivfpq_index* cix, cudaStream_t s) {
  auto* ix = const_cast<ivfpq_index*>(cix);
  std::lock_guard<std::mutex> lock(ix->sep_mutex);
  if (ix->cent_sep) return IVFPQ_OK;
  const int nlist = ix->nlist;
  float* sep = nullptr;
  IVFPQ_CUDA(cudaMalloc(&sep, size_t(nlist) * sizeof(float)));
  struct Guard {
    float*& p;
    ~Guard() {
      if (p) cudaFree(p);
    }
  } guard{sep};
  if (nlist == 1) {
    const float inf = INFINITY;
    IVFPQ_CUDA(cudaMemcpyAsync(sep, &inf, sizeof(float), cudaMemcpyHostToDevice, s));
  } else {
    Workspace ws(s);
    float* d2 = nullptr;
    int64_t* i2 = nullptr;
    float* mx = nullptr;
    IVFPQ_TRY(ws.alloc(&d2, size_t(nlist) * 2));
    IVFPQ_TRY(ws.alloc(&i2, size_t(nlist) * 2));
    IVFPQ_TRY(ws.alloc(&mx, 1));
    SelectOut o;
    o.kind = OutKind::Float;
    o.vals = d2;
    o.idx64 = i2;
    TcOperand xo;
    xo.hi = ix->cent_hi;
    xo.lo = ix->cent_lo;
    xo.norms = ix->cent_norms;
    IVFPQ_TRY(knn_by_tiles(ix->centroids, nlist, ix->centroids, nlist, ix->d, 2, o, s,
                           ix->cent_hi ? &xo : nullptr));
    size_t red_bytes = 0;
    IVFPQ_CUDA(cub::DeviceReduce::Max(nullptr, red_bytes, ix->cent_norms, mx, nlist, s));
    uint8_t* red_tmp = nullptr;
    IVFPQ_TRY(ws.alloc(&red_tmp, red_bytes));
    IVFPQ_CUDA(cub::DeviceReduce::Max(red_tmp, red_bytes, ix->cent_norms, mx, nlist, s));
    separation_kernel<<<unsigned(ceil_div(nlist, 256)), 256, 0, s>>>(d2, i2, nlist,
                                                                     ix->cent_norms, mx, sep);
    IVFPQ_LAUNCHED();
  }
  IVFPQ_CUDA(cudaStreamSynchronize(s));
  ix->cent_sep = sep;
  sep = nullptr;
  return IVFPQ_OK;
}

}  // namespace
}  // namespace ivfpq

extern "C" int ivfpq_residuals(const float* centroids, int nlist, int d, const float* x, int64_t n,
                               int32_t* list_ids, float* residuals, void* stream) {
  clear_error();
  IVFPQ_REQUIRE(d >= 1 && nlist >= 1, "ivfpq_residuals: bad sizes (d=%d nlist=%d)", d, nlist);
  IVFPQ_REQUIRE(n >= 0 && n < (int64_t(1) << 31), "ivfpq_residuals: n=%lld", (long long)n);
  if (n == 0) return IVFPQ_OK;
  IVFPQ_REQUIRE(centroids && x && list_ids && residuals, "ivfpq_residuals: null pointer");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  SelectOut o;
  o.kind = OutKind::Probes;
  o.idx32 = list_ids;
  IVFPQ_TRY(knn_by_tiles(x, n, centroids, nlist, d, 1, o, s));
  residual_kernel<<<grid1(n * d, 256), 256, 0, s>>>(x, n, d, centroids, nlist, list_ids,
                                                   residuals);
  IVFPQ_LAUNCHED();
  return IVFPQ_OK;
}

extern "C" int ivfpq_encode_hinted(const ivfpq_index* ix, const float* x, int64_t n,
                                   const int32_t* hint, int32_t* list_ids, uint8_t* codes,
                                   int64_t* n_searched, void* stream) {
  clear_error();
  IVFPQ_REQUIRE(ix, "ivfpq_encode_hinted: null index");
  IVFPQ_REQUIRE(n >= 0 && n < (int64_t(1) << 31), "ivfpq_encode_hinted: n=%lld", (long long)n);
  IVFPQ_REQUIRE(ix->dsub <= 32, "ivfpq_encode_hinted: d/m=%d above 32", ix->dsub);
  if (n_searched) *n_searched = 0;
  if (n == 0) return IVFPQ_OK;
  IVFPQ_REQUIRE(x && hint && list_ids && codes, "ivfpq_encode_hinted: null pointer");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  IVFPQ_TRY(centroid_separation(ix, s));
  Workspace ws(s);
  int *need = nullptr, *pos = nullptr;
  IVFPQ_TRY(ws.alloc(&need, size_t(n)));
  IVFPQ_TRY(ws.alloc(&pos, size_t(n)));
  hint_check_kernel<<<grid1(n * 32, 256), 256, 0, s>>>(x, n, ix->d, ix->centroids, ix->nlist,
                                                        ix->cent_sep, hint, list_ids, need);
  IVFPQ_LAUNCHED();
  size_t scan_bytes = 0;
  IVFPQ_CUDA(cub::DeviceScan::ExclusiveSum(nullptr, scan_bytes, need, pos, n, s));
  uint8_t* scan_tmp = nullptr;
  IVFPQ_TRY(ws.alloc(&scan_tmp, scan_bytes));
  IVFPQ_CUDA(cub::DeviceScan::ExclusiveSum(scan_tmp, scan_bytes, need, pos, n, s));
  int tail[2] = {0, 0};
  IVFPQ_CUDA(cudaMemcpyAsync(&tail[0], pos + n - 1, sizeof(int), cudaMemcpyDeviceToHost, s));
  IVFPQ_CUDA(cudaMemcpyAsync(&tail[1], need + n - 1, sizeof(int), cudaMemcpyDeviceToHost, s));
  IVFPQ_CUDA(cudaStreamSynchronize(s));
  const int64_t cnt = int64_t(tail[0]) + tail[1];
  if (cnt > 0) {
    // the rows whose hint could not be confirmed: a full nearest-centroid search
    int32_t *rows = nullptr, *found = nullptr;
    float* y = nullptr;
    IVFPQ_TRY(ws.alloc(&rows, size_t(cnt)));
    IVFPQ_TRY(ws.alloc(&found, size_t(cnt)));
    IVFPQ_TRY(ws.alloc(&y, size_t(cnt) * ix->d));
    compact_kernel<<<grid1(n, 256), 256, 0, s>>>(need, pos, n, rows);
    IVFPQ_LAUNCHED();
    gather_rows_kernel<<<grid1(cnt * ix->d, 256), 256, 0, s>>>(x, ix->d, rows, cnt, y);
    IVFPQ_LAUNCHED();
    SelectOut o;
    o.kind = OutKind::Probes;
    o.idx32 = found;
    TcOperand xo;
    xo.hi = ix->cent_hi;
    xo.lo = ix->cent_lo;
    xo.norms = ix->cent_norms;
    IVFPQ_TRY(knn_by_tiles(y, cnt, ix->centroids, ix->nlist, ix->d, 1, o, s,
                           ix->cent_hi ? &xo : nullptr));
    scatter_lists_kernel<<<grid1(cnt, 256), 256, 0, s>>>(rows, found, cnt, list_ids);
    IVFPQ_LAUNCHED();
  }
  encode_kernel<<<grid1(n * ix->m, 256), 256, 0, s>>>(x, n, ix->d, ix->m, ix->dsub, ix->dsub4,
                                                      ix->centroids, ix->nlist, list_ids,
                                                      ix->codebooks, codes);
  IVFPQ_LAUNCHED();
  if (n_searched) *n_searched = cnt;
  return IVFPQ_OK;
}
