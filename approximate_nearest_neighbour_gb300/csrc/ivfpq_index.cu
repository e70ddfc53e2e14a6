// IVF-PQ index storage: creation, the interleaved inverted-list layout and
// ivfpq_add, plus small index-level entry points.
//
// Source: IVFPQ build step 4 ("Custom 8-bit floating point value format for
// reducing shared memory bank conflict in approximate nearest neighbor
// search": store the list of each vector and its PQ code) and the list
// representation of "Billion-scale similarity search with GPUs", section 5
// (codes kept as sequential groups of b bytes per vector within lists).
//
// Layout used here (differs from the sequential groups on purpose): each list
// owns whole blocks of 32 vector slots. Inside a block the m code bytes of the
// vector in slot i are stored as 16-byte chunks, chunk c of all 32 slots
// together ([c][slot][16 bytes]); when m is not a multiple of 16 the remaining
// m % 16 bytes follow as [slot][m % 16 bytes]. So one 128-bit load per lane
// fetches a chunk for a whole warp with full coalescing. The bytes are also
// rotated per slot: sub-quantizers are grouped by 32 (group g covers
// [32g, 32g + gs)), and stored byte 32g + s of slot i holds code byte
// 32g + (i + s) mod gs. At scan step s lane i then reads sub-quantizer table
// (i + s) mod gs, so the 32 lanes of a warp read 32 different tables at
// every step (see scan.cuh for why that removes bank conflicts).
#include <cub/cub.cuh>

#include <algorithm>
#include <cstring>

#include "internal.h"
#include "layout.cuh"

namespace ivfpq {
namespace {

__global__ void cent_norms_kernel(const float* __restrict__ c, int64_t nlist, int d,
                                  float* __restrict__ out) {
  const int64_t l = int64_t(blockIdx.x) * blockDim.y + threadIdx.y;
  if (l >= nlist) return;
  float s = 0.f;
  for (int t = threadIdx.x; t < d; t += 32) {
    const float v = c[l * d + t];
    s = fmaf(v, v, s);
  }
#pragma unroll
  for (int o = 16; o >= 1; o /= 2) s += __shfl_xor_sync(kFullMask, s, o);
  if (threadIdx.x == 0) out[l] = s;
}

// [m][256][dsub] (input) -> [256][m][dsub4] (internal), dsub4 = dsub rounded
// up to a multiple of 4 with zero padding: reading the codewords of one
// reproduction value for consecutive sub-quantizers is then contiguous and
// can use 128-bit loads.
__global__ void transpose_codebooks_kernel(const float* __restrict__ in, int m, int dsub,
                                           int dsub4, float* __restrict__ out) {
  const int64_t n = int64_t(m) * 256 * dsub4;
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += int64_t(gridDim.x) * blockDim.x) {
    const int t = int(i % dsub4);
    const int64_t ej = i / dsub4;
    const int j = int(ej % m), e = int(ej / m);
    out[i] = t < dsub ? in[(int64_t(j) * 256 + e) * dsub + t] : 0.f;
  }
}

__global__ void histogram_kernel(const int32_t* __restrict__ list_ids, int64_t n, int nlist,
                                 int32_t* __restrict__ counts, int32_t* __restrict__ bad) {
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += int64_t(gridDim.x) * blockDim.x) {
    const int32_t l = list_ids[i];
    if (l < 0 || l >= nlist) {
      atomicOr(bad, 1);
    } else {
      // one atomic per distinct list among the active lanes of the warp
      const unsigned peers = __match_any_sync(__activemask(), l);
      if ((__ffs(peers) - 1) == int(threadIdx.x & 31)) atomicAdd(counts + l, __popc(peers));
    }
  }
}

__global__ void new_sizes_kernel(const int32_t* __restrict__ old_len,
                                 const int32_t* __restrict__ counts, int nlist,
                                 int32_t* __restrict__ new_len, int64_t* __restrict__ nblk) {
  for (int l = blockIdx.x * blockDim.x + threadIdx.x; l < nlist; l += gridDim.x * blockDim.x) {
    const int32_t len = old_len[l] + counts[l];
    new_len[l] = len;
    nblk[l] = (len + 31) / 32;
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) nblk[nlist] = 0;
}

// Copies every list's old blocks (codes and ids) to the list's new position.
__global__ void copy_lists_kernel(const int64_t* __restrict__ old_off,
                                  const int64_t* __restrict__ new_off,
                                  const uint8_t* __restrict__ old_codes,
                                  const int64_t* __restrict__ old_ids, uint8_t* __restrict__ codes,
                                  int64_t* __restrict__ ids, int m) {
  const int l = blockIdx.x;
  const int64_t b0 = old_off[l], nb = old_off[l + 1] - b0, nb0 = new_off[l];
  const int64_t n16 = nb * 32 * m / 16;
  const uint4* src = reinterpret_cast<const uint4*>(old_codes + b0 * 32 * m);
  uint4* dst = reinterpret_cast<uint4*>(codes + nb0 * 32 * m);
  for (int64_t i = threadIdx.x; i < n16; i += blockDim.x) dst[i] = src[i];
  for (int64_t i = threadIdx.x; i < nb * 32; i += blockDim.x)
    ids[nb0 * 32 + i] = old_ids[b0 * 32 + i];
}

// Places the i-th vector of the list-sorted order into its slot.
__global__ void scatter_kernel(const int32_t* __restrict__ sorted_list,
                               const int32_t* __restrict__ sorted_row, int64_t n,
                               const int32_t* __restrict__ old_len,
                               const int32_t* __restrict__ seg_start,
                               const int64_t* __restrict__ new_off,
                               const uint8_t* __restrict__ codes_in,
                               const int64_t* __restrict__ ids_in, uint8_t* __restrict__ codes,
                               int64_t* __restrict__ ids, int m) {
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += int64_t(gridDim.x) * blockDim.x) {
    const int l = sorted_list[i];
    const int64_t v = sorted_row[i];
    const int64_t pos = old_len[l] + (i - seg_start[l]);
    const int64_t slot = new_off[l] * 32 + pos;
    const int lane = int(slot & 31);
    uint8_t* blk = codes + (slot >> 5) * 32 * m;
    const uint8_t* src = codes_in + v * m;
    for (int s = 0; s < m; ++s) blk[stored_byte_offset(lane, s, m)] = src[stored_source_byte(lane, s, m)];
    ids[slot] = ids_in[v];
  }
}

__global__ void iota_kernel(int32_t* out, int64_t n) {
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += int64_t(gridDim.x) * blockDim.x)
    out[i] = int32_t(i);
}

unsigned grid_for(int64_t n, int threads) {
  return unsigned(std::max<int64_t>(1, std::min<int64_t>(ceil_div(n, threads), 65535LL * 16)));
}

// T1[l][e][j] = ||y_R||^2 + 2 <y_C, y_R> with y_C = centroid l restricted to
// sub-quantizer j's dimensions and y_R = reproduction value e of
// sub-quantizer j ("Billion-scale similarity search with GPUs", section 5:
// the term of the expanded distance that depends on the list and the code but
// not on the query). One thread per (l, e, j).
__global__ void term1_kernel(const float* __restrict__ cent, const float* __restrict__ cb_t,
                             int64_t nlist, int d, int m, int dsub, int dsub4,
                             float* __restrict__ t1) {
  const int64_t n = nlist * 256 * m;
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += int64_t(gridDim.x) * blockDim.x) {
    const int j = int(i % m);
    const int64_t le = i / m;
    const int e = int(le % 256);
    const int64_t l = le / 256;
    const float* c = cent + l * d + int64_t(j) * dsub;
    const float* y = cb_t + (int64_t(e) * m + j) * dsub4;
    float s = 0.f;
    for (int t = 0; t < dsub; ++t) s = fmaf(y[t], fmaf(2.f, c[t], y[t]), s);
    t1[i] = s;
  }
}

}  // namespace

bool use_precomputed(const ivfpq_index* ix) {
  if (ix->lut_type != IVFPQ_LUT_FP32 || ix->m * ix->dsub != ix->d) return false;
  const int key = ix->m * 100 + ix->dsub;
  const bool shape = key == 812 || key == 808 || key == 1608 || key == 1604;
  if (!shape || ix->precomputed == 0) return false;
  if (ix->precomputed == 1) return true;
  // automatic: where it measured faster (scan ms, 10,000 queries: m = 16, d/m = 8,
  // 1e7 vectors, 64 probes 12.1 -> 11.3; m = 8, d/m = 12, 1e9 vectors, 128
  // probes 23.9 -> 25.5, slower: the list table read outweighs the build)
  return key == 1608;
}

int build_term1(ivfpq_index* ix) {
  if (ix->term1) return IVFPQ_OK;
  const size_t n = size_t(ix->nlist) * 256 * ix->m;
  float* t = nullptr;
  if (cudaMalloc(&t, n * sizeof(float)) != cudaSuccess) {
    cudaGetLastError();
    set_error("precomputed-term tables: cannot allocate %zu bytes", n * sizeof(float));
    return IVFPQ_ERR_OOM;
  }
  term1_kernel<<<grid_for(int64_t(n), 256), 256, 0, 0>>>(ix->centroids, ix->codebooks, ix->nlist,
                                                        ix->d, ix->m, ix->dsub, ix->dsub4, t);
  IVFPQ_LAUNCHED();
  IVFPQ_CUDA(cudaStreamSynchronize(0));
  ix->term1 = t;
  return IVFPQ_OK;
}

}  // namespace ivfpq

using namespace ivfpq;

extern "C" int ivfpq_index_create(int d, int nlist, int m, int nbits, const float* centroids,
                                  const float* codebooks, ivfpq_index** out) {
  clear_error();
  IVFPQ_REQUIRE(out != nullptr, "ivfpq_index_create: out is null");
  *out = nullptr;
  IVFPQ_REQUIRE(d > 0 && nlist > 0 && m > 0, "ivfpq_index_create: bad sizes d=%d nlist=%d m=%d",
                d, nlist, m);
  IVFPQ_REQUIRE(nlist <= (1 << 24), "ivfpq_index_create: nlist=%d above 2^24", nlist);
  IVFPQ_REQUIRE(d % m == 0, "ivfpq_index_create: d=%d is not a multiple of m=%d", d, m);
  IVFPQ_REQUIRE(centroids && codebooks, "ivfpq_index_create: null pointer");
  if (nbits != 8 || m % 4 != 0 || m > IVFPQ_MAX_M) {
    set_error("ivfpq_index_create: unsupported nbits=%d / m=%d (need nbits=8, m a multiple of 4 "
              "up to %d)", nbits, m, IVFPQ_MAX_M);
    return IVFPQ_ERR_UNSUPPORTED;
  }
  ivfpq_index* ix = new ivfpq_index();
  ix->d = d;
  ix->nlist = nlist;
  ix->m = m;
  ix->nbits = nbits;
  ix->dsub = d / m;
  cudaGetDevice(&ix->device);
  auto fail = [&](int st) {
    ivfpq_index_destroy(ix);
    return st;
  };
  ix->dsub4 = (ix->dsub + 3) & ~3;
  const size_t cb_n = size_t(m) * 256 * ix->dsub;
  const size_t cb4_n = size_t(m) * 256 * ix->dsub4;
  float* cb_tmp = nullptr;
#define CREATE_CUDA(expr)                                                            \
  do {                                                                               \
    cudaError_t e_ = (expr);                                                         \
    if (e_ != cudaSuccess) {                                                         \
      set_error("ivfpq_index_create: %s: %s", #expr, cudaGetErrorString(e_));        \
      if (cb_tmp) cudaFree(cb_tmp);                                                  \
      return fail(e_ == cudaErrorMemoryAllocation ? IVFPQ_ERR_OOM : IVFPQ_ERR_CUDA); \
    }                                                                                \
  } while (0)
  CREATE_CUDA(cudaMalloc(&ix->centroids, size_t(nlist) * d * sizeof(float)));
  CREATE_CUDA(cudaMalloc(&ix->cent_norms, size_t(nlist) * sizeof(float)));
  CREATE_CUDA(cudaMalloc(&ix->codebooks, cb4_n * sizeof(float)));
  CREATE_CUDA(cudaMalloc(&cb_tmp, cb_n * sizeof(float)));
  CREATE_CUDA(cudaMalloc(&ix->list_len, size_t(nlist) * sizeof(int32_t)));
  CREATE_CUDA(cudaMalloc(&ix->list_block_off, size_t(nlist + 1) * sizeof(int64_t)));
  CREATE_CUDA(cudaMalloc(&ix->repaired, sizeof(unsigned long long)));
  CREATE_CUDA(cudaMemsetAsync(ix->repaired, 0, sizeof(unsigned long long), 0));
  CREATE_CUDA(cudaMemcpyAsync(ix->centroids, centroids, size_t(nlist) * d * sizeof(float),
                              cudaMemcpyDefault, 0));
  CREATE_CUDA(cudaMemcpyAsync(cb_tmp, codebooks, cb_n * sizeof(float), cudaMemcpyDefault, 0));
  CREATE_CUDA(cudaMemsetAsync(ix->list_len, 0, size_t(nlist) * sizeof(int32_t), 0));
  CREATE_CUDA(cudaMemsetAsync(ix->list_block_off, 0, size_t(nlist + 1) * sizeof(int64_t), 0));
  cent_norms_kernel<<<unsigned(ceil_div(nlist, 8)), dim3(32, 8), 0, 0>>>(ix->centroids, nlist, d,
                                                                         ix->cent_norms);
  CREATE_CUDA(cudaGetLastError());
  transpose_codebooks_kernel<<<grid_for(int64_t(cb4_n), 256), 256, 0, 0>>>(
      cb_tmp, m, ix->dsub, ix->dsub4, ix->codebooks);
  CREATE_CUDA(cudaGetLastError());
  if (l2_tc_available(d)) {
    const size_t nn = size_t(nlist) * tc_dpad(d);
    CREATE_CUDA(cudaMalloc(&ix->cent_hi, nn * sizeof(float)));
    CREATE_CUDA(cudaMalloc(&ix->cent_lo, nn * sizeof(float)));
    const int st = l2_tc_prepare(ix->centroids, nlist, d, ix->cent_hi, ix->cent_lo, ix->cent_norms, 0);
    if (st != IVFPQ_OK) {
      cudaFree(cb_tmp);
      return fail(st);
    }
  }
  CREATE_CUDA(cudaStreamSynchronize(0));
  cudaFree(cb_tmp);
  cb_tmp = nullptr;
  if (use_precomputed(ix)) {
    const int st = build_term1(ix);
    if (st != IVFPQ_OK) return fail(st);
  }
#undef CREATE_CUDA
  ix->h_list_len.assign(nlist, 0);
  *out = ix;
  return IVFPQ_OK;
}

extern "C" int ivfpq_index_destroy(ivfpq_index* ix) {
  if (!ix) return IVFPQ_OK;
  cudaDeviceSynchronize();
  cudaFree(ix->centroids);
  cudaFree(ix->cent_norms);
  cudaFree(ix->cent_hi);
  cudaFree(ix->cent_lo);
  cudaFree(ix->codebooks);
  cudaFree(ix->term1);
  cudaFree(ix->list_len);
  cudaFree(ix->list_block_off);
  cudaFree(ix->codes);
  cudaFree(ix->ids);
  cudaFree(ix->repaired);
  cudaFree(ix->cent_sep);
  for (auto& set : ix->ev_sets)
    for (auto& e : set.ev)
      if (e) cudaEventDestroy(e);
  delete ix;
  return IVFPQ_OK;
}

extern "C" int ivfpq_set_lut_type(ivfpq_index* ix, int lut_type) {
  clear_error();
  IVFPQ_REQUIRE(ix, "ivfpq_set_lut_type: null index");
  IVFPQ_REQUIRE(lut_type == IVFPQ_LUT_FP32 || lut_type == IVFPQ_LUT_FP16 ||
                    lut_type == IVFPQ_LUT_FP8,
                "ivfpq_set_lut_type: unknown type %d", lut_type);
  ix->lut_type = lut_type;
  return IVFPQ_OK;
}

extern "C" int ivfpq_set_precomputed(ivfpq_index* ix, int mode) {
  clear_error();
  IVFPQ_REQUIRE(ix, "ivfpq_set_precomputed: null index");
  IVFPQ_REQUIRE(mode >= -1 && mode <= 1, "ivfpq_set_precomputed: mode %d not in {-1, 0, 1}",
                mode);
  IVFPQ_CUDA(cudaDeviceSynchronize());  // no search of this index may be running
  ix->precomputed = mode;
  if (use_precomputed(ix)) IVFPQ_TRY(build_term1(ix));
  return IVFPQ_OK;
}

extern "C" int ivfpq_uses_precomputed(const ivfpq_index* ix) {
  return ix && use_precomputed(ix) && ix->term1 ? 1 : 0;
}

extern "C" int64_t ivfpq_ntotal(const ivfpq_index* ix) { return ix ? ix->ntotal : -1; }

extern "C" int ivfpq_add(ivfpq_index* ix, const uint8_t* codes, const int32_t* list_ids,
                         const int64_t* ids, int64_t n, void* stream) {
  clear_error();
  IVFPQ_REQUIRE(ix, "ivfpq_add: null index");
  IVFPQ_REQUIRE(n >= 0, "ivfpq_add: negative n");
  if (n == 0) return IVFPQ_OK;
  IVFPQ_REQUIRE(codes && list_ids && ids, "ivfpq_add: null pointer");
  IVFPQ_REQUIRE(n < (int64_t(1) << 31), "ivfpq_add: n=%lld above 2^31 - 1 per call", (long long)n);
  const int nlist = ix->nlist, m = ix->m;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Workspace ws(s);
  int32_t *counts, *bad, *new_len, *rows_in, *rows_sorted, *lists_sorted, *seg_start;
  int64_t *nblk, *new_off;
  IVFPQ_TRY(ws.alloc(&counts, nlist));
  IVFPQ_TRY(ws.alloc(&bad, 1));
  IVFPQ_TRY(ws.alloc(&new_len, nlist));
  IVFPQ_TRY(ws.alloc(&nblk, nlist + 1));
  IVFPQ_TRY(ws.alloc(&new_off, nlist + 1));
  IVFPQ_TRY(ws.alloc(&seg_start, nlist));
  IVFPQ_CUDA(cudaMemsetAsync(counts, 0, sizeof(int32_t) * nlist, s));
  IVFPQ_CUDA(cudaMemsetAsync(bad, 0, sizeof(int32_t), s));
  histogram_kernel<<<grid_for(n, 256), 256, 0, s>>>(list_ids, n, nlist, counts, bad);
  IVFPQ_LAUNCHED();
  new_sizes_kernel<<<grid_for(nlist, 256), 256, 0, s>>>(ix->list_len, counts, nlist, new_len, nblk);
  IVFPQ_LAUNCHED();
  // block offsets of the new layout: exclusive scan of the block counts
  size_t scan_bytes = 0;
  IVFPQ_CUDA(cub::DeviceScan::ExclusiveSum(nullptr, scan_bytes, nblk, new_off, nlist + 1, s));
  uint8_t* scan_tmp = nullptr;
  IVFPQ_TRY(ws.alloc(&scan_tmp, scan_bytes));
  IVFPQ_CUDA(cub::DeviceScan::ExclusiveSum(scan_tmp, scan_bytes, nblk, new_off, nlist + 1, s));
  // first position of each list among the new vectors sorted by list
  size_t seg_bytes = 0;
  IVFPQ_CUDA(cub::DeviceScan::ExclusiveSum(nullptr, seg_bytes, counts, seg_start, nlist, s));
  uint8_t* seg_tmp = nullptr;
  IVFPQ_TRY(ws.alloc(&seg_tmp, seg_bytes));
  IVFPQ_CUDA(cub::DeviceScan::ExclusiveSum(seg_tmp, seg_bytes, counts, seg_start, nlist, s));
  int64_t total_blocks = 0;
  int32_t h_bad = 0;
  IVFPQ_CUDA(cudaMemcpyAsync(&total_blocks, new_off + nlist, sizeof(int64_t),
                             cudaMemcpyDeviceToHost, s));
  IVFPQ_CUDA(cudaMemcpyAsync(&h_bad, bad, sizeof(int32_t), cudaMemcpyDeviceToHost, s));
  IVFPQ_CUDA(cudaStreamSynchronize(s));
  IVFPQ_REQUIRE(!h_bad, "ivfpq_add: a list id is outside [0, %d)", nlist);
  IVFPQ_REQUIRE(total_blocks * 32 < int64_t(0xffffffffLL),
                "ivfpq_add: the index would exceed 2^32 - 1 vector slots");

  // stable order of the new vectors by list (LSD radix sort is stable)
  IVFPQ_TRY(ws.alloc(&rows_in, n));
  IVFPQ_TRY(ws.alloc(&rows_sorted, n));
  IVFPQ_TRY(ws.alloc(&lists_sorted, n));
  iota_kernel<<<grid_for(n, 256), 256, 0, s>>>(rows_in, n);
  IVFPQ_LAUNCHED();
  int end_bit = 1;
  while ((1 << end_bit) < nlist) ++end_bit;
  size_t sort_bytes = 0;
  IVFPQ_CUDA(cub::DeviceRadixSort::SortPairs(nullptr, sort_bytes, list_ids, lists_sorted, rows_in,
                                             rows_sorted, n, 0, end_bit, s));
  uint8_t* sort_tmp = nullptr;
  IVFPQ_TRY(ws.alloc(&sort_tmp, sort_bytes));
  IVFPQ_CUDA(cub::DeviceRadixSort::SortPairs(sort_tmp, sort_bytes, list_ids, lists_sorted, rows_in,
                                             rows_sorted, n, 0, end_bit, s));

  uint8_t* new_codes = nullptr;
  int64_t* new_ids = nullptr;
  cudaError_t e1 = cudaMalloc(&new_codes, size_t(total_blocks) * 32 * m);
  cudaError_t e2 = e1 == cudaSuccess ? cudaMalloc(&new_ids, size_t(total_blocks) * 32 * 8)
                                     : cudaSuccess;
  if (e1 != cudaSuccess || e2 != cudaSuccess) {
    cudaGetLastError();
    cudaFree(new_codes);
    set_error("ivfpq_add: cannot allocate %lld blocks of list storage", (long long)total_blocks);
    return IVFPQ_ERR_OOM;
  }
  cudaError_t e = cudaSuccess;
  auto step = [&](cudaError_t r) {
    if (e == cudaSuccess && r != cudaSuccess) e = r;
  };
  step(cudaMemsetAsync(new_codes, 0, size_t(total_blocks) * 32 * m, s));
  step(cudaMemsetAsync(new_ids, 0xff, size_t(total_blocks) * 32 * 8, s));
  if (ix->nblocks > 0) {
    copy_lists_kernel<<<nlist, 256, 0, s>>>(ix->list_block_off, new_off, ix->codes, ix->ids,
                                            new_codes, new_ids, m);
    step(cudaGetLastError());
  }
  scatter_kernel<<<grid_for(n, 256), 256, 0, s>>>(lists_sorted, rows_sorted, n, ix->list_len,
                                                  seg_start, new_off, codes, ids, new_codes,
                                                  new_ids, m);
  step(cudaGetLastError());
  step(cudaMemcpyAsync(ix->list_len, new_len, sizeof(int32_t) * nlist, cudaMemcpyDeviceToDevice,
                       s));
  step(cudaMemcpyAsync(ix->list_block_off, new_off, sizeof(int64_t) * (nlist + 1),
                       cudaMemcpyDeviceToDevice, s));
  std::vector<int32_t> h_len(nlist);
  step(cudaMemcpyAsync(h_len.data(), new_len, sizeof(int32_t) * nlist, cudaMemcpyDeviceToHost, s));
  step(cudaStreamSynchronize(s));
  if (e != cudaSuccess) {
    cudaFree(new_codes);
    cudaFree(new_ids);
    set_error("ivfpq_add: %s", cudaGetErrorString(e));
    return IVFPQ_ERR_CUDA;
  }
  cudaFree(ix->codes);
  cudaFree(ix->ids);
  ix->codes = new_codes;
  ix->ids = new_ids;
  ix->nblocks = total_blocks;
  ix->ntotal += n;
  ix->max_list_len = 0;
  for (int l = 0; l < nlist; ++l) {
    ix->h_list_len[l] = h_len[l];
    ix->max_list_len = std::max<int64_t>(ix->max_list_len, h_len[l]);
  }
  ivfpq::update_list_units(ix);
  return IVFPQ_OK;
}
