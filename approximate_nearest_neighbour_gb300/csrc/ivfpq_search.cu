// Batched IVF-PQ search: coarse quantizer, fused table build + list scan +
// per-chunk selection, and the cross-chunk merge with id translation.
//
// Source: IVFPQ search steps 1-5 ("Custom 8-bit floating point value format
// for reducing shared memory bank conflict in approximate nearest neighbor
// search"); section 5 of "Billion-scale similarity search with GPUs" (tables
// per query x list, queries x lists processed independently, two-pass
// k-selection with subdivision factor f: here f = the number of list chunks
// per query).
#include <cub/cub.cuh>

#include <algorithm>

#include "internal.h"
#include "scan2.cuh"
#include "scan_lm.cuh"
#include "select_radix.cuh"

namespace ivfpq {

#define IVFPQ_EXTERN_SCAN(MW, K) \
  extern template int launch_scan_mw<MW, K>(const ScanParams&, int64_t, cudaStream_t);
#define IVFPQ_EXTERN_SCAN_ALL(K) \
  IVFPQ_EXTERN_SCAN(0, K) IVFPQ_EXTERN_SCAN(2, K) IVFPQ_EXTERN_SCAN(4, K) IVFPQ_EXTERN_SCAN(8, K)
IVFPQ_EXTERN_SCAN_ALL(32)
IVFPQ_EXTERN_SCAN_ALL(64)
IVFPQ_EXTERN_SCAN_ALL(128)
IVFPQ_EXTERN_SCAN_ALL(256)
IVFPQ_EXTERN_SCAN_ALL(512)
IVFPQ_EXTERN_SCAN_ALL(1024)
IVFPQ_EXTERN_SCAN_ALL(2048)
IVFPQ_EXTERN_SCAN(16, 32)
IVFPQ_EXTERN_SCAN(16, 64)
IVFPQ_EXTERN_SCAN(16, 128)
IVFPQ_EXTERN_SCAN(16, 256)

#define IVFPQ_EXTERN_SCAN2_1(MW, DS, KW, PRE) \
  extern template int launch_scan2<MW, DS, KW, PRE>(const ScanParams&, int64_t, cudaStream_t);
#define IVFPQ_EXTERN_SCAN2_KW(MW, DS, PRE)                                                  \
  IVFPQ_EXTERN_SCAN2_1(MW, DS, 32, PRE) IVFPQ_EXTERN_SCAN2_1(MW, DS, 64, PRE)               \
  IVFPQ_EXTERN_SCAN2_1(MW, DS, 128, PRE) IVFPQ_EXTERN_SCAN2_1(MW, DS, 256, PRE)
#define IVFPQ_EXTERN_SCAN2(MW, DS) \
  IVFPQ_EXTERN_SCAN2_KW(MW, DS, false) IVFPQ_EXTERN_SCAN2_KW(MW, DS, true)
IVFPQ_EXTERN_SCAN2_KW(8, 3, false)
IVFPQ_EXTERN_SCAN2_KW(8, 4, false)
IVFPQ_EXTERN_SCAN2(4, 8)
IVFPQ_EXTERN_SCAN2(4, 4)
IVFPQ_EXTERN_SCAN2(2, 12)
IVFPQ_EXTERN_SCAN2(2, 8)

// The register-codebook kernel (scan2.cuh) with KW-entry warp queues, for
// the (m, d/m) shapes it is built for, with precomputed-term tables when
// p.term1 is set (m <= 16 shapes); 1 = launched, 0 = not applicable.
template <int KW>
int try_scan2_kw(const ScanParams& p, int64_t nq, cudaStream_t s, int* launched) {
  *launched = 1;
  const int key = p.m * 100 + p.dsub;
  const bool pre = p.term1 != nullptr;
  switch (key) {
    case 3203: return launch_scan2<8, 3, KW, false>(p, nq, s);
    case 3204: return launch_scan2<8, 4, KW, false>(p, nq, s);
    case 1608:
      return pre ? launch_scan2<4, 8, KW, true>(p, nq, s) : launch_scan2<4, 8, KW, false>(p, nq, s);
    case 1604:
      return pre ? launch_scan2<4, 4, KW, true>(p, nq, s) : launch_scan2<4, 4, KW, false>(p, nq, s);
    case 812:
      return pre ? launch_scan2<2, 12, KW, true>(p, nq, s)
                 : launch_scan2<2, 12, KW, false>(p, nq, s);
    case 808:
      return pre ? launch_scan2<2, 8, KW, true>(p, nq, s) : launch_scan2<2, 8, KW, false>(p, nq, s);
  }
  *launched = 0;
  return IVFPQ_OK;
}

#define IVFPQ_EXTERN_SCAN_LM_LT(MW, DS, LT)                                           \
  extern template int launch_scan_lm<MW, DS, 1, 2, LT>(const LmParams&, cudaStream_t); \
  extern template int launch_scan_lm<MW, DS, 1, 4, LT>(const LmParams&, cudaStream_t); \
  extern template int launch_scan_lm<MW, DS, 1, 8, LT>(const LmParams&, cudaStream_t);
#define IVFPQ_EXTERN_SCAN_LM(MW, DS)                                                         \
  extern template int launch_scan_lm<MW, DS, 2, 0, IVFPQ_LUT_FP32>(const LmParams&,          \
                                                                   cudaStream_t);            \
  extern template int launch_scan_lm<MW, DS, 3, 0, IVFPQ_LUT_FP32>(const LmParams&,          \
                                                                   cudaStream_t);            \
  extern template int launch_scan_lm<MW, DS, 4, 0, IVFPQ_LUT_FP16>(const LmParams&,          \
                                                                   cudaStream_t);            \
  extern template int launch_scan_lm<MW, DS, 6, 0, IVFPQ_LUT_FP16>(const LmParams&,          \
                                                                   cudaStream_t);            \
  extern template int launch_scan_lm<MW, DS, 4, 0, IVFPQ_LUT_FP8>(const LmParams&,           \
                                                                  cudaStream_t);             \
  extern template int launch_scan_lm<MW, DS, 8, 0, IVFPQ_LUT_FP8>(const LmParams&,           \
                                                                  cudaStream_t);             \
  IVFPQ_EXTERN_SCAN_LM_LT(MW, DS, IVFPQ_LUT_FP32)                                            \
  IVFPQ_EXTERN_SCAN_LM_LT(MW, DS, IVFPQ_LUT_FP16)                                            \
  IVFPQ_EXTERN_SCAN_LM_LT(MW, DS, IVFPQ_LUT_FP8)
IVFPQ_EXTERN_SCAN_LM(8, 3)
IVFPQ_EXTERN_SCAN_LM(8, 4)
IVFPQ_EXTERN_SCAN_LM(4, 8)
IVFPQ_EXTERN_SCAN_LM(4, 4)
IVFPQ_EXTERN_SCAN_LM(2, 12)
IVFPQ_EXTERN_SCAN_LM(2, 8)

// The list-major kernel (scan_lm.cuh): the filter pass with G queries per
// table set (TQ = 0) or the bound pass with TQ-entry lane queues (G = 1).
template <int G, int TQ, int LT>
int try_scan_lm(const LmParams& p, cudaStream_t s, int* launched) {
  *launched = 1;
  switch (p.s.m * 100 + p.s.dsub) {
    case 3203: return launch_scan_lm<8, 3, G, TQ, LT>(p, s);
    case 3204: return launch_scan_lm<8, 4, G, TQ, LT>(p, s);
    case 1608: return launch_scan_lm<4, 8, G, TQ, LT>(p, s);
    case 1604: return launch_scan_lm<4, 4, G, TQ, LT>(p, s);
    case 812: return launch_scan_lm<2, 12, G, TQ, LT>(p, s);
    case 808: return launch_scan_lm<2, 8, G, TQ, LT>(p, s);
  }
  *launched = 0;
  return IVFPQ_OK;
}

// The bound pass with TQ-entry lane queues, tables of type LT.
template <int LT>
int launch_bound_pass(const LmParams& p, int tq, cudaStream_t s, int* launched) {
  switch (tq) {
    case 2: return try_scan_lm<1, 2, LT>(p, s, launched);
    case 4: return try_scan_lm<1, 4, LT>(p, s, launched);
    default: return try_scan_lm<1, 8, LT>(p, s, launched);
  }
}

bool scan2_shape(const ScanParams& p) {
  const int key = p.m * 100 + p.dsub;
  return p.lut_type == IVFPQ_LUT_FP32 && p.m * p.dsub == p.d && p.k <= IVFPQ_MAX_K &&
         (key == 3203 || key == 3204 || key == 1608 || key == 1604 || key == 812 || key == 808);
}

// Code words per vector as a template argument where a specialised kernel
// exists (m = 8, 16, 32; m = 64 for K <= 256); 0 selects the generic kernel.
template <int K>
int launch_scan_k(const ScanParams& p, int64_t nq, cudaStream_t s) {
  switch (p.m) {
    case 8: return launch_scan_mw<2, K>(p, nq, s);
    case 16: return launch_scan_mw<4, K>(p, nq, s);
    case 32: return launch_scan_mw<8, K>(p, nq, s);
    case 64:
      if constexpr (K <= 256) return launch_scan_mw<16, K>(p, nq, s);
      else return launch_scan_mw<0, K>(p, nq, s);
    default: return launch_scan_mw<0, K>(p, nq, s);
  }
}

namespace {

int queue_len(int k) {
  int K = 32;
  while (K < k) K *= 2;
  return K;
}

// The general kernel (scan.cuh): BlockSelect with K-entry queues.
int launch_scan_general(const ScanParams& p, int64_t nq, cudaStream_t s) {
  switch (queue_len(p.k)) {
    case 32: return launch_scan_k<32>(p, nq, s);
    case 64: return launch_scan_k<64>(p, nq, s);
    case 128: return launch_scan_k<128>(p, nq, s);
    case 256: return launch_scan_k<256>(p, nq, s);
    case 512: return launch_scan_k<512>(p, nq, s);
    case 1024: return launch_scan_k<1024>(p, nq, s);
    case 2048: return launch_scan_k<2048>(p, nq, s);
  }
  set_error("k=%d above %d", p.k, IVFPQ_MAX_K);
  return IVFPQ_ERR_INVALID_ARG;
}

// Queries whose result may have lost an entry to a short warp queue: some
// full queue (last key real) whose last key is not above the merged k-th
// key. kth: merged distances [nq, k] (row's k-th at kth[q * k + k - 1]).
// The number of flagged queries is added to *repaired.
__global__ void warp_queue_check_kernel(const uint32_t* __restrict__ pkeys, int64_t nq,
                                        int groups, int kw, const float* __restrict__ kth,
                                        int k, int* __restrict__ flags,
                                        unsigned long long* __restrict__ repaired) {
  const int64_t q = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  int f = 0;
  if (q < nq) {
    const uint32_t theta = __float_as_uint(kth[q * k + k - 1]);
    for (int g = 0; g < groups; ++g) {
      const uint32_t last = pkeys[(q * groups + g) * kw + kw - 1];
      f |= last != kSentinelKey && last <= theta;
    }
    flags[q] = f;
  }
  const unsigned c = __popc(__ballot_sync(kFullMask, f));
  if ((threadIdx.x & 31) == 0 && c) atomicAdd(repaired, (unsigned long long)c);
}

// *repaired += number of flagged queries
__global__ void count_flags_kernel(const int* __restrict__ flags, int64_t nq,
                                   unsigned long long* __restrict__ repaired) {
  const int64_t q = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  const int f = q < nq ? flags[q] : 0;
  const unsigned c = __popc(__ballot_sync(kFullMask, f != 0));
  if ((threadIdx.x & 31) == 0 && c) atomicAdd(repaired, (unsigned long long)c);
}

const size_t kMaxEventSets = 4096;

// Starts a new event set for this search (profiling only).
void begin_profile(const ivfpq_index* ix) {
  auto* mix = const_cast<ivfpq_index*>(ix);
  mix->cur_set = -1;
  if (!mix->profile || mix->ev_used >= kMaxEventSets) return;
  if (mix->ev_sets.size() <= mix->ev_used) mix->ev_sets.resize(mix->ev_used + 1);
  auto& set = mix->ev_sets[mix->ev_used];
  for (bool& r : set.recorded) r = false;
  mix->cur_set = int(mix->ev_used++);
}

void record(const ivfpq_index* ix, int i, cudaStream_t s) {
  auto* mix = const_cast<ivfpq_index*>(ix);
  if (mix->cur_set < 0) return;
  auto& set = mix->ev_sets[mix->cur_set];
  if (!set.ev[i] && cudaEventCreate(&set.ev[i]) != cudaSuccess) return;
  if (cudaEventRecord(set.ev[i], s) == cudaSuccess) set.recorded[i] = true;
}

// ---- list-major scan: planning and final selection ----------------------------

// Record of every item (one warp per item): its list, length, first block,
// queries and their bounds (the sentinel in the bound pass), and the
// residual of each of its queries to the list's centroid.
__global__ void lm_records_kernel(const LmParams p, int G, bool bound_pass, uint8_t* records) {
  const ScanParams& sp = p.s;
  const int lane = threadIdx.x & 31;
  const int nit = *p.n_items;
  const int warps = int(gridDim.x) * (blockDim.x >> 5);
  for (int it = int(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); it < nit; it += warps) {
    const int64_t pos = p.items[it];
    const bool pos_ok = dcheck(sp.dbg, pos >= 0 && pos < p.npairs, 0);
    const int l = pos_ok ? p.pair_list[pos] : 0;
    const bool list_ok = dcheck(sp.dbg, l >= 0 && l < sp.nlist, 1);
    const bool mine = pos_ok && list_ok && lane < G && pos + lane < p.npairs &&
                      p.pair_list[pos + lane] == l;
    const unsigned vm = __ballot_sync(kFullMask, mine);
    const int nq = __popc(vm);
    uint8_t* rec = records + int64_t(it) * p.rec_bytes;
    LmHead* h = reinterpret_cast<LmHead*>(rec);
    int qv = 0;
    if (mine) {
      qv = p.pair_query[pos + lane];
      if (!dcheck(sp.dbg, qv >= 0 && qv < sp.nq, 2)) qv = 0;
      h->q[lane] = qv;
      h->theta[lane] = bound_pass ? kSentinelKey : p.theta_key[int64_t(qv) * p.theta_stride];
    }
    if (lane == 0) {
      h->list = l;
      h->item = it;
      h->nq = nq;
      h->len = sp.list_len[l];
      h->boff = sp.list_block_off[l];
      dcheck(sp.dbg, h->boff >= 0 && h->boff + ((h->len + 31) >> 5) <= sp.nblocks, 3);
    }
    float* res = reinterpret_cast<float*>(rec + kLmHead);
    const float* c = sp.centroids + int64_t(l) * sp.d;
    for (int g = 0; g < nq; ++g) {
      const int qg = __shfl_sync(kFullMask, qv, g);
      const float* x = sp.queries + int64_t(qg) * sp.d;
      for (int t = lane; t < p.dpad; t += 32) res[g * p.dpad + t] = t < sp.d ? x[t] - c[t] : 0.f;
    }
  }
}


// probes[q][col] -> out[q]
__global__ void probe_column_kernel(const int32_t* __restrict__ probes, int64_t nq, int nprobe,
                                    int col, int32_t* __restrict__ out) {
  const int64_t q = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (q < nq) out[q] = probes[q * nprobe + col];
}

// (list, query) pairs of probes p0 .. p0 + per - 1; a list id outside
// [0, nlist) becomes nlist (sorted last, no item)
__global__ void lm_pairs_kernel(const int32_t* __restrict__ probes, int64_t nq, int nprobe,
                                int p0, int per, int nlist, int32_t* __restrict__ key,
                                int32_t* __restrict__ val) {
  const int64_t n = nq * per;
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += int64_t(gridDim.x) * blockDim.x) {
    const int64_t q = i / per;
    const int l = probes[q * nprobe + p0 + (i - q * per)];
    key[i] = (l >= 0 && l < nlist) ? l : nlist;
    val[i] = int32_t(q);
  }
}

// flag[i] = 1 where sorted pair i starts an item: its rank among the pairs
// of its list is a multiple of G (rank from a binary search for the list's
// first pair)
__global__ void lm_item_flags_kernel(const int32_t* __restrict__ skey, int64_t n, int G,
                                     int nlist, int32_t* __restrict__ flag) {
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += int64_t(gridDim.x) * blockDim.x) {
    const int32_t l = skey[i];
    int64_t lo = 0, hi = i;  // first index with skey == l lies in [lo, hi]
    while (lo < hi) {
      const int64_t mid = (lo + hi) >> 1;
      if (skey[mid] < l) lo = mid + 1;
      else hi = mid;
    }
    flag[i] = (l < nlist && (i - lo) % G == 0) ? 1 : 0;
  }
}

// items[pos[i]] = i for the flagged pairs; *n_items = their number
__global__ void lm_items_kernel(const int32_t* __restrict__ flag, const int32_t* __restrict__ pos,
                                int64_t n, int32_t* __restrict__ items, int* __restrict__ n_items) {
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += int64_t(gridDim.x) * blockDim.x) {
    if (flag[i]) items[pos[i]] = int32_t(i);
    if (i == n - 1) *n_items = pos[i] + flag[i];
  }
}

// theta[r] = the k-th smallest of row r's len keys (the sentinel when fewer
// than k keys are below it): one warp per row, a binary search over the
// 32-bit key range for the least v with at least k keys <= v.
// The bound pass scans each query's nearest list in chunks of `chunk` codes
// (a multiple of 32), one item per chunk, so that a long list (the largest of
// a Zipf mixture holds ~1e6 codes) is spread over several blocks.
constexpr int kBoundChunkMin = 32768;
constexpr int kBoundChunksMax = 4;

// cnt[q] = chunks of query q's nearest list (at least 1)
__global__ void bound_chunks_kernel(const int32_t* __restrict__ probes, int64_t nq, int nprobe,
                                    const int32_t* __restrict__ list_len, int nlist, int chunk,
                                    int32_t* __restrict__ cnt) {
  const int64_t q = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (q >= nq) return;
  const int l = probes[q * nprobe];
  const int len = (l >= 0 && l < nlist) ? list_len[l] : 0;
  cnt[q] = max(1, (len + chunk - 1) / chunk);
}

// Records of the bound pass (one warp per query, one record per chunk of its
// nearest list, at item off[q] + c); *n_items = the number of items.
__global__ void bound_records_kernel(const LmParams p, int nprobe, int chunk,
                                     const int32_t* __restrict__ off,
                                     const int32_t* __restrict__ cnt, uint8_t* records,
                                     int* __restrict__ n_items) {
  const ScanParams& sp = p.s;
  const int lane = threadIdx.x & 31;
  const int64_t q = int64_t(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (q >= sp.nq) return;  // the same for the whole warp
  if (q == sp.nq - 1 && lane == 0) *n_items = off[q] + cnt[q];
  const int l0 = sp.probes[q * nprobe];
  const bool valid = dcheck(sp.dbg, l0 >= -1 && l0 < sp.nlist, 1) && l0 >= 0 && l0 < sp.nlist;
  const int l = valid ? l0 : 0;
  const int total = valid ? sp.list_len[l] : 0;
  const int64_t boff = sp.list_block_off[l];
  const float* x = sp.queries + q * sp.d;
  const float* c = sp.centroids + int64_t(l) * sp.d;
  for (int ch = 0; ch < cnt[q]; ++ch) {
    const int it = off[q] + ch;
    uint8_t* rec = records + int64_t(it) * p.rec_bytes;
    if (lane == 0) {
      LmHead* h = reinterpret_cast<LmHead*>(rec);
      h->list = l;
      h->item = it;
      h->nq = 1;
      h->len = max(0, min(chunk, total - ch * chunk));
      h->boff = boff + int64_t(ch) * (chunk / 32);
      h->q[0] = int(q);
      h->theta[0] = kSentinelKey;
    }
    float* res = reinterpret_cast<float*>(rec + kLmHead);
    for (int t = lane; t < p.dpad; t += 32) res[t] = t < sp.d ? x[t] - c[t] : 0.f;
  }
}

// Sort keys of the bound pass's items: len[i] = item i's code count (-1 past
// the last item), idx[i] = i.
__global__ void bound_order_keys_kernel(const uint8_t* __restrict__ records, int rec_bytes,
                                        const int* __restrict__ n_items, int64_t max_items,
                                        int32_t* __restrict__ len, int32_t* __restrict__ idx) {
  const int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= max_items) return;
  len[i] = i < *n_items ? reinterpret_cast<const LmHead*>(records + i * rec_bytes)->len : -1;
  idx[i] = int32_t(i);
}

// Row r holds cnt[r] * per keys from keys + off[r] * per.
__global__ void lm_theta_kernel(const uint32_t* __restrict__ keys, int64_t rows,
                                const int32_t* __restrict__ off, const int32_t* __restrict__ cnt,
                                int per, int k, uint32_t* __restrict__ theta) {
  const int lane = threadIdx.x & 31;
  const int64_t row = int64_t(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (row >= rows) return;  // the same for the whole warp
  const uint32_t* kr = keys + int64_t(off[row]) * per;
  const int len = cnt[row] * per;
  uint32_t lo = 0, hi = kSentinelKey;
  while (lo < hi) {
    const uint32_t mid = lo + ((hi - lo) >> 1);
    int c = 0;
    for (int i = lane; i < len; i += 32) c += kr[i] <= mid ? 1 : 0;
#pragma unroll
    for (int o = 16; o >= 1; o /= 2) c += __shfl_xor_sync(kFullMask, c, o);
    if (c >= k) hi = mid;
    else lo = mid + 1;
  }
  if (lane == 0) theta[row] = lo;
}

// The k smallest of a query's nearest-list result (k entries, ascending,
// (+inf, -1) padded) and its candidates from the other lists; one block per
// query, a bitonic sort of the <= k + cap entries in shared memory. A query
// whose candidates overflowed the buffer is flagged for the full rescan.
// With `only` set, just the queries with only[q] == 2 (those the radix
// selection below could not finish).
__global__ void lm_final_kernel(const float* __restrict__ pre_d, const int64_t* __restrict__ pre_i,
                                int k, const uint32_t* __restrict__ ckey,
                                const int64_t* __restrict__ cid, const int* __restrict__ ccount,
                                int cap, float* __restrict__ out_d, int64_t* __restrict__ out_i,
                                int* flags, const int* only) {
  extern __shared__ uint32_t lmf_smem[];
  const int64_t q = blockIdx.x;
  if (only && only[q] != 2) return;  // the same for the whole block
  const int cnt = ccount[q];
  const int n2 = max(0, min(cnt, cap));
  const int total = k + n2;
  int T = 32;
  while (T < total) T *= 2;
  uint32_t* sk = lmf_smem;
  uint32_t* sv = lmf_smem + T;
  for (int i = threadIdx.x; i < T; i += blockDim.x) {
    uint32_t key = kSentinelKey;
    if (i < k) {
      if (pre_i && pre_i[q * k + i] >= 0) key = __float_as_uint(pre_d[q * k + i]);
    } else if (i < total) {
      key = ckey[q * cap + (i - k)];
    }
    sk[i] = key;
    sv[i] = uint32_t(i);
  }
  __syncthreads();
  for (int size = 2; size <= T; size *= 2) {
    for (int st = size / 2; st >= 1; st /= 2) {
      for (int c = threadIdx.x; c < T / 2; c += blockDim.x) {
        const int lo = 2 * c - (c & (st - 1));
        const int hi = lo + st;
        const bool up = (lo & size) == 0;
        const uint32_t a = sk[lo], b = sk[hi];
        if ((a > b) == up) {
          sk[lo] = b;
          sk[hi] = a;
          const uint32_t t = sv[lo];
          sv[lo] = sv[hi];
          sv[hi] = t;
        }
      }
      __syncthreads();
    }
  }
  for (int i = threadIdx.x; i < k; i += blockDim.x) {
    const uint32_t key = sk[i];
    const uint32_t src = sv[i];
    out_d[q * k + i] = dist_key_to_float(key);
    out_i[q * k + i] = key == kSentinelKey ? int64_t(-1)
                       : src < uint32_t(k) ? pre_i[q * k + src]
                                           : cid[q * cap + (src - k)];
  }
  if (threadIdx.x == 0) flags[q] = cnt > cap ? 1 : 0;
}

// The k smallest of each query's candidates for long k: a radix bound of the
// k-th (select_radix.cuh), the candidates under it gathered into a buffer of
// B entries and sorted there (the full bitonic sort of all k + cap entries
// took 0.82 ms per 10,000 queries at k = 1000). flags[q] = 1 where the
// candidates overflowed (the full rescan writes that query), 2 where more
// than B lie under the bound (lm_final_kernel sorts them all), else 0.
__global__ void __launch_bounds__(radix::kRThreads)
lm_final_radix_kernel(int k, const uint32_t* __restrict__ ckey, const int64_t* __restrict__ cid,
                      const int* __restrict__ ccount, int cap, int B, float* __restrict__ out_d,
                      int64_t* __restrict__ out_i, int* __restrict__ flags) {
  extern __shared__ uint32_t lmr_smem[];
  uint32_t* hist = lmr_smem;
  uint32_t* sk = hist + radix::kRBins;
  uint32_t* sv = sk + B;
  __shared__ radix::RadixShared sh;
  const int64_t q = blockIdx.x;
  const int cnt = ccount[q];
  if (cnt > cap) {  // the same for the whole block
    if (threadIdx.x == 0) flags[q] = 1;
    return;
  }
  const int n2 = max(cnt, 0);
  const uint32_t* kr = ckey + q * cap;
  const uint32_t theta = radix::radix_theta(hist, sh, uint32_t(k), [&](auto f) {
    for (int i = threadIdx.x; i < n2; i += radix::kRThreads) f(kr[i]);
  });
  if (threadIdx.x == 0) sh.count = 0;
  __syncthreads();
  for (int i = threadIdx.x; i < n2; i += radix::kRThreads) {
    const uint32_t key = kr[i];
    if (key <= theta) {
      const uint32_t pos = atomicAdd(&sh.count, 1u);
      if (pos < uint32_t(B)) {
        sk[pos] = key;
        sv[pos] = uint32_t(i);
      }
    }
  }
  __syncthreads();
  const uint32_t n = sh.count;
  if (n > uint32_t(B)) {  // the same for the whole block
    if (threadIdx.x == 0) flags[q] = 2;
    return;
  }
  uint32_t P = 32;
  while (P < n) P <<= 1;
  for (uint32_t i = n + threadIdx.x; i < P; i += radix::kRThreads) {
    sk[i] = kSentinelKey;
    sv[i] = kSentinelIdx;
  }
  __syncthreads();
  radix::bitonic_sort(sk, sv, P);
  for (int i = threadIdx.x; i < k; i += radix::kRThreads) {
    const uint32_t key = uint32_t(i) < P ? sk[i] : kSentinelKey;
    out_d[q * k + i] = dist_key_to_float(key);
    out_i[q * k + i] = key == kSentinelKey ? int64_t(-1) : cid[q * cap + sv[i]];
  }
  if (threadIdx.x == 0) flags[q] = 0;
}

int coarse_stage(const ivfpq_index* ix, const float* queries, int64_t nq, int nprobe,
                 int32_t* probes, float* coarse, cudaStream_t s) {
  SelectOut o;
  o.kind = OutKind::Probes;
  o.idx32 = probes;
  o.vals = coarse;
  TcOperand xo;
  xo.hi = ix->cent_hi;
  xo.lo = ix->cent_lo;
  xo.norms = ix->cent_norms;
  return knn_by_tiles(queries, nq, ix->centroids, ix->nlist, ix->d, nprobe, o, s,
                      ix->cent_hi ? &xo : nullptr);
}

// Lists per block: enough blocks to give every SM several waves.
void plan_chunks(int64_t nq, int nprobe, int* per_chunk, int* nchunks) {
  const int64_t target = int64_t(num_sms()) * 3 * 8;
  int64_t c = std::max<int64_t>(1, std::min<int64_t>(nprobe, ceil_div(target, std::max<int64_t>(nq, 1))));
  int pc = int(ceil_div(nprobe, c));
  *per_chunk = pc;
  *nchunks = int(ceil_div(nprobe, pc));
}

ScanParams scan_params(const ivfpq_index* ix, const float* queries, int64_t nq, int nprobe,
                       const int32_t* probes, int k) {
  ScanParams p;
  p.queries = queries;
  p.centroids = ix->centroids;
  p.codebooks_t = ix->codebooks;
  p.probes = probes;
  p.list_len = ix->list_len;
  p.list_block_off = ix->list_block_off;
  p.codes = ix->codes;
  p.d = ix->d;
  p.m = ix->m;
  p.dsub = ix->dsub;
  p.dsub4 = ix->dsub4;
  p.nlist = ix->nlist;
  p.nprobe = nprobe;
  p.k = k;
  p.lut_type = ix->lut_type;
  p.nq = nq;
  p.nblocks = ix->nblocks;
#ifdef IVFPQ_DEBUG_CHECKS
  if (device_status_word(&p.dbg) != IVFPQ_OK) p.dbg = nullptr;
#endif
  plan_chunks(nq, nprobe, &p.per_chunk, &p.nchunks);
  return p;
}

// Re-scans, with the general kernel and full-length queues, the queries
// flagged in `flags` (device, [nq]) and overwrites their results.
int repair_stage(const ScanParams& p0, int64_t nq, int* flags, const SelectOut& o, Workspace& ws,
                 cudaStream_t s) {
  ScanParams r = p0;
  r.term1 = nullptr;
  plan_chunks(nq, r.nprobe, &r.per_chunk, &r.nchunks);
  r.qmask = flags;
  const size_t nr = size_t(nq) * r.nchunks * r.k;
  IVFPQ_TRY(ws.alloc(&r.pkeys, nr));
  IVFPQ_TRY(ws.alloc(&r.pidx, nr));
  IVFPQ_TRY(launch_scan_general(r, nq, s));
  SelectOut ro = o;
  ro.row_mask = flags;
  const int64_t rlen = int64_t(r.nchunks) * r.k;
  return select_pairs(r.pkeys, r.pidx, nq, rlen, r.k, 1, rlen, ro, s);
}

// The list scan organised by query: one block per (query, chunk of lists).
int scan_stage_qm(const ivfpq_index* ix, const float* queries, int64_t nq, int nprobe,
                  const int32_t* probes, int k, float* out_dist, int64_t* out_ids,
                  cudaStream_t s, bool timed) {
  ScanParams p = scan_params(ix, queries, nq, nprobe, probes, k);
  if (use_precomputed(ix)) p.term1 = ix->term1;
  Workspace ws(s);
  SelectOut o;
  o.kind = OutKind::Dist;
  o.vals = out_dist;
  o.idx64 = out_ids;
  o.id_map = ix->ids;
  auto* mix = const_cast<ivfpq_index*>(ix);
  if (!scan2_shape(p)) {
    const size_t np = size_t(nq) * p.nchunks * k;
    IVFPQ_TRY(ws.alloc(&p.pkeys, np));
    IVFPQ_TRY(ws.alloc(&p.pidx, np));
    if (timed) record(ix, 2, s);
    IVFPQ_TRY(launch_scan_general(p, nq, s));
    mix->last_scan_kernel.store("ivfpq_scan_kernel");
    if (timed) record(ix, 3, s);
    const int64_t len = int64_t(p.nchunks) * k;
    IVFPQ_TRY(select_pairs(p.pkeys, p.pidx, nq, len, k, 1, len, o, s));
    if (timed) record(ix, 4, s);
    return IVFPQ_OK;
  }
  // register-codebook kernel: per-warp queues of kw entries, unmerged; at
  // most kScan2MaxLists lists per block
  if (p.per_chunk > kScan2MaxLists) {
    p.per_chunk = kScan2MaxLists;
    p.nchunks = int(ceil_div(nprobe, kScan2MaxLists));
  }
  const int kw = scan2_kw(k);
  const int groups = p.nchunks * kScan2Warps;
  const size_t np = size_t(nq) * groups * kw;
  IVFPQ_TRY(ws.alloc(&p.pkeys, np));
  IVFPQ_TRY(ws.alloc(&p.pidx, np));
  if (timed) record(ix, 2, s);
  int launched = 0;
  switch (kw) {
    case 32: IVFPQ_TRY(try_scan2_kw<32>(p, nq, s, &launched)); break;
    case 64: IVFPQ_TRY(try_scan2_kw<64>(p, nq, s, &launched)); break;
    case 128: IVFPQ_TRY(try_scan2_kw<128>(p, nq, s, &launched)); break;
    default: IVFPQ_TRY(try_scan2_kw<256>(p, nq, s, &launched)); break;
  }
  IVFPQ_REQUIRE(launched, "scan: no register-codebook kernel for m=%d d/m=%d", p.m, p.dsub);
  mix->last_scan_kernel.store("ivfpq_scan2_kernel");
  if (timed) record(ix, 3, s);
  IVFPQ_TRY(merge_sorted_runs(p.pkeys, p.pidx, nq, groups, kw, k, o, s));
  if (kw < k) {
    // repair the queries whose merged result a short queue may have cut
    int* flags = nullptr;
    IVFPQ_TRY(ws.alloc(&flags, size_t(nq)));
    warp_queue_check_kernel<<<unsigned(ceil_div(nq, 256)), 256, 0, s>>>(
        p.pkeys, nq, groups, kw, out_dist, k, flags, ix->repaired);
    IVFPQ_LAUNCHED();
    IVFPQ_TRY(repair_stage(p, nq, flags, o, ws, s));
  }
  if (timed) record(ix, 4, s);
  return IVFPQ_OK;
}

// Whether a search takes the list-major scan: its shapes (as the
// register-codebook scan, fp32 tables, direct tables), at least two probes,
// and (automatic mode) on average at least two queries per probed list.
bool use_list_major(const ivfpq_index* ix, int64_t nq, int nprobe) {
  if (ix->scan_mode == 0 || nprobe < 2 || nq < 1 || ix->precomputed == 1) return false;
  ScanParams p;
  p.m = ix->m;
  p.dsub = ix->dsub;
  p.d = ix->d;
  p.k = 1;
  p.lut_type = ix->lut_type;
  p.lut_type = IVFPQ_LUT_FP32;  // by list: fp32, binary16 or E4M3 tables, the same shapes
  if (!scan2_shape(p)) return false;
  if (ix->scan_mode == 1) return true;
  return double(nq) * nprobe >= 2.0 * ix->nlist;
}

// (list, query) pairs of probes [p0, p0 + per) sorted by list and cut into
// items of up to G pairs of one list (into lp's pair and item arrays).
int plan_items(const int32_t* probes, int64_t nq, int nprobe, int p0, int per, int G, int nlist,
               Workspace& ws, cudaStream_t s, LmParams& lp) {
  const int64_t npairs = nq * per;
  IVFPQ_REQUIRE(npairs < (int64_t(1) << 31), "scan: %lld (list, query) pairs", (long long)npairs);
  int32_t *key = nullptr, *val = nullptr, *skey = nullptr, *sval = nullptr;
  int32_t *flag = nullptr, *pos = nullptr, *items = nullptr;
  int* n_items = nullptr;
  IVFPQ_TRY(ws.alloc(&key, size_t(npairs)));
  IVFPQ_TRY(ws.alloc(&val, size_t(npairs)));
  IVFPQ_TRY(ws.alloc(&skey, size_t(npairs)));
  IVFPQ_TRY(ws.alloc(&sval, size_t(npairs)));
  IVFPQ_TRY(ws.alloc(&flag, size_t(npairs)));
  IVFPQ_TRY(ws.alloc(&pos, size_t(npairs)));
  IVFPQ_TRY(ws.alloc(&items, size_t(npairs)));
  IVFPQ_TRY(ws.alloc(&n_items, 1));
  const unsigned pg = unsigned(std::max<int64_t>(1, std::min<int64_t>(ceil_div(npairs, 256),
                                                                    int64_t(num_sms()) * 16)));
  lm_pairs_kernel<<<pg, 256, 0, s>>>(probes, nq, nprobe, p0, per, nlist, key, val);
  IVFPQ_LAUNCHED();
  int end_bit = 1;
  while ((int64_t(1) << end_bit) <= nlist) ++end_bit;
  size_t sort_bytes = 0, scan_bytes = 0;
  IVFPQ_CUDA(cub::DeviceRadixSort::SortPairs(nullptr, sort_bytes, key, skey, val, sval, npairs, 0,
                                             end_bit, s));
  IVFPQ_CUDA(cub::DeviceScan::ExclusiveSum(nullptr, scan_bytes, flag, pos, npairs, s));
  uint8_t* tmp = nullptr;
  IVFPQ_TRY(ws.alloc(&tmp, std::max(sort_bytes, scan_bytes)));
  IVFPQ_CUDA(cub::DeviceRadixSort::SortPairs(tmp, sort_bytes, key, skey, val, sval, npairs, 0,
                                             end_bit, s));
  lm_item_flags_kernel<<<pg, 256, 0, s>>>(skey, npairs, G, nlist, flag);
  IVFPQ_LAUNCHED();
  IVFPQ_CUDA(cub::DeviceScan::ExclusiveSum(tmp, scan_bytes, flag, pos, npairs, s));
  lm_items_kernel<<<pg, 256, 0, s>>>(flag, pos, npairs, items, n_items);
  IVFPQ_LAUNCHED();
  lp.pair_list = skey;
  lp.pair_query = sval;
  lp.items = items;
  lp.n_items = n_items;
  lp.npairs = npairs;
  return IVFPQ_OK;
}

// The filter pass scans a list longer than kLmUnitMin codes in chunks
// (units) of unit_len codes, at most kLmMaxChunks per record, so that the
// few items of a long list (the largest of a Zipf mixture holds ~1e6 codes)
// do not keep a few blocks busy after the rest have finished.
constexpr int64_t kLmUnitMin = 65536;

// cnt[r] = units of record r (0 past the last record)
__global__ void lm_unit_count_kernel(const uint8_t* __restrict__ records, int rec_bytes,
                                     const int* __restrict__ n_items, int64_t nmax, int unit_len,
                                     int32_t* __restrict__ cnt) {
  const int64_t r = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (r >= nmax) return;
  int c = 0;
  if (r < *n_items) {
    const int len = reinterpret_cast<const LmHead*>(records + r * rec_bytes)->len;
    c = max(1, min(kLmMaxChunks, (len + unit_len - 1) / unit_len));
  }
  cnt[r] = c;
}

// units[off[r] + c] = r * kLmMaxChunks + c for c < cnt[r]; *n_units = total
// (at most cap: the rest are dropped and counted as a debug-check failure,
// which the host's bound excludes)
__global__ void lm_units_kernel(const int32_t* __restrict__ cnt, const int32_t* __restrict__ off,
                                int64_t nmax, int64_t cap, int32_t* __restrict__ units,
                                int* __restrict__ n_units, int* dbg) {
  const int64_t r = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (r >= nmax) return;
  if (r == nmax - 1) {
    const int64_t total = int64_t(off[r]) + cnt[r];
    dcheck(dbg, total <= cap, 12);
    *n_units = int(min(total, cap));
  }
  for (int c = 0; c < cnt[r]; ++c)
    if (off[r] + c < cap) units[off[r] + c] = int32_t(r * kLmMaxChunks + c);
}

// Item records (scan_lm.cuh, lm_records_kernel) for the items of lp, after
// lp's bounds are set; room for one record per pair (the item count stays on
// the device).
int make_records(LmParams& lp, int G, bool bound_pass, Workspace& ws, cudaStream_t s) {
  lp.dpad = (lp.s.d + 3) & ~3;
  lp.rec_bytes = lm_record_bytes(G, lp.s.d);
  uint8_t* rec = nullptr;
  IVFPQ_TRY(ws.alloc(&rec, size_t(std::max<int64_t>(lp.npairs, 1)) * lp.rec_bytes));
  const unsigned rg = unsigned(std::max<int64_t>(
      1, std::min<int64_t>(ceil_div(lp.npairs, 8), int64_t(num_sms()) * 16)));
  lm_records_kernel<<<rg, 256, 0, s>>>(lp, G, bound_pass, rec);
  IVFPQ_LAUNCHED();
  lp.records = rec;
  return IVFPQ_OK;
}

// The list scan organised by list (scan_lm.cuh): a bound pass over every
// query's nearest list, a filter pass over all its lists, one selection per
// query over its candidates, and the full rescan of queries whose candidates
// overflowed.
int scan_stage_lm(const ivfpq_index* ix, const float* queries, int64_t nq, int nprobe,
                  const int32_t* probes, int k, float* out_dist, int64_t* out_ids,
                  cudaStream_t s) {
  auto* mix = const_cast<ivfpq_index*>(ix);
  Workspace ws(s);
  const ScanParams base = scan_params(ix, queries, nq, nprobe, probes, k);
  // 1. bound pass: per query and chunk of its nearest list, 512 lane queues
  //    of tq (512 * tq >= 2k), and the k-th smallest of their entries
  const int tq = k <= 512 ? 2 : k <= 1024 ? 4 : 8;
  LmParams bp;
  bp.s = base;
  int32_t *bcnt = nullptr, *boffs = nullptr;
  int* bn_items = nullptr;
  IVFPQ_TRY(ws.alloc(&bcnt, size_t(nq)));
  IVFPQ_TRY(ws.alloc(&boffs, size_t(nq)));
  IVFPQ_TRY(ws.alloc(&bn_items, 1));
  // chunks of at least 32,768 codes, at most 4 per query
  int64_t chunk = std::max<int64_t>(kBoundChunkMin, ceil_div(ix->max_list_len, kBoundChunksMax));
  chunk = ceil_div(chunk, 32) * 32;
  IVFPQ_REQUIRE(chunk < (int64_t(1) << 30), "scan: list of %lld vectors", (long long)ix->max_list_len);
  bound_chunks_kernel<<<unsigned(ceil_div(nq, 256)), 256, 0, s>>>(probes, nq, nprobe, ix->list_len,
                                                                 ix->nlist, int(chunk), bcnt);
  IVFPQ_LAUNCHED();
  {
    size_t sb = 0;
    IVFPQ_CUDA(cub::DeviceScan::ExclusiveSum(nullptr, sb, bcnt, boffs, nq, s));
    uint8_t* st = nullptr;
    IVFPQ_TRY(ws.alloc(&st, sb));
    IVFPQ_CUDA(cub::DeviceScan::ExclusiveSum(st, sb, bcnt, boffs, nq, s));
  }
  const int64_t max_items = nq * std::max<int64_t>(1, ceil_div(ix->max_list_len, chunk));
  bp.dpad = (base.d + 3) & ~3;
  bp.rec_bytes = lm_record_bytes(1, base.d);
  bp.n_items = bn_items;
  IVFPQ_TRY(ws.alloc(&bp.records_w, size_t(max_items) * bp.rec_bytes));
  bp.records = bp.records_w;
  bound_records_kernel<<<unsigned(ceil_div(nq, 8)), 256, 0, s>>>(bp, nprobe, int(chunk), boffs,
                                                                bcnt, bp.records_w, bn_items);
  IVFPQ_LAUNCHED();
  // items by decreasing length where list lengths are skewed (the longest
  // over 4x the mean): block b takes items b, b + B, ..., so each block's
  // total exceeds the mean by at most one item (in query order the Zipf-sized
  // lists left some blocks several long chunks: billion bound pass and
  // planning 1.82 -> 1.02 ms; with even lists the sort only costs, large
  // 0.56 -> 0.64 ms)
  if (ix->nlist > 0 && ix->max_list_len > 4 * ceil_div(ix->ntotal, int64_t(ix->nlist))) {
    int32_t *ilen = nullptr, *ilen_s = nullptr, *iidx = nullptr, *order = nullptr;
    IVFPQ_TRY(ws.alloc(&ilen, size_t(max_items)));
    IVFPQ_TRY(ws.alloc(&ilen_s, size_t(max_items)));
    IVFPQ_TRY(ws.alloc(&iidx, size_t(max_items)));
    IVFPQ_TRY(ws.alloc(&order, size_t(max_items)));
    bound_order_keys_kernel<<<unsigned(ceil_div(max_items, 256)), 256, 0, s>>>(
        bp.records_w, bp.rec_bytes, bn_items, max_items, ilen, iidx);
    IVFPQ_LAUNCHED();
    size_t sb = 0;
    IVFPQ_CUDA(cub::DeviceRadixSort::SortPairsDescending(nullptr, sb, ilen, ilen_s, iidx, order,
                                                         int(max_items), 0, 32, s));
    uint8_t* st = nullptr;
    IVFPQ_TRY(ws.alloc(&st, sb));
    IVFPQ_CUDA(cub::DeviceRadixSort::SortPairsDescending(st, sb, ilen, ilen_s, iidx, order,
                                                         int(max_items), 0, 32, s));
    bp.order = order;
  }
  const int64_t plen = int64_t(kLmWarps) * 32 * tq;  // keys per item
  IVFPQ_TRY(ws.alloc(&bp.part_key, size_t(max_items) * plen));
  int launched = 0;
  const bool half = ix->lut_type == IVFPQ_LUT_FP16;
  const bool e4m3 = ix->lut_type == IVFPQ_LUT_FP8;
  if (half) IVFPQ_TRY(launch_bound_pass<IVFPQ_LUT_FP16>(bp, tq, s, &launched));
  else if (e4m3) IVFPQ_TRY(launch_bound_pass<IVFPQ_LUT_FP8>(bp, tq, s, &launched));
  else IVFPQ_TRY(launch_bound_pass<IVFPQ_LUT_FP32>(bp, tq, s, &launched));
  IVFPQ_REQUIRE(launched, "scan: no list-major kernel for m=%d d/m=%d", ix->m, ix->dsub);
  uint32_t* theta = nullptr;
  IVFPQ_TRY(ws.alloc(&theta, size_t(nq)));
  lm_theta_kernel<<<unsigned(ceil_div(nq, 8)), 256, 0, s>>>(bp.part_key, nq, boffs, bcnt,
                                                            int(plen), k, theta);
  IVFPQ_LAUNCHED();
  // 2. filter pass over all the probed lists
  LmParams lp;
  lp.s = base;
  // table sets per item (fp32: one query each, binary16: two); automatic:
  // the fastest measured (search ms, 10,000 queries, 2 / 3 sets: fp32 large
  // 13.02 / 12.29; binary16 billion 21.40 / 20.06, large 10.73 / 10.66, mid
  // 7.72 / 8.45)
  // (E4M3: four queries per set, at most two sets)
  const int sets = e4m3 ? std::min(ix->lm_group ? ix->lm_group : 2, 2)
                        : ix->lm_group ? ix->lm_group : (half && ix->m == 16) ? 2 : 3;
  const int G = sets * (e4m3 ? 4 : half ? 2 : 1);
  IVFPQ_TRY(plan_items(probes, nq, nprobe, 0, nprobe, G, ix->nlist, ws, s, lp));
  const int cap = std::max(1024, 2 * k);
  lp.theta_key = theta;
  lp.theta_stride = 1;
  lp.ids = ix->ids;
  lp.cap = cap;
  IVFPQ_TRY(make_records(lp, G, false, ws, s));
  // chunks where the longest list is over 5% of a block's mean share of the
  // codes scanned (estimated from the mean list length): billion (1e9 codes,
  // Zipf, nprobe 128) 0.19, filter 12.03 -> 11.21 ms; mid (1e7, Zipf,
  // nprobe 64) 0.03, where chunking measured 5.25 -> 5.45 ms
  const double block_share = double(nq) * nprobe * (double(ix->ntotal) / std::max(1, ix->nlist)) /
                             (double(G) * num_sms());
  if (ix->unit_len > 0 && double(ix->max_list_len) > 0.05 * block_share) {
    // units: at most kLmMaxChunks per record, and beyond one per record at
    // most the lists' extra chunks once per group of G of the nq queries
    const int64_t nrec = std::max<int64_t>(lp.npairs, 1);
    const int64_t cap = std::min<int64_t>(nrec * kLmMaxChunks, nrec + ix->unit_extra * ceil_div(nq, G));
    IVFPQ_REQUIRE(cap < (int64_t(1) << 31) / kLmMaxChunks, "scan: %lld work units", (long long)cap);
    int32_t *ucnt = nullptr, *uoff = nullptr, *units = nullptr;
    int* n_units = nullptr;
    IVFPQ_TRY(ws.alloc(&ucnt, size_t(nrec)));
    IVFPQ_TRY(ws.alloc(&uoff, size_t(nrec)));
    IVFPQ_TRY(ws.alloc(&units, size_t(cap)));
    IVFPQ_TRY(ws.alloc(&n_units, 1));
    const unsigned ug = unsigned(ceil_div(nrec, 256));
    lm_unit_count_kernel<<<ug, 256, 0, s>>>(lp.records, lp.rec_bytes, lp.n_items, nrec,
                                            int(ix->unit_len), ucnt);
    IVFPQ_LAUNCHED();
    size_t sb = 0;
    IVFPQ_CUDA(cub::DeviceScan::ExclusiveSum(nullptr, sb, ucnt, uoff, nrec, s));
    uint8_t* st = nullptr;
    IVFPQ_TRY(ws.alloc(&st, sb));
    IVFPQ_CUDA(cub::DeviceScan::ExclusiveSum(st, sb, ucnt, uoff, nrec, s));
    lm_units_kernel<<<ug, 256, 0, s>>>(ucnt, uoff, nrec, cap, units, n_units, lp.s.dbg);
    IVFPQ_LAUNCHED();
    lp.units = units;
    lp.n_units = n_units;
    lp.unit_len = int(ix->unit_len);
  }
  IVFPQ_TRY(ws.alloc(&lp.ckey, size_t(nq) * cap));
  IVFPQ_TRY(ws.alloc(&lp.cid, size_t(nq) * cap));
  IVFPQ_TRY(ws.alloc(&lp.ccount, size_t(nq)));
  IVFPQ_CUDA(cudaMemsetAsync(lp.ccount, 0, size_t(nq) * sizeof(int), s));
  // stage timing: the bound pass and the planning count as stage 1, the
  // filter kernel alone as stage 2
  record(ix, 2, s);
  if (e4m3) {
    if (G >= 8) IVFPQ_TRY((try_scan_lm<8, 0, IVFPQ_LUT_FP8>(lp, s, &launched)));
    else IVFPQ_TRY((try_scan_lm<4, 0, IVFPQ_LUT_FP8>(lp, s, &launched)));
  } else if (half) {
    if (G >= 6) IVFPQ_TRY((try_scan_lm<6, 0, IVFPQ_LUT_FP16>(lp, s, &launched)));
    else IVFPQ_TRY((try_scan_lm<4, 0, IVFPQ_LUT_FP16>(lp, s, &launched)));
  } else {
    if (G >= 3) IVFPQ_TRY((try_scan_lm<3, 0, IVFPQ_LUT_FP32>(lp, s, &launched)));
    else IVFPQ_TRY((try_scan_lm<2, 0, IVFPQ_LUT_FP32>(lp, s, &launched)));
  }
  IVFPQ_REQUIRE(launched, "scan: no list-major kernel for m=%d d/m=%d", ix->m, ix->dsub);
  mix->last_scan_kernel.store("ivfpq_scan_lm_kernel");
  record(ix, 3, s);
  // 3. the k smallest candidates of each query
  int* flags = nullptr;
  IVFPQ_TRY(ws.alloc(&flags, size_t(nq)));
  int T = 32;
  while (T < k + cap) T *= 2;
  const size_t fsm = size_t(T) * 8;
  IVFPQ_TRY(set_dynamic_smem(lm_final_kernel, fsm));
  if (k > 256) {
    // a radix bound, then the full sort only for the queries it flags 2
    int B = 32;
    while (B < 2 * k) B *= 2;
    const size_t rsm = (size_t(radix::kRBins) + 2 * size_t(B)) * 4;
    IVFPQ_TRY(set_dynamic_smem(lm_final_radix_kernel, rsm));
    lm_final_radix_kernel<<<unsigned(nq), radix::kRThreads, rsm, s>>>(
        k, lp.ckey, lp.cid, lp.ccount, cap, B, out_dist, out_ids, flags);
    IVFPQ_LAUNCHED_K(lm_final_radix_kernel, rsm, radix::kRThreads);
  }
  lm_final_kernel<<<unsigned(nq), 256, fsm, s>>>(nullptr, nullptr, k, lp.ckey, lp.cid, lp.ccount,
                                                 cap, out_dist, out_ids, flags,
                                                 k > 256 ? flags : nullptr);
  IVFPQ_LAUNCHED_K(lm_final_kernel, fsm, 256);
  // 4. queries whose candidates overflowed: full rescan
  count_flags_kernel<<<unsigned(ceil_div(nq, 256)), 256, 0, s>>>(flags, nq, ix->repaired);
  IVFPQ_LAUNCHED();
  SelectOut o;
  o.kind = OutKind::Dist;
  o.vals = out_dist;
  o.idx64 = out_ids;
  o.id_map = ix->ids;
  IVFPQ_TRY(repair_stage(base, nq, flags, o, ws, s));
  record(ix, 4, s);
  return IVFPQ_OK;
}

int scan_stage(const ivfpq_index* ix, const float* queries, int64_t nq, int nprobe,
               const int32_t* probes, int k, float* out_dist, int64_t* out_ids, cudaStream_t s) {
  if (use_list_major(ix, nq, nprobe))
    return scan_stage_lm(ix, queries, nq, nprobe, probes, k, out_dist, out_ids, s);
  return scan_stage_qm(ix, queries, nq, nprobe, probes, k, out_dist, out_ids, s, true);
}

int check_common(const ivfpq_index* ix, const float* queries, int64_t nq, int nprobe,
                 const char* who) {
  IVFPQ_REQUIRE(ix, "%s: null index", who);
  IVFPQ_REQUIRE(nq >= 0, "%s: negative nq", who);
  IVFPQ_REQUIRE(nq < (int64_t(1) << 31), "%s: nq=%lld too large", who, (long long)nq);
  IVFPQ_REQUIRE(nprobe >= 1 && nprobe <= ix->nlist && nprobe <= IVFPQ_MAX_K,
                "%s: nprobe=%d outside [1, min(nlist=%d, %d)]", who, nprobe, ix->nlist,
                IVFPQ_MAX_K);
  IVFPQ_REQUIRE(queries || nq == 0, "%s: null queries", who);
  return IVFPQ_OK;
}

void reset_events(const ivfpq_index* ix) { begin_profile(ix); }

// Row r of a [rows, k + 1] result without the entry whose id is self[r] (or
// without its last entry when self[r] is absent) -> [rows, k]. One thread per
// row.
__global__ void drop_self_kernel(const float* __restrict__ d1, const int64_t* __restrict__ i1,
                                 int64_t rows, int k, const int64_t* __restrict__ self,
                                 float* __restrict__ d, int64_t* __restrict__ id) {
  const int64_t r = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (r >= rows) return;
  const int64_t me = self[r];
  const float* dr = d1 + r * (k + 1);
  const int64_t* ir = i1 + r * (k + 1);
  int o = 0;
  bool dropped = false;
  for (int j = 0; j <= k && o < k; ++j) {
    if (!dropped && ir[j] == me && me >= 0) {
      dropped = true;
      continue;
    }
    d[r * k + o] = dr[j];
    id[r * k + o] = ir[j];
    ++o;
  }
}

}  // namespace

void update_list_units(ivfpq_index* ix) {
  ix->unit_len = 0;
  ix->unit_extra = 0;
  if (ix->max_list_len <= kLmUnitMin) return;
  ix->unit_len = ceil_div(std::max(kLmUnitMin, ceil_div(ix->max_list_len, kLmMaxChunks)), 32) * 32;
  for (const int64_t len : ix->h_list_len)
    ix->unit_extra += std::max<int64_t>(0, ceil_div(len, ix->unit_len) - 1);
}

}  // namespace ivfpq

using namespace ivfpq;

extern "C" int ivfpq_search(const ivfpq_index* ix, const float* queries, int64_t nq, int nprobe,
                            int k, float* out_dist, int64_t* out_ids, void* stream) {
  clear_error();
  IVFPQ_TRY(check_common(ix, queries, nq, nprobe, "ivfpq_search"));
  IVFPQ_REQUIRE(k >= 1 && k <= IVFPQ_MAX_K, "ivfpq_search: k=%d outside [1, %d]", k, IVFPQ_MAX_K);
  if (nq == 0) return IVFPQ_OK;
  IVFPQ_REQUIRE(out_dist && out_ids, "ivfpq_search: null output");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  reset_events(ix);
  Workspace ws(s);
  int32_t* probes;
  IVFPQ_TRY(ws.alloc(&probes, size_t(nq) * nprobe));
  record(ix, 0, s);
  IVFPQ_TRY(coarse_stage(ix, queries, nq, nprobe, probes, nullptr, s));
  record(ix, 1, s);
  return scan_stage(ix, queries, nq, nprobe, probes, k, out_dist, out_ids, s);
}

extern "C" int ivfpq_knn_graph(const ivfpq_index* ix, const float* x, const int64_t* self_ids,
                               int64_t n, int nprobe, int k, float* out_dist, int64_t* out_ids,
                               void* stream) {
  clear_error();
  IVFPQ_TRY(check_common(ix, x, n, nprobe, "ivfpq_knn_graph"));
  IVFPQ_REQUIRE(k >= 1 && k < IVFPQ_MAX_K, "ivfpq_knn_graph: k=%d outside [1, %d]", k,
                IVFPQ_MAX_K - 1);
  if (n == 0) return IVFPQ_OK;
  IVFPQ_REQUIRE(self_ids && out_dist && out_ids, "ivfpq_knn_graph: null pointer");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  reset_events(ix);
  // batches of queries bound the temporary memory
  const int64_t batch = std::min<int64_t>(n, 32768);
  Workspace ws(s);
  int32_t* probes = nullptr;
  float* d1 = nullptr;
  int64_t* i1 = nullptr;
  IVFPQ_TRY(ws.alloc(&probes, size_t(batch) * nprobe));
  IVFPQ_TRY(ws.alloc(&d1, size_t(batch) * (k + 1)));
  IVFPQ_TRY(ws.alloc(&i1, size_t(batch) * (k + 1)));
  for (int64_t b0 = 0; b0 < n; b0 += batch) {
    const int64_t rows = std::min(batch, n - b0);
    const float* xb = x + b0 * ix->d;
    IVFPQ_TRY(coarse_stage(ix, xb, rows, nprobe, probes, nullptr, s));
    IVFPQ_TRY(scan_stage(ix, xb, rows, nprobe, probes, k + 1, d1, i1, s));
    drop_self_kernel<<<unsigned(ceil_div(rows, 256)), 256, 0, s>>>(
        d1, i1, rows, k, self_ids + b0, out_dist + b0 * k, out_ids + b0 * k);
    IVFPQ_LAUNCHED();
  }
  return IVFPQ_OK;
}

extern "C" int ivfpq_search_probes(const ivfpq_index* ix, const float* queries, int64_t nq,
                                   int nprobe, int32_t* out_probes, float* out_coarse,
                                   void* stream) {
  clear_error();
  IVFPQ_TRY(check_common(ix, queries, nq, nprobe, "ivfpq_search_probes"));
  if (nq == 0) return IVFPQ_OK;
  IVFPQ_REQUIRE(out_probes, "ivfpq_search_probes: null output");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  reset_events(ix);
  record(ix, 0, s);
  IVFPQ_TRY(coarse_stage(ix, queries, nq, nprobe, out_probes, out_coarse, s));
  record(ix, 1, s);
  return IVFPQ_OK;
}

extern "C" int ivfpq_search_preassigned(const ivfpq_index* ix, const float* queries, int64_t nq,
                                        int nprobe, const int32_t* probes, int k,
                                        float* out_dist, int64_t* out_ids, void* stream) {
  clear_error();
  IVFPQ_REQUIRE(ix, "ivfpq_search_preassigned: null index");
  IVFPQ_REQUIRE(nq >= 0 && nq < (int64_t(1) << 31), "ivfpq_search_preassigned: bad nq");
  IVFPQ_REQUIRE(nprobe >= 1 && nprobe <= (1 << 20), "ivfpq_search_preassigned: bad nprobe=%d",
                nprobe);
  IVFPQ_REQUIRE(k >= 1 && k <= IVFPQ_MAX_K, "ivfpq_search_preassigned: k=%d outside [1, %d]", k,
                IVFPQ_MAX_K);
  if (nq == 0) return IVFPQ_OK;
  IVFPQ_REQUIRE(queries && probes && out_dist && out_ids, "ivfpq_search_preassigned: null pointer");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  reset_events(ix);
  return scan_stage(ix, queries, nq, nprobe, probes, k, out_dist, out_ids, s);
}

extern "C" int ivfpq_set_profiling(ivfpq_index* ix, int enable) {
  clear_error();
  IVFPQ_REQUIRE(ix, "ivfpq_set_profiling: null index");
  ix->profile = enable != 0;
  ix->ev_used = 0;
  ix->cur_set = -1;
  return IVFPQ_OK;
}

extern "C" int ivfpq_set_scan_mode(ivfpq_index* ix, int mode, int group) {
  clear_error();
  IVFPQ_REQUIRE(ix, "ivfpq_set_scan_mode: null index");
  IVFPQ_REQUIRE(mode >= -1 && mode <= 1, "ivfpq_set_scan_mode: mode=%d outside [-1, 1]", mode);
  IVFPQ_REQUIRE(group >= -1 && group <= 3,
                "ivfpq_set_scan_mode: group=%d (0 keeps the current, -1 automatic, else 1 to 3)",
                group);
  ix->scan_mode = mode;
  if (group) ix->lm_group = group < 0 ? 0 : group;
  return IVFPQ_OK;
}

extern "C" int ivfpq_repaired_queries(const ivfpq_index* ix, int64_t* count, void* stream) {
  clear_error();
  IVFPQ_REQUIRE(ix && count, "ivfpq_repaired_queries: null pointer");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned long long h = 0;
  IVFPQ_CUDA(cudaMemcpyAsync(&h, ix->repaired, sizeof(h), cudaMemcpyDeviceToHost, s));
  IVFPQ_CUDA(cudaMemsetAsync(ix->repaired, 0, sizeof(h), s));
  IVFPQ_CUDA(cudaStreamSynchronize(s));
  *count = int64_t(h);
  return IVFPQ_OK;
}

extern "C" const char* ivfpq_last_scan_kernel(const ivfpq_index* ix) {
  return ix ? ix->last_scan_kernel.load() : nullptr;
}

extern "C" int ivfpq_stage_times(const ivfpq_index* ix, float* ms, int* nsearches) {
  clear_error();
  IVFPQ_REQUIRE(ix && ms, "ivfpq_stage_times: null pointer");
  for (int i = 0; i < 4; ++i) ms[i] = 0.f;
  if (nsearches) *nsearches = int(ix->ev_used);
  // stage i spans events (i, i+1); the planning stage has no events of its own
  for (size_t k = 0; k < ix->ev_used; ++k) {
    const auto& set = ix->ev_sets[k];
    for (int i = 0; i < 4; ++i) {
      if (!set.recorded[i] || !set.recorded[i + 1]) continue;
      IVFPQ_CUDA(cudaEventSynchronize(set.ev[i + 1]));
      float t = 0.f;
      IVFPQ_CUDA(cudaEventElapsedTime(&t, set.ev[i], set.ev[i + 1]));
      ms[i] += t;
    }
  }
  return IVFPQ_OK;
}
