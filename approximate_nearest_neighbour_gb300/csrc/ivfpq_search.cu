// Batched IVF-PQ search: coarse quantizer, fused table build + list scan +
// per-chunk selection, and the cross-chunk merge with id translation.
//
// Source: IVFPQ search steps 1-5 ("Custom 8-bit floating point value format
// for reducing shared memory bank conflict in approximate nearest neighbor
// search"); section 5 of "Billion-scale similarity search with GPUs" (tables
// per query x list, queries x lists processed independently, two-pass
// k-selection with subdivision factor f: here f = the number of list chunks
// per query).
#include <algorithm>

#include "internal.h"
#include "scan2.cuh"

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

int scan_stage(const ivfpq_index* ix, const float* queries, int64_t nq, int nprobe,
               const int32_t* probes, int k, float* out_dist, int64_t* out_ids, cudaStream_t s) {
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
  if (use_precomputed(ix)) p.term1 = ix->term1;
  plan_chunks(nq, nprobe, &p.per_chunk, &p.nchunks);
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
    record(ix, 2, s);
    IVFPQ_TRY(launch_scan_general(p, nq, s));
    mix->last_scan_kernel.store("ivfpq_scan_kernel");
    record(ix, 3, s);
    const int64_t len = int64_t(p.nchunks) * k;
    IVFPQ_TRY(select_pairs(p.pkeys, p.pidx, nq, len, k, 1, len, o, s));
    record(ix, 4, s);
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
  record(ix, 2, s);
  int launched = 0;
  switch (kw) {
    case 32: IVFPQ_TRY(try_scan2_kw<32>(p, nq, s, &launched)); break;
    case 64: IVFPQ_TRY(try_scan2_kw<64>(p, nq, s, &launched)); break;
    case 128: IVFPQ_TRY(try_scan2_kw<128>(p, nq, s, &launched)); break;
    default: IVFPQ_TRY(try_scan2_kw<256>(p, nq, s, &launched)); break;
  }
  IVFPQ_REQUIRE(launched, "scan: no register-codebook kernel for m=%d d/m=%d", p.m, p.dsub);
  mix->last_scan_kernel.store("ivfpq_scan2_kernel");
  record(ix, 3, s);
  IVFPQ_TRY(merge_sorted_runs(p.pkeys, p.pidx, nq, groups, kw, k, o, s));
  if (kw < k) {
    // repair the queries whose merged result a short queue may have cut
    int* flags = nullptr;
    IVFPQ_TRY(ws.alloc(&flags, size_t(nq)));
    warp_queue_check_kernel<<<unsigned(ceil_div(nq, 256)), 256, 0, s>>>(
        p.pkeys, nq, groups, kw, out_dist, k, flags, ix->repaired);
    IVFPQ_LAUNCHED();
    ScanParams r = p;
    r.qmask = flags;
    const size_t nr = size_t(nq) * p.nchunks * k;
    IVFPQ_TRY(ws.alloc(&r.pkeys, nr));
    IVFPQ_TRY(ws.alloc(&r.pidx, nr));
    IVFPQ_TRY(launch_scan_general(r, nq, s));
    SelectOut ro = o;
    ro.row_mask = flags;
    const int64_t rlen = int64_t(p.nchunks) * k;
    IVFPQ_TRY(select_pairs(r.pkeys, r.pidx, nq, rlen, k, 1, rlen, ro, s));
  }
  record(ix, 4, s);
  return IVFPQ_OK;
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
