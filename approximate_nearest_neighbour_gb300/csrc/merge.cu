// knn_merge: the final k-selection over the results of several index shards.
//
// Source: sharding ("Billion-scale similarity search with GPUs", section 5,
// multi-GPU: each shard holds a part of the database and answers every query;
// the partial results are combined by an additional round of k-selection).
// Candidates of a row are the S * k_in (distance, id) pairs of the S shards;
// the k smallest distances are kept with their ids.
#include "internal.h"

namespace ivfpq {
namespace {

// keys[r * L + c] = key of shard (c / k_in)'s entry c % k_in of row r,
// idx = c, L = S * k_in.
__global__ void merge_gather_kernel(const float* __restrict__ dists, int64_t nq, int nshards,
                                    int k_in, uint32_t* __restrict__ keys,
                                    uint32_t* __restrict__ idx) {
  const int64_t L = int64_t(nshards) * k_in;
  const int64_t t = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (t >= nq * L) return;
  const int64_t r = t / L;
  const int c = int(t - r * L);
  const int s = c / k_in, i = c - s * k_in;
  keys[t] = float_to_key(dists[(int64_t(s) * nq + r) * k_in + i]);
  idx[t] = uint32_t(c);
}

}  // namespace
}  // namespace ivfpq

using namespace ivfpq;

extern "C" int knn_merge(const float* dists, const int64_t* ids, int64_t nq, int nshards,
                         int k_in, int k, float* out_dist, int64_t* out_ids, void* stream) {
  clear_error();
  IVFPQ_REQUIRE(nq >= 0 && nshards >= 1 && k_in >= 1,
                "knn_merge: bad sizes (nq=%lld nshards=%d k_in=%d)", (long long)nq, nshards,
                k_in);
  IVFPQ_REQUIRE(k >= 1 && k <= IVFPQ_MAX_K, "knn_merge: k=%d outside [1, %d]", k, IVFPQ_MAX_K);
  IVFPQ_REQUIRE(int64_t(nshards) * k_in < (int64_t(1) << 31),
                "knn_merge: nshards * k_in = %lld too large", (long long)nshards * k_in);
  IVFPQ_REQUIRE(nq < (int64_t(1) << 31), "knn_merge: nq=%lld too large", (long long)nq);
  if (nq == 0) return IVFPQ_OK;
  IVFPQ_REQUIRE(dists && ids && out_dist && out_ids, "knn_merge: null pointer");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int64_t L = int64_t(nshards) * k_in;
  Workspace ws(s);
  uint32_t *keys = nullptr, *idx = nullptr;
  IVFPQ_TRY(ws.alloc(&keys, size_t(nq * L)));
  IVFPQ_TRY(ws.alloc(&idx, size_t(nq * L)));
  merge_gather_kernel<<<unsigned(ceil_div(nq * L, 256)), 256, 0, s>>>(dists, nq, nshards, k_in,
                                                                      keys, idx);
  IVFPQ_LAUNCHED();
  SelectOut o;
  o.kind = OutKind::Merge;
  o.vals = out_dist;
  o.idx64 = out_ids;
  o.id_map = ids;
  o.merge_rows = nq;
  o.merge_kin = k_in;
  return select_pairs(keys, idx, nq, L, k, 1, L, o, s);
}
