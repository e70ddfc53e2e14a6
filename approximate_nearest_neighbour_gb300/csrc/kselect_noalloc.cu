// kselect_noalloc: the row-wise k-selection of kselect for callers that must
// not allocate device memory during a call. Its two-pass plan keeps the
// per-chunk partial results in one fixed, file-scope device array instead of
// the stream-ordered pool that kselect draws its workspace from.
//
// The array (kScratchPairs (key, index) pairs, 8 MiB) exists on every GPU that
// loads this library, for as long as the library stays loaded. Host code may
// not use the array's name as a device address (on the host it names a
// stand-in object), so the first call on each device looks up the real
// address with cudaGetSymbolAddress while that device is current and keeps it
// for later calls.
#include <algorithm>
#include <mutex>

#include "internal.h"

namespace ivfpq {
namespace {

constexpr int64_t kScratchPairs = int64_t(1) << 20;  // 1,048,576 (key, index) pairs

static __device__ __align__(256) uint32_t g_kselect_scratch[2 * kScratchPairs];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
uint32_t* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_kselect_scratch on the current device (set up once per
// device).
int scratch_address(uint32_t** out) {
  int dev = 0;
  IVFPQ_CUDA(cudaGetDevice(&dev));
  IVFPQ_REQUIRE(dev >= 0 && dev < kMaxDevices, "kselect_noalloc: device %d not supported", dev);
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    IVFPQ_CUDA(cudaGetSymbolAddress(&p, g_kselect_scratch));
    g_scratch_ptr[dev] = static_cast<uint32_t*>(p);
  }
  *out = g_scratch_ptr[dev];
  return IVFPQ_OK;
}

int queue_len(int k) {
  int K = 32;
  while (K < k) K *= 2;
  return K;
}

}  // namespace
}  // namespace ivfpq

using namespace ivfpq;

extern "C" int kselect_noalloc(const float* vals, int64_t rows, int64_t cols, int k,
                               float* out_vals, int64_t* out_idx, void* stream) {
  clear_error();
  IVFPQ_REQUIRE(rows >= 0 && cols >= 0, "kselect_noalloc: negative size (rows=%lld, cols=%lld)",
                (long long)rows, (long long)cols);
  IVFPQ_REQUIRE(k >= 1 && k <= IVFPQ_MAX_K, "kselect_noalloc: k=%d outside [1, %d]", k,
                IVFPQ_MAX_K);
  IVFPQ_REQUIRE(cols < int64_t(0xffffffffLL), "kselect_noalloc: cols=%lld too large",
                (long long)cols);
  IVFPQ_REQUIRE(rows < (int64_t(1) << 31), "kselect_noalloc: rows=%lld too large",
                (long long)rows);
  IVFPQ_REQUIRE(rows * k <= kScratchPairs,
                "kselect_noalloc: rows * k = %lld exceeds the fixed scratch of %lld pairs",
                (long long)(rows * k), (long long)kScratchPairs);
  if (rows == 0) return IVFPQ_OK;
  IVFPQ_REQUIRE(out_vals && out_idx && (vals || cols == 0), "kselect_noalloc: null pointer");
  uint32_t* scratch = nullptr;
  IVFPQ_TRY(scratch_address(&scratch));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  SelectOut out;
  out.kind = OutKind::Float;
  out.vals = out_vals;
  out.idx64 = out_idx;

  // The same plan as kselect, with the number of chunks capped so that the
  // partial results fit the fixed scratch.
  const int64_t target_blocks = 4 * int64_t(num_sms());
  const int64_t min_chunk = std::max<int64_t>(16384, 8 * int64_t(queue_len(k)));
  int64_t chunks = 1;
  if (rows < target_blocks && cols > 2 * min_chunk)
    chunks = std::min(ceil_div(target_blocks, rows), ceil_div(cols, min_chunk));
  chunks = std::min(chunks, kScratchPairs / (rows * k));
  if (chunks <= 1) return select_rows(vals, rows, cols, k, 1, std::max<int64_t>(cols, 1), out, s);
  const int64_t chunk_len = ceil_div(ceil_div(cols, chunks), 4) * 4;
  chunks = ceil_div(cols, chunk_len);
  // The first pass writes every (row, chunk, i < k) entry that the second pass
  // reads, so nothing left in the scratch by an earlier call is ever used.
  uint32_t* pk = scratch;
  uint32_t* pi = scratch + kScratchPairs;
  SelectOut part;
  part.kind = OutKind::Partial;
  part.pkeys = pk;
  part.pidx = pi;
  IVFPQ_TRY(select_rows(vals, rows, cols, k, chunks, chunk_len, part, s));
  const int64_t len = chunks * k;
  return select_pairs(pk, pi, rows, len, k, 1, len, out, s);
}
