// Thread-local error messages and status names of the C ABI.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <mutex>

#include "common.cuh"

namespace ivfpq {

static thread_local char g_err[1024] = {0};

void set_error(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
}

void clear_error() { g_err[0] = 0; }

static std::atomic<unsigned long long> g_launches{0};
void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

static std::atomic<unsigned long long> g_ws_allocs{0};
void count_workspace_alloc() { g_ws_allocs.fetch_add(1, std::memory_order_relaxed); }

// One status word per device, allocated on first use and kept while the
// library is loaded. Kernels whose bounded waits expire set bit 0; the
// debug build's bounds checks set bit 1 and bit 8 + the check's id.
static std::mutex g_status_mu;
static int* g_status[64] = {};

int device_status_word(int** out) {
  int dev = 0;
  IVFPQ_CUDA(cudaGetDevice(&dev));
  IVFPQ_REQUIRE(dev >= 0 && dev < 64, "device %d not supported", dev);
  std::lock_guard<std::mutex> lock(g_status_mu);
  if (!g_status[dev]) {
    int* p = nullptr;
    IVFPQ_CUDA(cudaMalloc(&p, sizeof(int)));
    IVFPQ_CUDA(cudaMemset(p, 0, sizeof(int)));
    g_status[dev] = p;
  }
  *out = g_status[dev];
  return IVFPQ_OK;
}

}  // namespace ivfpq

extern "C" int ivfpq_device_check(void* stream) {
  using namespace ivfpq;
  clear_error();
  int* w = nullptr;
  IVFPQ_TRY(device_status_word(&w));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int h = 0;
  IVFPQ_CUDA(cudaMemcpyAsync(&h, w, sizeof(int), cudaMemcpyDeviceToHost, s));
  IVFPQ_CUDA(cudaStreamSynchronize(s));
  if (h != 0) {
    IVFPQ_CUDA(cudaMemsetAsync(w, 0, sizeof(int), s));
    IVFPQ_CUDA(cudaStreamSynchronize(s));
    if (h & 1) {
      set_error("a kernel's bounded wait expired: results of the calls since the last check "
                "are invalid");
      return IVFPQ_ERR_TIMEOUT;
    }
    set_error("device bounds checks failed (check mask 0x%x): results of the calls since the "
              "last check are invalid", unsigned(h) >> 8);
    return IVFPQ_ERR_DEVICE_CHECK;
  }
  return IVFPQ_OK;
}

extern "C" const char* ivfpq_last_error(void) { return ivfpq::g_err; }

extern "C" uint64_t ivfpq_kernel_launches(void) { return ivfpq::g_launches.load(); }

extern "C" uint64_t ivfpq_workspace_allocations(void) { return ivfpq::g_ws_allocs.load(); }

extern "C" const char* ivfpq_status_string(int status) {
  switch (status) {
    case IVFPQ_OK: return "IVFPQ_OK";
    case IVFPQ_ERR_INVALID_ARG: return "IVFPQ_ERR_INVALID_ARG";
    case IVFPQ_ERR_UNSUPPORTED: return "IVFPQ_ERR_UNSUPPORTED";
    case IVFPQ_ERR_OOM: return "IVFPQ_ERR_OOM";
    case IVFPQ_ERR_CUDA: return "IVFPQ_ERR_CUDA";
    case IVFPQ_ERR_DEVICE_CHECK: return "IVFPQ_ERR_DEVICE_CHECK";
    case IVFPQ_ERR_TIMEOUT: return "IVFPQ_ERR_TIMEOUT";
  }
  return "IVFPQ_ERR_UNKNOWN";
}
