// Thread-local error messages and status names of the C ABI.
#include <atomic>
#include <cstdarg>
#include <cstdio>

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

}  // namespace ivfpq

extern "C" const char* ivfpq_last_error(void) { return ivfpq::g_err; }

extern "C" uint64_t ivfpq_kernel_launches(void) { return ivfpq::g_launches.load(); }

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
