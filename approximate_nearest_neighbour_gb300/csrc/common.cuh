// Shared host/device helpers of libivfpq_gb300: status handling, the
// thread-local error message, workspace allocation and small device utilities.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <cstdarg>
#include <cstdio>
#include <string>

#include "ivfpq.h"

namespace ivfpq {

// ---- error reporting --------------------------------------------------------
void set_error(const char* fmt, ...);
void clear_error();

#define IVFPQ_REQUIRE(cond, ...)                   \
  do {                                             \
    if (!(cond)) {                                 \
      ::ivfpq::set_error(__VA_ARGS__);             \
      return IVFPQ_ERR_INVALID_ARG;                \
    }                                              \
  } while (0)

#define IVFPQ_CUDA(expr)                                                        \
  do {                                                                          \
    cudaError_t e_ = (expr);                                                    \
    if (e_ != cudaSuccess) {                                                    \
      ::ivfpq::set_error("%s failed: %s (%s:%d)", #expr, cudaGetErrorString(e_), \
                         __FILE__, __LINE__);                                   \
      return e_ == cudaErrorMemoryAllocation ? IVFPQ_ERR_OOM : IVFPQ_ERR_CUDA;  \
    }                                                                           \
  } while (0)

#define IVFPQ_TRY(expr)              \
  do {                               \
    int s_ = (expr);                 \
    if (s_ != IVFPQ_OK) return s_;   \
  } while (0)

// Number of kernels this library has launched (all threads, all devices).
void count_launch();
// Number of workspace allocations the library has made (all threads).
void count_workspace_alloc();

// Checks (and counts) the launch that was just enqueued.
#define IVFPQ_LAUNCHED()             \
  do {                               \
    ::ivfpq::count_launch();         \
    IVFPQ_CUDA(cudaGetLastError());  \
  } while (0)

// Same, and on failure reports the kernel's resource attributes.
#define IVFPQ_LAUNCHED_K(kern, smem, threads)                                                  \
  do {                                                                                         \
    ::ivfpq::count_launch();                                                                   \
    cudaError_t e_ = cudaGetLastError();                                                       \
    if (e_ != cudaSuccess) {                                                                   \
      cudaFuncAttributes a_{};                                                                 \
      cudaFuncGetAttributes(&a_, (const void*)(kern));                                         \
      cudaGetLastError();                                                                      \
      ::ivfpq::set_error("launch failed: %s (%s:%d; threads=%d smem=%zu; kernel regs=%d "      \
                         "max_threads=%d max_dyn_smem=%d static_smem=%zu local=%zu)",          \
                         cudaGetErrorString(e_), __FILE__, __LINE__, int(threads),            \
                         size_t(smem), a_.numRegs, a_.maxThreadsPerBlock,                      \
                         a_.maxDynamicSharedSizeBytes, a_.sharedSizeBytes, a_.localSizeBytes); \
      return IVFPQ_ERR_CUDA;                                                                   \
    }                                                                                          \
  } while (0)

// ---- stream-ordered workspace --------------------------------------------------
// Frees its allocations on the stream (stream-ordered) when it goes out of
// scope, so a failing call never leaks workspace.
class Workspace {
 public:
  explicit Workspace(cudaStream_t s) : s_(s) {}
  ~Workspace() {
    for (int i = 0; i < n_; ++i) cudaFreeAsync(p_[i], s_);
  }
  template <class T>
  int alloc(T** out, size_t count) {
    *out = nullptr;
    if (count == 0) return IVFPQ_OK;
    if (n_ == kMax) {
      set_error("internal: too many workspace buffers");
      return IVFPQ_ERR_CUDA;
    }
    void* p = nullptr;
    cudaError_t e = cudaMallocAsync(&p, count * sizeof(T), s_);
    if (e != cudaSuccess) {
      cudaGetLastError();
      set_error("workspace allocation of %zu bytes failed: %s", count * sizeof(T),
                cudaGetErrorString(e));
      return IVFPQ_ERR_OOM;
    }
    count_workspace_alloc();
    p_[n_++] = p;
    *out = static_cast<T*>(p);
    return IVFPQ_OK;
  }

 private:
  static const int kMax = 48;
  cudaStream_t s_;
  void* p_[kMax];
  int n_ = 0;
};

// Raises a kernel's dynamic shared-memory limit to `bytes`. The kernel's
// attributes are read first: that loads its module (kernels are loaded lazily
// on first use), and an attribute set before the module is loaded was seen
// to be ignored by the first launch.
template <class Kern>
int set_dynamic_smem(Kern kern, size_t bytes) {
  cudaFuncAttributes a{};
  IVFPQ_CUDA(cudaFuncGetAttributes(&a, reinterpret_cast<const void*>(kern)));
  if (size_t(a.maxDynamicSharedSizeBytes) < bytes)
    IVFPQ_CUDA(cudaFuncSetAttribute(reinterpret_cast<const void*>(kern),
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, int(bytes)));
  return IVFPQ_OK;
}

inline int num_sms() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 1;
  }
  return n;
}

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// ---- device utilities ---------------------------------------------------------
constexpr unsigned kFullMask = 0xffffffffu;
constexpr uint32_t kSentinelKey = 0xffffffffu;
constexpr uint32_t kSentinelIdx = 0xffffffffu;

// Order-preserving map from fp32 to uint32 (negative values flip all bits,
// non-negative values flip the sign bit): a < b as floats iff key(a) < key(b)
// as unsigned integers (with -0 ordered just below +0). +inf maps to
// 0xff800000, below the sentinel key 0xffffffff.
__device__ __forceinline__ uint32_t float_to_key(float f) {
  uint32_t u = __float_as_uint(f);
  return u ^ (uint32_t(int32_t(u) >> 31) | 0x80000000u);
}
__device__ __forceinline__ float key_to_float(uint32_t k) {
  if (k == kSentinelKey) return __int_as_float(0x7f800000);
  return __uint_as_float(k ^ (uint32_t(int32_t(~k) >> 31) | 0x80000000u));
}

// Device bounds checks of the debug build (-DIVFPQ_DEBUG_CHECKS): dcheck
// returns ok; when ok is false it records check `id` in the device status
// word (bit 1 = a check failed, bit 8 + id = which) and the caller skips
// the access it guards. Kernels never trap or return early on a failed
// check (their block barriers stay matched); ivfpq_device_check reports
// IVFPQ_ERR_DEVICE_CHECK. In the normal build the check and its condition
// compile away.
#ifdef IVFPQ_DEBUG_CHECKS
__device__ __forceinline__ bool dcheck(int* word, bool ok, int id) {
  if (!ok && word) atomicOr(word, 2 | (1 << (8 + id)));
  return ok;
}
#else
__device__ __forceinline__ bool dcheck(int*, bool, int) { return true; }
#endif

// Distances produced by the list scan are sums of non-negative terms, so
// their raw fp32 bits already order correctly as unsigned integers; the
// sentinel 0xffffffff lies above +inf (0x7f800000).
__device__ __forceinline__ float dist_key_to_float(uint32_t k) {
  return k == kSentinelKey ? __int_as_float(0x7f800000) : __uint_as_float(k);
}

}  // namespace ivfpq
