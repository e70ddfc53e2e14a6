// Device helpers of the radix-bound selection (select_radix.cu; the by-list
// scan's final selection in ivfpq_search.cu): one block of kRThreads threads
// per row locates a bound theta of the row's k-th smallest key by a 4,096-bin
// histogram of the keys' top 12 bits and, within the k-th's bin, a histogram
// of the next 12 bits; at least k keys are <= theta (the end of a 256-key
// sub-bin). bitonic_sort sorts (key, value) pairs in shared memory.
#pragma once

#include "common.cuh"

namespace ivfpq {
namespace radix {

constexpr int kRThreads = 512;
constexpr int kRBins = 4096, kRShift = 20, kRSub = 8, kRPer = kRBins / kRThreads;

struct RadixShared {
  uint32_t part[kRThreads / 32];
  uint32_t bin, before, theta, count;
};

// The bin in which the running count of hist reaches `target` (>= 1): the
// thread holding it writes sh.bin and sh.before (the count below that bin).
// Block-wide (one barrier inside); hist is only read.
__device__ __forceinline__ void radix_find(const uint32_t* hist, RadixShared& sh, uint32_t target) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t h[kRPer], sum = 0;
#pragma unroll
  for (int i = 0; i < kRPer; ++i) {
    h[i] = hist[threadIdx.x * kRPer + i];
    sum += h[i];
  }
  uint32_t inc = sum;
#pragma unroll
  for (int o = 1; o < 32; o *= 2) {
    const uint32_t v = __shfl_up_sync(kFullMask, inc, o);
    if (lane >= o) inc += v;
  }
  if (lane == 31) sh.part[warp] = inc;
  __syncthreads();
  uint32_t run = inc - sum;
  for (int w = 0; w < warp; ++w) run += sh.part[w];
  if (run < target && run + sum >= target) {
#pragma unroll
    for (int i = 0; i < kRPer; ++i) {
      if (run + h[i] >= target) {
        sh.bin = threadIdx.x * kRPer + i;
        sh.before = run;
        break;
      }
      run += h[i];
    }
  }
}

// theta for the k smallest of the keys that for_each(f) hands to f (each
// thread its share; called twice): at least k keys are <= theta. Block-wide,
// block-uniform result; kSentinelKey when there are fewer than k keys or the
// k-th lies in the top bin (NaN keys and the sentinel's).
template <class ForEach>
__device__ uint32_t radix_theta(uint32_t* hist, RadixShared& sh, uint32_t k, ForEach for_each) {
  for (int b = threadIdx.x; b < kRBins; b += kRThreads) hist[b] = 0;
  if (threadIdx.x == 0) {
    sh.bin = kRBins - 1;
    sh.before = 0;
    sh.theta = kSentinelKey;
  }
  __syncthreads();
  for_each([&](uint32_t key) { atomicAdd(&hist[key >> kRShift], 1u); });
  __syncthreads();
  radix_find(hist, sh, k);
  __syncthreads();
  const uint32_t bin = sh.bin;
  if (bin == kRBins - 1) return kSentinelKey;  // block-uniform
  const uint32_t need = k - sh.before;         // >= 1 keys of the bin, in order
  __syncthreads();                              // every thread has read sh.bin / before
  for (int b = threadIdx.x; b < kRBins; b += kRThreads) hist[b] = 0;
  __syncthreads();
  for_each([&](uint32_t key) {
    if ((key >> kRShift) == bin) atomicAdd(&hist[(key >> kRSub) & (kRBins - 1)], 1u);
  });
  __syncthreads();
  radix_find(hist, sh, need);  // sh.bin is now the sub-bin
  __syncthreads();
  const uint32_t theta = (bin << kRShift) | (sh.bin << kRSub) | ((1u << kRSub) - 1u);
  __syncthreads();  // sh is reused by the caller
  return theta;
}

// Ascending bitonic sort of n = power of two (key, value) pairs in shared
// memory. Block-wide.
__device__ __forceinline__ void bitonic_sort(uint32_t* sk, uint32_t* sv, uint32_t n) {
  for (uint32_t size = 2; size <= n; size <<= 1) {
    for (uint32_t stride = size >> 1; stride > 0; stride >>= 1) {
      for (uint32_t t = threadIdx.x; t < n / 2; t += kRThreads) {
        const uint32_t a = 2 * t - (t & (stride - 1));
        const uint32_t b = a + stride;
        const uint32_t ka = sk[a], kb = sk[b];
        if ((ka > kb) == ((a & size) == 0)) {
          const uint32_t va = sv[a];
          sk[a] = kb;
          sk[b] = ka;
          sv[a] = sv[b];
          sv[b] = va;
        }
      }
      __syncthreads();
    }
  }
}

}  // namespace radix
}  // namespace ivfpq
