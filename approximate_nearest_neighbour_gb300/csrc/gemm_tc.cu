// Squared-L2 distance tiles on the 5th-generation tensor cores:
//   D[i, j] = ||q_i||^2 + ||x_j||^2 - 2 <q_i, x_j>
// with <q_i, x_j> from 3xTF32 split accumulation (q = q_hi + q_lo, x = x_hi +
// x_lo, hi = x rounded to TF32, lo = x - hi, and <q,x> ~ q_hi.x_hi + q_hi.x_lo
// + q_lo.x_hi; Ootomo & Yokota's error-corrected TF32 scheme), which keeps
// the dot product at fp32 accuracy.
//
// Source: the GEMM form of exact brute-force distances and of the coarse
// quantizer ("Billion-scale similarity search with GPUs", section 5, exact
// search; "Faiss GPU: k-select that never leaves registers", Step 5).
//
// Kernel organisation (one CTA per SM, 10 warps):
//  * warp 0, one thread: TMA producer. Loads the CTA's 128-query tile of
//    q_hi / q_lo once (all of K), then streams 128-row tiles of x_hi / x_lo
//    through an NSTAGE ring, one 32-column (128-byte, 128B-swizzled) K chunk
//    per stage;
//  * warp 1: allocates 256 TMEM columns (two 128-column fp32 accumulators)
//    and, one thread, issues tcgen05.mma kind::tf32 (M = 128, N = 128, K = 8)
//    three times per K step, committing stage releases and finished
//    accumulators to mbarriers;
//  * warps 2..9: epilogue. Thread t of warps w and w + 4 owns TMEM lane
//    (query row) 32 * (w % 4) + t, one warp of the pair the first 64
//    accumulator columns, the other the last 64. Three modes: write D; keep
//    per-row minima over column groups; or keep only the entries at or below
//    a per-row bound, appended to the (row, CTA, half) segment of a candidate
//    buffer with a register counter (no atomics).
// Every mbarrier wait is bounded: on expiry the CTA records an error in
// *err, stops issuing work, waits (bounded) for its copies and MMAs in
// flight, frees its TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "internal.h"

namespace ivfpq {
namespace {

constexpr int TM = 128, TN = 128, TKC = 32;  // rows per tile, fp32 per K chunk
constexpr int kChunkBytes = TM * TKC * 4;    // 16 KB: one 128 x 32 fp32 tile
constexpr int kTmemCols = 256;
constexpr uint32_t kSpinLimit = 1u << 22;

// ---- PTX wrappers -------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
// Waits for the phase of the given parity to complete; false after the spin
// limit.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity,
                                          uint32_t limit = kSpinLimit) {
  for (uint32_t i = 0; i < limit; ++i) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    if (done) return true;
  }
  return false;
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, rows of
// 128 bytes, 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr) {
  return uint64_t((addr & 0x3FFFFu) >> 4) | (uint64_t(1) << 16) | (uint64_t(1024 >> 4) << 32) |
         (uint64_t(1) << 46) | (uint64_t(2) << 61);
}
// Instruction descriptor: D fp32, A and B TF32, both K-major, N = TN, M = TM.
constexpr uint32_t kIdesc = (1u << 4) | (2u << 7) | (2u << 10) | (uint32_t(TN >> 3) << 17) |
                            (uint32_t(TM >> 4) << 24);
__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(kIdesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
// 32 consecutive accumulator columns of the warp's 32 TMEM lanes into
// registers, without waiting for the load (tmem_wait_ld does).
__device__ __forceinline__ void tmem_ld32_nowait(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

enum TcMode : int {
  kModeTile = 0,      // write D
  kModeGroupMin = 1,  // per-row minima of u over column groups
  kModeFilter = 2     // per-row candidate segments of entries with u <= bound
};

// u[i, j] = ||x_j||^2 - 2 <q_i, x_j> = D[i, j] - ||q_i||^2 (the same order per
// row as D); the filter and group-minimum modes work on u.
struct TcArgs {
  const float* qnorm;  // [nq]
  const float* xnorm;  // [n]
  int nq, n;
  int ntiles_n;        // ceil(n / TN)
  int nsplit;          // CTAs per query tile (contiguous runs of column tiles)
  int* err;
  // tile mode
  float* D;            // [nq, ldd]
  int64_t ldd;
  // group-minimum mode: gmin[i * G + split * TN + c] = min over the CTA's
  // columns j = c (mod TN) of u[i, j], G = nsplit * TN (+inf if none)
  float* gmin;
  // filter mode: entries with u[i, j] <= bound[i * bound_stride] (widened by
  // a few ulps) go to segment (i, split * 2 + half) of cap_s packed
  // (key of D << 32 | j) entries, half = which 64 columns of each tile;
  // scnt[i * nseg + seg] = entries found (may exceed cap_s: overflow).
  const float* bound;
  int64_t bound_stride;
  uint64_t* cand;
  int* scnt;
  int cap_s;
};

template <int KC, int NSTAGE>
struct TcSmem {
  static constexpr int kA = 2 * KC * kChunkBytes;   // q_hi, q_lo, all K chunks
  static constexpr int kB = NSTAGE * 2 * kChunkBytes;
  static constexpr int kBars = 1024;
  static constexpr int kTotal = kA + kB + kBars + 1024;  // + alignment slack
};

constexpr int kEpiWarps = 8;                    // two per TMEM lane group
constexpr int kTcThreads = (2 + kEpiWarps) * 32;  // producer, MMA, epilogue

template <int KC, int NSTAGE, int MODE>
__global__ void __launch_bounds__(kTcThreads, 1)
l2_tc_kernel(const __grid_constant__ CUtensorMap mq_hi, const __grid_constant__ CUtensorMap mq_lo,
             const __grid_constant__ CUtensorMap mx_hi, const __grid_constant__ CUtensorMap mx_lo,
             const TcArgs a) {
  extern __shared__ uint8_t tc_smem_raw[];
  // 1024-byte alignment for the 128B-swizzled tiles
  const uint32_t raw = smem_u32(tc_smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = tc_smem_raw + (base - raw);
  const uint32_t sA_hi = base, sA_lo = base + KC * kChunkBytes;
  const uint32_t sB = base + 2 * KC * kChunkBytes;  // stage s: hi at +2s*chunk, lo at +(2s+1)*chunk
  const uint32_t bars = base + TcSmem<KC, NSTAGE>::kA + TcSmem<KC, NSTAGE>::kB;
  const uint32_t bar_a = bars;
  auto bar_full = [&](int s) { return bars + 8 + 8 * s; };
  auto bar_empty = [&](int s) { return bars + 8 + 8 * NSTAGE + 8 * s; };
  auto bar_accf = [&](int b) { return bars + 8 + 16 * NSTAGE + 8 * b; };
  auto bar_acce = [&](int b) { return bars + 8 + 16 * NSTAGE + 16 + 8 * b; };
  uint32_t* tmem_slot =
      reinterpret_cast<uint32_t*>(gbase + (bars - base) + 8 + 16 * NSTAGE + 32);
  volatile int* abort_flag =
      reinterpret_cast<volatile int*>(gbase + (bars - base) + 8 + 16 * NSTAGE + 40);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qt = blockIdx.x / a.nsplit, split = blockIdx.x % a.nsplit;
  const int t_per = (a.ntiles_n + a.nsplit - 1) / a.nsplit;
  const int t0 = split * t_per;
  const int t1 = min(a.ntiles_n, t0 + t_per);
  const int ntiles = max(0, t1 - t0);

  if (threadIdx.x == 0) {
    mbar_init(bar_a, 1);
    for (int s = 0; s < NSTAGE; ++s) {
      mbar_init(bar_full(s), 1);
      mbar_init(bar_empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_accf(b), 1);
      mbar_init(bar_acce(b), kEpiWarps);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  auto fail = [&]() {
    atomicExch(a.err, 1);
    *abort_flag = 1;
  };

  if (warp == 0 && lane == 0) {
    // ---- TMA producer ----
    mbar_expect_tx(bar_a, 2 * KC * kChunkBytes);
    for (int kc = 0; kc < KC; ++kc) {
      tma_load_2d(sA_hi + kc * kChunkBytes, &mq_hi, kc * TKC, qt * TM, bar_a);
      tma_load_2d(sA_lo + kc * kChunkBytes, &mq_lo, kc * TKC, qt * TM, bar_a);
    }
    int it = 0;
    for (int i = 0; i < ntiles && !*abort_flag; ++i) {
      for (int kc = 0; kc < KC; ++kc, ++it) {
        const int s = it % NSTAGE;
        if (!mbar_wait(bar_empty(s), ((it / NSTAGE) & 1) ^ 1)) {
          fail();
          break;
        }
        mbar_expect_tx(bar_full(s), 2 * kChunkBytes);
        tma_load_2d(sB + (2 * s) * kChunkBytes, &mx_hi, kc * TKC, (t0 + i) * TN, bar_full(s));
        tma_load_2d(sB + (2 * s + 1) * kChunkBytes, &mx_lo, kc * TKC, (t0 + i) * TN,
                    bar_full(s));
      }
    }
    // the last NSTAGE stages armed may still be landing: wait for them
    const int last = it;
    for (int j = max(0, last - NSTAGE); j < last; ++j)
      mbar_wait(bar_full(j % NSTAGE), (j / NSTAGE) & 1);
    mbar_wait(bar_a, 0);
  } else if (warp == 1 && lane == 0) {
    // ---- MMA issuer ----
    bool ok = mbar_wait(bar_a, 0);
    if (!ok) fail();
    int it = 0;
    int committed = 0;  // accumulator phases committed
    for (int i = 0; i < ntiles && ok && !*abort_flag; ++i) {
      const int ab = i & 1;
      if (!mbar_wait(bar_acce(ab), ((i >> 1) & 1) ^ 1)) {
        fail();
        break;
      }
      tc_fence_after();
      const uint32_t d_tmem = tmem + uint32_t(ab * TN);
      for (int kc = 0; kc < KC; ++kc, ++it) {
        const int s = it % NSTAGE;
        if (!mbar_wait(bar_full(s), (it / NSTAGE) & 1)) {
          fail();
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t ahi = smem_desc(sA_hi + kc * kChunkBytes);
        const uint64_t alo = smem_desc(sA_lo + kc * kChunkBytes);
        const uint64_t bhi = smem_desc(sB + (2 * s) * kChunkBytes);
        const uint64_t blo = smem_desc(sB + (2 * s + 1) * kChunkBytes);
#pragma unroll
        for (int k8 = 0; k8 < TKC / 8; ++k8) {
          const uint64_t adv = uint64_t(k8 * 32) >> 4;  // 8 fp32 = 32 bytes
          const uint32_t first = (kc == 0 && k8 == 0) ? 0u : 1u;
          mma_tf32(d_tmem, alo + adv, bhi + adv, first);
          mma_tf32(d_tmem, ahi + adv, blo + adv, 1u);
          mma_tf32(d_tmem, ahi + adv, bhi + adv, 1u);
        }
        mma_commit(bar_empty(s));
      }
      if (!ok) break;
      mma_commit(bar_accf(ab));
      ++committed;
    }
    // on an early exit, let the issued MMAs finish before TMEM is freed
    if (committed > 0) mbar_wait(bar_accf((committed - 1) & 1), ((committed - 1) >> 1) & 1);
  } else if (warp >= 2) {
    // ---- epilogue: warp w reads TMEM lanes 32 * (w % 4) .. +32 (its rows)
    // and the 64 accumulator columns of its half ----
    const int lg = warp & 3;
    const int half = (warp - 2) >> 2;
    const int row = 32 * lg + lane;
    const int q = qt * TM + row;
    const bool live = q < a.nq;
    const float qn = live ? __ldg(a.qnorm + q) : 0.f;
    constexpr int NC = TN / 32 / 2;  // 32-column chunks per half
    float gm[MODE == kModeGroupMin ? NC * 32 : 1];
    if constexpr (MODE == kModeGroupMin) {
#pragma unroll
      for (int j = 0; j < NC * 32; ++j) gm[j] = INFINITY;
    }
    float bnd = -INFINITY;  // rows past nq keep nothing
    int cnt = 0;
    uint64_t* seg = nullptr;
    if constexpr (MODE == kModeFilter) {
      if (live) {
        const float t = __ldg(a.bound + int64_t(q) * a.bound_stride);
        bnd = t + fabsf(t) * 1e-6f;
      }
      seg = a.cand + (int64_t(q) * (2 * a.nsplit) + 2 * split + half) * a.cap_s;
    }
    for (int i = 0; i < ntiles && !*abort_flag; ++i) {
      const int ab = i & 1;
      if (!mbar_wait(bar_accf(ab), (i >> 1) & 1)) {
        fail();
        break;
      }
      tc_fence_after();
      const int col0 = (t0 + i) * TN;
      if constexpr (MODE == kModeFilter) {
        if (col0 + TN <= a.n) {
          // a full tile: both accumulator chunks of this half loaded before one
          // wait; lane j holds the norm of column j of each chunk and hands it
          // to the other lanes by shuffle; four partial pass masks keep the
          // compare chain short; a warp with no passing entry skips the appends
          uint32_t r0[32], r1[32];
          const uint32_t ta = tmem + (uint32_t(32 * lg) << 16) + uint32_t(ab * TN + half * 64);
          tmem_ld32_nowait(ta, r0);
          tmem_ld32_nowait(ta + 32, r1);
          const int cb0 = col0 + half * 64;
          const float xr0 = __ldg(a.xnorm + cb0 + lane);
          const float xr1 = __ldg(a.xnorm + cb0 + 32 + lane);
          tmem_wait_ld();
          uint32_t m0[4] = {0, 0, 0, 0}, m1[4] = {0, 0, 0, 0};
          float u0[32], u1[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            u0[j] = fmaf(-2.f, __uint_as_float(r0[j]), __shfl_sync(kFullMask, xr0, j));
            u1[j] = fmaf(-2.f, __uint_as_float(r1[j]), __shfl_sync(kFullMask, xr1, j));
            m0[j & 3] |= uint32_t(u0[j] <= bnd) << j;
            m1[j & 3] |= uint32_t(u1[j] <= bnd) << j;
          }
          const uint32_t mk0 = (m0[0] | m0[1]) | (m0[2] | m0[3]);
          const uint32_t mk1 = (m1[0] | m1[1]) | (m1[2] | m1[3]);
          if (__any_sync(kFullMask, (mk0 | mk1) != 0u)) {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              if ((mk0 >> j) & 1u) {
                if (cnt < a.cap_s)
                  seg[cnt] = (uint64_t(float_to_key(u0[j] + qn)) << 32) | uint32_t(cb0 + j);
                ++cnt;
              }
            }
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              if ((mk1 >> j) & 1u) {
                if (cnt < a.cap_s)
                  seg[cnt] = (uint64_t(float_to_key(u1[j] + qn)) << 32) | uint32_t(cb0 + 32 + j);
                ++cnt;
              }
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_acce(ab));
          continue;
        }
      }
#pragma unroll
      for (int cc = 0; cc < NC; ++cc) {
        const int c = half * NC + cc;
        float v[32];
        tmem_ld32(tmem + (uint32_t(32 * lg) << 16) + uint32_t(ab * TN + c * 32), v);
        const int cb = col0 + c * 32;
        const bool full = cb + 32 <= a.n;
        // norms of the chunk's columns (0 past n); the filter's full-chunk
        // path reads them inline instead
        float xn[32];
        if (MODE != kModeFilter || !full) {
#pragma unroll
          for (int j = 0; j < 32; ++j) xn[j] = cb + j < a.n ? __ldg(a.xnorm + cb + j) : 0.f;
        }
        if constexpr (MODE == kModeTile) {
          float* drow = a.D + int64_t(q) * a.ldd;
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = fmaf(-2.f, v[j], qn + xn[j]);
          if (live) {
            const bool vec = (a.ldd % 4) == 0 && ((reinterpret_cast<uintptr_t>(a.D) & 15) == 0);
            if (vec && cb + 32 <= a.n) {
              float4* o = reinterpret_cast<float4*>(drow + cb);
#pragma unroll
              for (int j = 0; j < 8; ++j)
                o[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
            } else {
#pragma unroll
              for (int j = 0; j < 32; ++j)
                if (cb + j < a.n) drow[cb + j] = v[j];
            }
          }
        } else if constexpr (MODE == kModeGroupMin) {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float u = fmaf(-2.f, v[j], xn[j]);
            if (cb + j < a.n) gm[cc * 32 + j] = fminf(gm[cc * 32 + j], u);
          }
        } else if (full) {
          // full chunk: the pass mask first (no branch per entry), then the
          // appends of this lane's few passing entries
          uint32_t mk = 0;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            v[j] = fmaf(-2.f, v[j], __ldg(a.xnorm + cb + j));
            mk |= uint32_t(v[j] <= bnd) << j;
          }
          if (mk != 0) {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              if ((mk >> j) & 1u) {
                if (cnt < a.cap_s)
                  seg[cnt] = (uint64_t(float_to_key(v[j] + qn)) << 32) | uint32_t(cb + j);
                ++cnt;
              }
            }
          }
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float u = fmaf(-2.f, v[j], xn[j]);
            if (u <= bnd && cb + j < a.n) {
              if (cnt < a.cap_s)
                seg[cnt] = (uint64_t(float_to_key(u + qn)) << 32) | uint32_t(cb + j);
              ++cnt;
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_acce(ab));
    }
    if constexpr (MODE == kModeGroupMin) {
      if (live) {
        float* g = a.gmin + int64_t(q) * (int64_t(a.nsplit) * TN) + split * TN + half * NC * 32;
#pragma unroll
        for (int j = 0; j < NC * 32; ++j) g[j] = gm[j];
      }
    }
    if constexpr (MODE == kModeFilter) {
      if (live) a.scnt[int64_t(q) * (2 * a.nsplit) + 2 * split + half] = cnt;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols)
                 : "memory");
  }
}

// A barrier expecting one arrival that never comes: the wait expires after
// `spins` tries and the block records it, as the distance kernel does.
__global__ void wait_timeout_kernel(uint32_t spins, int* err) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    if (!mbar_wait(smem_u32(&bar), 0, spins)) atomicExch(err, 1);
  }
}

// ---- operand preparation ------------------------------------------------------------
// hi = x rounded to TF32 (10 explicit mantissa bits, to nearest, ties away),
// lo = x - hi (exact in fp32); rows padded with zeros to dpad columns; norms
// = sum of squares in fp32.
__global__ void tc_prepare_kernel(const float* __restrict__ x, int64_t rows, int d, int dpad,
                                  float* __restrict__ hi, float* __restrict__ lo,
                                  float* __restrict__ norms) {
  const int64_t r = int64_t(blockIdx.x) * blockDim.y + threadIdx.y;
  if (r >= rows) return;
  float s = 0.f;
  for (int t = threadIdx.x; t < dpad; t += 32) {
    const float v = t < d ? x[r * d + t] : 0.f;
    uint32_t h;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(h) : "f"(v));
    const float hv = __uint_as_float(h);
    hi[r * dpad + t] = hv;
    lo[r * dpad + t] = v - hv;
    s = fmaf(v, v, s);
  }
#pragma unroll
  for (int o = 16; o >= 1; o /= 2) s += __shfl_xor_sync(kFullMask, s, o);
  if (threadIdx.x == 0 && norms) norms[r] = s;
}

// ---- host side ------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

int encode_fn(PFN_cuTensorMapEncodeTiled_v12000* out) {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    cudaGetLastError();
  });
  if (!g_encode) {
    set_error("cuTensorMapEncodeTiled is not available from the driver");
    return IVFPQ_ERR_CUDA;
  }
  *out = g_encode;
  return IVFPQ_OK;
}

int make_map(CUtensorMap* m, const float* p, int64_t rows, int dpad) {
  PFN_cuTensorMapEncodeTiled_v12000 enc;
  IVFPQ_TRY(encode_fn(&enc));
  cuuint64_t dims[2] = {cuuint64_t(dpad), cuuint64_t(rows)};
  cuuint64_t strides[1] = {cuuint64_t(dpad) * 4};
  cuuint32_t box[2] = {TKC, TM};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(p), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_error("cuTensorMapEncodeTiled failed (%d) for a %lld x %d operand", int(r),
              (long long)rows, dpad);
    return IVFPQ_ERR_CUDA;
  }
  return IVFPQ_OK;
}

template <int KC, int MODE>
int launch_tc(const CUtensorMap& qh, const CUtensorMap& ql, const CUtensorMap& xh,
              const CUtensorMap& xl, const TcArgs& args, int qtiles, cudaStream_t s) {
  // as many 32 KB stages as fit beside the resident query tile (224 KB total)
  constexpr int NSTAGE = (224 * 1024 - 2 * KC * kChunkBytes) / (2 * kChunkBytes);
  auto kern = l2_tc_kernel<KC, NSTAGE, MODE>;
  const size_t smem = TcSmem<KC, NSTAGE>::kTotal;
  IVFPQ_TRY(set_dynamic_smem(kern, smem));
  kern<<<unsigned(qtiles * args.nsplit), kTcThreads, smem, s>>>(qh, ql, xh, xl, args);
  IVFPQ_LAUNCHED_K(kern, smem, kTcThreads);
  return IVFPQ_OK;
}

template <int MODE>
int launch_mode(int kc, const CUtensorMap& qh, const CUtensorMap& ql, const CUtensorMap& xh,
                const CUtensorMap& xl, const TcArgs& args, int qtiles, cudaStream_t s) {
  switch (kc) {
    case 1: return launch_tc<1, MODE>(qh, ql, xh, xl, args, qtiles, s);
    case 2: return launch_tc<2, MODE>(qh, ql, xh, xl, args, qtiles, s);
    case 3: return launch_tc<3, MODE>(qh, ql, xh, xl, args, qtiles, s);
    case 4: return launch_tc<4, MODE>(qh, ql, xh, xl, args, qtiles, s);
  }
  set_error("tensor-core distances need d <= 128");
  return IVFPQ_ERR_UNSUPPORTED;
}

}  // namespace

bool l2_tc_available(int d) {
  if (d <= 0 || d > 128) return false;
  static int cc = -1;
  if (cc < 0) {
    int dev = 0, maj = 0, min_ = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&maj, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&min_, cudaDevAttrComputeCapabilityMinor, dev);
    cc = maj * 10 + min_;
  }
  return cc == 103;
}

int tc_dpad(int d) { return (d + TKC - 1) / TKC * TKC; }

int l2_tc_prepare(const float* x, int64_t rows, int d, float* hi, float* lo, float* norms,
                  cudaStream_t s) {
  if (rows == 0) return IVFPQ_OK;
  dim3 block(32, 8);
  tc_prepare_kernel<<<unsigned(ceil_div(rows, 8)), block, 0, s>>>(x, rows, d, tc_dpad(d), hi, lo,
                                                                  norms);
  IVFPQ_LAUNCHED();
  return IVFPQ_OK;
}

namespace {
// nsplit = 0: enough CTAs for several waves.
int run_tc(const float* qhi, const float* qlo, int64_t nq, const float* xhi, const float* xlo,
           int64_t n, int d, int mode, TcArgs& args, cudaStream_t s) {
  const int dpad = tc_dpad(d);
  CUtensorMap mqh, mql, mxh, mxl;
  IVFPQ_TRY(make_map(&mqh, qhi, nq, dpad));
  IVFPQ_TRY(make_map(&mql, qlo, nq, dpad));
  IVFPQ_TRY(make_map(&mxh, xhi, n, dpad));
  IVFPQ_TRY(make_map(&mxl, xlo, n, dpad));
  args.nq = int(nq);
  args.n = int(n);
  args.ntiles_n = int(ceil_div(n, TN));
  const int qtiles = int(ceil_div(nq, TM));
  const int kc = dpad / TKC;
  switch (mode) {
    case kModeTile: return launch_mode<kModeTile>(kc, mqh, mql, mxh, mxl, args, qtiles, s);
    case kModeGroupMin:
      return launch_mode<kModeGroupMin>(kc, mqh, mql, mxh, mxl, args, qtiles, s);
    default: return launch_mode<kModeFilter>(kc, mqh, mql, mxh, mxl, args, qtiles, s);
  }
}

int default_split(int64_t nq, int64_t n) {
  const int64_t qtiles = ceil_div(nq, TM), ntiles = ceil_div(n, TN), sms = num_sms();
  const int64_t s0 = std::max<int64_t>(1, std::min<int64_t>(ntiles, ceil_div(8 * sms, qtiles)));
  // long CTAs (at least 64 column tiles each): up to twice the CTAs where
  // that fills the last wave better (flat 1e6 x 128 with 10,000 queries: 16
  // per query tile left the ninth wave 30 % full); short ones keep s0, their
  // start-up (query tile load, TMEM allocation) outweighs the tail (the
  // large workload's coarse pass took 1.43 -> 1.56 ms with twice the CTAs)
  if (ntiles / s0 < 64) return int(s0);
  int64_t best = s0;
  double best_fill = 0.0;
  for (int64_t sv = s0; sv <= std::min(ntiles, 2 * s0); ++sv) {
    const int64_t ctas = qtiles * sv;
    const double fill = double(ctas) / double(ceil_div(ctas, sms) * sms);
    if (fill > best_fill + 1e-9) {
      best_fill = fill;
      best = sv;
    }
  }
  return int(best);
}
}  // namespace

int tc_filter_split(int64_t nq, int64_t n) { return default_split(nq, n); }

int l2_tc_tiles(const float* qhi, const float* qlo, const float* qnorm, int64_t nq,
                const float* xhi, const float* xlo, const float* xnorm, int64_t n, int d,
                float* D, int64_t ldd, int* err, cudaStream_t s) {
  if (nq == 0 || n == 0) return IVFPQ_OK;
  TcArgs args{};
  args.qnorm = qnorm;
  args.xnorm = xnorm;
  args.D = D;
  args.ldd = ldd;
  args.err = err;
  args.nsplit = default_split(nq, n);
  return run_tc(qhi, qlo, nq, xhi, xlo, n, d, kModeTile, args, s);
}

int l2_tc_group_min(const float* qhi, const float* qlo, int64_t nq, const float* xhi,
                    const float* xlo, const float* xnorm, int64_t n, int d, int nsplit,
                    float* gmin, int* err, cudaStream_t s) {
  if (nq == 0 || n == 0) return IVFPQ_OK;
  TcArgs args{};
  args.xnorm = xnorm;
  args.err = err;
  args.gmin = gmin;
  args.nsplit = nsplit;
  return run_tc(qhi, qlo, nq, xhi, xlo, n, d, kModeGroupMin, args, s);
}

int l2_tc_filter(const float* qhi, const float* qlo, const float* qnorm, int64_t nq,
                 const float* xhi, const float* xlo, const float* xnorm, int64_t n, int d,
                 const float* bound, int64_t bound_stride, int nsplit, uint64_t* cand, int* scnt,
                 int cap_s, int* err, cudaStream_t s) {
  if (nq == 0 || n == 0) return IVFPQ_OK;
  TcArgs args{};
  args.qnorm = qnorm;
  args.xnorm = xnorm;
  args.err = err;
  args.bound = bound;
  args.bound_stride = bound_stride;
  args.nsplit = nsplit;
  args.cand = cand;
  args.scnt = scnt;
  args.cap_s = cap_s;
  return run_tc(qhi, qlo, nq, xhi, xlo, n, d, kModeFilter, args, s);
}

}  // namespace ivfpq

extern "C" int ivfpq_selftest_wait_timeout(int spins, void* stream) {
  using namespace ivfpq;
  clear_error();
  IVFPQ_REQUIRE(spins >= 1 && spins <= (1 << 20), "spins=%d outside [1, 2^20]", spins);
  int* w = nullptr;
  IVFPQ_TRY(device_status_word(&w));
  wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(uint32_t(spins), w);
  IVFPQ_LAUNCHED();
  return IVFPQ_OK;
}
