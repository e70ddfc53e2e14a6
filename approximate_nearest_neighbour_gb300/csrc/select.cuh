// Register-resident k-selection: WarpSelect and BlockSelect.
//
// Source: "Billion-scale similarity search with GPUs", section 4.
//  * lane-stride register arrays: element i of an array of length 32*R lives
//    in register i / 32 of lane i % 32;
//  * compare-swap by butterfly shuffles for strides < 32 and inside a lane for
//    strides that are multiples of 32;
//  * Algorithm 1 (odd-size merge: a bitonic merge whose first comparator stage
//    is reversed, so that two ascending arrays can be merged directly) and
//    Algorithm 2 (sort built from it);
//  * Algorithm 3 (WarpSelect): per-lane thread queues of length T, a warp
//    queue of K = k rounded up to a multiple of 32, a ballot after each round
//    of insertions, and an odd-size merge of the (sorted) thread queues into
//    the warp queue when any lane's largest thread-queue key T_0 has dropped
//    below the largest warp-queue key (the second invariant).
// BlockSelect runs one WarpSelect per warp over interleaved parts of a row and
// merges the warp queues in shared memory with the same merge network.
//
// Keys are uint32 (an order-preserving image of the fp32 value, see
// common.cuh) and the carried index is uint32; the sentinel key 0xffffffff
// plays the role of +infinity and is larger than every real key, including
// the image of +inf. All array lengths here are powers of two, so the
// networks need no dummy elements; k that is not a power of two is handled
// by rounding K up.
#pragma once

#include "common.cuh"

namespace ivfpq {

// (k, v) of this lane against the partner lane (lane ^ x): the lower lane of
// the pair keeps the smaller key, the upper lane the larger. Both lanes take
// the partner's element under the same condition, so equal keys never
// duplicate or lose an element.
__device__ __forceinline__ void cx_shfl(uint32_t& k, uint32_t& v, int x, bool lower) {
  uint32_t pk = __shfl_xor_sync(kFullMask, k, x);
  uint32_t pv = __shfl_xor_sync(kFullMask, v, x);
  bool take = lower ? (pk < k) : (pk > k);
  k = take ? pk : k;
  v = take ? pv : v;
}

// In-lane compare-swap: (ak, av) is the lower position.
__device__ __forceinline__ void cx_reg(uint32_t& ak, uint32_t& av, uint32_t& bk, uint32_t& bv) {
  bool s = bk < ak;
  uint32_t tk = s ? bk : ak, tv = s ? bv : av;
  bk = s ? ak : bk;
  bv = s ? av : bv;
  ak = tk;
  av = tv;
}

// Half-cleaner cascade (strides 16R .. 1): sorts a bitonic lane-stride array
// of 32R elements ascending.
template <int R>
__device__ __forceinline__ void bitonic_clean(uint32_t (&k)[R], uint32_t (&v)[R], int lane) {
#pragma unroll
  for (int sr = R / 2; sr >= 1; sr /= 2) {
#pragma unroll
    for (int r = 0; r < R; ++r)
      if ((r & sr) == 0) cx_reg(k[r], v[r], k[r + sr], v[r + sr]);
  }
#pragma unroll
  for (int s = 16; s >= 1; s /= 2) {
    bool lower = (lane & s) == 0;
#pragma unroll
    for (int r = 0; r < R; ++r) cx_shfl(k[r], v[r], s, lower);
  }
}

// Algorithm 2 for a power-of-two length 32R: for block sizes 2, 4, .., 32R a
// reversed (mirror) stage followed by half-cleaners inside each block.
template <int R>
__device__ __forceinline__ void bitonic_sort(uint32_t (&k)[R], uint32_t (&v)[R], int lane) {
#pragma unroll
  for (int size = 2; size <= 32; size *= 2) {
    bool lower = (lane & (size / 2)) == 0;
#pragma unroll
    for (int r = 0; r < R; ++r) cx_shfl(k[r], v[r], size - 1, lower);
#pragma unroll
    for (int s = size / 4; s >= 1; s /= 2) {
      bool lw = (lane & s) == 0;
#pragma unroll
      for (int r = 0; r < R; ++r) cx_shfl(k[r], v[r], s, lw);
    }
  }
#pragma unroll
  for (int rs = 2; rs <= R; rs *= 2) {  // registers per block
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int off = r & (rs - 1);
      if (off < rs / 2) {
        const int r2 = r - off + rs - 1 - off;
        // (r, lane) pairs with (r2, 31 - lane); (r2, lane) with (r, 31 - lane).
        uint32_t ak = __shfl_xor_sync(kFullMask, k[r2], 31);
        uint32_t av = __shfl_xor_sync(kFullMask, v[r2], 31);
        uint32_t bk = __shfl_xor_sync(kFullMask, k[r], 31);
        uint32_t bv = __shfl_xor_sync(kFullMask, v[r], 31);
        bool t1 = ak < k[r];
        bool t2 = bk > k[r2];
        k[r] = t1 ? ak : k[r];
        v[r] = t1 ? av : v[r];
        k[r2] = t2 ? bk : k[r2];
        v[r2] = t2 ? bv : v[r2];
      }
    }
#pragma unroll
    for (int sr = rs / 4; sr >= 1; sr /= 2) {
#pragma unroll
      for (int r = 0; r < R; ++r)
        if ((r & sr) == 0) cx_reg(k[r], v[r], k[r + sr], v[r + sr]);
    }
#pragma unroll
    for (int s = 16; s >= 1; s /= 2) {
      bool lw = (lane & s) == 0;
#pragma unroll
      for (int r = 0; r < R; ++r) cx_shfl(k[r], v[r], s, lw);
    }
  }
}

// Algorithm 1 on the warp queue W (32R, ascending) and an ascending array S
// (32T): the reversed first stage pairs W[32R-1-i] with S[i]; afterwards W
// holds the 32R smallest of both and S the rest, each bitonic, and one
// half-cleaner cascade per side sorts them.
template <int R, int T>
__device__ __forceinline__ void merge_queues(uint32_t (&wk)[R], uint32_t (&wv)[R],
                                             uint32_t (&sk)[T], uint32_t (&sv)[T], int lane) {
  constexpr int C = R < T ? R : T;
#pragma unroll
  for (int r = 0; r < C; ++r) {
    uint32_t wkp = __shfl_xor_sync(kFullMask, wk[R - 1 - r], 31);
    uint32_t wvp = __shfl_xor_sync(kFullMask, wv[R - 1 - r], 31);
    uint32_t skp = __shfl_xor_sync(kFullMask, sk[r], 31);
    uint32_t svp = __shfl_xor_sync(kFullMask, sv[r], 31);
    bool ts = wkp > sk[r];
    bool tw = skp < wk[R - 1 - r];
    sk[r] = ts ? wkp : sk[r];
    sv[r] = ts ? wvp : sv[r];
    wk[R - 1 - r] = tw ? skp : wk[R - 1 - r];
    wv[R - 1 - r] = tw ? svp : wv[R - 1 - r];
  }
  bitonic_clean<R>(wk, wv, lane);
  bitonic_clean<T>(sk, sv, lane);
}

// WarpSelect state of one warp. The thread queue of a lane is kept in
// ascending register order, so tk[T-1] is the lane's largest key (T_0 in the
// paper's numbering) and the T registers of the 32 lanes form a lane-stride
// array directly.
template <int K, int T>
struct WarpSelect {
  static_assert(K % 32 == 0 && (K & (K - 1)) == 0, "K: power of two >= 32");
  static_assert((T & (T - 1)) == 0, "T: power of two");
  static constexpr int R = K / 32;
  uint32_t wk[R], wv[R];
  uint32_t tk[T], tv[T];
  uint32_t wmax;  // largest warp-queue key, W_{K-1}
  int lane;

  __device__ __forceinline__ void init(int lane_id) {
    lane = lane_id;
#pragma unroll
    for (int r = 0; r < R; ++r) {
      wk[r] = kSentinelKey;
      wv[r] = kSentinelIdx;
    }
#pragma unroll
    for (int r = 0; r < T; ++r) {
      tk[r] = kSentinelKey;
      tv[r] = kSentinelIdx;
    }
    wmax = kSentinelKey;
  }

  // Lane's largest thread-queue key: candidates not below it are rejected.
  __device__ __forceinline__ uint32_t threshold() const { return tk[T - 1]; }

  __device__ __forceinline__ void merge() {
    bitonic_sort<T>(tk, tv, lane);
    merge_queues<R, T>(wk, wv, tk, tv, lane);
    wmax = __shfl_sync(kFullMask, wk[R - 1], 31);
  }

  // One candidate per lane (pass the sentinel key for "none"). Must be called
  // by all 32 lanes together. A key not below the warp queue's largest can
  // never enter it (that largest key only decreases), so it is rejected as
  // well as one not below the lane's own largest: on a stream of good
  // candidates (a query's nearest list) this keeps the thread queues from
  // filling with keys the next merge would discard.
  __device__ __forceinline__ void add(uint32_t key, uint32_t idx) {
    bool pass = key < min(tk[T - 1], wmax);
    if (__any_sync(kFullMask, pass)) {
      if (pass) {
        tk[T - 1] = key;
        tv[T - 1] = idx;
#pragma unroll
        for (int i = T - 1; i > 0; --i) cx_reg(tk[i - 1], tv[i - 1], tk[i], tv[i]);
      }
      if (__any_sync(kFullMask, tk[T - 1] < wmax)) merge();
    }
  }

  // Final sort and merge: afterwards the warp queue holds the K smallest.
  __device__ __forceinline__ void finalize() { merge(); }
};

// BlockSelect reduction: every warp has finalized its WarpSelect; warps
// combine their queues pairwise through shared memory (sk/sv hold NW*K
// entries). Warp 0 ends with the block's K smallest, ascending. All threads
// of the block must call this.
template <int K, int T, int NW>
__device__ __forceinline__ void block_merge(WarpSelect<K, T>& ws, uint32_t* sk, uint32_t* sv,
                                            int warp) {
  constexpr int R = K / 32;
  if (NW == 1) return;
  const int lane = ws.lane;
#pragma unroll
  for (int r = 0; r < R; ++r) {
    sk[warp * K + 32 * r + lane] = ws.wk[r];
    sv[warp * K + 32 * r + lane] = ws.wv[r];
  }
  __syncthreads();
#pragma unroll
  for (int h = 1; h < NW; h *= 2) {
    if ((warp % (2 * h)) == 0 && warp + h < NW) {
      const uint32_t* ok = sk + (warp + h) * K;
      const uint32_t* ov = sv + (warp + h) * K;
      // reversed stage: W[K-1-i] against O[i]; W keeps the smaller.
#pragma unroll
      for (int r = 0; r < R; ++r) {
        uint32_t k2 = ok[32 * r + 31 - lane];
        uint32_t v2 = ov[32 * r + 31 - lane];
        bool t = k2 < ws.wk[R - 1 - r];
        ws.wk[R - 1 - r] = t ? k2 : ws.wk[R - 1 - r];
        ws.wv[R - 1 - r] = t ? v2 : ws.wv[R - 1 - r];
      }
      bitonic_clean<R>(ws.wk, ws.wv, lane);
    }
    __syncthreads();
    if ((warp % (2 * h)) == 0 && warp + h < NW) {
#pragma unroll
      for (int r = 0; r < R; ++r) {
        sk[warp * K + 32 * r + lane] = ws.wk[r];
        sv[warp * K + 32 * r + lane] = ws.wv[r];
      }
    }
    __syncthreads();
  }
}

// Thread-queue length used with each warp-queue length.
template <int K>
struct ThreadQ {
  static constexpr int value = K <= 128 ? 2 : (K <= 256 ? 4 : 8);
};

}  // namespace ivfpq
