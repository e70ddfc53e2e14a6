// List scan with the codebook held in registers and double-buffered tables.
//
// Same computation as ivfpq_scan_kernel (scan.cuh; sources: "Billion-scale
// similarity search with GPUs", section 5, tables T_1..T_b and their use in
// the list scan; "Custom 8-bit floating point value format ...", search steps
// 2-5 and Eq. (1)), organised for the shapes where it pays:
//  * 16 warps per block, one block per SM (two 64 KB table buffers);
//  * the 256 x m codewords (d floats each row) are split over the 512
//    threads and kept in registers for the whole block (d/2 floats per
//    thread), so building a table reads no memory but the centroid: thread
//    (warp w, lane i) owns sub-quantizer jj = i mod GS of the group and the
//    reproduction values e = (s*16 + w) * QQ + i / GS, QQ = 32 / GS;
//  * the table of list i+1 is built into one buffer while list i is scanned
//    with the other, so each probed list costs one block barrier;
//  * the block's probe list (list id, length, first block) is staged in
//    shared memory once, and each warp loads its first code block of list
//    i+1 before the barrier that ends list i, so no list starts with a chain
//    of dependent global loads; the list two ahead is streamed into L2 with
//    bulk prefetches, and (m = 32) the centroid slice of the next table is
//    loaded a list early;
//  * for m < 32 a warp scores 16 / MW of its blocks per iteration; for
//    m = 32 the tables are built with packed fp32x2 arithmetic;
//  * optionally (ivfpq_set_precomputed, m <= 16) the table of a list is the
//    stored list term plus the query's term, the list's exact coarse
//    distance being added to its distances;
//  * each warp keeps only its own KW best (WarpSelect with a KW-entry warp
//    queue, KW < k allowed) and writes them out unmerged; the cross-chunk
//    merge selects the k best of all warps' entries. That is exact unless a
//    warp's k-th-best contribution was cut off by its short queue, which the
//    merge detects (a full warp queue whose last key is not above the merged
//    k-th key) and repairs by scanning that query again with full-length
//    queues (ivfpq_search.cu).
// The shared-memory table layout, the rotated code layout and the look-up
// addressing are those of scan.cuh.
#pragma once

#include "scan.cuh"

namespace ivfpq {

constexpr int kScan2Warps = 16;
constexpr int kScan2MaxLists = 256;  // probed lists per block (per query chunk)

template <int MW, int DS>
struct Scan2Shape {
  static constexpr int M = 4 * MW;
  static_assert(M <= 32, "one group of sub-quantizers");
  static constexpr int GS = M;  // group size: all sub-quantizers
  static constexpr int QQ = 32 / GS;
  static constexpr int LOG_GS = GS == 32 ? 5 : GS == 16 ? 4 : GS == 8 ? 3 : 2;
  static constexpr int STEPS = 256 / (kScan2Warps * QQ);  // values per thread
  static constexpr int REPS = 64 / GS;                     // copies of a table in a row
  static constexpr int DS4 = (DS + 3) & ~3;
};

template <int MW, int DS, int KW, bool PRE>
__global__ void __launch_bounds__(kScan2Warps * 32, 1)
ivfpq_scan2_kernel(const ScanParams p) {
  using Sh = Scan2Shape<MW, DS>;
  constexpr int T = ThreadQ<KW>::value;
  constexpr int NW = kScan2Warps;
  constexpr int m = Sh::M;
  extern __shared__ __align__(16) uint32_t scan2_smem[];
  float* buf0 = reinterpret_cast<float*>(scan2_smem);
  float* buf1 = buf0 + kGroupWords;

  const int64_t q = int64_t(blockIdx.x) / p.nchunks;
  const int chunk = int(int64_t(blockIdx.x) % p.nchunks);
  if (p.qmask && !p.qmask[q]) return;  // the same for the whole block
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int jj = lane & (Sh::GS - 1), qq = lane >> Sh::LOG_GS;

  // this thread's codewords and query slice
  float cw[Sh::STEPS][DS];
#pragma unroll
  for (int s = 0; s < Sh::STEPS; ++s) {
    const int e = (s * NW + warp) * Sh::QQ + qq;
    const float* c = p.codebooks_t + (int64_t(e) * m + jj) * Sh::DS4;
#pragma unroll
    for (int t = 0; t < DS; ++t) cw[s][t] = __ldg(c + t);
  }
  float xs[DS];
  const float* x = p.queries + q * p.d + jj * DS;
#pragma unroll
  for (int t = 0; t < DS; ++t) xs[t] = __ldg(x + t);

  // precomputed terms: this thread's entries of the query's table
  // -2 <x^(jj), y_R(e)> (the codewords are not needed after this)
  float t3[PRE ? Sh::STEPS : 1];
  if constexpr (PRE) {
#pragma unroll
    for (int s = 0; s < Sh::STEPS; ++s) {
      float a = 0.f;
#pragma unroll
      for (int t = 0; t < DS; ++t) a = fmaf(xs[t], cw[s][t], a);
      t3[s] = -2.f * a;
    }
  }

  // table of list l into buf (fp32 entries, one per 4-byte slot): the direct
  // ||r^(jj) - y_R(e)||^2, or with precomputed terms T1[l][e][jj] + t3 (the
  // list's ||x - y_C||^2 is added to every distance of the list instead)
  // m = 32: the centroid slice of the list whose table is built next is
  // loaded one list early (scan ms 15.70 -> 15.48 on 2e8 vectors; it spills
  // registers for m <= 16, which load it in the build)
  constexpr bool CPF = MW == 8 && !PRE;
  float cnx[DS];
  auto load_cent = [&](int l) {
    if constexpr (CPF) {
      if (l >= 0) {
        const float* cl = p.centroids + int64_t(l) * p.d + jj * DS;
#pragma unroll
        for (int t = 0; t < DS; ++t) cnx[t] = __ldg(cl + t);
      }
    }
  };
  auto build = [&](int l, float* buf) {
    float r[DS];
    if constexpr (CPF) {
#pragma unroll
      for (int t = 0; t < DS; ++t) r[t] = xs[t] - cnx[t];
    } else if constexpr (!PRE) {
      const float* cl = p.centroids + int64_t(l) * p.d + jj * DS;
#pragma unroll
      for (int t = 0; t < DS; ++t) r[t] = xs[t] - __ldg(cl + t);
    }
    const float* t1 = p.term1 + int64_t(l) * 256 * m + jj;
    // m = 32: two table entries at a time with packed fp32x2 arithmetic
    // (scan ms 16.05 -> 15.67 on 2e8 vectors; slower for m = 8, so not there)
    constexpr bool PACKED = !PRE && MW == 8 && Sh::STEPS % 2 == 0;
    float tv2[PACKED ? Sh::STEPS : 1];
    if constexpr (PACKED) {
#pragma unroll
      for (int s = 0; s < Sh::STEPS; s += 2) {
        unsigned long long acc = 0ull;
#pragma unroll
        for (int t = 0; t < DS; ++t) {
          unsigned long long c2, r2, df;
          asm("mov.b64 %0, {%1, %2};" : "=l"(c2) : "f"(cw[s][t]), "f"(cw[s + 1][t]));
          asm("mov.b64 %0, {%1, %1};" : "=l"(r2) : "f"(r[t]));
          asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(df) : "l"(r2), "l"(c2));
          asm("fma.rn.f32x2 %0, %1, %1, %2;" : "=l"(acc) : "l"(df), "l"(acc));
        }
        asm("mov.b64 {%0, %1}, %2;" : "=f"(tv2[s]), "=f"(tv2[s + 1]) : "l"(acc));
      }
    }
#pragma unroll
    for (int s = 0; s < Sh::STEPS; ++s) {
      const int e = (s * NW + warp) * Sh::QQ + qq;
      float Tv = 0.f;
      if constexpr (PRE) {
        Tv = __ldg(t1 + e * m) + t3[s];
      } else if constexpr (PACKED) {
        Tv = tv2[s];
      } else {
#pragma unroll
        for (int t = 0; t < DS; ++t) {
          const float df = r[t] - cw[s][t];
          Tv = fmaf(df, df, Tv);
        }
      }
      float* row = buf + e * 64 + jj;
#pragma unroll
      for (int rep = 0; rep < Sh::REPS; ++rep)
        row[Sh::GS * ((rep + qq) & (Sh::REPS - 1))] = Tv;
    }
  };

  WarpSelect<KW, T> ws;
  ws.init(lane);
  const int p0 = chunk * p.per_chunk;
  const int n = max(0, min(p.nprobe, p0 + p.per_chunk) - p0);  // <= kScan2MaxLists
  const uint32_t lane4 = uint32_t(lane) * 4;

  // the block's lists: id (-1 if out of range), length, first block
  int* s_list = reinterpret_cast<int*>(scan2_smem + 2 * kGroupWords);
  int* s_len = s_list + kScan2MaxLists;
  int64_t* s_boff = reinterpret_cast<int64_t*>(s_len + kScan2MaxLists);
  float* s_c2 = reinterpret_cast<float*>(s_boff + kScan2MaxLists);
  for (int i = tid; i < n; i += NW * 32) {
    const int l = p.probes[q * p.nprobe + p0 + i];
    const bool v = l >= 0 && l < p.nlist;
    const int len = v ? p.list_len[l] : 0;
    const int64_t boff = v ? p.list_block_off[l] : 0;
    const bool in_range = dcheck(p.dbg, boff >= 0 && boff + ((len + 31) >> 5) <= p.nblocks, 8);
    s_list[i] = v ? l : -1;
    s_len[i] = in_range ? len : 0;
    s_boff[i] = boff;
  }
  if constexpr (PRE) {
    // ||x - y_C||^2 of each list, one warp per list (exact form, fp32)
    const float* xq = p.queries + q * p.d;
    for (int i = warp; i < n; i += NW) {
      const int l = p.probes[q * p.nprobe + p0 + i];
      float a = 0.f;
      if (l >= 0 && l < p.nlist) {
        const float* c = p.centroids + int64_t(l) * p.d;
        for (int t = lane; t < p.d; t += 32) {
          const float df = __ldg(xq + t) - __ldg(c + t);
          a = fmaf(df, df, a);
        }
      }
#pragma unroll
      for (int o = 16; o >= 1; o /= 2) a += __shfl_xor_sync(kFullMask, a, o);
      if (lane == 0) s_c2[i] = a;
    }
  }
  __syncthreads();

  if (tid == 0 && n > 0 && s_list[0] >= 0) prefetch_list(p, s_list[0], m);
  if (tid == 0 && n > 1 && s_list[1] >= 0) prefetch_list(p, s_list[1], m);
  if (n > 0) load_cent(s_list[0]);
  if (n > 0 && s_list[0] >= 0) build(s_list[0], buf0);
  if (n > 1) load_cent(s_list[1]);
  // R = 16 / MW blocks per warp and iteration (blocks b, b + 16, ..., all
  // congruent to the warp mod 16): 2 x 16 code words per lane, R
  // independent sums, the loop overhead shared by R blocks
  // (16 / MW measured faster than 8 / MW: scan ms 24.9 -> 23.9 for m = 8,
  // d/m = 12 and 12.5 -> 12.1 for m = 16, d/m = 8, although those two spill a
  // few bytes in the rarely taken merge path)
  constexpr int R = MW >= 8 ? 1 : (KW >= 128 ? 8 : 16) / MW;  // longer queues: fewer registers
  uint32_t c0[R][MW], c1[R][MW];
  auto load_group = [&](const uint8_t* lc, int b, int nb, uint32_t (&c)[R][MW]) {
#pragma unroll
    for (int r = 0; r < R; ++r)
      if (b + r * NW < nb) load_codes<MW>(lc + int64_t(b + r * NW) * 32 * m, lane, c[r]);
  };
  if (n > 0) load_group(p.codes + s_boff[0] * 32 * m, warp, (s_len[0] + 31) >> 5, c0);
  __syncthreads();

  for (int i = 0; i < n; ++i) {
    float* cur = (i & 1) ? buf1 : buf0;
    float* nxt = (i & 1) ? buf0 : buf1;
    if (i + 1 < n) {
      // two lists ahead (2e8 vectors x 10,000 queries x 64 probes, scan ms: none
      // 20.0, one 15.8-16.8 depending on the GPU, two 16.0-16.05 on every GPU
      // measured, four 16.5)
      if (tid == 0 && i + 2 < n && s_list[i + 2] >= 0) prefetch_list(p, s_list[i + 2], m);
      if (s_list[i + 1] >= 0) build(s_list[i + 1], nxt);
      if (i + 2 < n) load_cent(s_list[i + 2]);
    }
    const int len = s_len[i];
    const int64_t boff = s_boff[i];
    const int nb = (len + 31) >> 5;
    const uint8_t* lcodes = p.codes + boff * 32 * m;
    const char* lut_bytes = reinterpret_cast<const char*>(cur);
    const float c2 = PRE ? s_c2[i] : 0.f;
    for (int b = warp; b < nb; b += R * NW) {
      load_group(lcodes, b + R * NW, nb, c1);
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const int br = b + r * NW;  // the same in every lane
        if (br < nb) {
          float dist = adc_sum<MW, IVFPQ_LUT_FP32>(c0[r], lut_bytes, lane4);
          if constexpr (PRE) dist = fmaxf(dist + c2, 0.f);  // keys are raw bits of d >= 0
          const bool valid = br * 32 + lane < len;
          ws.add(valid ? __float_as_uint(dist) : kSentinelKey,
                 uint32_t((boff + br) * 32 + lane));
        }
      }
#pragma unroll
      for (int r = 0; r < R; ++r)
#pragma unroll
        for (int w = 0; w < MW; ++w) c0[r][w] = c1[r][w];
    }
    // this warp's first blocks of the next list, before the barrier
    if (i + 1 < n) load_group(p.codes + s_boff[i + 1] * 32 * m, warp, (s_len[i + 1] + 31) >> 5, c0);
    __syncthreads();  // cur may be overwritten next; nxt is complete
  }
  ws.finalize();
  // this warp's KW best, ascending (sentinel-padded)
  const int64_t o = ((q * p.nchunks + chunk) * NW + warp) * KW;
  if (!dcheck(p.dbg, q < p.nq || p.nq == 0, 9)) return;  // after the last barrier
#pragma unroll
  for (int r = 0; r < KW / 32; ++r) {
    p.pkeys[o + 32 * r + lane] = ws.wk[r];
    p.pidx[o + 32 * r + lane] = ws.wv[r];
  }
}

// two table buffers and the staged probe list
inline size_t scan2_smem_bytes() { return size_t(2) * kGroupWords * 4 + kScan2MaxLists * 20; }

// Warp-queue length: each warp's share of the k best is about k / 16 (with a
// binomial spread of about sqrt(k / 16)), so these leave a wide margin; a
// query whose share overflowed anyway is repaired by the caller.
inline int scan2_kw(int k) { return k <= 128 ? 32 : k <= 256 ? 64 : k <= 1024 ? 128 : 256; }

template <int MW, int DS, int KW, bool PRE>
int launch_scan2(const ScanParams& p, int64_t nq, cudaStream_t s) {
  auto kern = ivfpq_scan2_kernel<MW, DS, KW, PRE>;
  const size_t smem = scan2_smem_bytes();
  IVFPQ_TRY(set_dynamic_smem(kern, smem));
  const int64_t blocks = nq * p.nchunks;
  kern<<<unsigned(blocks), kScan2Warps * 32, smem, s>>>(p);
  IVFPQ_LAUNCHED_K(kern, smem, kScan2Warps * 32);
  return IVFPQ_OK;
}

}  // namespace ivfpq

#define IVFPQ_INST_SCAN2(MW, DS, KW, PRE)                                                  \
  template int ivfpq::launch_scan2<MW, DS, KW, PRE>(const ivfpq::ScanParams&, int64_t,      \
                                                    cudaStream_t);
