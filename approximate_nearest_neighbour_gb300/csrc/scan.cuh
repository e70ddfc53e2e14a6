// Fused ADC lookup-table build, inverted-list scan and per-chunk k-selection.
//
// Source: "Billion-scale similarity search with GPUs", section 5 -- the
// tables T_1..T_b of 256 entries per sub-quantizer (a distance is b look-ups
// and additions), the tables kept in shared memory, queries x lists processed
// independently, and the two-pass k-selection (k results per chunk of lists,
// then a final k-selection); "Custom 8-bit floating point value format ...",
// search steps 2-5 and Eq. (1): residual r = q - c, F(y_j) = ||r_j - codeword||^2,
// R = sum_j F(y_j).
//
// One thread block handles one query and a chunk of `per_chunk` of its probed
// lists. For each list it forms the residual, builds all m tables in shared
// memory, and its 8 warps scan the list's 32-vector blocks (warp w takes
// blocks w, w+8, ...); lane i of a warp computes the distance of the vector in
// slot i and inserts it into the warp's WarpSelect. The warp queues survive
// across the chunk's lists; at the end they are merged (BlockSelect) and the
// chunk's k best (distance, slot) pairs are written out.
//
// Shared-memory table layout (fp32): tables are grouped by 32; a group is a
// 256 x 64 array of 4-byte words, row e = reproduction value, and column c
// holds the table of sub-quantizer 32g + (c mod gs). At step s of a group,
// lane i reads column i + s of row code_byte. Word (e, c) sits in bank
// (64 e + c) mod 32 = c mod 32, and i + s takes 32 distinct values mod 32
// across the warp, so every look-up instruction is free of bank conflicts
// whatever the code bytes are. (A plain table per sub-quantizer, entry e in
// word e, gives up to 7 conflicts per look-up in fp32 and 3 in fp16, as the
// 8-bit-float page computes.) The code bytes are stored pre-rotated
// (layout.cuh) so that the byte lane i needs at step s is simply stored byte s.
#pragma once

#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "internal.h"
#include "layout.cuh"
#include "select.cuh"

namespace ivfpq {

struct ScanParams {
  const float* queries;      // [nq, d]
  const float* centroids;    // [nlist, d]
  const float* codebooks_t;  // [256, m, dsub4], zero-padded
  const int32_t* probes;     // [nq, nprobe]
  const int32_t* list_len;   // [nlist]
  const int64_t* list_block_off;  // [nlist + 1]
  const uint8_t* codes;      // blocks of 32 * m bytes
  uint32_t* pkeys;           // [nq, nchunks, k] (scan2: [nq, nchunks, warps, kw])
  uint32_t* pidx;
  int d, m, dsub, dsub4, nlist, nprobe, per_chunk, nchunks, k;
  int lut_type;              // IVFPQ_LUT_FP32 / FP16 / FP8
  const int* qmask = nullptr;  // if set, only queries q with qmask[q] != 0 are scanned
  const float* term1 = nullptr;  // precomputed list terms [nlist, 256, m] (register-codebook scan)
  int64_t nq = 0;              // queries of the batch (debug checks)
  int64_t nblocks = 0;         // code blocks stored (debug checks)
  int* dbg = nullptr;          // device status word of the debug build, else null
};

constexpr int kScanWarps = 8;
constexpr int kGroupWords = 256 * 64;  // one group of up to 32 tables

inline size_t scan_smem_bytes(int m, int dsub4, int K) {
  const size_t lut = size_t((m + 31) / 32) * kGroupWords * 4;
  const size_t merge = size_t(kScanWarps) * K * 8;
  return (lut > merge ? lut : merge) + size_t(m) * dsub4 * 4;
}

__device__ __forceinline__ uint4 ld_code16(const uint8_t* p) {
  return __ldcs(reinterpret_cast<const uint4*>(p));
}
__device__ __forceinline__ uint2 ld_code8(const uint8_t* p) {
  return __ldcs(reinterpret_cast<const uint2*>(p));
}
__device__ __forceinline__ uint32_t ld_code4(const uint8_t* p) {
  return __ldcs(reinterpret_cast<const unsigned int*>(p));
}

// Asks the TMA unit to stream [p, p + bytes) from HBM into L2 (no completion
// to wait for; the later loads of the scan hit L2). p and bytes are multiples
// of 16.
__device__ __forceinline__ void prefetch_l2(const uint8_t* p, int64_t bytes) {
  for (int64_t o = 0; o < bytes; o += 65536) {
    const uint32_t n = uint32_t(bytes - o < 65536 ? bytes - o : 65536);
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p + o), "r"(n) : "memory");
  }
}

__device__ __forceinline__ void prefetch_list(const ScanParams& p, int l, int m) {
  if (l < 0 || l >= p.nlist) return;
  const int64_t nb = (int64_t(p.list_len[l]) + 31) >> 5;
  if (nb > 0) prefetch_l2(p.codes + p.list_block_off[l] * 32 * m, nb * 32 * m);
}

// Stored code words of slot `lane` in a block (MW = m / 4 words).
template <int MW>
__device__ __forceinline__ void load_codes(const uint8_t* blk, int lane, uint32_t (&w)[MW]) {
  constexpr int NF = MW / 4, RW = MW % 4;
#pragma unroll
  for (int c = 0; c < NF; ++c) {
    const uint4 v = ld_code16(blk + c * 512 + lane * 16);
    w[4 * c] = v.x;
    w[4 * c + 1] = v.y;
    w[4 * c + 2] = v.z;
    w[4 * c + 3] = v.w;
  }
  const uint8_t* rp = blk + NF * 512 + lane * (4 * RW);
  if (RW == 1) {
    w[4 * NF] = ld_code4(rp);
  } else if (RW == 2) {
    const uint2 v = ld_code8(rp);
    w[4 * NF] = v.x;
    w[4 * NF + 1] = v.y;
  } else if (RW == 3) {
    w[4 * NF] = ld_code4(rp);
    w[4 * NF + 1] = ld_code4(rp + 4);
    w[4 * NF + 2] = ld_code4(rp + 8);
  }
}

// One table entry of the given storage type at a byte address (each entry
// occupies a 4-byte slot; binary16 and E4M3 values sit in its low bytes).
template <int LT>
__device__ __forceinline__ float lut_load(const char* addr) {
  if constexpr (LT == IVFPQ_LUT_FP32) {
    return *reinterpret_cast<const float*>(addr);
  } else if constexpr (LT == IVFPQ_LUT_FP16) {
    return __half2float(*reinterpret_cast<const __half*>(addr));
  } else {
    const __nv_fp8_storage_t b = *reinterpret_cast<const __nv_fp8_storage_t*>(addr);
    return __half2float(__half(__nv_cvt_fp8_to_halfraw(b, __NV_E4M3)));
  }
}

// Sum of the m table entries selected by the stored code words. The byte
// offset of entry (code byte e, column lane + s) is e*256 + 4*lane + 4*s; one
// byte permute builds e*256 + 4*lane from the code word and lane4 = 4*lane,
// and 4*s (plus the group offset) is a constant. Sums are in fp32 for every
// table type (E4M3 sums are scaled by the caller).
template <int MW, int LT>
__device__ __forceinline__ float adc_sum(const uint32_t (&w)[MW], const char* lut_bytes,
                                         uint32_t lane4) {
  // four independent accumulation chains keep the adds off the critical path
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int s = 0; s < 4 * MW; ++s) {
    const uint32_t off = __byte_perm(w[s >> 2], lane4, 0x5504u | (uint32_t(s & 3) << 4));
    acc[s & 3] += lut_load<LT>(lut_bytes + off + ((s >> 5) * kGroupWords + (s & 31)) * 4);
  }
  return (acc[0] + acc[1]) + (acc[2] + acc[3]);
}

// Converts the fp32 tables in place to the storage type (all words of the
// groups; every thread of the block takes part). binary16: round to nearest
// even. E4M3: one scale per table set, s = max T / 448 (the largest finite
// E4M3 value), entries stored as E4M3(T / s) with round-to-nearest-even and
// saturation; *scale receives s. Ends with the block synchronized.
__device__ __forceinline__ void quantize_lut(uint32_t* lut, int nwords, int lut_type,
                                             float* scale, uint32_t* red, int tid) {
  if (lut_type == IVFPQ_LUT_FP16) {
    for (int i = tid; i < nwords; i += kScanWarps * 32)
      lut[i] = __half_as_ushort(__float2half_rn(__uint_as_float(lut[i])));
    __syncthreads();
    return;
  }
  // E4M3: block-wide maximum first (entries are >= 0, so their bits order
  // like unsigned integers)
  uint32_t mx = 0;
  for (int i = tid; i < nwords; i += kScanWarps * 32) mx = max(mx, lut[i]);
#pragma unroll
  for (int o = 16; o >= 1; o /= 2) mx = max(mx, __shfl_xor_sync(kFullMask, mx, o));
  if (tid == 0) *red = 0;
  __syncthreads();
  if ((tid & 31) == 0) atomicMax(red, mx);
  __syncthreads();
  const float tmax = __uint_as_float(*red);
  const float s = tmax > 0.f ? tmax / 448.f : 1.f;
  const float inv = tmax > 0.f ? 448.f / tmax : 1.f;
  for (int i = tid; i < nwords; i += kScanWarps * 32) {
    const float v = __uint_as_float(lut[i]) * inv;
    lut[i] = uint32_t(__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3));
  }
  if (tid == 0) *scale = s;
  __syncthreads();
}

// Scans blocks warp, warp + NW, ... of one list with tables of type LT.
template <int MW, int LT, class WS>
__device__ __forceinline__ void scan_list(WS& ws, const uint8_t* lcodes, int64_t boff, int nb,
                                          int len, int m, const char* lut_bytes,
                                          uint32_t lane4, float scale, int warp, int lane) {
  constexpr int NW = kScanWarps;
  uint32_t cur[MW], nxt[MW];
  int b = warp;
  if (b < nb) load_codes<MW>(lcodes + int64_t(b) * 32 * m, lane, cur);
  for (; b < nb; b += NW) {
    const int bn = b + NW;
    if (bn < nb) load_codes<MW>(lcodes + int64_t(bn) * 32 * m, lane, nxt);
    float dist = adc_sum<MW, LT>(cur, lut_bytes, lane4);
    if (LT == IVFPQ_LUT_FP8) dist *= scale;
    const bool valid = b * 32 + lane < len;
    ws.add(valid ? __float_as_uint(dist) : kSentinelKey, uint32_t((boff + b) * 32 + lane));
#pragma unroll
    for (int w = 0; w < MW; ++w) cur[w] = nxt[w];
  }
}

// Residual r = q - c_l into shared memory as [m][dsub4], zero-padded.
__device__ __forceinline__ void residual(float* res, const ScanParams& p, int64_t q, int l,
                                         int m, int tid) {
  const float* x = p.queries + q * p.d;
  const float* c = p.centroids + int64_t(l) * p.d;
  for (int i = tid; i < m * p.dsub4; i += kScanWarps * 32) {
    const int j = i / p.dsub4, t = i - j * p.dsub4;
    res[i] = t < p.dsub ? x[j * p.dsub + t] - c[j * p.dsub + t] : 0.f;
  }
}

// Tables of group g (sub-quantizers [32g, 32g + GS)) when GS is a power of
// two and dsub4 = 4*NV: lane -> table jj = lane % GS (fixed, so its residual
// slice stays in registers) and value e = (it + lane) / GS; each entry is
// computed once and stored to its 64/GS columns, lane i starting at a
// different copy so the 32 stores of one instruction hit 32 distinct banks.
template <int GS, int NV>
__device__ __forceinline__ void build_group(float* base, const float* res, const float* cbt,
                                            int m, int g, int warp, int lane) {
  constexpr int REPS = 64 / GS;
  constexpr int LOG_GS = GS == 32 ? 5 : GS == 16 ? 4 : GS == 8 ? 3 : 2;
  const int jj = lane & (GS - 1), qq = lane >> LOG_GS;
  const int j = 32 * g + jj;
  float4 rr[NV];
  const float4* r4 = reinterpret_cast<const float4*>(res) + j * NV;
#pragma unroll
  for (int i = 0; i < NV; ++i) rr[i] = r4[i];
  const float4* cb4 = reinterpret_cast<const float4*>(cbt);
#pragma unroll 2
  for (int it = warp * 32; it < 256 * GS; it += kScanWarps * 32) {
    const int e = (it + lane) >> LOG_GS;
    const float4* c = cb4 + (e * m + j) * NV;
    float T = 0.f;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const float4 cv = __ldg(c + i);
      float df = rr[i].x - cv.x;
      T = fmaf(df, df, T);
      df = rr[i].y - cv.y;
      T = fmaf(df, df, T);
      df = rr[i].z - cv.z;
      T = fmaf(df, df, T);
      df = rr[i].w - cv.w;
      T = fmaf(df, df, T);
    }
    float* row = base + e * 64 + jj;
#pragma unroll
    for (int s = 0; s < REPS; ++s) row[GS * ((s + qq) & (REPS - 1))] = T;
  }
}

// Any group size / dsub4: every (row, column) word is computed directly.
__device__ __forceinline__ void build_group_generic(float* base, const float* res,
                                                    const float* cbt, int m, int dsub4, int g,
                                                    int warp, int lane) {
  const int gs = group_size(g, m);
  const int nv = dsub4 >> 2;
  const float4* cb4 = reinterpret_cast<const float4*>(cbt);
  const float4* r4 = reinterpret_cast<const float4*>(res);
  for (int it = warp * 32 + lane; it < kGroupWords; it += kScanWarps * 32) {
    const int e = it >> 6, col = it & 63;
    const int j = 32 * g + col % gs;
    float T = 0.f;
    for (int i = 0; i < nv; ++i) {
      const float4 cv = __ldg(cb4 + (e * m + j) * nv + i);
      const float4 rv = r4[j * nv + i];
      float df = rv.x - cv.x;
      T = fmaf(df, df, T);
      df = rv.y - cv.y;
      T = fmaf(df, df, T);
      df = rv.z - cv.z;
      T = fmaf(df, df, T);
      df = rv.w - cv.w;
      T = fmaf(df, df, T);
    }
    base[it] = T;
  }
}

template <int GS>
__device__ __forceinline__ void build_group_nv(float* base, const float* res, const float* cbt,
                                               int m, int dsub4, int g, int warp, int lane) {
  switch (dsub4 >> 2) {
    case 1: build_group<GS, 1>(base, res, cbt, m, g, warp, lane); break;
    case 2: build_group<GS, 2>(base, res, cbt, m, g, warp, lane); break;
    case 3: build_group<GS, 3>(base, res, cbt, m, g, warp, lane); break;
    case 4: build_group<GS, 4>(base, res, cbt, m, g, warp, lane); break;
    default: build_group_generic(base, res, cbt, m, dsub4, g, warp, lane); break;
  }
}

// All m tables of the residual into `lut` (MW > 0: m = 4*MW known).
template <int MW>
__device__ __forceinline__ void build_lut(float* lut, const float* res, const float* cbt,
                                          int m, int dsub4, int warp, int lane) {
  if constexpr (MW > 0) {
    constexpr int NG = (4 * MW + 31) / 32;
    constexpr int GS = 4 * MW < 32 ? 4 * MW : 32;
    static_assert((GS & (GS - 1)) == 0, "power-of-two group");
#pragma unroll
    for (int g = 0; g < NG; ++g)
      build_group_nv<GS>(lut + g * kGroupWords, res, cbt, m, dsub4, g, warp, lane);
  } else {
    const int ng = (m + 31) >> 5;
    for (int g = 0; g < ng; ++g)
      build_group_generic(lut + g * kGroupWords, res, cbt, m, dsub4, g, warp, lane);
  }
}

// Blocks per SM that the shared-memory tables allow (64 KB per group of 32
// sub-quantizers, 64 KB of block-merge area up to K = 1024), given to the
// compiler so that registers do not become the tighter limit.
template <int MW, int K>
constexpr int scan_min_blocks() {
  return (MW > 0 && MW <= 8 && K <= 1024) ? 3 : 1;
}

template <int MW, int K>
__global__ void __launch_bounds__(kScanWarps * 32, (scan_min_blocks<MW, K>()))
ivfpq_scan_kernel(const ScanParams p) {
  constexpr int T = ThreadQ<K>::value;
  constexpr int NW = kScanWarps;
  extern __shared__ __align__(16) uint32_t scan_smem[];
  const int m = MW > 0 ? 4 * MW : p.m;
  const int ngroups = (m + 31) >> 5;
  float* lut = reinterpret_cast<float*>(scan_smem);
  const int lut_words = ngroups * kGroupWords;
  const int merge_words = NW * K * 2;
  float* res = reinterpret_cast<float*>(scan_smem) + (lut_words > merge_words ? lut_words : merge_words);

  const int64_t q = int64_t(blockIdx.x) / p.nchunks;
  const int chunk = int(int64_t(blockIdx.x) % p.nchunks);
  if (p.qmask && !p.qmask[q]) return;  // the same for the whole block
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  WarpSelect<K, T> ws;
  ws.init(lane);
  __shared__ float lut_scale;  // E4M3 tables: the scale of the current table set
  __shared__ uint32_t lut_red;
  const int p0 = chunk * p.per_chunk;
  const int p1 = min(p.nprobe, p0 + p.per_chunk);
  const int32_t* qprobes = p.probes + q * p.nprobe;
  const char* lut_bytes = reinterpret_cast<const char*>(lut);
  const uint32_t lane4 = uint32_t(lane) * 4;
  if (tid == 0 && p0 < p1) prefetch_list(p, qprobes[p0], m);

  for (int pi = p0; pi < p1; ++pi) {
    const int l = qprobes[pi];
    if (tid == 0 && pi + 1 < p1) prefetch_list(p, qprobes[pi + 1], m);
    if (l < 0 || l >= p.nlist) continue;  // same value for the whole block
    __syncthreads();  // the previous list's scan no longer reads the tables
    residual(res, p, q, l, m, tid);
    __syncthreads();
    build_lut<MW>(lut, res, p.codebooks_t, m, p.dsub4, warp, lane);
    __syncthreads();
    if (p.lut_type != IVFPQ_LUT_FP32)
      quantize_lut(scan_smem, lut_words, p.lut_type, &lut_scale, &lut_red, tid);
    const int64_t boff = p.list_block_off[l];
    const bool in_range = dcheck(
        p.dbg, boff >= 0 && boff + ((int64_t(p.list_len[l]) + 31) >> 5) <= p.nblocks, 10);
    const int len = in_range ? p.list_len[l] : 0;
    const int nb = (len + 31) >> 5;
    const uint8_t* lcodes = p.codes + boff * 32 * m;
    if constexpr (MW > 0) {
      if (p.lut_type == IVFPQ_LUT_FP32)
        scan_list<MW, IVFPQ_LUT_FP32>(ws, lcodes, boff, nb, len, m, lut_bytes, lane4, 1.f, warp,
                                      lane);
      else if (p.lut_type == IVFPQ_LUT_FP16)
        scan_list<MW, IVFPQ_LUT_FP16>(ws, lcodes, boff, nb, len, m, lut_bytes, lane4, 1.f, warp,
                                      lane);
      else
        scan_list<MW, IVFPQ_LUT_FP8>(ws, lcodes, boff, nb, len, m, lut_bytes, lane4, lut_scale,
                                     warp, lane);
    } else {
      const char* lut_lane = lut_bytes + lane4;
      for (int b = warp; b < nb; b += NW) {
        const uint8_t* blk = lcodes + int64_t(b) * 32 * m;
        float dist = 0.f;
        for (int s0 = 0; s0 < m; s0 += 4) {
          const uint32_t word =
              *reinterpret_cast<const uint32_t*>(blk + stored_byte_offset(lane, s0, m));
#pragma unroll
          for (int bb = 0; bb < 4; ++bb) {
            const int s = s0 + bb;
            const uint32_t byte = (word >> (8 * bb)) & 0xffu;
            const char* a = lut_lane + ((s >> 5) * kGroupWords + int(byte) * 64 + (s & 31)) * 4;
            dist += p.lut_type == IVFPQ_LUT_FP32   ? lut_load<IVFPQ_LUT_FP32>(a)
                    : p.lut_type == IVFPQ_LUT_FP16 ? lut_load<IVFPQ_LUT_FP16>(a)
                                                   : lut_load<IVFPQ_LUT_FP8>(a);
          }
        }
        if (p.lut_type == IVFPQ_LUT_FP8) dist *= lut_scale;
        const bool valid = b * 32 + lane < len;
        ws.add(valid ? __float_as_uint(dist) : kSentinelKey, uint32_t((boff + b) * 32 + lane));
      }
    }
  }
  ws.finalize();
  __syncthreads();  // the table area is reused for the block merge
  block_merge<K, T, NW>(ws, scan_smem, scan_smem + NW * K, warp);
  if (warp == 0) {
    const int64_t o = (q * p.nchunks + chunk) * p.k;
#pragma unroll
    for (int r = 0; r < K / 32; ++r) {
      const int i = 32 * r + lane;
      if (i < p.k) {
        p.pkeys[o + i] = ws.wk[r];
        p.pidx[o + i] = ws.wv[r];
      }
    }
  }
}

template <int MW, int K>
int launch_scan_mw(const ScanParams& p, int64_t nq, cudaStream_t s) {
  auto kern = ivfpq_scan_kernel<MW, K>;
  const size_t smem = scan_smem_bytes(p.m, p.dsub4, K);
  IVFPQ_TRY(set_dynamic_smem(kern, smem));
  const int64_t blocks = nq * p.nchunks;
  kern<<<unsigned(blocks), kScanWarps * 32, smem, s>>>(p);
  IVFPQ_LAUNCHED_K(kern, smem, kScanWarps * 32);
  return IVFPQ_OK;
}

}  // namespace ivfpq

#define IVFPQ_INST_SCAN(MW, K) \
  template int ivfpq::launch_scan_mw<MW, K>(const ivfpq::ScanParams&, int64_t, cudaStream_t);
