// List-major ADC scan: the queries that probe one inverted list are scanned
// together, so one load of a code block and one byte permute per code byte
// serve the tables of G queries.
//
// Same computation as the other list scans ("Billion-scale similarity search
// with GPUs", section 5: tables T_1..T_b per query and list, b look-ups and
// additions per code; "Custom 8-bit floating point value format ...", search
// steps 2-5 and Eq. (1)); the section's queries x lists work is organised by
// list instead of by query:
//  * a work item is one list and up to G of the queries that probe it (the
//    (list, query) pairs sorted by list, cut into groups of G); items run in
//    list order, so the blocks working at one time share lists in L2;
//  * one persistent block of 16 warps per SM takes items blockIdx.x,
//    blockIdx.x + gridDim.x, ...; the 256 x m codewords stay in registers
//    for the whole kernel (d/2 floats per thread, as in scan2.cuh);
//  * shared memory holds the item's table sets (one query's fp32 tables,
//    two queries' binary16 or four queries' E4M3 entries per 32-bit word),
//    each a 256 x 64-word array whose two 32-column halves are the double
//    buffer: item t is scanned from half t & 1 while item t + 1's tables are
//    built into the other half; a
//    column c of a half holds table c mod m, lane i reads column
//    (i & ~(m-1)) | ((i + s) & (m-1)) at stored position s (table
//    (i + s) mod m, the sub-quantizer of that stored byte), so the 32 lanes
//    of a look-up hit 32 banks; the query and the half are immediates;
//  * selection is a filter: every query has a bound theta, and a code whose
//    distance is at most theta is appended, with its id, to the query's
//    candidate buffer (one atomic per warp and query); the k smallest
//    candidates are the query's result, and a query whose buffer overflows
//    is scanned again by the general kernel;
//  * a long list's records may be cut into units of unit_len codes (up to 16
//    per record), so one list's items do not keep a few blocks busy alone;
//  * the bound comes from a first pass of the same kernel over every query's
//    nearest list alone (TQ > 0; one item per query and chunk of that list,
//    the chunks at least 32,768 codes long and at most 4 per list, so a long
//    list is spread over blocks): each lane keeps the TQ smallest distances
//    of the codes it scores (a sorted register queue, no communication
//    between lanes) and writes them out; the k-th smallest of the query's
//    512 * TQ distances per chunk (512 * TQ >= k) is at least the k-th
//    smallest of the list (a lane that saw more than TQ of the list's k
//    smallest only makes it larger), hence at least the query's final k-th
//    distance.
#pragma once

#include <type_traits>

#include "scan2.cuh"

namespace ivfpq {

constexpr int kLmWarps = 16;
constexpr int kLmSlots = 3;  // item descriptors in flight: scanned, built, fetched
constexpr int kLmMaxG = 8;   // queries per item at most
constexpr int kLmMaxChunks = 16;  // chunks of one record at most

struct LmParams {
  ScanParams s;                // tables, lists, codes, shapes (nprobe unused)
  const int32_t* pair_list;    // [npairs] list of each (list, query) pair, sorted
  const int32_t* pair_query;   // [npairs] query of each pair
  const int32_t* items;        // [n_items] first pair of each item
  const int* n_items;          // device scalar
  int64_t npairs;
  // filter pass: bound of query q (raw bits of a distance >= 0, or the
  // sentinel for none) at theta_key[q * theta_stride]
  const uint32_t* theta_key;
  int theta_stride;
  const int64_t* ids;          // slot -> id
  uint32_t* ckey;              // [nq, cap] candidate distances (raw bits)
  int64_t* cid;                // [nq, cap] candidate ids
  int* ccount;                 // [nq] candidates appended (may exceed cap)
  int cap;
  // bound pass: lane i of warp w's TQ smallest distances for item it at
  // part_key[((it * 16 + w) * 32 + i) * TQ ..], ascending, sentinel-padded
  uint32_t* part_key;
  // item records (lm_records_kernel, bound_records_kernel): rec_bytes each
  const uint8_t* records;
  uint8_t* records_w = nullptr;  // the same, for the kernels that write them
  // the kernel's i-th item is record order[i] (null: record i)
  const int32_t* order = nullptr;
  // long lists in chunks (null: one unit of work per record): unit i is chunk
  // units[i] % kLmMaxChunks (codes [c * unit_len, (c + 1) * unit_len)) of
  // record units[i] / kLmMaxChunks; *n_units units
  const int32_t* units = nullptr;
  const int* n_units = nullptr;
  int unit_len = 0;
  int rec_bytes;
  int dpad;                    // d rounded up to a multiple of 4
};

// Head of an item record; the G residuals x_q - c_list (dpad floats each)
// follow at byte kLmHead.
struct LmHead {
  int list, len, nq, item;  // item: its index (the bound pass writes by item)
  int64_t boff;
  int q[kLmMaxG];
  uint32_t theta[kLmMaxG];
  float scale[kLmMaxG];  // E4M3 tables: each query's table scale (set by the build)
};
constexpr int kLmHead = 128;
static_assert(sizeof(LmHead) <= kLmHead, "record head");

inline int lm_record_bytes(int G, int d) { return kLmHead + G * ((d + 3) & ~3) * 4; }

__device__ __forceinline__ void lm_cp_async16(void* smem, const void* gmem) {
  const uint32_t sa = uint32_t(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sa), "l"(gmem) : "memory");
}

// Column byte offsets of stored positions 4a .. 4a + 3 for lane `lane`, one
// per byte (each below 128).
template <int GS>
__device__ __forceinline__ uint32_t lm_lane_columns(int lane, int a) {
  uint32_t r = 0;
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    const int s = 4 * a + b;
    const uint32_t c = uint32_t((lane & ~(GS - 1)) | ((lane + s) & (GS - 1)));
    r |= (c * 4u) << (8 * b);
  }
  return r;
}

template <int SEL>
__device__ __forceinline__ uint32_t lm_prmt(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "n"(SEL));
  return r;
}

// Table look-ups of one slot for GG queries: acc[g][s & 3] += T_g[row(s)][col(s)]
// for every stored position s. The row is code byte s & 3 of word s / 4,
// the column byte offset byte s & 3 of lcol[s / 4]; one prmt puts them at
// bytes 1 and 0 (its two upper bytes are copies of the sign of a column
// byte, zero). Table set g of half P is at byte g * 65536 + 128 * P.
template <int MW, int GG, int P, int S = 0>
__device__ __forceinline__ void lm_lookups(const uint32_t (&w)[MW], const char* tab,
                                           const uint32_t (&lcol)[MW], float (&acc)[GG][4]) {
  if constexpr (S < 4 * MW) {
    constexpr int SEL = 0xCC00 | ((S & 3) << 4) | (4 + (S & 3));
    const uint32_t off = lm_prmt<SEL>(w[S >> 2], lcol[S >> 2]);
#pragma unroll
    for (int g = 0; g < GG; ++g)
      acc[g][S & 3] += *reinterpret_cast<const float*>(tab + off + g * 65536 + 128 * P);
    lm_lookups<MW, GG, P, S + 1>(w, tab, lcol, acc);
  }
}

// binary16 tables: word (row, column) of table set g holds the entries of
// queries 2g (low half) and 2g + 1 (high half); each is added to its fp32
// sum (mixed-precision add: exact conversion, one rounding). NC sums per
// query (4, or 2 with three table sets, where 4 would spill registers).
template <int MW, int NS, int NC, int P, int S = 0>
__device__ __forceinline__ void lm_lookups_h(const uint32_t (&w)[MW], const char* tab,
                                             const uint32_t (&lcol)[MW], float (&acc)[2 * NS][4]) {
  if constexpr (S < 4 * MW) {
    constexpr int SEL = 0xCC00 | ((S & 3) << 4) | (4 + (S & 3));
    const uint32_t off = lm_prmt<SEL>(w[S >> 2], lcol[S >> 2]);
#pragma unroll
    for (int g = 0; g < NS; ++g) {
      const uint32_t v = *reinterpret_cast<const uint32_t*>(tab + off + g * 65536 + 128 * P);
      asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
          "add.rn.f32.f16 %0, lo, %0;\n\tadd.rn.f32.f16 %1, hi, %1;\n\t}"
          : "+f"(acc[2 * g][S % NC]), "+f"(acc[2 * g + 1][S % NC])
          : "r"(v));
    }
    lm_lookups_h<MW, NS, NC, P, S + 1>(w, tab, lcol, acc);
  }
}

// E4M3 tables: word (row, column) of table set g holds the entries of queries
// 4g .. 4g + 3 (byte i: query 4g + i), each decoded exactly to binary16 and
// added to its query's fp32 sum (mixed-precision add, one rounding).
__device__ __forceinline__ void lm_add_h2(float& a, float& b, uint32_t h2) {
  asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
      "add.rn.f32.f16 %0, lo, %0;\n\tadd.rn.f32.f16 %1, hi, %1;\n\t}"
      : "+f"(a), "+f"(b)
      : "r"(h2));
}
template <int MW, int NS, int NC, int P, int S = 0>
__device__ __forceinline__ void lm_lookups_q8(const uint32_t (&w)[MW], const char* tab,
                                              const uint32_t (&lcol)[MW], float (&acc)[4 * NS][4]) {
  if constexpr (S < 4 * MW) {
    constexpr int SEL = 0xCC00 | ((S & 3) << 4) | (4 + (S & 3));
    const uint32_t off = lm_prmt<SEL>(w[S >> 2], lcol[S >> 2]);
#pragma unroll
    for (int g = 0; g < NS; ++g) {
      const uint32_t v = *reinterpret_cast<const uint32_t*>(tab + off + g * 65536 + 128 * P);
      const __half2_raw h01 =
          __nv_cvt_fp8x2_to_halfraw2(__nv_fp8x2_storage_t(v & 0xffffu), __NV_E4M3);
      const __half2_raw h23 = __nv_cvt_fp8x2_to_halfraw2(__nv_fp8x2_storage_t(v >> 16), __NV_E4M3);
      lm_add_h2(acc[4 * g][S % NC], acc[4 * g + 1][S % NC],
                uint32_t(h01.x) | (uint32_t(h01.y) << 16));
      lm_add_h2(acc[4 * g + 2][S % NC], acc[4 * g + 3][S % NC],
                uint32_t(h23.x) | (uint32_t(h23.y) << 16));
    }
    lm_lookups_q8<MW, NS, NC, P, S + 1>(w, tab, lcol, acc);
  }
}

// Per-query partial sums of one code block (acc[q][s & 3] over positions s).
template <int NA>
struct LmAcc {
  float v[NA][4];
};

// Appends (dist, id of slot) to query q's candidates where `pass` holds.
// All 32 lanes call it together.
__device__ __forceinline__ void lm_append(const LmParams& p, int q, bool pass, float dist,
                                          uint32_t slot, int lane) {
  const unsigned mask = __ballot_sync(kFullMask, pass);
  if (mask == 0u) return;
  const int leader = __ffs(mask) - 1;
  int base = 0;
  if (lane == leader) base = atomicAdd(p.ccount + q, __popc(mask));
  base = __shfl_sync(kFullMask, base, leader);
  if (pass) {
    const int pos = base + __popc(mask & ((1u << lane) - 1u));
    if (pos < p.cap &&
        dcheck(p.s.dbg, int64_t(slot) < p.s.nblocks * 32 && q >= 0 && q < p.s.nq, 5)) {
      const int64_t o = int64_t(q) * p.cap + pos;
      p.ckey[o] = __float_as_uint(dist);
      p.cid[o] = p.ids[slot];
    }
  }
}

// Code blocks in flight per warp. The bound pass (one query per item, a few
// look-ups per code) gains from a deep ring with short codes; the filter
// pass does not: billion (m = 8, binary16) planning / filter ms at 10,000
// queries, depth 2: 1.34 / 12.03, bound 8: 0.90, filter 3: 12.88, filter 4:
// 14.59; mid (m = 16) filter 6.05 at 2, 7.01 at 3 (with register spills).
__host__ __device__ constexpr int lm_prefetch_depth(int MW, int TQ) {
  return TQ > 0 && MW < 8 ? 16 / MW : 2;
}

template <int MW, int DS, int G, int TQ, int LT>
__global__ void __launch_bounds__(kLmWarps * 32, 1) ivfpq_scan_lm_kernel(const LmParams p) {
  static_assert(TQ == 0 || G == 1, "the bound pass takes one query per item");
  static_assert(LT == IVFPQ_LUT_FP32 || LT == IVFPQ_LUT_FP16 || LT == IVFPQ_LUT_FP8,
                "fp32, binary16 or E4M3 tables");
  static_assert(G <= kLmMaxG, "record head");
  constexpr bool H = LT == IVFPQ_LUT_FP16;
  constexpr bool Q8 = LT == IVFPQ_LUT_FP8;
  constexpr int QPS = Q8 ? 4 : H ? 2 : 1;     // queries per table set (entries per word)
  constexpr int NS = (G + QPS - 1) / QPS;      // table sets
  using Sh = Scan2Shape<MW, DS>;
  constexpr int NW = kLmWarps;
  constexpr int m = Sh::M;
  constexpr int GS = Sh::GS;
  constexpr int QQ = 32 / GS;
  constexpr int STEPS = 256 / (NW * QQ);
  constexpr int REPS = 32 / GS;
  static_assert(kScan2Warps == NW, "codeword ownership as in scan2.cuh");
  extern __shared__ __align__(16) uint32_t lm_smem[];
  float* tab = reinterpret_cast<float*>(lm_smem);  // NS x [256][64] 4-byte words
  uint8_t* slots = reinterpret_cast<uint8_t*>(lm_smem + NS * kGroupWords);
  auto head = [&](int slot) -> const LmHead& {
    return *reinterpret_cast<const LmHead*>(slots + slot * p.rec_bytes);
  };
  auto resid = [&](int slot) {
    return reinterpret_cast<const float*>(slots + slot * p.rec_bytes + kLmHead);
  };
  const ScanParams& sp = p.s;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int jj = lane & (GS - 1), qq = lane / GS;
  const int nit = p.units ? *p.n_units : *p.n_items;
  int j = blockIdx.x;
  if (j >= nit) return;  // the same for the whole block
  const int B = gridDim.x;

  // this thread's codewords (as scan2.cuh)
  float cw[STEPS][DS];
#pragma unroll
  for (int s = 0; s < STEPS; ++s) {
    const int e = (s * NW + warp) * QQ + qq;
    const float* c = sp.codebooks_t + (int64_t(e) * m + jj) * Sh::DS4;
#pragma unroll
    for (int t = 0; t < DS; ++t) cw[s][t] = __ldg(c + t);
  }
  uint32_t lcol[MW];
#pragma unroll
  for (int a = 0; a < MW; ++a) lcol[a] = lm_lane_columns<GS>(lane, a);

  // record of item it into slot: asynchronous copies by warp 0, completed
  // before the barrier that ends the iteration
  // where item it is (warp 0): its unit, its place in `order`, or it; read
  // a step before the fetch that needs it, so the load does not stall warp 0
  auto locate = [&](int it) {
    if (warp != 0 || it >= nit) return 0;
    return p.units ? p.units[it] : p.order ? p.order[it] : it;
  };
  // copies item it's record (record `at`, or chunk at % kLmMaxChunks of
  // record at / kLmMaxChunks) into slot; returns the chunk, -1 if none
  auto fetch = [&](int it, int slot, int at) {
    if (warp != 0 || it >= nit) return -1;
    int r = at, c = -1;
    if (p.units) {
      r = at / kLmMaxChunks;
      c = at % kLmMaxChunks;
      if (!dcheck(sp.dbg, r >= 0 && r < *p.n_items, 11)) r = 0;
    }
    const uint8_t* src = p.records + int64_t(r) * p.rec_bytes;
    uint8_t* dst = slots + slot * p.rec_bytes;
    for (int q = lane; q < p.rec_bytes / 16; q += 32) lm_cp_async16(dst + 16 * q, src + 16 * q);
    asm volatile("cp.async.commit_group;" ::: "memory");
    return c;
  };
  auto fetch_wait = [&]() {
    if (warp == 0) asm volatile("cp.async.wait_all;" ::: "memory");
  };
  // after fetch_wait: narrows the record in slot to chunk c of its list
  // (warp 0, before the barrier that publishes the slot)
  auto set_chunk = [&](int slot, int c) {
    if (warp != 0 || c < 0) return;  // the same for the whole warp
    __syncwarp();
    if (lane == 0) {
      LmHead& h = *reinterpret_cast<LmHead*>(slots + slot * p.rec_bytes);
      h.boff += int64_t(c) * (p.unit_len / 32);
      h.len = max(0, min(p.unit_len, h.len - c * p.unit_len));
    }
  };

  // tables of the queries of the item in `slot` into half P
  auto entry = [&](const float (&r)[DS], int s) {
    float Tv = 0.f;
#pragma unroll
    for (int t = 0; t < DS; ++t) {
      const float df = r[t] - cw[s][t];
      Tv = fmaf(df, df, Tv);
    }
    return Tv;
  };
  auto build = [&](int slot, int P) {
    const LmHead& d = head(slot);
    const int nq = d.nq;
    const float* rs = resid(slot);
    if constexpr (Q8) {
      // E4M3: one scale per query's table, s = max T / 448 (the largest
      // finite E4M3 value), entries E4M3(T * 448 / max T) (round to nearest
      // even, saturating). The block-wide maximum first: each warp's maximum
      // of its entries, then the entries again, quantized.
      float* wmax = reinterpret_cast<float*>(slots + kLmSlots * p.rec_bytes);  // [NW][kLmMaxG]
#pragma unroll
      for (int q = 0; q < G; ++q) {
        if (q >= nq) break;
        float r[DS];
#pragma unroll
        for (int t = 0; t < DS; ++t) r[t] = rs[q * p.dpad + jj * DS + t];
        float mx = 0.f;
#pragma unroll
        for (int s = 0; s < STEPS; ++s) mx = fmaxf(mx, entry(r, s));
#pragma unroll
        for (int o = 16; o >= 1; o /= 2) mx = fmaxf(mx, __shfl_xor_sync(kFullMask, mx, o));
        if (lane == 0) wmax[warp * kLmMaxG + q] = mx;
      }
      __syncthreads();
      LmHead* hw = reinterpret_cast<LmHead*>(slots + slot * p.rec_bytes);
#pragma unroll
      for (int g = 0; g < NS; ++g) {
        if (4 * g >= nq) break;
        uint32_t word[STEPS];
#pragma unroll
        for (int s = 0; s < STEPS; ++s) word[s] = 0u;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int q = 4 * g + i;
          if (q < nq) {
            float tmax = 0.f;
#pragma unroll
            for (int w = 0; w < NW; ++w) tmax = fmaxf(tmax, wmax[w * kLmMaxG + q]);
            const float inv = tmax > 0.f ? 448.f / tmax : 1.f;
            if (tid == 0) hw->scale[q] = tmax > 0.f ? tmax / 448.f : 1.f;
            float r[DS];
#pragma unroll
            for (int t = 0; t < DS; ++t) r[t] = rs[q * p.dpad + jj * DS + t];
#pragma unroll
            for (int s = 0; s < STEPS; ++s)
              word[s] |= uint32_t(__nv_cvt_float_to_fp8(entry(r, s) * inv, __NV_SATFINITE,
                                                        __NV_E4M3))
                         << (8 * i);
          } else {
            // a missing query of the set: entries 448 and, in the scan, bound 0
            if (tid == 0 && q < kLmMaxG) hw->scale[q] = 1.f;
#pragma unroll
            for (int s = 0; s < STEPS; ++s) word[s] |= 0x7Eu << (8 * i);
          }
        }
        uint32_t* tg = reinterpret_cast<uint32_t*>(tab) + g * kGroupWords + 32 * P + jj;
#pragma unroll
        for (int s = 0; s < STEPS; ++s) {
          const int e = (s * NW + warp) * QQ + qq;
          uint32_t* row = tg + e * 64;
          if (dcheck(sp.dbg, e >= 0 && e < 256, 7)) {
#pragma unroll
            for (int rep = 0; rep < REPS; ++rep) row[GS * ((rep + qq) & (REPS - 1))] = word[s];
          }
        }
      }
      return;
    }
#pragma unroll
    for (int g = 0; g < NS; ++g) {
      if ((H ? 2 * g : g) >= nq) break;
      float r[DS], r2[DS];
#pragma unroll
      for (int t = 0; t < DS; ++t) r[t] = rs[(H ? 2 * g : g) * p.dpad + jj * DS + t];
      const bool two = H && 2 * g + 1 < nq;
      if constexpr (H) {
#pragma unroll
        for (int t = 0; t < DS; ++t) r2[t] = two ? rs[(2 * g + 1) * p.dpad + jj * DS + t] : 0.f;
      }
      uint32_t* tg = reinterpret_cast<uint32_t*>(tab) + g * kGroupWords + 32 * P + jj;
#pragma unroll
      for (int s = 0; s < STEPS; ++s) {
        const int e = (s * NW + warp) * QQ + qq;
        uint32_t word;
        if constexpr (H) {
          // a missing second query gets +inf entries: its sums never pass
          const float T0 = entry(r, s);
          const float T1 = two ? entry(r2, s) : INFINITY;
          word = uint32_t(__half_as_ushort(__float2half_rn(T0))) |
                 (uint32_t(__half_as_ushort(__float2half_rn(T1))) << 16);
        } else {
          word = __float_as_uint(entry(r, s));
        }
        uint32_t* row = tg + e * 64;
        if (dcheck(sp.dbg, e >= 0 && e < 256, 7)) {
#pragma unroll
          for (int rep = 0; rep < REPS; ++rep) row[GS * ((rep + qq) & (REPS - 1))] = word;
        }
      }
    }
  };

  // code blocks in flight per warp: PD = 2 is a double buffer (block b is
  // scored while b + NW loads, then copied over); PD > 2 a ring of PD blocks
  // (b, b + NW, ..., b + (PD-1) NW) whose slot is refilled with the block PD NW
  // further on as soon as its look-ups have read it, so PD - 1 loads overlap
  // each block's scoring (with short codes and few look-ups per code, one
  // load in flight does not cover the memory latency); the ring's unrolled
  // loop spills where the double buffer does not (m = 32)
  constexpr int PD = lm_prefetch_depth(MW, TQ);
  constexpr int PF = PD == 2 ? 1 : PD;  // blocks loaded before the scan
  uint32_t cr[PD][MW];
  auto first_codes = [&](int slot) {
    const LmHead& d = head(slot);
    const int nb = (d.len + 31) >> 5;
    const bool in_range = d.boff >= 0 && d.boff + nb <= sp.nblocks;  // checked in scan
#pragma unroll
    for (int u = 0; u < PF; ++u)
      if (warp + u * NW < nb && in_range)
        load_codes<MW>(sp.codes + (d.boff + warp + u * NW) * 32 * m, lane, cr[u]);
  };
  // the item's codes into L2 (its list, or the chunk of it)
  auto prefetch = [&](int slot) {
    const LmHead& d = head(slot);
    const int64_t nb = (int64_t(d.len) + 31) >> 5;
    if (nb > 0 && d.boff >= 0 && d.boff + nb <= sp.nblocks)
      prefetch_l2(sp.codes + d.boff * 32 * m, nb * 32 * m);
  };

  // bound pass: this lane's TQ smallest of the current item, ascending
  uint32_t tq[TQ ? TQ : 1];
#pragma unroll
  for (int i = 0; i < (TQ ? TQ : 1); ++i) tq[i] = kSentinelKey;

  // scan of the item in `slot` (its descriptor read into registers) from half P
  const char* tab_bytes = reinterpret_cast<const char*>(tab);
  auto scan = [&](int slot, auto Pc, auto GGc) {
    constexpr int P = decltype(Pc)::value;
    constexpr int GG = decltype(GGc)::value;
    const LmHead& d = head(slot);
    const int len = d.len;
    const int64_t boff = d.boff;
    const int nqi = d.nq;
    int qv[GG];
    uint32_t th[GG];
    float sc[GG];
#pragma unroll
    for (int g = 0; g < GG; ++g) {
      // fp32 items are scanned with exactly their query count (GG = nqi);
      // binary16 / E4M3 ones in whole sets of 2 / 4, so the last set may be
      // short: a missing query has +inf / 448 table entries and bound 0, so
      // nothing passes
      const bool live = QPS == 1 || g < nqi;
      qv[g] = live ? d.q[g] : d.q[0];
      th[g] = live ? d.theta[g] : 0u;
      sc[g] = Q8 ? d.scale[g] : 1.f;
    }
    const bool in_range =
        dcheck(sp.dbg, boff >= 0 && boff + ((len + 31) >> 5) <= sp.nblocks, 4);
    const int nb = in_range ? (len + 31) >> 5 : 0;
    const uint8_t* lcodes = sp.codes + boff * 32 * m;
    // partial sums of a code block from its code words w
    auto score = [&](const uint32_t (&w)[MW]) {
      LmAcc<QPS * ((GG + QPS - 1) / QPS)> acc;
#pragma unroll
      for (auto& a : acc.v) a[0] = a[1] = a[2] = a[3] = 0.f;
      if constexpr (Q8) lm_lookups_q8<MW, (GG + 3) / 4, (GG > 4 ? 2 : 4), P>(w, tab_bytes, lcol, acc.v);
      else if constexpr (H) lm_lookups_h<MW, (GG + 1) / 2, (GG > 4 ? 2 : 4), P>(w, tab_bytes, lcol, acc.v);
      else lm_lookups<MW, GG, P>(w, tab_bytes, lcol, acc.v);
      return acc;
    };
    auto select = [&](const auto& acc, int b) {
      const bool valid = b * 32 + lane < len;
      const uint32_t slot_id = uint32_t((boff + b) * 32 + lane);
#pragma unroll
      for (int g = 0; g < GG; ++g) {
        float dist = (acc.v[g][0] + acc.v[g][1]) + (acc.v[g][2] + acc.v[g][3]);
        if constexpr (Q8) dist *= sc[g];
        if constexpr (TQ > 0) {
          const uint32_t key = valid ? __float_as_uint(dist) : kSentinelKey;
          if (key < tq[TQ - 1]) {
            tq[TQ - 1] = key;
#pragma unroll
            for (int i = TQ - 1; i > 0; --i) {
              const uint32_t lo = tq[i - 1], hi = tq[i];
              tq[i - 1] = min(lo, hi);
              tq[i] = max(lo, hi);
            }
          }
        } else {
          lm_append(p, qv[g], valid && __float_as_uint(dist) <= th[g], dist, slot_id, lane);
        }
      }
    };
    if constexpr (PD == 2) {
      for (int b = warp; b < nb; b += NW) {
        if (b + NW < nb) load_codes<MW>(lcodes + int64_t(b + NW) * 32 * m, lane, cr[1]);
        select(score(cr[0]), b);
#pragma unroll
        for (int w = 0; w < MW; ++w) cr[0][w] = cr[1][w];
      }
    } else {
      for (int b0 = warp; b0 < nb; b0 += PD * NW) {
#pragma unroll
        for (int u = 0; u < PD; ++u) {
          const int b = b0 + u * NW;
          if (b >= nb) break;  // the same for the whole warp
          const auto acc = score(cr[u]);
          if (b + PD * NW < nb) load_codes<MW>(lcodes + int64_t(b + PD * NW) * 32 * m, lane, cr[u]);
          select(acc, b);
        }
      }
    }
    if constexpr (TQ > 0) {
      uint32_t* o = p.part_key + ((int64_t(d.item) * NW + warp) * 32 + lane) * TQ;
#pragma unroll
      for (int i = 0; i < TQ; ++i) {
        o[i] = tq[i];
        tq[i] = kSentinelKey;
      }
    }
  };

  const int c0 = fetch(j, 0, locate(j));
  const int c1 = fetch(j + B, 1, locate(j + B));
  int at_next = locate(j + 2 * B);
  fetch_wait();
  set_chunk(0, c0);
  set_chunk(1, c1);
  __syncthreads();
  build(0, 0);
  first_codes(0);
  if (tid == 0 && j + B < nit) prefetch(1);
  __syncthreads();

  int t = 0;
  auto step = [&](auto Pc) {
    constexpr int P = decltype(Pc)::value;
    const int cur = t % kLmSlots, nxt = (t + 1) % kLmSlots, fil = (t + 2) % kLmSlots;
    const bool more = j + B < nit;
    const int cf = fetch(j + 2 * B, fil, at_next);
    at_next = locate(j + 3 * B);
    if (more) build(nxt, 1 - P);
    const int nqc = head(cur).nq;
    if (TQ > 0 || nqc >= G) {
      scan(cur, Pc, std::integral_constant<int, G>{});
    } else if constexpr (Q8) {
      // E4M3: whole table sets (quadruples of queries)
      if constexpr (G > 4) {
        if (nqc > 4) scan(cur, Pc, std::integral_constant<int, 8>{});
        else scan(cur, Pc, std::integral_constant<int, 4>{});
      } else {
        scan(cur, Pc, std::integral_constant<int, 4>{});
      }
    } else if constexpr (H) {
      // binary16: whole table sets (pairs of queries)
      if constexpr (G > 4) {
        if (nqc > 4) scan(cur, Pc, std::integral_constant<int, 6>{});
        else if (nqc > 2) scan(cur, Pc, std::integral_constant<int, 4>{});
        else scan(cur, Pc, std::integral_constant<int, 2>{});
      } else if constexpr (G > 2) {
        if (nqc > 2) scan(cur, Pc, std::integral_constant<int, 4>{});
        else scan(cur, Pc, std::integral_constant<int, 2>{});
      } else {
        scan(cur, Pc, std::integral_constant<int, 2>{});
      }
    } else {
      if constexpr (G > 2) {
        if (nqc == 2) scan(cur, Pc, std::integral_constant<int, 2>{});
        else scan(cur, Pc, std::integral_constant<int, 1>{});
      } else {
        scan(cur, Pc, std::integral_constant<int, 1>{});
      }
    }
    if (more) first_codes(nxt);
    fetch_wait();
    set_chunk(fil, cf);
    __syncthreads();  // half P may be rebuilt next; slot fil is complete
    if (tid == 0 && j + 2 * B < nit) prefetch(fil);
    j += B;
    ++t;
  };
  while (j < nit) {
    step(std::integral_constant<int, 0>{});
    if (j < nit) step(std::integral_constant<int, 1>{});
  }
}

inline size_t scan_lm_smem_bytes(int sets, int rec_bytes) {
  return size_t(sets) * kGroupWords * 4 + size_t(kLmSlots) * rec_bytes;
}

template <int MW, int DS, int G, int TQ, int LT>
int launch_scan_lm(const LmParams& p, cudaStream_t s) {
  auto kern = ivfpq_scan_lm_kernel<MW, DS, G, TQ, LT>;
  const int qps = LT == IVFPQ_LUT_FP8 ? 4 : LT == IVFPQ_LUT_FP16 ? 2 : 1;
  const int sets = (G + qps - 1) / qps;
  // E4M3 tables: the warps' table maxima follow the item records
  const size_t smem = scan_lm_smem_bytes(sets, p.rec_bytes) +
                      (LT == IVFPQ_LUT_FP8 ? size_t(kLmWarps) * kLmMaxG * 4 : 0);
  IVFPQ_TRY(set_dynamic_smem(kern, smem));
  kern<<<unsigned(num_sms()), kLmWarps * 32, smem, s>>>(p);
  IVFPQ_LAUNCHED_K(kern, smem, kLmWarps * 32);
  return IVFPQ_OK;
}

}  // namespace ivfpq

#define IVFPQ_INST_SCAN_LM(MW, DS, G, TQ, LT) \
  template int ivfpq::launch_scan_lm<MW, DS, G, TQ, LT>(const ivfpq::LmParams&, cudaStream_t);
