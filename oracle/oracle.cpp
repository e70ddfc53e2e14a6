// Plain, slow CPU oracle for batched IVF-PQ search, exact flat k-NN and
// row-wise k-selection.
//
// TEST INFRASTRUCTURE ONLY. Nothing in the product library may include, link,
// load or call this file. Only the tests, the package smoke check and the CPU
// baseline leg of the benchmark use it. It shares no code with the CUDA path.
//
// Arithmetic is IEEE double unless a function says otherwise. Every ordering is
// lexicographic on (value, index), so results are deterministic and do not
// depend on the thread count.
//
// Sources (all from the pages on billion-scale similarity search):
//  * "Billion-scale similarity search with GPUs" (Johnson, Douze, Jegou):
//      - IVFADC lookup tables and the cost of the list scan (section 5, the
//        paragraphs after Eq. (10)): tables T_1..T_b of 256 entries, a distance
//        is b look-ups and additions.
//      - odd-size merging network (Algorithm 1, Figure 1), odd-size sort
//        (Algorithm 2), WarpSelect (Algorithm 3, Figure 2, three invariants).
//  * "Custom 8-bit floating point value format for reducing shared memory bank
//    conflict in approximate nearest neighbor search" (Ootomo):
//      - IVFPQ build steps 1-4 and search steps 1-5, Eq. (1): R = sum_j F(y_j).
//  * "Faiss GPU: k-select that never leaves registers" (reading guide):
//      - the coarse quantizer is a brute-force nearest-centroid search (Step 5).

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <thread>
#include <utility>
#include <vector>

namespace {

const double kInf = std::numeric_limits<double>::infinity();

// Run f(begin, end) over [0, n) split into contiguous chunks, one per thread.
// Each output element is written by exactly one chunk, so results do not
// depend on the number of threads.
template <class F>
void parallel_for(int64_t n, int nthreads, F f) {
  if (nthreads <= 1 || n <= 1) {
    f(int64_t(0), n);
    return;
  }
  int64_t nt = std::min<int64_t>(nthreads, n);
  std::vector<std::thread> pool;
  int64_t per = (n + nt - 1) / nt;
  for (int64_t t = 0; t < nt; ++t) {
    int64_t b = t * per, e = std::min(n, b + per);
    if (b >= e) break;
    pool.emplace_back([=]() { f(b, e); });
  }
  for (auto& th : pool) th.join();
}

struct Cand {
  double d;
  int64_t id;
};
inline bool cand_less(const Cand& a, const Cand& b) {
  return a.d < b.d || (a.d == b.d && a.id < b.id);
}

// Squared L2 distance written out as its definition: sum_t (a_t - b_t)^2.
inline double sq_l2(const float* a, const float* b, int d) {
  double s = 0.0;
  for (int t = 0; t < d; ++t) {
    double diff = double(a[t]) - double(b[t]);
    s += diff * diff;
  }
  return s;
}

// Coarse quantizer for one query: exact distances to every centroid, full sort
// by (distance, list id), first nprobe kept.
void coarse_one(const float* q, int d, const float* cent, int64_t nlist,
                int nprobe, int32_t* out_list, double* out_dist) {
  std::vector<Cand> all(nlist);
  for (int64_t c = 0; c < nlist; ++c) all[c] = {sq_l2(q, cent + c * d, d), c};
  std::sort(all.begin(), all.end(), cand_less);
  for (int p = 0; p < nprobe; ++p) {
    out_list[p] = int32_t(all[p].id);
    if (out_dist) out_dist[p] = all[p].d;
  }
}

// ADC lookup table for one query residual r (length d): for sub-quantizer j
// and reproduction value e, T[j][e] is the squared distance between the j-th
// sub-vector of r (dims [j*dsub, (j+1)*dsub)) and codeword e of sub-quantizer j.
// Codebook layout: cb[(j*256 + e)*dsub + t].
void lut_one(const double* r, int d, const float* cb, int m, double* T) {
  int dsub = d / m;
  for (int j = 0; j < m; ++j) {
    const double* rj = r + j * dsub;
    for (int e = 0; e < 256; ++e) {
      const float* c = cb + (int64_t(j) * 256 + e) * dsub;
      double s = 0.0;
      for (int t = 0; t < dsub; ++t) {
        double diff = rj[t] - double(c[t]);
        s += diff * diff;
      }
      T[j * 256 + e] = s;
    }
  }
}

// --- IEEE binary16, written from the format's definition -------------------
// 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits; subnormals have
// exponent field 0 and value 2^-14 * f/1024. Rounding is to nearest, ties to
// even; magnitudes that round above the largest finite value become infinity.
uint16_t f16_encode(double x) {
  uint16_t sign = std::signbit(x) ? 0x8000 : 0;
  double a = std::fabs(x);
  if (std::isnan(x)) return 0x7E00;
  if (std::isinf(a)) return sign | 0x7C00;
  if (a == 0.0) return sign;
  int e;
  double fr = std::frexp(a, &e);  // a = fr * 2^e, fr in [0.5, 1)
  int exp_unbiased = e - 1;       // a = (2*fr) * 2^(e-1), 2*fr in [1, 2)
  double scaled;
  int biased;
  if (exp_unbiased < -14) {  // subnormal range: units of 2^-24
    scaled = a * std::ldexp(1.0, 24);
    biased = 0;
  } else {
    scaled = (2.0 * fr - 1.0) * 1024.0;  // fraction in units of 2^-10
    biased = exp_unbiased + 15;
  }
  double fl = std::floor(scaled);
  double rem = scaled - fl;
  uint32_t q = uint32_t(fl);
  if (rem > 0.5 || (rem == 0.5 && (q & 1u))) q += 1;
  uint32_t bits;
  if (biased == 0) {
    bits = q;  // q == 1024 carries into the smallest normal, which is correct
  } else {
    bits = (uint32_t(biased) << 10) + q;  // fraction overflow carries into exp
  }
  if (bits >= 0x7C00) return sign | 0x7C00;
  return uint16_t(sign | bits);
}

double f16_decode(uint16_t h) {
  int s = (h >> 15) & 1, ex = (h >> 10) & 0x1F, fr = h & 0x3FF;
  double v;
  if (ex == 0)
    v = std::ldexp(double(fr), -24);
  else if (ex == 31)
    v = fr ? std::numeric_limits<double>::quiet_NaN() : kInf;
  else
    v = std::ldexp(1.0 + fr / 1024.0, ex - 15);
  return s ? -v : v;
}

// --- 8-bit float, 1 sign / 4 exponent / 3 mantissa bits (E4M3) -------------
// Bias 7; exponent field 0 is subnormal (2^-6 * m/8); the pattern with all
// exponent and mantissa bits set is NaN, so the largest finite magnitude is
// 2^8 * 1.75 = 448 and there is no infinity. Encoding rounds to nearest, ties
// to even, and saturates finite overflow to +-448.
double e4m3_decode(uint8_t b) {
  int s = (b >> 7) & 1, ex = (b >> 3) & 0xF, fr = b & 0x7;
  double v;
  if (ex == 0xF && fr == 0x7)
    v = std::numeric_limits<double>::quiet_NaN();
  else if (ex == 0)
    v = std::ldexp(double(fr), -9);
  else
    v = std::ldexp(1.0 + fr / 8.0, ex - 7);
  return s ? -v : v;
}

uint8_t e4m3_encode(double x) {
  if (std::isnan(x)) return 0x7F;
  uint8_t sign = std::signbit(x) ? 0x80 : 0;
  double a = std::fabs(x);
  // Candidates are the 127 non-negative finite codes, in increasing order of
  // value (codes 0x00..0x7E are monotone in value). Pick the nearest; on a tie
  // pick the one with an even mantissa (the even code).
  if (a >= 448.0) return sign | 0x7E;
  int lo = 0, hi = 0x7E;
  while (lo < hi) {  // first code with value >= a
    int mid = (lo + hi) / 2;
    if (e4m3_decode(uint8_t(mid)) >= a)
      hi = mid;
    else
      lo = mid + 1;
  }
  int up = lo;
  if (e4m3_decode(uint8_t(up)) == a || up == 0) return uint8_t(sign | up);
  int dn = up - 1;
  double dup = e4m3_decode(uint8_t(up)) - a, ddn = a - e4m3_decode(uint8_t(dn));
  int pick;
  if (ddn < dup)
    pick = dn;
  else if (dup < ddn)
    pick = up;
  else
    pick = (dn & 1) ? up : dn;
  return uint8_t(sign | pick);
}

// Reduced-precision table variants. lut_type 0 keeps the exact table.
// lut_type 1: each entry rounded to binary16 (nearest, ties to even).
// lut_type 2: one scale per table set s = max_{j,e} T / 448; each entry is
// stored as e4m3(T / s) and read back as s * decode(code).
void quantize_lut(double* T, int m, int lut_type) {
  int n = m * 256;
  if (lut_type == 1) {
    for (int i = 0; i < n; ++i) T[i] = f16_decode(f16_encode(T[i]));
  } else if (lut_type == 2) {
    double mx = 0.0;
    for (int i = 0; i < n; ++i) mx = std::max(mx, T[i]);
    if (mx <= 0.0) return;
    double s = mx / 448.0;
    for (int i = 0; i < n; ++i) T[i] = s * e4m3_decode(e4m3_encode(T[i] / s));
  }
}

// --- sorting networks -----------------------------------------------------
// Comparator (lo, hi, step): after it, position lo holds the smaller value.
struct Comp {
  int lo, hi, step;
};

int ceil_log2(int x) {
  int l = 0;
  while ((1 << l) < x) ++l;
  return l;
}

// Odd-size merge of a sorted left array (positions base .. base+lL-1) with a
// sorted right array (positions base+lL .. base+lL+lR-1). Both are padded to
// N = 2^ceil(log2(max(lL, lR))) with dummies: the left array at its start, the
// right array at its end. The network is a bitonic merge of the 2N padded
// positions whose first stage is reversed (mirror comparisons), followed by
// half-cleaners of stride N/2 .. 1 inside each half; comparisons that touch a
// dummy are elided. Returns the number of parallel steps used (step0 is the
// index of the first step).
int odd_merge(int base, int lL, int lR, int step0, std::vector<Comp>* out) {
  if (lL == 0 || lR == 0) return 0;
  int N = 1 << ceil_log2(std::max(lL, lR));
  int padL = N - lL;
  // padded position p in [0, 2N) -> real position, or -1 for a dummy
  auto real = [&](int p) -> int {
    if (p < N) return p < padL ? -1 : base + (p - padL);
    int r = p - N;
    return r < lR ? base + lL + r : -1;
  };
  int step = step0;
  for (int i = 0; i < N; ++i) {
    int a = real(i), b = real(2 * N - 1 - i);
    if (a >= 0 && b >= 0) out->push_back({a, b, step});
  }
  ++step;
  for (int s = N / 2; s >= 1; s /= 2) {
    for (int half = 0; half < 2; ++half) {
      for (int i = 0; i < N; ++i) {
        if (i & s) continue;
        int a = real(half * N + i), b = real(half * N + i + s);
        if (a >= 0 && b >= 0) out->push_back({a, b, step});
      }
    }
    ++step;
  }
  return step - step0;
}

// Odd-size sort: sort the left ceil(l/2) and right floor(l/2) elements in
// parallel, then merge them with the odd-size merge.
int odd_sort(int base, int l, int step0, std::vector<Comp>* out) {
  if (l <= 1) return 0;
  int lL = (l + 1) / 2, lR = l / 2;
  int sL = odd_sort(base, lL, step0, out);
  int sR = odd_sort(base + lL, lR, step0, out);
  int s = std::max(sL, sR);
  return s + odd_merge(base, lL, lR, step0 + s, out);
}

template <class K>
void apply_network(const std::vector<Comp>& net, K* v) {
  for (const Comp& c : net)
    if (v[c.hi] < v[c.lo]) std::swap(v[c.lo], v[c.hi]);
}

// Lexicographic (value, index) key used by the WarpSelect simulation.
struct Key {
  double v;
  int64_t i;
  bool operator<(const Key& o) const { return v < o.v || (v == o.v && i < o.i); }
  bool operator==(const Key& o) const { return v == o.v && i == o.i; }
};

}  // namespace

extern "C" {

// ===== coarse quantizer ======================================================
// Exact squared L2 distance of each query to every centroid, full sort by
// (distance, list id); the first nprobe list ids and distances are returned.
// q: nq*d, cent: nlist*d (row-major fp32); out_list: nq*nprobe; out_dist may be
// null. Returns 0, or -1 on invalid arguments.
int oracle_coarse(const float* q, int64_t nq, int d, const float* cent,
                  int64_t nlist, int nprobe, int32_t* out_list,
                  double* out_dist, int nthreads) {
  if (nq < 0 || d <= 0 || nlist <= 0 || nprobe <= 0 || nprobe > nlist)
    return -1;
  parallel_for(nq, nthreads, [&](int64_t b, int64_t e) {
    for (int64_t i = b; i < e; ++i)
      coarse_one(q + i * d, d, cent, nlist, nprobe, out_list + i * nprobe,
                 out_dist ? out_dist + i * nprobe : nullptr);
  });
  return 0;
}

// ===== lookup table and ADC =================================================
// T (m*256 doubles, [j][e]) for one residual r (d doubles).
void oracle_lut(const double* r, int d, const float* cb, int m, double* T) {
  lut_one(r, d, cb, m, T);
}

// Apply a reduced-precision table variant in place (0 fp32/exact, 1 binary16,
// 2 E4M3 with one scale per table set).
void oracle_quantize_lut(double* T, int m, int lut_type) {
  quantize_lut(T, m, lut_type);
}

// R = sum over sub-quantizers j (in order 0..m-1) of T[j][code[j]].
double oracle_adc(const double* T, int m, const uint8_t* code) {
  double s = 0.0;
  for (int j = 0; j < m; ++j) s += T[j * 256 + code[j]];
  return s;
}

uint16_t oracle_f16_encode(double x) { return f16_encode(x); }
double oracle_f16_decode(uint16_t h) { return f16_decode(h); }
uint8_t oracle_e4m3_encode(double x) { return e4m3_encode(x); }
double oracle_e4m3_decode(uint8_t b) { return e4m3_decode(b); }

// ===== IVF-PQ search =========================================================
// Inverted lists in compressed form: list l holds vectors
// [list_off[l], list_off[l+1]); their m-byte codes are stored as sequential
// groups of m bytes (codes[v*m + j]) and their user ids in ids[v].
// For each query: probes = forced_probes row (if given) or the nprobe nearest
// centroids (oracle_coarse); for each probe l, r = q - c_l, the table T is
// built (oracle_lut) and optionally reduced (lut_type); each vector of list l
// gets distance sum_j T[j][code_j]; all candidates of all probes are pooled and
// the k smallest by (distance, id) are written in ascending order. Missing
// results are (+inf, -1). out_probes (nq*nprobe, may be null) receives the
// probes used.
int oracle_ivfpq_search(const float* q, int64_t nq, int d, const float* cent,
                        int64_t nlist, const float* cb, int m,
                        const int64_t* list_off, const uint8_t* codes,
                        const int64_t* ids, int nprobe, int k, int lut_type,
                        const int32_t* forced_probes, double* out_dist,
                        int64_t* out_ids, int32_t* out_probes, int nthreads) {
  if (nq < 0 || d <= 0 || m <= 0 || d % m || nlist <= 0 || nprobe <= 0 ||
      nprobe > nlist || k <= 0 || lut_type < 0 || lut_type > 2)
    return -1;
  parallel_for(nq, nthreads, [&](int64_t b, int64_t e) {
    std::vector<int32_t> probes(nprobe);
    std::vector<double> r(d), T(size_t(m) * 256);
    std::vector<Cand> cand;
    for (int64_t qi = b; qi < e; ++qi) {
      const float* x = q + qi * d;
      if (forced_probes)
        std::copy(forced_probes + qi * nprobe,
                  forced_probes + (qi + 1) * nprobe, probes.begin());
      else
        coarse_one(x, d, cent, nlist, nprobe, probes.data(), nullptr);
      if (out_probes)
        std::copy(probes.begin(), probes.end(), out_probes + qi * nprobe);
      cand.clear();
      for (int p = 0; p < nprobe; ++p) {
        int64_t l = probes[p];
        for (int t = 0; t < d; ++t)
          r[t] = double(x[t]) - double(cent[l * d + t]);
        lut_one(r.data(), d, cb, m, T.data());
        quantize_lut(T.data(), m, lut_type);
        for (int64_t v = list_off[l]; v < list_off[l + 1]; ++v) {
          const uint8_t* c = codes + v * m;
          double s = 0.0;
          for (int j = 0; j < m; ++j) s += T[j * 256 + c[j]];
          cand.push_back({s, ids[v]});
        }
      }
      int64_t kk = std::min<int64_t>(k, int64_t(cand.size()));
      std::partial_sort(cand.begin(), cand.begin() + kk, cand.end(), cand_less);
      for (int i = 0; i < k; ++i) {
        out_dist[qi * k + i] = i < kk ? cand[i].d : kInf;
        out_ids[qi * k + i] = i < kk ? cand[i].id : -1;
      }
    }
  });
  return 0;
}

// ===== exact flat k-NN ========================================================
// For every (query, database row): sum_t (q_t - y_t)^2 written out directly;
// the k smallest by (distance, row index), ascending; missing -> (+inf, -1).
int oracle_flat_knn(const float* db, int64_t n, int d, const float* q,
                    int64_t nq, int k, double* out_dist, int64_t* out_ids,
                    int nthreads) {
  if (n < 0 || nq < 0 || d <= 0 || k <= 0) return -1;
  parallel_for(nq, nthreads, [&](int64_t b, int64_t e) {
    std::vector<Cand> cand(n);
    for (int64_t qi = b; qi < e; ++qi) {
      for (int64_t i = 0; i < n; ++i)
        cand[i] = {sq_l2(q + qi * d, db + i * d, d), i};
      int64_t kk = std::min<int64_t>(k, n);
      std::partial_sort(cand.begin(), cand.begin() + kk, cand.end(), cand_less);
      for (int i = 0; i < k; ++i) {
        out_dist[qi * k + i] = i < kk ? cand[i].d : kInf;
        out_ids[qi * k + i] = i < kk ? cand[i].id : -1;
      }
    }
  });
  return 0;
}

// ===== row-wise k-selection ===================================================
// The k smallest values of each row of vals (rows*cols fp32) with their column
// index, ordered by (value, column); rows shorter than k are padded with
// (+inf, -1). Values are copied, not recomputed, so out_vals is exact.
int oracle_kselect(const float* vals, int64_t rows, int64_t cols, int k,
                   float* out_vals, int64_t* out_idx, int nthreads) {
  if (rows < 0 || cols < 0 || k <= 0) return -1;
  parallel_for(rows, nthreads, [&](int64_t b, int64_t e) {
    std::vector<Cand> row(cols);
    for (int64_t r = b; r < e; ++r) {
      for (int64_t c = 0; c < cols; ++c) row[c] = {double(vals[r * cols + c]), c};
      int64_t kk = std::min<int64_t>(k, cols);
      std::partial_sort(row.begin(), row.begin() + kk, row.end(), cand_less);
      for (int i = 0; i < k; ++i) {
        out_vals[r * k + i] = i < kk ? float(row[i].d)
                                     : std::numeric_limits<float>::infinity();
        out_idx[r * k + i] = i < kk ? row[i].id : -1;
      }
    }
  });
  return 0;
}

// ===== sorting networks (Algorithms 1 and 2) ================================
// Writes up to cap comparators as (lo, hi, step) triples into out and the
// number of parallel steps into *nsteps. Returns the number of comparators, or
// -1 if cap is too small.
int oracle_odd_merge_network(int lL, int lR, int32_t* out, int cap,
                             int* nsteps) {
  std::vector<Comp> net;
  *nsteps = odd_merge(0, lL, lR, 0, &net);
  if (int(net.size()) > cap) return -1;
  for (size_t i = 0; i < net.size(); ++i) {
    out[3 * i] = net[i].lo;
    out[3 * i + 1] = net[i].hi;
    out[3 * i + 2] = net[i].step;
  }
  return int(net.size());
}

int oracle_odd_sort_network(int l, int32_t* out, int cap, int* nsteps) {
  std::vector<Comp> net;
  *nsteps = odd_sort(0, l, 0, &net);
  if (int(net.size()) > cap) return -1;
  for (size_t i = 0; i < net.size(); ++i) {
    out[3 * i] = net[i].lo;
    out[3 * i + 1] = net[i].hi;
    out[3 * i + 2] = net[i].step;
  }
  return int(net.size());
}

// ===== WarpSelect, simulated on the host (Algorithm 3) =======================
// 32 simulated lanes. Lane j takes a[32i + j]. Each lane keeps a thread queue
// of t keys ordered largest first (T_0 >= T_1 >= ...); the warp keeps a queue
// of K = k rounded up to a multiple of 32 keys, smallest first. All start at a
// +inf sentinel. A new key larger than the lane's T_0 is rejected; otherwise
// it replaces T_0 and is moved to its sorted place. After each group of 32 a
// vote checks whether any lane has T_0 < W_{K-1} (the second invariant
// broken); if so the thread queues (read as one unsorted lane-stride array of
// 32t keys) are sorted with the odd-size sort and merged with the warp queue
// by the odd-size merge: the K smallest become the warp queue, the next 32t
// go back to the thread queues. A final sort and merge follows the last
// element. Keys are (value, index) pairs compared lexicographically.
//
// After every group the three invariants are checked against the multiset of
// keys seen so far; the function returns 0 and the k smallest in
// out_vals/out_idx (ascending), 1..3 if invariant 1..3 failed, or -1 on bad
// arguments. *n_merges counts the merges triggered by the vote.
int oracle_warpselect_sim(const float* vals, int64_t n, int k, int t,
                          float* out_vals, int64_t* out_idx,
                          int64_t* n_merges) {
  if (k <= 0 || t <= 0 || n < 0) return -1;
  const int L = 32;
  const int K = (k + L - 1) / L * L;
  const Key sentinel{kInf, std::numeric_limits<int64_t>::max()};
  std::vector<std::vector<Key>> tq(L, std::vector<Key>(t, sentinel));
  std::vector<Key> wq(K, sentinel);
  std::vector<Comp> sort_net, merge_net;
  odd_sort(0, L * t, 0, &sort_net);
  odd_merge(0, K, L * t, 0, &merge_net);
  std::vector<Key> seen;
  int64_t merges = 0;

  auto merge = [&]() {
    // thread queues as a lane-stride array: element r*32 + j is register r of
    // lane j, where register r holds T_{t-1-r} (so each lane's registers are
    // ascending, as after a merge).
    std::vector<Key> all(K + L * t);
    for (int i = 0; i < K; ++i) all[i] = wq[i];
    for (int r = 0; r < t; ++r)
      for (int j = 0; j < L; ++j) all[K + r * L + j] = tq[j][t - 1 - r];
    apply_network(sort_net, all.data() + K);
    apply_network(merge_net, all.data());
    for (int i = 0; i < K; ++i) wq[i] = all[i];
    for (int r = 0; r < t; ++r)
      for (int j = 0; j < L; ++j) tq[j][t - 1 - r] = all[K + r * L + j];
  };

  auto check = [&]() -> int {
    std::vector<Key> s = seen;
    std::sort(s.begin(), s.end());
    size_t kk = std::min<size_t>(size_t(k), s.size());
    // invariant 1: no lane's T_0 is among the k smallest seen
    for (int j = 0; j < L; ++j)
      for (size_t i = 0; i < kk; ++i)
        if (tq[j][0] == s[i]) return 1;
    // invariant 2: every T_0 is greater than every warp queue key
    for (int j = 0; j < L; ++j)
      if (tq[j][0] < wq[K - 1]) return 2;
    // invariant 3: every key among the k smallest seen is held somewhere
    for (size_t i = 0; i < kk; ++i) {
      bool found = false;
      for (int w = 0; w < K && !found; ++w) found = wq[w] == s[i];
      for (int j = 0; j < L && !found; ++j)
        for (int r = 0; r < t && !found; ++r) found = tq[j][r] == s[i];
      if (!found) return 3;
    }
    return 0;
  };

  for (int64_t g = 0; g < n; g += L) {
    for (int j = 0; j < L && g + j < n; ++j) {
      Key a{double(vals[g + j]), g + j};
      seen.push_back(a);
      std::vector<Key>& T = tq[j];
      if (T[0] < a) continue;  // rejected: larger than T_0
      T[0] = a;
      for (int r = 0; r + 1 < t; ++r)
        if (T[r] < T[r + 1]) std::swap(T[r], T[r + 1]);
    }
    bool vote = false;
    for (int j = 0; j < L; ++j) vote = vote || tq[j][0] < wq[K - 1];
    if (vote) {
      merge();
      ++merges;
    }
    int bad = check();
    if (bad) return bad;
  }
  merge();
  if (n_merges) *n_merges = merges;
  for (int i = 0; i < k; ++i) {
    bool real = i < K && wq[i].v != kInf;
    out_vals[i] = real ? float(wq[i].v) : std::numeric_limits<float>::infinity();
    out_idx[i] = real ? wq[i].i : -1;
  }
  return 0;
}

// ===== index-building helpers (input preparation, not the search path) =======
// Product-quantizer training by Lloyd iterations, one sub-quantizer at a time
// on sub-vectors [j*dsub, (j+1)*dsub) of x (n*d residuals). Codewords start at
// the sub-vectors of rows init[0..255]. Each iteration assigns every point to
// its nearest codeword (ties to the lower index) and moves each codeword to the
// mean of its points; a codeword with no points keeps its position. obj
// (niter+1 entries, may be null) receives the total squared quantization error
// of each assignment pass, the last one after the final update.
int oracle_pq_train(const float* x, int64_t n, int d, int m, int niter,
                    const int64_t* init, float* cb_out, double* obj,
                    int nthreads) {
  if (n < 256 || d <= 0 || m <= 0 || d % m || niter < 0) return -1;
  int dsub = d / m;
  if (obj)
    for (int i = 0; i <= niter; ++i) obj[i] = 0.0;
  std::vector<int> assign(n);
  for (int j = 0; j < m; ++j) {
    std::vector<double> cw(256 * size_t(dsub));
    for (int e = 0; e < 256; ++e)
      for (int t = 0; t < dsub; ++t)
        cw[e * dsub + t] = x[init[e] * d + j * dsub + t];
    for (int it = 0; it <= niter; ++it) {
      std::vector<double> part(std::max(1, nthreads), 0.0);
      int64_t per = (n + std::max(1, nthreads) - 1) / std::max(1, nthreads);
      parallel_for(n, nthreads, [&](int64_t b, int64_t e) {
        double acc = 0.0;
        for (int64_t i = b; i < e; ++i) {
          const float* xi = x + i * d + j * dsub;
          double best = kInf;
          int bi = 0;
          for (int c = 0; c < 256; ++c) {
            double s = 0.0;
            for (int t = 0; t < dsub; ++t) {
              double diff = double(xi[t]) - cw[c * dsub + t];
              s += diff * diff;
            }
            if (s < best) {
              best = s;
              bi = c;
            }
          }
          assign[i] = bi;
          acc += best;
        }
        part[b / per] = acc;
      });
      if (obj)
        for (double v : part) obj[it] += v;
      if (it == niter) break;
      std::vector<double> sum(256 * size_t(dsub), 0.0);
      std::vector<int64_t> cnt(256, 0);
      for (int64_t i = 0; i < n; ++i) {
        int c = assign[i];
        ++cnt[c];
        for (int t = 0; t < dsub; ++t)
          sum[c * dsub + t] += x[i * d + j * dsub + t];
      }
      for (int c = 0; c < 256; ++c)
        if (cnt[c])
          for (int t = 0; t < dsub; ++t)
            cw[c * dsub + t] = sum[c * dsub + t] / double(cnt[c]);
    }
    for (int e = 0; e < 256; ++e)
      for (int t = 0; t < dsub; ++t)
        cb_out[(int64_t(j) * 256 + e) * dsub + t] = float(cw[e * dsub + t]);
  }
  return 0;
}

// Product-quantizer encoding: for each row of x and each sub-quantizer j, the
// index of the nearest codeword (ties to the lower index).
int oracle_pq_encode(const float* x, int64_t n, int d, int m, const float* cb,
                     uint8_t* codes, int nthreads) {
  if (n < 0 || d <= 0 || m <= 0 || d % m) return -1;
  int dsub = d / m;
  parallel_for(n, nthreads, [&](int64_t b, int64_t e) {
    for (int64_t i = b; i < e; ++i)
      for (int j = 0; j < m; ++j) {
        const float* xi = x + i * d + j * dsub;
        double best = kInf;
        int bi = 0;
        for (int c = 0; c < 256; ++c) {
          double s = sq_l2(xi, cb + (int64_t(j) * 256 + c) * dsub, dsub);
          if (s < best) {
            best = s;
            bi = c;
          }
        }
        codes[i * m + j] = uint8_t(bi);
      }
  });
  return 0;
}

}  // extern "C"
