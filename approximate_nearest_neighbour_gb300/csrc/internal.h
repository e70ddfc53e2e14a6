// Internal host-side interfaces shared by the translation units of
// libivfpq_gb300 (not part of the C ABI).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>
#include <vector>

#include "common.cuh"

namespace ivfpq {

// ---- k-selection launchers (select_k*.cu, kselect.cu) -------------------------
enum class OutKind {
  Float,    // fp32 value (from an order-preserving key) + int64 column index
  Dist,     // fp32 distance (raw non-negative key) + int64 id looked up in id_map
  Probes,   // int32 column index + optional fp32 value
  Partial,  // raw (key, index) pairs, k per (row, chunk)
  Merge     // fp32 value (order-preserving key) + int64 id of candidate c of row r:
            // id_map[((c / merge_kin) * merge_rows + r) * merge_kin + c % merge_kin]
};

struct SelectOut {
  OutKind kind = OutKind::Float;
  float* vals = nullptr;          // Float / Dist / Probes (optional)
  int64_t* idx64 = nullptr;       // Float / Dist
  int32_t* idx32 = nullptr;       // Probes
  const int64_t* id_map = nullptr;  // Dist: slot -> id
  uint32_t* pkeys = nullptr;      // Partial: [rows][chunks][k]
  uint32_t* pidx = nullptr;
  const int* row_mask = nullptr;  // if set, rows with row_mask[row] == 0 are skipped
  int64_t merge_rows = 0;         // Merge: rows per input set
  int merge_kin = 0;              // Merge: candidates per row per input set
};

// Rows of fp32 values: row r holds vals[r*cols .. r*cols+cols). The columns of
// each row are split into `chunks` ranges of `chunk_len` (chunks > 1 only
// with OutKind::Partial). K = power of two >= max(32, k).
int select_rows(const float* vals, int64_t rows, int64_t cols, int k, int64_t chunks,
                int64_t chunk_len, const SelectOut& out, cudaStream_t s);

// Rows of (key, index) pairs of length len: keys[r*len + i], idx[r*len + i].
int select_pairs(const uint32_t* keys, const uint32_t* idx, int64_t rows, int64_t len, int k,
                 int64_t chunks, int64_t chunk_len, const SelectOut& out, cudaStream_t s);

// Radix-bound selection, one block per row (select_radix.cu).
// bound[r] = a float >= the k-th smallest of row r of vals (+inf if none).
int row_kth_bound(const float* vals, int64_t rows, int64_t cols, int k, float* bound,
                  cudaStream_t s);
// The k smallest entries of each row's candidate segments (as
// select_candidates), sorted; flags[r] = 1 where row r was not written (an
// overflowed segment, or too many entries tie around the bound), else 0.
int cand_radix_select(const uint64_t* cand, const int* scnt, int nseg, int cap_s, int64_t rows,
                      int k, const SelectOut& out, int* flags, cudaStream_t s);
// Each row's len (key, index) pairs sorted, the first k written (len <= 8192).
int sort_pairs_rows(const uint32_t* keys, const uint32_t* idx, int64_t rows, int len, int k,
                    const SelectOut& out, cudaStream_t s);

// The k smallest of each row's `runs` runs of kw (key, index) pairs, each run
// sorted ascending (rows of runs * kw entries): a bitonic merge tree in shared
// memory (the pair selection when runs * kw exceeds 8,192).
int merge_sorted_runs(const uint32_t* pk, const uint32_t* pi, int64_t rows, int runs, int kw, int k,
                      const SelectOut& out, cudaStream_t s);

// Two-level selection over long rows when there are few rows: a first pass
// per column chunk into workspace, then a pass over the chunk winners.
int kselect_device(const float* vals, int64_t rows, int64_t cols, int k, const SelectOut& out,
                   cudaStream_t s);

// ---- squared-L2 distance tiles (distance.cu) -----------------------------------
// D[i*ldd + j] = sum_t (Q[i*d + t] - X[j*d + t])^2 for i < nq, j < n.
int l2_distance_tile(const float* Q, int64_t nq, const float* X, int64_t n, int d, float* D,
                     int64_t ldd, cudaStream_t s);

// The current device's status word (abi_util.cu): kernels with bounded waits
// set it when a wait expires; ivfpq_device_check reads and clears it.
int device_status_word(int** out);

// ---- tensor-core distance tiles (gemm_tc.cu) -------------------------------------
// Operands for 3xTF32 distances: hi/lo split rows padded to tc_dpad(d) columns
// and fp32 squared norms.
struct TcOperand {
  const float* hi = nullptr;
  const float* lo = nullptr;
  const float* norms = nullptr;
};
bool l2_tc_available(int d);
int tc_dpad(int d);
int l2_tc_prepare(const float* x, int64_t rows, int d, float* hi, float* lo, float* norms,
                  cudaStream_t s);
// D[i*ldd + j] = ||q_i||^2 + ||x_j||^2 - 2 <q_i, x_j> (3xTF32) for i < nq, j < n.
int l2_tc_tiles(const float* qhi, const float* qlo, const float* qnorm, int64_t nq,
                const float* xhi, const float* xlo, const float* xnorm, int64_t n, int d,
                float* D, int64_t ldd, int* err, cudaStream_t s);
// u[i, j] = ||x_j||^2 - 2 <q_i, x_j> (= D[i, j] - ||q_i||^2, so each row is
// ordered as D). Group-minimum pass over n columns with nsplit CTAs per
// 128-row query tile: gmin[i * G + g] = min of u[i, j] over group g of the
// columns, G = 128 * nsplit groups (column position mod 128 within each CTA's
// contiguous run of column tiles); +inf for an empty group.
int l2_tc_group_min(const float* qhi, const float* qlo, int64_t nq, const float* xhi,
                    const float* xlo, const float* xnorm, int64_t n, int d, int nsplit,
                    float* gmin, int* err, cudaStream_t s);
// Filter pass: row i keeps the entries with u[i, j] <= bound[i * bound_stride]
// (widened by a few ulps) as packed (order-preserving key of D << 32 | j) in
// nseg = 2 * nsplit segments of cap_s entries:
// cand[(i * nseg + seg) * cap_s ..], scnt[i * nseg + seg] = entries found (a
// count above cap_s means entries were dropped).
int l2_tc_filter(const float* qhi, const float* qlo, const float* qnorm, int64_t nq,
                 const float* xhi, const float* xlo, const float* xnorm, int64_t n, int d,
                 const float* bound, int64_t bound_stride, int nsplit, uint64_t* cand, int* scnt,
                 int cap_s, int* err, cudaStream_t s);
// CTAs per query tile that l2_tc_tiles would use for nq x n.
int tc_filter_split(int64_t nq, int64_t n);

// k-selection (k <= 256) over the candidate segments of l2_tc_filter; a row
// with an overflowed segment is selected over exact distances between row i
// of Q and all n rows of X instead (select_cand.cu).
int select_candidates(const uint64_t* cand, const int* scnt, int nseg, int cap_s, int64_t rows,
                      const float* Q, const float* X, int64_t n, int d, int k,
                      const SelectOut& out, cudaStream_t s);
// Whether searches of this index use the precomputed-term tables (the
// register-codebook scan, fp32 tables, m <= 16 when automatic), and their
// construction (ivfpq_index.cu).
bool use_precomputed(const ivfpq_index* ix);
int build_term1(ivfpq_index* ix);
// unit_len and unit_extra of the index from its list lengths
// (ivfpq_search.cu; called whenever the lists change).
void update_list_units(ivfpq_index* ix);

// ---- flat / coarse search on distance tiles (flat.cu) ----------------------------
// k nearest rows of X for each row of Q under squared L2; output as SelectOut
// (Float with column ids, or Probes).
// xop: precomputed tensor-core operands of X (may be null).
int knn_by_tiles(const float* Q, int64_t nq, const float* X, int64_t n, int d, int k,
                 const SelectOut& out, cudaStream_t s, const TcOperand* xop = nullptr);

}  // namespace ivfpq

// ---- the index -------------------------------------------------------------------------
struct ivfpq_index {
  int d = 0, nlist = 0, m = 0, nbits = 8, dsub = 0, dsub4 = 0;
  std::atomic<const char*> last_scan_kernel{nullptr};  // static name, for reports
  int lut_type = IVFPQ_LUT_FP32;
  int device = 0;
  float* centroids = nullptr;   // [nlist, d]
  float* cent_norms = nullptr;  // [nlist]
  float* codebooks = nullptr;   // [256, m, dsub4], zero-padded to dsub4 = roundup(dsub, 4)
  // precomputed list terms ||y_R||^2 + 2 <y_C, y_R> per (list, reproduction
  // value, sub-quantizer), [nlist, 256, m]; null unless the precomputed-term
  // tables are in use (precomputed: -1 automatic, 0 off, 1 on)
  float* term1 = nullptr;
  int precomputed = -1;
  // list scan organisation: -1 automatic, 0 by query, 1 by list (list-major,
  // where its shapes apply); table sets per by-list item (0 automatic)
  int scan_mode = -1;
  int lm_group = 0;
  // tensor-core operands of the centroids (null when that path is unavailable)
  float* cent_hi = nullptr;     // [nlist, tc_dpad(d)]
  float* cent_lo = nullptr;
  // inverted lists, interleaved in blocks of 32 vectors
  int64_t ntotal = 0;
  int64_t nblocks = 0;
  int32_t* list_len = nullptr;        // [nlist]
  int64_t* list_block_off = nullptr;  // [nlist + 1], in blocks
  uint8_t* codes = nullptr;           // [nblocks, 32 * m]
  int64_t* ids = nullptr;             // [nblocks * 32], -1 on padding slots
  std::vector<int64_t> h_list_len;    // host mirror of list_len
  int64_t max_list_len = 0;
  // by-list filter pass: lists longer than unit_len codes are scanned in
  // chunks of unit_len (0: no list is); unit_extra = the sum over lists of
  // their chunks beyond the first (set by ivfpq::update_list_units)
  int64_t unit_len = 0, unit_extra = 0;
  // queries re-scanned with full-length queues since the last read
  // (ivfpq_repaired_queries); device int64
  unsigned long long* repaired = nullptr;
  // per centroid, a lower bound (with rounding margins) of the squared
  // distance to its nearest other centroid; computed on the first hinted
  // encode (ivfpq_encode_hinted) under sep_mutex
  float* cent_sep = nullptr;
  std::mutex sep_mutex;
  // optional per-stage timing: one set of 5 events per profiled search
  struct EventSet {
    cudaEvent_t ev[5] = {nullptr, nullptr, nullptr, nullptr, nullptr};
    bool recorded[5] = {false, false, false, false, false};
  };
  bool profile = false;
  std::vector<EventSet> ev_sets;
  size_t ev_used = 0;
  int cur_set = -1;
};
