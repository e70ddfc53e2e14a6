/*
 * ivfpq.h -- C ABI of the GB300 (sm_103a) batched IVF-PQ search library
 * (libivfpq_gb300.so).
 *
 * The library implements the search path of the method described in
 * "Billion-scale similarity search with GPUs" (Johnson, Douze, Jegou): a
 * coarse quantizer, per-(query, list) ADC lookup tables, a scan of the PQ codes
 * in the probed inverted lists, and register-resident k-selection (WarpSelect /
 * BlockSelect) merged across lists. Exact brute-force k-NN and stand-alone
 * row-wise k-selection are exposed too.
 *
 * Conventions for every entry point:
 *  - Array pointers are DEVICE pointers (for example torch tensors'
 *    data_ptr()) unless stated otherwise; matrices are row-major and densely
 *    packed. `stream` is a cudaStream_t (NULL = the legacy default stream).
 *  - Calls enqueue work on `stream` and return without synchronizing, except
 *    ivfpq_add, which synchronizes `stream` once (it needs the new list sizes
 *    on the host to size the list storage), ivfpq_device_check,
 *    ivfpq_set_precomputed and the training calls (kmeans_lloyd, pq_train),
 *    which return host results.
 *  - Argument errors are detected on the host before any work is enqueued; in
 *    that case nothing is written and IVFPQ_ERR_INVALID_ARG (or
 *    IVFPQ_ERR_UNSUPPORTED) is returned. CUDA errors return IVFPQ_ERR_CUDA,
 *    failed workspace allocations IVFPQ_ERR_OOM. ivfpq_last_error() gives a
 *    message for the most recent failure on the calling thread.
 *  - Distances are squared L2 distances. Results are ordered by ascending
 *    distance; when fewer than k results exist the tail is (+inf, -1). The
 *    order of equal distances is unspecified.
 *  - Workspace is taken from the device's stream-ordered memory pool
 *    (cudaMallocAsync) on `stream` and returned on the same stream.
 *  - Search calls on one index may run concurrently on different streams;
 *    ivfpq_add must not overlap a search of the same index.
 */
#ifndef IVFPQ_GB300_H
#define IVFPQ_GB300_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct ivfpq_index ivfpq_index; /* opaque; owned by the library */

typedef enum {
  IVFPQ_OK = 0,
  IVFPQ_ERR_INVALID_ARG = -1,
  IVFPQ_ERR_UNSUPPORTED = -2,
  IVFPQ_ERR_OOM = -3,
  IVFPQ_ERR_CUDA = -4,
  IVFPQ_ERR_DEVICE_CHECK = -5,
  IVFPQ_ERR_TIMEOUT = -6
} ivfpq_status;

/* Storage type of the ADC lookup tables built in shared memory. */
typedef enum {
  IVFPQ_LUT_FP32 = 0, /* IEEE binary32 */
  IVFPQ_LUT_FP16 = 1, /* IEEE binary16, round to nearest even */
  IVFPQ_LUT_FP8 = 2   /* 1 sign / 4 exponent / 3 mantissa bits (E4M3), one
                         fp32 scale per table set */
} ivfpq_lut_type;

#define IVFPQ_MAX_K 2048  /* largest k accepted by every search entry point */
#define IVFPQ_MAX_M 64    /* largest number of sub-quantizers */

/*
 * ivfpq_index_create -- an empty IVF-PQ index.
 * Source: IVFADC ("Billion-scale similarity search with GPUs", section 5:
 * coarse quantizer q1 with |C1| centroids, product quantizer with b
 * sub-quantizers of 256 reproduction values each; b any multiple of 4 up to 64).
 *  d          vector dimension, > 0, multiple of m
 *  nlist      number of inverted lists / coarse centroids, 1 .. 2^24
 *  m          number of sub-quantizers (bytes per code): a multiple of 4, <= 64
 *  nbits      bits per sub-quantizer index; must be 8
 *  centroids  device fp32 [nlist, d]
 *  codebooks  device fp32 [m, 256, d/m]: codebooks[(j*256 + e)*(d/m) + t] is
 *             dimension t of reproduction value e of sub-quantizer j, which
 *             quantizes dimensions [j*d/m, (j+1)*d/m) of the residual
 *  out        receives the handle
 * The inputs are copied (synchronously, on the legacy default stream); the
 * caller keeps ownership of them. Errors: INVALID_ARG, UNSUPPORTED (nbits != 8,
 * m not a multiple of 4 or > 64), OOM, CUDA.
 */
int ivfpq_index_create(int d, int nlist, int m, int nbits, const float* centroids,
                       const float* codebooks, ivfpq_index** out);

/* ivfpq_index_destroy -- frees the index (synchronizes the device first).
 * NULL is accepted. */
int ivfpq_index_destroy(ivfpq_index* index);

/*
 * ivfpq_set_lut_type -- storage type of the lookup tables used by later
 * searches (ivfpq_lut_type). Source: fp32 / fp16 tables ("Billion-scale
 * similarity search with GPUs", section 5, the paragraph on T_i in shared
 * memory); 8-bit float tables ("Custom 8-bit floating point value format for
 * reducing shared memory bank conflict in approximate nearest neighbor
 * search", title and the paragraph on the norm2 fragment lookup table).
 * Errors: INVALID_ARG for an unknown type.
 */
int ivfpq_set_lut_type(ivfpq_index* index, int lut_type);

/*
 * ivfpq_add -- appends n encoded vectors to the inverted lists.
 * Source: IVFPQ build step 4 ("Custom 8-bit floating point ..." page): store
 * each vector's list and its PQ code; codes are kept as sequential groups of m
 * bytes per vector within lists ("Billion-scale similarity search with GPUs",
 * section 5). The library stores them interleaved in blocks of 32 vectors.
 *  codes     device uint8 [n, m], row-major
 *  list_ids  device int32 [n], each in [0, nlist)
 *  ids       device int64 [n], the ids returned by searches
 * Vectors keep their relative order inside each list (earlier rows first).
 * The inputs are copied; they may be freed once `stream` has completed.
 * Synchronizes `stream`. Errors: INVALID_ARG (also when a list id is out of
 * range; then the index is unchanged), OOM, CUDA.
 */
int ivfpq_add(ivfpq_index* index, const uint8_t* codes, const int32_t* list_ids,
              const int64_t* ids, int64_t n, void* stream);

/* ivfpq_ntotal -- number of vectors stored (host value), or -1 for NULL. */
int64_t ivfpq_ntotal(const ivfpq_index* index);

/*
 * ivfpq_search -- batched IVF-PQ search.
 * Source: IVFPQ search steps 1-5 and Eq. (1) ("Custom 8-bit floating point
 * ..." page); lookup tables T_1..T_b and their use in the list scan, two-pass
 * k-selection ("Billion-scale similarity search with GPUs", section 5).
 * For each query: the nprobe nearest centroids (the order of equal
 * distances is unspecified), per probed list the table T_j[e] = ||r^(j) - codeword_j(e)||^2 of the
 * residual r = query - centroid, the distance sum_j T_j[code_j] of every
 * stored vector, and the k smallest over all probed lists.
 *  queries   device fp32 [nq, d]
 *  nprobe    1 .. min(nlist, IVFPQ_MAX_K);  k  1 .. IVFPQ_MAX_K
 *  out_dist  device fp32 [nq, k];  out_ids  device int64 [nq, k]
 * Errors: INVALID_ARG, OOM, CUDA.
 */
int ivfpq_search(const ivfpq_index* index, const float* queries, int64_t nq, int nprobe,
                 int k, float* out_dist, int64_t* out_ids, void* stream);

/*
 * ivfpq_search_probes -- the coarse-quantizer stage alone: for each query the
 * nprobe nearest list ids (ascending distance) and their
 * squared distances. Same source and argument rules as ivfpq_search.
 *  out_probes  device int32 [nq, nprobe];  out_coarse  device fp32 [nq, nprobe]
 *  (out_coarse may be NULL)
 */
int ivfpq_search_probes(const ivfpq_index* index, const float* queries, int64_t nq,
                        int nprobe, int32_t* out_probes, float* out_coarse, void* stream);

/*
 * ivfpq_search_preassigned -- lookup-table build, list scan and k-selection
 * for caller-given probes (the stages after the coarse quantizer).
 *  probes  device int32 [nq, nprobe], each in [0, nlist); a list given twice
 *          for one query contributes its vectors twice; an id outside
 *          [0, nlist) (for example -1 as padding) is skipped
 * Other arguments as ivfpq_search.
 */
int ivfpq_search_preassigned(const ivfpq_index* index, const float* queries, int64_t nq,
                             int nprobe, const int32_t* probes, int k, float* out_dist,
                             int64_t* out_ids, void* stream);

/*
 * ivfpq_set_profiling / ivfpq_stage_times -- optional per-stage timing (not
 * part of the method; a measurement aid). Enabling (or disabling) clears the
 * history. While enabled, each search entry point records CUDA events on its
 * `stream` around its stages (up to 4096 searches are kept).
 * ivfpq_stage_times waits for the recorded events and writes, summed over
 * the recorded searches, the milliseconds of [0] coarse quantizer (distances
 * + top-nprobe), [1] planning (by-list scan: the bound pass over each
 * query's nearest list, the (list, query) items and their records),
 * [2] the list-scan kernel (lookup tables + list scan + per-chunk selection
 * or candidate filter), [3] merge / final selection and rescans into
 * ms[0..3], and the number of recorded searches into *nsearches (may be
 * NULL). Stages that did not run contribute 0.
 */
int ivfpq_set_profiling(ivfpq_index* index, int enable);
int ivfpq_stage_times(const ivfpq_index* index, float* ms, int* nsearches);

/*
 * ivfpq_set_precomputed -- lookup tables from precomputed terms.
 * Source: "Billion-scale similarity search with GPUs", section 5: the
 * residual distance ||x - y_C - y_R||^2 expands into ||x - y_C||^2 (the
 * coarse distance, per query and list), ||y_R||^2 + 2 <y_C, y_R> (per list and
 * code: a table of 256 x m entries per list, computed once) and
 * -2 <x, y_R> (per query: one table of 256 x m entries for all its lists), so
 * a list's table is the sum of a stored table and the query's table instead
 * of 256 x d multiply-adds. The stored tables take nlist x 256 x m x 4 bytes
 * of device memory.
 *  mode  -1 automatic (default: on for fp32 tables with m = 16, d/m = 8,
 *           where it measured faster), 0 off, 1 on where supported (fp32
 *           tables, m = 8 with d/m in {12, 8}, m = 16 with d/m in {8, 4})
 * Synchronizes the device; must not overlap a search of the index. Results
 * equal those of the direct tables up to fp32 rounding (distances are
 * clamped at 0). Errors: INVALID_ARG, OOM, CUDA.
 */
int ivfpq_set_precomputed(ivfpq_index* index, int mode);

/*
 * ivfpq_set_scan_mode -- how later searches of the index organise the list
 * scan; results are the same either way (up to the order of equal distances).
 * Source: "Billion-scale similarity search with GPUs", section 5: queries x
 * lists are independent work, taken there query by query.
 *  mode   -1 automatic (default): by list where the shapes allow it (fp32,
 *            binary16 or E4M3 tables, direct tables, (m, d/m) in {(32,3), (32,4),
 *            (16,8), (16,4), (8,12), (8,8)}, nprobe >= 2) and the batch
 *            probes every list twice or more on average, else by query;
 *          0 by query: one thread block per (query, chunk of its lists);
 *          1 by list where the shapes allow it: the queries that probe a
 *            list are scanned together, up to `group` table sets of them
 *            per item, each query keeping the codes within a bound taken
 *            from its nearest list (scanned first); a query with more such
 *            codes than its buffer holds is scanned again by query
 *  group  table sets per by-list item: 1 to 3 (a set holds one query's fp32
 *         tables, two queries' binary16 tables or four queries' E4M3 tables;
 *         E4M3 items take at most 2 sets), -1 automatic (default: 3, or 2 for
 *         binary16 tables with m = 16 and for E4M3 tables), 0 keeps the
 *         current value
 * Errors: INVALID_ARG.
 */
int ivfpq_set_scan_mode(ivfpq_index* index, int mode, int group);

/* ivfpq_uses_precomputed -- 1 if searches of the index currently use the
 * precomputed-term tables, else 0. */
int ivfpq_uses_precomputed(const ivfpq_index* index);

/* ivfpq_last_scan_kernel -- name of the list-scan kernel family that the
 * most recent search of this index launched ("ivfpq_scan_lm_kernel": the
 * by-list scan of ivfpq_set_scan_mode; "ivfpq_scan2_kernel": by query,
 * codebook in registers, double-buffered fp32 tables, used for fp32 tables
 * with (m, d/m) in {(32,3), (32,4), (16,8), (16,4), (8,12), (8,8)};
 * "ivfpq_scan_kernel": the general kernel), or NULL before the first search;
 * a measurement aid. */
const char* ivfpq_last_scan_kernel(const ivfpq_index* index);

/* ivfpq_kernel_launches -- number of CUDA kernels this library has launched
 * since it was loaded (all threads); a measurement aid. */
uint64_t ivfpq_kernel_launches(void);

/* ivfpq_workspace_allocations -- number of temporary device allocations
 * (stream-ordered workspace) the library has made since it was loaded (all
 * threads); lets a caller check that an entry point allocated nothing. */
uint64_t ivfpq_workspace_allocations(void);

/*
 * flat_knn -- exact brute-force k-NN under squared L2.
 * Source: exact search by a GEMM-form distance ||x||^2 - 2<x, y> + ||y||^2
 * followed by k-selection ("Billion-scale similarity search with GPUs",
 * sections 4-5, "as with exact search").
 *  db       device fp32 [n, d];  queries  device fp32 [nq, d]
 *  k        1 .. IVFPQ_MAX_K
 *  out_dist device fp32 [nq, k];  out_ids  device int64 [nq, k] (row index in db)
 * Errors: INVALID_ARG, OOM, CUDA.
 */
int flat_knn(const float* db, int64_t n, int d, const float* queries, int64_t nq, int k,
             float* out_dist, int64_t* out_ids, void* stream);

/*
 * kselect -- the k smallest values of each row with their column index.
 * Source: WarpSelect ("Billion-scale similarity search with GPUs", section 4,
 * Algorithm 3) with BlockSelect (several warps, queues merged in shared memory)
 * for long rows. With at least 4 rows per SM and at least 32768 columns, a
 * row's k smallest are instead taken from the values at or below a bound read
 * off a histogram of the row's first values (a shared buffer, one sort); a
 * row with too many such values (many equal values) is redone by the queues.
 * Results are the same either way; equal values may come in any order.
 *  vals      device fp32 [rows, cols]; +-inf allowed, NaN not supported
 *  k         1 .. IVFPQ_MAX_K;  cols < 2^32 - 1
 *  out_vals  device fp32 [rows, k];  out_idx  device int64 [rows, k]
 * Errors: INVALID_ARG, OOM, CUDA.
 */
int kselect(const float* vals, int64_t rows, int64_t cols, int k, float* out_vals,
            int64_t* out_idx, void* stream);

/*
 * kselect_noalloc -- kselect for callers that cannot allocate device memory
 * while they run. No passage of the pages corresponds to it; it exists for
 * callers such as a process whose device memory is fully reserved up front by
 * another allocator, or a latency-critical loop that may not wait on an
 * allocator. kselect takes its two-pass workspace from the stream-ordered
 * pool; this variant allocates nothing: its partial results live in one fixed
 * 8 MiB device array that every GPU loading the library holds until the
 * library is unloaded.
 *  Arguments, layout and results as kselect (the caller passes inputs and
 *  outputs). Limit: rows * k <= 1,048,576; larger problems return
 *  IVFPQ_ERR_INVALID_ARG with a message naming the limit.
 *  The first call on a device sets up the array's device address on that
 *  device (a runtime symbol lookup); make that first call before any stream
 *  capture. All calls on one device share that device's array, so calls whose
 *  work overlaps on the GPU (for example on two streams) race and must be
 *  ordered by the caller. Nothing left in the array by an earlier call is read.
 */
int kselect_noalloc(const float* vals, int64_t rows, int64_t cols, int k, float* out_vals,
                    int64_t* out_idx, void* stream);

/*
 * ivfpq_knn_graph -- approximate k-nearest-neighbour graph of a vector set:
 * every vector searched as a query against an index holding the same set
 * ("Billion-scale similarity search with GPUs", section 6, k-NN graph).
 *  x         device fp32 [n, d]: the vectors (as added to the index)
 *  self_ids  device int64 [n]: the id under which x[i] was added; that id is
 *            removed from row i (if the search did not return it, the row's
 *            (k+1)-th neighbour is dropped instead)
 *  nprobe, k as ivfpq_search, 1 <= k < IVFPQ_MAX_K
 *  out_dist  device fp32 [n, k], out_ids device int64 [n, k]
 * Queries run in batches of 32,768. Errors: as ivfpq_search.
 */
int ivfpq_knn_graph(const ivfpq_index* index, const float* x, const int64_t* self_ids, int64_t n,
                    int nprobe, int k, float* out_dist, int64_t* out_ids, void* stream);

/*
 * kmeans_lloyd -- Lloyd k-means (coarse quantizer training).
 * Source: "Billion-scale similarity search with GPUs", section 6: k-means
 * alternates a k = 1 nearest-centroid search over all points with a centroid
 * update.
 *  x          device fp32 [n, d], k <= n < 2^31, d >= 1
 *  init       device int64 [k]: row indices of x that seed the centroids
 *  niter      number of updates (>= 0); niter + 1 assignment passes
 *  centroids  device fp32 [k, d] (out)
 *  assign     device int32 [n] (out, may be NULL): the final assignment
 * A row holding NaN has no finite distance: the search may leave it without a
 * centroid (assignment -1, the row joins no cluster) or assign it at distance
 * NaN (its cluster's mean and the objective become NaN); either way nothing
 * outside the arguments is read or written.
 *  objective  HOST fp64 [niter + 1] (out, may be NULL): sum of squared
 *             distances to the assigned centroid at each assignment pass
 * The update is the mean of each cluster's points summed in fp64 in
 * increasing point order (deterministic); an empty cluster keeps its
 * centroid. Synchronizes `stream`. Errors: INVALID_ARG (also an init index
 * outside [0, n)), OOM, CUDA.
 */
int kmeans_lloyd(const float* x, int64_t n, int d, int k, int niter, const int64_t* init,
                 float* centroids, int32_t* assign, double* objective, void* stream);

/*
 * pq_train -- product quantizer training: for each of the m sub-spaces
 * (dimensions [j*d/m, (j+1)*d/m)), kmeans_lloyd with 256 centroids on the
 * points' sub-vectors (train on residuals x - centroid of x's list for IVF-PQ).
 * Source: "Custom 8-bit floating point value format ...", index construction
 * step 3 (256 codewords per sub-space); "Billion-scale similarity search with
 * GPUs", sections 5-6.
 *  x          device fp32 [n, d], 256 <= n < 2^31, d % m == 0
 *  init       device int64 [256]: the rows whose sub-vectors seed every
 *             sub-quantizer's codewords
 *  codebooks  device fp32 [m, 256, d/m] (out), the layout ivfpq_index_create takes
 *  objective  HOST fp64 [niter + 1] (may be NULL): summed over sub-quantizers
 * Synchronizes `stream`. Errors: INVALID_ARG, OOM, CUDA.
 */
int pq_train(const float* x, int64_t n, int d, int m, int niter, const int64_t* init,
             float* codebooks, double* objective, void* stream);

/*
 * ivfpq_encode -- IVF-PQ codes of a batch of vectors, for ivfpq_add.
 * Source: "Custom 8-bit floating point value format ...", index construction
 * steps 1-3 (nearest centroid, residual, nearest codeword per sub-space).
 *  x         device fp32 [n, index d]
 *  list_ids  device int32 [n] (out): nearest centroid (exact distances); a
 *            row holding NaN may get -1 (no finite distance to any centroid),
 *            which ivfpq_add rejects
 *  codes     device uint8 [n, m] (out): per sub-space, the codeword nearest
 *            to the residual's sub-vector (fp32 distances, lowest index on
 *            ties); zeros for a row with list -1
 * Asynchronous. Errors: INVALID_ARG (also d/m > 32), OOM, CUDA.
 */
int ivfpq_encode(const ivfpq_index* index, const float* x, int64_t n, int32_t* list_ids,
                 uint8_t* codes, void* stream);

/*
 * ivfpq_residuals -- nearest coarse centroid of each vector and the residual
 * (vector minus that centroid), the training input of the product quantizer.
 * Source: "Custom 8-bit floating point value format ...", index construction
 * steps 1-2 (each vector belongs to the cluster of its nearest centroid; the
 * residual is the vector minus the centroid); "Billion-scale similarity
 * search with GPUs", section 5 (the product quantizer encodes residuals).
 *  centroids  device fp32 [nlist, d];  x  device fp32 [n, d], n < 2^31
 *  list_ids   device int32 [n] (out): nearest centroid (exact distances;
 *             equal distances go to either centroid); a row holding NaN
 *             may get -1 (no finite distance to any centroid)
 *  residuals  device fp32 [n, d] (out): x - centroids[list_ids]; NaN for a
 *             row with list -1
 * Asynchronous. Errors: INVALID_ARG, OOM, CUDA.
 */
int ivfpq_residuals(const float* centroids, int nlist, int d, const float* x, int64_t n,
                    int32_t* list_ids, float* residuals, void* stream);

/*
 * ivfpq_encode_hinted -- ivfpq_encode for callers that know a likely list of
 * each vector (the previous assignment of an iterative clustering, or the
 * cluster a vector was drawn from). Same results as ivfpq_encode: the hint h
 * of row r is accepted only when 4 ||x_r - c_h||^2 is below a lower bound of
 * the squared distance from c_h to its nearest other centroid, which proves
 * by the triangle inequality that c_h is the nearest centroid and the only
 * one (Elkan, "Using the triangle inequality to accelerate k-means", ICML
 * 2003, Lemma 1); every other row (a wrong, doubtful or out-of-range hint)
 * gets the full nearest-centroid search of ivfpq_encode. The first call on an
 * index computes the centroids' separations once (a k = 2 search of the
 * centroids among themselves) and keeps them with the index.
 *  hint        device int32 [n]: a list id per row (any value accepted)
 *  n_searched  HOST int64 (out, may be NULL): rows that needed the full search
 * Other arguments as ivfpq_encode. Synchronizes `stream` (the number of rows
 * to search sizes that search). Errors: INVALID_ARG, OOM, CUDA.
 */
int ivfpq_encode_hinted(const ivfpq_index* index, const float* x, int64_t n, const int32_t* hint,
                        int32_t* list_ids, uint8_t* codes, int64_t* n_searched, void* stream);

/*
 * ivfpq_repaired_queries -- the number of queries that searches of this
 * index re-scanned since the previous call (or since creation), then resets
 * it; a measurement aid. The register-codebook list scan keeps per warp a
 * queue shorter than k; a query for which one warp may have held more of the
 * k best than its queue is detected after the merge and scanned again with
 * full-length queues, so results do not depend on it. Synchronizes `stream`;
 * searches still running on other streams may not be counted yet.
 *  count  HOST int64 (out)
 * Errors: INVALID_ARG, CUDA.
 */
int ivfpq_repaired_queries(const ivfpq_index* index, int64_t* count, void* stream);

/*
 * knn_merge -- final k-selection over the results of S index shards.
 * Source: sharding ("Billion-scale similarity search with GPUs", section 5,
 * multi-GPU): every shard holds part of the database and answers all queries;
 * an additional round of k-selection combines their k results per query.
 *  dists   device fp32 [nshards, nq, k_in]: shard s's distances of query q,
 *          ascending or not (order is not required); +inf marks a missing entry
 *  ids     device int64 [nshards, nq, k_in]: the matching ids (global ids,
 *          -1 for missing entries)
 *  k       1 .. IVFPQ_MAX_K; k > nshards * k_in pads with (+inf, -1)
 *  out_dist device fp32 [nq, k], out_ids device int64 [nq, k]: the k smallest
 *          distances of each query over all shards, ascending, with their ids
 * Ties are broken arbitrarily. Errors: INVALID_ARG, OOM, CUDA.
 */
int knn_merge(const float* dists, const int64_t* ids, int64_t nq, int nshards, int k_in, int k,
              float* out_dist, int64_t* out_ids, void* stream);

/* ivfpq_device_check -- synchronises `stream` and reports whether any kernel
 * of this library on the current device gave up a bounded wait since the
 * last check (the tensor-core distance pipeline waits on its own copies and
 * MMAs with an iteration limit; on expiry it stops, releases its resources
 * and sets a per-device status word instead of hanging). Clears the word.
 * Returns IVFPQ_OK, or IVFPQ_ERR_TIMEOUT (the results of the calls since the
 * previous check are then invalid), or IVFPQ_ERR_CUDA. */
int ivfpq_device_check(void* stream);

/* ivfpq_selftest_wait_timeout -- launches one block that waits, with an
 * iteration limit of `spins`, on a barrier phase that nothing completes, the
 * same bounded wait the distance pipeline uses; the block records the expiry
 * in the status word and returns. A host-visible check of that mechanism:
 * ivfpq_device_check then returns IVFPQ_ERR_TIMEOUT. spins: 1 .. 2^20. */
int ivfpq_selftest_wait_timeout(int spins, void* stream);

/* ivfpq_last_error -- message for the most recent failure on this thread
 * (empty string if none). The pointer stays valid until the next call into
 * the library from this thread. */
const char* ivfpq_last_error(void);

/* ivfpq_status_string -- a static name for a status code. */
const char* ivfpq_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* IVFPQ_GB300_H */
