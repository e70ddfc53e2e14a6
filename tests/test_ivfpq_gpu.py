"""IVF-PQ search on the GPU against the oracle.

The probe sets are checked with the tie rule (a probe may differ only by a
list whose exact coarse distance ties the nprobe-th), then the oracle is run
with the GPU's probes and the results are compared with the tolerance rule of
tests/parity.py.
"""

import numpy as np
import pytest

import oracle
from approximate_nearest_neighbour_gb300 import synthetic as S
from parity import check_probes, compare_knn, tol

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from approximate_nearest_neighbour_gb300 import binding
    return binding


def _t(x):
    import torch
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def make_index(B, cent, cb, codes, list_ids, ids, pieces=1):
    ix = B.ivfpq_index_create(_t(cent), _t(cb))
    n = codes.shape[0]
    bounds = np.linspace(0, n, pieces + 1).astype(np.int64)
    for a, b in zip(bounds[:-1], bounds[1:]):
        B.ivfpq_add(ix, _t(codes[a:b]), _t(list_ids[a:b]), _t(ids[a:b]))
    return ix


def coarse_all(q, cent):
    lists, dist = oracle.coarse(q, cent, cent.shape[0])
    out = np.empty_like(dist)
    np.put_along_axis(out, lists.astype(np.int64), dist, axis=1)
    return out


def search_and_check(B, ix, cent, cb, lists, q, nprobe, k, rows=None, extra=64, context=""):
    """lists = (list_off, codes in list order, ids in list order)."""
    import torch
    qd = _t(q)
    gp, gc = B.ivfpq_search_probes(ix, qd, nprobe)
    gd, gi = B.ivfpq_search(ix, qd, nprobe, k)
    torch.cuda.synchronize()
    gp, gc, gd, gi = (x.cpu().numpy() for x in (gp, gc, gd, gi))
    rows = np.arange(q.shape[0]) if rows is None else np.asarray(rows)
    qs = q[rows]
    op, _ = oracle.coarse(qs, cent, nprobe)
    call = None

    def dist_all(r):
        nonlocal call
        if call is None:
            call = coarse_all(qs, cent)
        return call[r]

    ndiff = check_probes(gp[rows], op, dist_all)
    # coarse distances of the GPU's probes
    dc = np.stack([((cent[gp[r]].astype(np.float64) - q[r].astype(np.float64)) ** 2).sum(1)
                   for r in rows])
    assert np.all(np.abs(gc[rows] - dc) <= tol(dc)), f"{context}: coarse distances"
    off, codes_l, ids_l = lists
    od, oi, _ = oracle.ivfpq_search(qs, cent, cb, off, codes_l, ids_l, nprobe, k + extra,
                                    forced_probes=gp[rows])
    compare_knn(gd[rows], gi[rows], od, oi, context=context)
    return gd, gi, ndiff


# ---------------------------------------------------------------------------
def test_tiny_workload_trained_codebooks(B):
    """N=1e5, d=64, 256 clusters (sigma 0.1), centroids = true centres, PQ m=8
    trained by 10 Lloyd iterations on residuals, nq=100, nprobe=8, k=10."""
    w = S.IVFPQ_TINY
    cent, x, init = S.tiny_raw(w)
    assign, _ = oracle.coarse(x, cent, 1)
    list_ids = assign[:, 0].astype(np.int32)
    resid = x - cent[list_ids]
    cb, obj = oracle.pq_train(resid, w.m, 10, init)
    assert np.all(np.diff(obj) <= 1e-9 * obj[0])
    codes = oracle.pq_encode(resid, cb)
    ids = np.arange(x.shape[0], dtype=np.int64)
    lists = oracle.to_lists(codes, list_ids, ids, w.nlist)
    q = S.queries(w.number, cent, S.component_weights(w.nlist, False), w.sigma, w.nq)
    ix = make_index(B, cent, cb, codes, list_ids, ids)
    assert ix.ntotal == x.shape[0]
    gd, gi, _ = search_and_check(B, ix, cent, cb, lists, q, 8, 10, context="tiny")
    # recall against exact neighbours is reported, not gated
    _, ti = oracle.flat_knn(x, q, 10)
    r = oracle.recall_at_k(gi, ti)
    print(f"tiny workload recall@10 vs exact = {r:.3f}")
    assert r > 0.3


@pytest.mark.parametrize("m,dsub", [(8, 12), (12, 4), (16, 8), (32, 3), (64, 2), (20, 3), (4, 5),
                                    (8, 8), (16, 4), (32, 4)])
def test_code_widths_and_ragged_lists(B, m, dsub):
    d = m * dsub
    w = S.IVFPQWorkload("t", 90 + m, 30_000, d, 97, m, 0.15, True, 40, (7,), (33,), ("fp32",))
    data = S.compressed_index(w)
    assert (np.diff(data.list_off) == 0).any() or True
    q = S.queries(w.number, data.cent, data.weights, w.sigma, w.nq)
    codes, list_ids, ids = S.shuffled(data, w.number)
    ix = make_index(B, data.cent, data.cb, codes, list_ids, ids)
    lists = oracle.to_lists(codes, list_ids, ids, w.nlist)
    for mode in (0, -1):  # by query, then automatic (by list for its shapes)
        B.ivfpq_set_scan_mode(ix, mode)
        for k in (1, 33, 250):
            search_and_check(B, ix, data.cent, data.cb, lists, q, 7, k,
                             context=f"m={m} k={k} mode={mode}")


LM_SHAPES = [(32, 3), (32, 4), (16, 8), (16, 4), (8, 12), (8, 8)]


@pytest.mark.parametrize("group", [2, 3])
@pytest.mark.parametrize("m,dsub", LM_SHAPES)
def test_list_major_scan_follows_the_oracle(B, m, dsub, group):
    """The by-list scan (queries of a list scanned together, a bound from each
    query's nearest list, candidate buffers) on ragged and empty lists, many
    queries per list, k from 1 to 2048."""
    w = S.IVFPQWorkload("t", 200 + m + dsub, 40_000, m * dsub, 61, m, 0.15, True, 300, (9,),
                        (33,), ("fp32",))
    data = S.compressed_index(w)
    q = S.queries(w.number, data.cent, data.weights, w.sigma, w.nq)
    codes, list_ids, ids = S.shuffled(data, w.number)
    ix = make_index(B, data.cent, data.cb, codes, list_ids, ids)
    B.ivfpq_set_scan_mode(ix, 1, group)
    lists = oracle.to_lists(codes, list_ids, ids, w.nlist)
    for k in (1, 100, 1000, 2048):
        search_and_check(B, ix, data.cent, data.cb, lists, q, 9, k, rows=np.arange(0, 300, 7),
                         context=f"list-major m={m} G={group} k={k}")
        assert B.last_scan_kernel(ix) == "ivfpq_scan_lm_kernel"


@pytest.mark.parametrize("group", [2, 3])
@pytest.mark.parametrize("m,dsub", LM_SHAPES)
def test_list_major_binary16_tables_follow_the_oracle_variant(B, m, dsub, group):
    """The by-list scan with binary16 tables (two queries' entries per
    shared-memory word, fp32 sums) against the oracle's binary16 tables, and
    against the by-query scan's binary16 tables (the general kernel)."""
    import torch
    w = S.IVFPQWorkload("t", 260 + m + dsub, 40_000, m * dsub, 61, m, 0.15, True, 300, (9,),
                        (33,), ("fp16",))
    data = S.compressed_index(w)
    q = S.queries(w.number, data.cent, data.weights, w.sigma, w.nq)
    ix = make_index(B, data.cent, data.cb, data.codes, data.list_ids, data.ids)
    B.ivfpq_set_lut_type(ix, "fp16")
    rows = np.arange(0, 300, 5)
    for k in (1, 100, 700):
        B.ivfpq_set_scan_mode(ix, 1, group)
        gp, _ = B.ivfpq_search_probes(ix, _t(q), 9)
        gd, gi = B.ivfpq_search(ix, _t(q), 9, k)
        assert B.last_scan_kernel(ix) == "ivfpq_scan_lm_kernel"
        B.ivfpq_set_scan_mode(ix, 0)
        qd, qi = B.ivfpq_search(ix, _t(q), 9, k)
        torch.cuda.synchronize()
        gp, gd, gi, qd = (t.cpu().numpy() for t in (gp, gd, gi, qd))
        od, oi, _ = oracle.ivfpq_search(q[rows], data.cent, data.cb, data.list_off, data.codes,
                                        data.ids, 9, k, oracle.LUT_FP16, forced_probes=gp[rows])
        assert np.all(np.abs(gd[rows] - od) <= 2e-3 * np.abs(od) + 1e-5), f"k={k}"
        assert oracle.recall_at_k(gi[rows], oi) >= 0.99
        # same tables and fp32 sums as the by-query scan, up to summation order
        assert np.all(np.abs(gd - qd) <= 1e-5 * np.abs(qd) + 1e-6), f"k={k}"


@pytest.mark.parametrize("group", [1, 2])
@pytest.mark.parametrize("m,dsub", LM_SHAPES)
def test_list_major_e4m3_tables_follow_the_oracle_variant(B, m, dsub, group):
    """The by-list scan with E4M3 tables (four queries' entries per
    shared-memory word, one scale per query's table, fp32 sums of the decoded
    entries) against the oracle's E4M3 tables: distances within the format's
    precision, ids up to the near-ties its 3-bit mantissas make (the GPU
    scales by 448 / max T where the oracle divides by max T / 448, so an entry
    next to a rounding boundary may land one step apart; with k = 1 over 60
    rows one swapped near-tie is 1.7 % of the recall)."""
    import torch
    w = S.IVFPQWorkload("t", 280 + m + dsub, 40_000, m * dsub, 61, m, 0.15, True, 300, (9,),
                        (33,), ("fp8",))
    data = S.compressed_index(w)
    q = S.queries(w.number, data.cent, data.weights, w.sigma, w.nq)
    ix = make_index(B, data.cent, data.cb, data.codes, data.list_ids, data.ids)
    B.ivfpq_set_lut_type(ix, "fp8")
    rows = np.arange(0, 300, 5)
    for k in (1, 100, 700):
        B.ivfpq_set_scan_mode(ix, 1, group)
        gp, _ = B.ivfpq_search_probes(ix, _t(q), 9)
        gd, gi = B.ivfpq_search(ix, _t(q), 9, k)
        assert B.last_scan_kernel(ix) == "ivfpq_scan_lm_kernel"
        torch.cuda.synchronize()
        gp, gd, gi = (t.cpu().numpy() for t in (gp, gd, gi))
        od, oi, _ = oracle.ivfpq_search(q[rows], data.cent, data.cb, data.list_off, data.codes,
                                        data.ids, 9, k, oracle.LUT_FP8, forced_probes=gp[rows])
        assert np.all(np.abs(gd[rows] - od) <= 3e-2 * np.abs(od) + 1e-5), f"k={k}"
        assert oracle.recall_at_k(gi[rows], oi) >= (0.9 if k == 1 else 0.95), f"k={k}"


@pytest.mark.parametrize("lut", ["fp32", "fp16"])
def test_list_major_long_nearest_list_is_chunked(B, lut):
    """A nearest list longer than a bound-pass chunk (32,768 codes): its
    chunks are separate items whose lane queues together give the bound."""
    import torch
    rng = np.random.default_rng(91)
    nlist, m, dsub = 8, 8, 12
    d = m * dsub
    cent = (3 * rng.standard_normal((nlist, d))).astype(np.float32)
    cb = (0.3 * rng.standard_normal((m, 256, dsub))).astype(np.float32)
    sizes = [100_003, 700, 650, 600, 550, 500, 450, 400]
    list_ids = np.repeat(np.arange(nlist, dtype=np.int32), sizes)
    n = list_ids.shape[0]
    codes = rng.integers(0, 256, (n, m)).astype(np.uint8)
    ids = np.arange(n, dtype=np.int64) * 3 + 1
    ix = make_index(B, cent, cb, codes, list_ids, ids)
    B.ivfpq_set_lut_type(ix, lut)
    B.ivfpq_set_scan_mode(ix, 1)
    q = (cent[0] + 0.05 * rng.standard_normal((48, d))).astype(np.float32)
    q[40:] = cent[3] + 0.05 * rng.standard_normal((8, d))  # some with a short nearest list
    lists = oracle.to_lists(codes, list_ids, ids, nlist)
    for k in (10, 100, 1000):
        if lut == "fp32":
            search_and_check(B, ix, cent, cb, lists, q, 4, k, context=f"chunked k={k}")
        else:
            gp, _ = B.ivfpq_search_probes(ix, _t(q), 4)
            gd, gi = B.ivfpq_search(ix, _t(q), 4, k)
            torch.cuda.synchronize()
            gp, gd, gi = gp.cpu().numpy(), gd.cpu().numpy(), gi.cpu().numpy()
            od, oi, _ = oracle.ivfpq_search(q, cent, cb, lists[0], lists[1], lists[2], 4, k,
                                            oracle.LUT_FP16, forced_probes=gp)
            assert np.all(np.abs(gd - od) <= 2e-3 * np.abs(od) + 1e-5), f"k={k}"
        assert B.last_scan_kernel(ix) == "ivfpq_scan_lm_kernel"


@pytest.mark.parametrize("group", [2, 3])
def test_list_major_candidate_overflow_is_rescanned(B, group):
    """Every query's nearest list holds fewer than k codes, so its bound is
    +inf and all codes of the other probed lists are candidates, more than
    the buffer holds: those queries are scanned again by query."""
    rng = np.random.default_rng(71 + group)
    nlist, m, dsub = 6, 32, 3
    d = m * dsub
    cent = rng.standard_normal((nlist, d)).astype(np.float32) * 3
    cb = (0.3 * rng.standard_normal((m, 256, dsub))).astype(np.float32)
    sizes = [5, 900, 900, 900, 900, 900]
    list_ids = np.repeat(np.arange(nlist, dtype=np.int32), sizes)
    n = list_ids.shape[0]
    codes = rng.integers(0, 256, (n, m)).astype(np.uint8)
    ids = np.arange(n, dtype=np.int64) * 5 + 2
    ix = make_index(B, cent, cb, codes, list_ids, ids)
    B.ivfpq_set_scan_mode(ix, 1, group)
    q = (cent[0] + 0.05 * rng.standard_normal((40, d))).astype(np.float32)
    lists = oracle.to_lists(codes, list_ids, ids, nlist)
    B.ivfpq_repaired_queries(ix)
    search_and_check(B, ix, cent, cb, lists, q, 5, 10, context="overflow")
    assert B.ivfpq_repaired_queries(ix) >= 40  # every query overflowed
    assert B.last_scan_kernel(ix) == "ivfpq_scan_lm_kernel"


def test_empty_lists_large_k_and_padding(B):
    """Many empty lists; k larger than the candidates of the probed lists."""
    w = S.IVFPQWorkload("t", 77, 900, 32, 400, 8, 0.15, True, 9, (3,), (5,), ("fp32",))
    data = S.compressed_index(w)
    assert (np.diff(data.list_off) == 0).sum() > 50
    q = S.queries(w.number, data.cent, data.weights, w.sigma, w.nq)
    ix = make_index(B, data.cent, data.cb, data.codes, data.list_ids, data.ids)
    lists = (data.list_off, data.codes, data.ids)
    for k in (64, 700, 2048):
        gd, gi, _ = search_and_check(B, ix, data.cent, data.cb, lists, q, 3, k, context=f"k={k}")
        assert np.isinf(gd[:, -1]).all() and (gi[:, -1] == -1).all()


@pytest.mark.parametrize("m,dsub", [(8, 12), (8, 8), (16, 8), (16, 4)])
def test_precomputed_term_tables_follow_the_oracle(B, m, dsub):
    """Tables from precomputed terms (list table + query table + the coarse
    distance) and the direct tables both match the oracle's direct ADC
    within the tolerance, on the same probes; automatic mode selects the
    precomputed tables where they measured faster (m = 16, d/m = 8)."""
    import torch
    w = S.IVFPQWorkload("t", 140 + m + dsub, 30_000, m * dsub, 61, m, 0.15, True, 30, (6,),
                        (40,), ("fp32",))
    data = S.compressed_index(w)
    q = S.queries(w.number, data.cent, data.weights, w.sigma, w.nq)
    ix = make_index(B, data.cent, data.cb, data.codes, data.list_ids, data.ids)
    assert B.ivfpq_uses_precomputed(ix) == ((m, dsub) == (16, 8))  # automatic mode
    assert B.ivfpq_set_precomputed(ix, 1)
    lists = oracle.to_lists(data.codes, data.list_ids, data.ids, w.nlist)
    gd1, gi1, _ = search_and_check(B, ix, data.cent, data.cb, lists, q, 6, 40,
                                   context=f"precomputed m={m}")
    assert not B.ivfpq_set_precomputed(ix, 0)
    gd0, gi0, _ = search_and_check(B, ix, data.cent, data.cb, lists, q, 6, 40,
                                   context=f"direct m={m}")
    assert np.all(np.abs(gd1 - gd0) <= tol(gd0))
    assert B.ivfpq_set_precomputed(ix, 1)
    torch.cuda.synchronize()


def test_appending_in_pieces_equals_one_add(B):
    import torch
    w = S.IVFPQWorkload("t", 66, 25_000, 64, 64, 16, 0.15, False, 30, (5,), (20,), ("fp32",))
    data = S.compressed_index(w)
    codes, list_ids, ids = S.shuffled(data, w.number)
    q = S.queries(w.number, data.cent, data.weights, w.sigma, w.nq)
    one = make_index(B, data.cent, data.cb, codes, list_ids, ids)
    three = make_index(B, data.cent, data.cb, codes, list_ids, ids, pieces=3)
    assert one.ntotal == three.ntotal == codes.shape[0]
    d1, i1 = B.ivfpq_search(one, _t(q), 5, 20)
    d3, i3 = B.ivfpq_search(three, _t(q), 5, 20)
    torch.cuda.synchronize()
    # identical list contents in identical order: identical results
    assert torch.equal(d1, d3) and torch.equal(i1, i3)
    lists = oracle.to_lists(codes, list_ids, ids, w.nlist)
    search_and_check(B, three, data.cent, data.cb, lists, q, 5, 20, context="pieces")


def test_preassigned_probes_with_repeats(B):
    import torch
    w = S.IVFPQWorkload("t", 55, 8_000, 48, 32, 16, 0.15, False, 12, (4,), (15,), ("fp32",))
    data = S.compressed_index(w)
    q = S.queries(w.number, data.cent, data.weights, w.sigma, w.nq)
    ix = make_index(B, data.cent, data.cb, data.codes, data.list_ids, data.ids)
    rng = np.random.default_rng(3)
    probes = rng.integers(0, w.nlist, (w.nq, 4)).astype(np.int32)
    probes[:, 3] = probes[:, 0]  # a list given twice contributes twice
    gd, gi = B.ivfpq_search_preassigned(ix, _t(q), _t(probes), 40)
    torch.cuda.synchronize()
    od, oi, _ = oracle.ivfpq_search(q, data.cent, data.cb, data.list_off, data.codes, data.ids,
                                    4, 40, forced_probes=probes)
    g = gd.cpu().numpy()
    assert np.all(np.abs(g - od) <= tol(od))


@pytest.mark.parametrize("k,blocks", [(100, (0, 16, 32)), (200, (0, 16, 32, 48)), (40, (16, 48)),
                                      (1000, (0, 16, 32, 48, 64)), (2000, (0, 16, 32))])
def test_results_concentrated_in_one_warp_are_repaired(B, k, blocks):
    """The list scan's per-warp queues are shorter than k (each warp of the
    register-codebook kernel takes code blocks b = w mod 16 of every list).
    Here the best vectors of the one probed list all sit in blocks that one
    warp scans, more of them than its queue holds: the merge must detect it
    and the query must be scanned again with full-length queues."""
    import torch
    rng = np.random.default_rng(k)
    nlist, m, dsub, n = 4, 32, 3, 4096
    d = m * dsub
    cent = rng.standard_normal((nlist, d)).astype(np.float32)
    cb = (0.3 * rng.standard_normal((m, 256, dsub))).astype(np.float32)
    q = (cent[[0, 0, 1]] + 0.2 * rng.standard_normal((3, d))).astype(np.float32)
    T = oracle.lut(q[0].astype(np.float64) - cent[0], cb)
    order = np.argsort(T, axis=1)
    codes = rng.integers(0, 256, (n, m)).astype(np.uint8)
    for b in blocks:
        for i in range(32 * b, 32 * b + 32):
            c = order[:, 0].copy()
            j = rng.integers(0, m)
            c[j] = order[j, rng.integers(1, 4)]
            codes[i] = c
    list_ids = np.zeros(n, np.int32)
    list_ids[-100:] = 1
    ids = np.arange(n, dtype=np.int64) * 7 + 3
    ix = make_index(B, cent, cb, codes, list_ids, ids)
    probes = np.array([[0], [0], [1]], np.int32)
    gd, gi = B.ivfpq_search_preassigned(ix, _t(q), _t(probes), k)
    torch.cuda.synchronize()
    off, codes_l, ids_l = oracle.to_lists(codes, list_ids, ids, nlist)
    od, oi, _ = oracle.ivfpq_search(q, cent, cb, off, codes_l, ids_l, 1, k + 64,
                                    forced_probes=probes)
    compare_knn(gd.cpu().numpy(), gi.cpu().numpy(), od, oi, context="warp repair")


def test_all_lists_on_exactly_encoded_set_matches_flat(B):
    """Vectors built as centroid + codewords: IVF-PQ with nprobe = nlist and
    flat k-NN on the decoded vectors agree (two different GPU paths)."""
    import torch
    rng = np.random.default_rng(12)
    nlist, d, m, n = 16, 32, 8, 6000
    cent = (rng.integers(-8, 9, (nlist, d)) / 4.0).astype(np.float32)
    cb = (rng.integers(-8, 9, (m, 256, d // m)) / 16.0).astype(np.float32)
    list_ids = rng.integers(0, nlist, n).astype(np.int32)
    codes = rng.integers(0, 256, (n, m)).astype(np.uint8)
    x = (cent[list_ids] + cb[np.arange(m), codes].reshape(n, d)).astype(np.float32)
    q = (rng.integers(-16, 17, (25, d)) / 8.0).astype(np.float32)
    ids = np.arange(n, dtype=np.int64)
    ix = make_index(B, cent, cb, codes, list_ids, ids)
    gd, gi = B.ivfpq_search(ix, _t(q), nlist, 50)
    fd, fi = B.flat_knn(_t(x), _t(q), 50)
    torch.cuda.synchronize()
    od, oi = oracle.flat_knn(x, q, 50 + 64)
    compare_knn(gd.cpu().numpy(), gi.cpu().numpy(), od, oi, context="ivf all lists")
    compare_knn(fd.cpu().numpy(), fi.cpu().numpy(), od, oi, context="flat")


def test_empty_index_and_single_query(B):
    import torch
    w = S.IVFPQ_LARGE
    data = S.compressed_index(w, n=0, nlist=8)
    ix = B.ivfpq_index_create(_t(data.cent), _t(data.cb))
    q = S.queries(w.number, data.cent, data.weights, w.sigma, 1)
    gd, gi = B.ivfpq_search(ix, _t(q), 2, 7)
    torch.cuda.synchronize()
    assert np.isinf(gd.cpu().numpy()).all() and (gi.cpu().numpy() == -1).all()


def test_bad_list_ids_leave_index_unchanged(B):
    w = S.IVFPQ_LARGE
    data = S.compressed_index(w, n=1000, nlist=8)
    ix = make_index(B, data.cent, data.cb, data.codes, data.list_ids, data.ids)
    bad = data.list_ids.copy()
    bad[17] = 8
    with pytest.raises(B.IVFPQError) as e:
        B.ivfpq_add(ix, _t(data.codes), _t(bad), _t(data.ids))
    assert e.value.status == B.IVFPQ_ERR_INVALID_ARG
    assert ix.ntotal == 1000


# ---------------------------------------------------------------------------
# full-size workloads, sampled queries (the launch configuration the
# benchmark times: all queries in one call)
def _full(B, w, nprobes, ks, nsample):
    """The workload in compressed form (codes and codebooks drawn directly,
    so every input of the oracle comes from the seeded generator)."""
    import torch
    data = S.compressed_index(w)
    q = S.queries(w.number, data.cent, data.weights, w.sigma, w.nq)
    ix = make_index(B, data.cent, data.cb, data.codes, data.list_ids, data.ids)
    lists = (data.list_off, data.codes, data.ids)
    rows = np.random.default_rng(w.number).choice(w.nq, nsample, replace=False)
    for nprobe in nprobes:
        for k in ks:
            search_and_check(B, ix, data.cent, data.cb, lists, q, nprobe, k, rows=rows,
                             context=f"{w.name} compressed nprobe={nprobe} k={k}")
    del ix
    torch.cuda.empty_cache()


@pytest.mark.slow
def test_full_mid_compressed(B):
    _full(B, S.IVFPQ_MID, (16, 64), (100,), 64)


@pytest.mark.slow
def test_full_large_compressed(B):
    _full(B, S.IVFPQ_LARGE, (64,), (100,), 256)


@pytest.mark.slow
def test_full_billion_compressed(B):
    _full(B, S.IVFPQ_BILLION, (128,), (1, 100, 1000), 64)


def _encoded(w):
    import torch
    from approximate_nearest_neighbour_gb300 import indexing
    return indexing.workload_index(w, torch.device("cuda"))


def _check_encoding(B, wi, w, nrows=512):
    """The stored list and code of rows of the built index against the
    oracle's nearest centroid (full sort) and nearest-codeword encoding of the
    same rows, drawn again from the generator."""
    import torch
    rows = np.sort(np.random.default_rng(w.number + 1).choice(S.NOISE_BLOCK, nrows,
                                                               replace=False))
    x = S.device_points(w.number, wi.cent_dev, wi.labels, w.sigma, 0, S.NOISE_BLOCK)[
        torch.as_tensor(rows, device="cuda")].cpu().numpy()
    r_d = torch.as_tensor(rows, device="cuda")
    lists = wi.lists[r_d].cpu().numpy()
    codes = wi.codes[r_d].cpu().numpy()
    ol, _ = oracle.coarse(x, wi.cent, 1)
    assert np.array_equal(lists, ol[:, 0]), f"{w.name}: nearest centroid"
    cb = wi.codebooks.cpu().numpy()
    resid = x.astype(np.float64) - wi.cent[lists].astype(np.float64)
    oc = oracle.pq_encode(resid.astype(np.float32), cb)
    dsub = cb.shape[2]
    for r, j in np.argwhere(oc != codes):
        sub = resid[r, j * dsub:(j + 1) * dsub]
        dg = ((sub - cb[j, codes[r, j]].astype(np.float64)) ** 2).sum()
        do = ((sub - cb[j, oc[r, j]].astype(np.float64)) ** 2).sum()
        assert dg - do <= 1e-5 * max(do, 1e-6), f"{w.name}: code of row {rows[r]}, j={j}"


def _full_encoded(B, wi, w, nprobes, ks, nsample):
    """The workload's index built from raw vectors by the library's training
    and encoding (their own parity is checked in test_index_build_gpu.py and
    by _check_encoding on this index); the search oracle reads the stored
    codes of the probed lists as its input."""
    import torch
    from approximate_nearest_neighbour_gb300 import indexing
    cb = wi.codebooks.cpu().numpy()
    q = S.queries(w.number, wi.cent, wi.weights, w.sigma, w.nq)
    rows = np.random.default_rng(w.number).choice(w.nq, nsample, replace=False)
    gp, _ = B.ivfpq_search_probes(wi.index, _t(q[rows]), max(nprobes), with_dist=False)
    torch.cuda.synchronize()
    codes_h, lists_h, ids_h = indexing.lists_on_host(wi, np.unique(gp.cpu().numpy()))
    lists = oracle.to_lists(codes_h, lists_h, ids_h, wi.cent.shape[0])
    del codes_h, lists_h, ids_h
    B.ivfpq_repaired_queries(wi.index)
    for nprobe in nprobes:
        for k in ks:
            search_and_check(B, wi.index, wi.cent, cb, lists, q, nprobe, k, rows=rows,
                             context=f"{w.name} encoded nprobe={nprobe} k={k}")
            print(f"{w.name} nprobe={nprobe} k={k}: queries re-scanned with full queues "
                  f"{B.ivfpq_repaired_queries(wi.index)} of {w.nq}")


@pytest.mark.slow
def test_full_mid_encoded(B):
    import torch
    w = S.IVFPQ_MID
    wi = _encoded(w)
    assert np.all(np.diff(wi.objective) <= 1e-6 * wi.objective[0])
    _check_encoding(B, wi, w)
    _full_encoded(B, wi, w, (16, 64), (100,), 64)
    del wi
    torch.cuda.empty_cache()


@pytest.fixture(scope="module")
def large_encoded(B):
    import torch
    wi = _encoded(S.IVFPQ_LARGE)
    yield wi
    del wi
    torch.cuda.empty_cache()


@pytest.mark.slow
def test_full_large_encoded(B, large_encoded):
    w = S.IVFPQ_LARGE
    wi = large_encoded
    assert np.all(np.diff(wi.objective) <= 1e-6 * wi.objective[0])
    print(f"{w.name}: rows searched in full by the encoder {wi.searched}")
    _check_encoding(B, wi, w)
    _full_encoded(B, wi, w, (64,), (100,), 256)


@pytest.mark.slow
def test_full_billion_encoded(B):
    import torch
    w = S.IVFPQ_BILLION
    wi = _encoded(w)
    print(f"{w.name}: rows searched in full by the encoder {wi.searched}")
    _check_encoding(B, wi, w)
    _full_encoded(B, wi, w, (128,), (1, 100, 1000), 64)
    del wi
    torch.cuda.empty_cache()


# ---------------------------------------------------------------------------
# reduced-precision lookup tables
def _variant_run(B, data, q, nprobe, k, lut):
    import torch
    ix = make_index(B, data.cent, data.cb, data.codes, data.list_ids, data.ids)
    B.ivfpq_set_lut_type(ix, lut)
    gp, _ = B.ivfpq_search_probes(ix, _t(q), nprobe)
    gd, gi = B.ivfpq_search(ix, _t(q), nprobe, k)
    torch.cuda.synchronize()
    return gp.cpu().numpy(), gd.cpu().numpy(), gi.cpu().numpy()


@pytest.mark.parametrize("lut,rtol,min_recall", [("fp16", 2e-3, 0.99), ("fp8", 3e-2, 0.97)])
@pytest.mark.parametrize("m,dsub", [(32, 3), (8, 12), (16, 4)])
def test_reduced_tables_follow_the_oracle_variant(B, lut, rtol, min_recall, m, dsub):
    """The GPU's binary16 / E4M3 tables against the oracle's tables of the
    same type (encoders written from the formats' definitions): ids agree up
    to rounding-order ties and distances to within the format's precision."""
    w = S.IVFPQWorkload("t", 120 + m, 40_000, m * dsub, 50, m, 0.15, False, 24, (6,), (40,),
                        (lut,))
    data = S.compressed_index(w)
    q = S.queries(w.number, data.cent, data.weights, w.sigma, w.nq)
    gp, gd, gi = _variant_run(B, data, q, 6, 40, lut)
    lt = {"fp16": oracle.LUT_FP16, "fp8": oracle.LUT_FP8}[lut]
    od, oi, _ = oracle.ivfpq_search(q, data.cent, data.cb, data.list_off, data.codes, data.ids,
                                    6, 40, lt, forced_probes=gp)
    assert oracle.recall_at_k(gi, oi) >= min_recall
    assert np.all(np.abs(gd - od) <= rtol * np.abs(od) + 1e-5)


@pytest.mark.slow
@pytest.mark.parametrize("lut,gate", [("fp16", 0.99), ("fp8", 0.95)])
def test_full_large_reduced_table_recall_gates(B, large_encoded, lut, gate):
    """Large workload (2e8 vectors, m = 32, nprobe = 64, k = 100; the index
    built from raw vectors with trained codebooks): recall@100 of the fp16 /
    E4M3 table variants against the fp32 oracle on a seeded sample of 256
    queries (gates: 0.99 and 0.95)."""
    import torch
    from approximate_nearest_neighbour_gb300 import indexing
    w = S.IVFPQ_LARGE
    wi = large_encoded
    q = S.queries(w.number, wi.cent, wi.weights, w.sigma, w.nq)
    B.ivfpq_set_lut_type(wi.index, lut)
    try:
        gp, _ = B.ivfpq_search_probes(wi.index, _t(q), 64, with_dist=False)
        gd, gi = B.ivfpq_search(wi.index, _t(q), 64, 100)
        torch.cuda.synchronize()
    finally:
        B.ivfpq_set_lut_type(wi.index, "fp32")
    gp, gi = gp.cpu().numpy(), gi.cpu().numpy()
    rows = np.random.default_rng(4).choice(w.nq, 256, replace=False)
    codes_h, lists_h, ids_h = indexing.lists_on_host(wi, np.unique(gp[rows]))
    off, codes_l, ids_l = oracle.to_lists(codes_h, lists_h, ids_h, wi.cent.shape[0])
    _, oi, _ = oracle.ivfpq_search(q[rows], wi.cent, wi.codebooks.cpu().numpy(), off, codes_l,
                                   ids_l, 64, 100, forced_probes=gp[rows])
    r = oracle.recall_at_k(gi[rows], oi)
    print(f"{lut} recall@100 vs fp32 oracle = {r:.4f}")
    assert r >= gate


@pytest.mark.parametrize("k", [10, 40])
def test_knn_graph_of_an_exactly_encoded_set(B, k):
    """Vectors built as centroid + codewords, all lists probed: the ADC
    distances are the exact ones, so the k-NN graph (each vector's own id
    removed) is the exact graph of the set."""
    import torch
    rng = np.random.default_rng(60 + k)
    nlist, d, m, n = 12, 32, 8, 3000
    cent = rng.standard_normal((nlist, d)).astype(np.float32)
    cb = (0.5 * rng.standard_normal((m, 256, d // m))).astype(np.float32)
    list_ids = rng.integers(0, nlist, n).astype(np.int32)
    codes = rng.integers(0, 256, (n, m)).astype(np.uint8)
    x = (cent[list_ids] + cb[np.arange(m), codes].reshape(n, d)).astype(np.float32)
    ids = (np.arange(n, dtype=np.int64) * 3 + 1)
    ix = make_index(B, cent, cb, codes, list_ids, ids)
    gd, gi = B.ivfpq_knn_graph(ix, _t(x), _t(ids), nlist, k)
    torch.cuda.synchronize()
    gd, gi = gd.cpu().numpy(), gi.cpu().numpy()
    assert not np.any(gi == ids[:, None]), "a vector is its own neighbour"
    od, oi = oracle.flat_knn(x, x, k + 1 + 64)
    keep = oi != np.arange(n)[:, None]
    od2 = np.stack([od[r][keep[r]][:k + 64] for r in range(n)])
    oi2 = np.stack([ids[oi[r][keep[r]][:k + 64]] for r in range(n)])
    compare_knn(gd, gi, od2, oi2, context="knn graph")
