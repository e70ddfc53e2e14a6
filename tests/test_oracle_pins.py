"""Pins for the CPU oracle (no GPU).

Each test checks the oracle against something other than itself: the values
the pages print for a worked example (tests/golden), exact arithmetic on
dyadic inputs, closed-form identities, library routines (numpy, scipy, torch
CPU casts) for special cases, and the 0-1 principle for sorting networks.
"""

import math
import os

import numpy as np
import pytest
import scipy.spatial.distance as ssd
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


def _golden_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append([int(x) for x in line.split()])
    return rows


# --------------------------------------------------------------------------
# number formats
def test_f16_encode_matches_numpy_round_to_nearest_even():
    g = _rng(1)
    vals = list(g.standard_normal(4000) * 10.0 ** g.uniform(-9, 5, 4000))
    one = 1.0
    vals += [one + 2 ** -11, one + 3 * 2 ** -11, 2 ** -25, 3 * 2 ** -25, 2 ** -24, 65504.0,
             65519.0, 65520.0, 1e6, -0.0, 0.0, 2 ** -14 - 2 ** -25, -(2 ** -14) + 2 ** -26]
    for v in vals:
        assert oracle.f16_encode(v) == int(np.float16(np.float64(v)).view(np.uint16)), v


def test_f16_decode_all_codes():
    codes = np.arange(65536, dtype=np.uint16)
    ref = codes.view(np.float16).astype(np.float64)
    for h in range(0, 65536, 7):
        got = oracle.f16_decode(h)
        if math.isnan(ref[h]):
            assert math.isnan(got)
        else:
            assert got == ref[h], h


def test_e4m3_decode_all_codes_matches_torch_and_definition():
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for b in range(256):
        got = oracle.e4m3_decode(b)
        if math.isnan(ref[b]):
            assert math.isnan(got), b
        else:
            assert got == ref[b], b
    # the format's defining values
    assert oracle.e4m3_decode(0x7E) == 448.0
    assert oracle.e4m3_decode(0x01) == 2.0 ** -9
    assert oracle.e4m3_decode(0x08) == 2.0 ** -6
    assert math.isnan(oracle.e4m3_decode(0x7F))


def test_e4m3_encode_matches_torch_cast():
    codes = torch.arange(0, 0x7F, dtype=torch.uint8)
    vals = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    mids = (vals[1:] + vals[:-1]) / 2  # exact ties
    g = _rng(2)
    rand = g.uniform(0, 448, 5000)
    tiny = g.uniform(0, 2 ** -5, 2000)
    allv = np.concatenate([vals, mids, rand, tiny, -rand[:500], -mids]).astype(np.float32)
    ref = torch.from_numpy(allv).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    for v, r in zip(allv, ref):
        assert oracle.e4m3_encode(float(v)) == int(r), float(v)
    # saturation of finite overflow (stated behaviour of the encoder)
    assert oracle.e4m3_encode(1000.0) == 0x7E
    assert oracle.e4m3_encode(-1e9) == 0xFE


# --------------------------------------------------------------------------
# lookup table and ADC
@pytest.mark.parametrize("d,m", [(24, 8), (96, 32), (128, 16), (64, 8), (96, 8)])
def test_adc_equals_squared_distance_to_decoded_residual(d, m):
    """Eq. (1) of the 8-bit-float page: sum_j F(y_j) is the squared L2 norm of
    the residual difference."""
    g = _rng(d * 100 + m)
    cb = (g.standard_normal((m, 256, d // m)) * 0.3).astype(np.float32)
    for _ in range(20):
        r = g.standard_normal(d) * 0.5
        code = g.integers(0, 256, m).astype(np.uint8)
        T = oracle.lut(r, cb)
        decoded = cb[np.arange(m), code].reshape(-1).astype(np.float64)
        ref = float(np.linalg.norm(r - decoded)) ** 2
        assert abs(oracle.adc(T, code) - ref) <= 1e-12 * ref


def test_quantized_lut_fp16_is_binary16_round_trip():
    g = _rng(3)
    T = g.uniform(0, 10, (16, 256))
    Q = oracle.quantize_lut(T, oracle.LUT_FP16)
    ref = T.astype(np.float16).astype(np.float64)
    assert np.array_equal(Q, ref)


def test_quantized_lut_fp8_scale_and_rounding():
    g = _rng(4)
    T = g.uniform(0, 448, (8, 256)).astype(np.float32).astype(np.float64)
    T[3, 17] = 448.0  # scale s = max / 448 = 1, so T / s is exact
    Q = oracle.quantize_lut(T, oracle.LUT_FP8)
    ref = torch.from_numpy(T.astype(np.float32)).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(Q, ref)
    assert Q[3, 17] == 448.0
    normal = T >= 2 ** -6
    assert np.all(np.abs(Q - T)[normal] <= 2 ** -4 * T[normal])


@pytest.mark.parametrize("top", [3.7, 0.01 * 448, 37 * 448, 2.0 ** -3])
def test_quantized_lut_fp8_applies_one_scale_per_table_set(top):
    """Tables whose largest entry is not 448: s = max T / 448, every entry is
    stored as E4M3(T / s) and read back times s (one fp32 scale per table
    set). The expected values go through torch's float8_e4m3fn cast of T / s,
    so an oracle that stored T * s, or did not multiply back, fails."""
    g = _rng(int(top * 1000) % 997)
    T = g.uniform(0, 1, (32, 256)) * top
    T[5, 200] = top  # the maximum
    T[0, 0] = 0.0
    s = top / 448.0
    ref = torch.from_numpy(T / s).to(torch.float8_e4m3fn).to(torch.float64).numpy() * s
    Q = oracle.quantize_lut(T, oracle.LUT_FP8)
    assert np.array_equal(Q, ref)
    assert Q[5, 200] == top and Q[0, 0] == 0.0
    # relative rounding of E4M3 normals is at most 2^-4
    normal = T / s >= 2 ** -6
    assert np.all(np.abs(Q - T)[normal] <= 2 ** -4 * T[normal])
    assert not np.array_equal(Q, T)


def test_quantized_lut_fp8_all_zero_table_is_unchanged():
    T = np.zeros((8, 256))
    assert np.array_equal(oracle.quantize_lut(T, oracle.LUT_FP8), T)


# --------------------------------------------------------------------------
# IVF-PQ end to end on exactly representable data
def _dyadic_index(seed, nlist, d, m, n, nq):
    g = _rng(seed)
    cent = (g.integers(-8, 9, (nlist, d)) / 4.0).astype(np.float32)
    cb = (g.integers(-8, 9, (m, 256, d // m)) / 16.0).astype(np.float32)
    list_ids = g.integers(0, nlist, n).astype(np.int32)
    codes = g.integers(0, 256, (n, m)).astype(np.uint8)
    x = cent[list_ids] + cb[np.arange(m), codes].reshape(n, d)
    q = (g.integers(-16, 17, (nq, d)) / 8.0).astype(np.float32)
    return cent, cb, list_ids, codes, x.astype(np.float32), q


@pytest.mark.parametrize("k", [1, 10, 37, 600])
def test_ivfpq_all_lists_equals_flat_knn_on_exactly_encoded_set(k):
    """Vectors built as centroid + concatenated codewords are encoded exactly,
    so IVF-PQ with nprobe = nlist must equal brute-force search."""
    nlist, d, m, n = 4, 8, 4, 500
    cent, cb, list_ids, codes, x, q = _dyadic_index(5, nlist, d, m, n, 7)
    ids = np.arange(n, dtype=np.int64)
    off, codes_l, ids_l = oracle.to_lists(codes, list_ids, ids, nlist)
    dI, iI, _ = oracle.ivfpq_search(q, cent, cb, off, codes_l, ids_l, nlist, k)
    dF, iF = oracle.flat_knn(x, q, k)
    assert np.array_equal(iI, iF)
    assert np.array_equal(dI, dF)
    if k > n:
        assert np.all(iI[:, n:] == -1) and np.all(np.isinf(dI[:, n:]))


def test_ivfpq_some_lists_equals_restricted_brute_force():
    nlist, d, m, n, nprobe, k = 16, 12, 4, 2000, 5, 25
    cent, cb, list_ids, codes, x, q = _dyadic_index(6, nlist, d, m, n, 9)
    ids = np.arange(n, dtype=np.int64) * 3 + 11  # user ids differ from rows
    off, codes_l, ids_l = oracle.to_lists(codes, list_ids, ids, nlist)
    dI, iI, probes = oracle.ivfpq_search(q, cent, cb, off, codes_l, ids_l, nprobe, k)
    # probes: exact distances (dyadic, so exact in double), ties to lower id
    dc = ssd.cdist(q.astype(np.float64), cent.astype(np.float64), "sqeuclidean")
    for i in range(q.shape[0]):
        order = np.lexsort((np.arange(nlist), dc[i]))
        assert np.array_equal(probes[i], order[:nprobe])
        sel = np.isin(list_ids, probes[i])
        dx = ssd.cdist(q[i:i + 1].astype(np.float64), x[sel].astype(np.float64), "sqeuclidean")[0]
        uid = ids[sel]
        o = np.lexsort((uid, dx))[:k]
        assert np.array_equal(iI[i], uid[o])
        assert np.array_equal(dI[i], dx[o])


def test_ivfpq_forced_probes_are_used():
    nlist, d, m, n = 8, 8, 2, 400
    cent, cb, list_ids, codes, x, q = _dyadic_index(7, nlist, d, m, n, 4)
    ids = np.arange(n, dtype=np.int64)
    off, codes_l, ids_l = oracle.to_lists(codes, list_ids, ids, nlist)
    forced = np.tile(np.array([[6, 1]], np.int32), (q.shape[0], 1))
    _, iI, probes = oracle.ivfpq_search(q, cent, cb, off, codes_l, ids_l, 2, n, forced_probes=forced)
    assert np.array_equal(probes, forced)
    for row in iI:
        got = set(row[row >= 0].tolist())
        assert got == set(np.nonzero(np.isin(list_ids, [6, 1]))[0].tolist())


# --------------------------------------------------------------------------
# coarse quantizer
def test_coarse_distances_match_expanded_form_and_argmin():
    g = _rng(8)
    q = g.standard_normal((50, 96)).astype(np.float32)
    cent = g.standard_normal((300, 96)).astype(np.float32)
    lists, dist = oracle.coarse(q, cent, 300)
    q64, c64 = q.astype(np.float64), cent.astype(np.float64)
    expanded = (q64 * q64).sum(1)[:, None] - 2 * q64 @ c64.T + (c64 * c64).sum(1)[None, :]
    got = np.take_along_axis(expanded, lists.astype(np.int64), 1)
    assert np.allclose(dist, got, rtol=1e-10, atol=1e-10)
    assert np.all(np.diff(dist, axis=1) >= 0)
    assert np.array_equal(lists[:, 0], ssd.cdist(q64, c64, "sqeuclidean").argmin(1))
    for row in lists:
        assert sorted(row.tolist()) == list(range(300))


# --------------------------------------------------------------------------
# flat k-NN and k-selection
def test_flat_knn_matches_cdist_with_index_tie_break():
    g = _rng(9)
    db = (g.integers(-6, 7, (700, 16)) / 4.0).astype(np.float32)
    q = (g.integers(-6, 7, (11, 16)) / 4.0).astype(np.float32)
    for k in (1, 50, 700, 900):
        dF, iF = oracle.flat_knn(db, q, k)
        dd = ssd.cdist(q.astype(np.float64), db.astype(np.float64), "sqeuclidean")
        o = np.argsort(dd, axis=1, kind="stable")[:, :k]
        kk = min(k, 700)
        assert np.array_equal(iF[:, :kk], o[:, :kk])
        assert np.array_equal(dF[:, :kk], np.take_along_axis(dd, o, 1)[:, :kk])
        assert np.all(iF[:, kk:] == -1)


@pytest.mark.parametrize("kind", ["normal", "ties", "equal", "sorted", "reverse", "inf"])
@pytest.mark.parametrize("k", [1, 33, 200, 256, 300])
def test_kselect_equals_stable_full_sort(kind, k):
    from approximate_nearest_neighbour_gb300 import synthetic
    vals = synthetic.random_rows(6, 256, seed=k, kind=kind)
    ov, oi = oracle.kselect(vals, k)
    o = np.argsort(vals, axis=1, kind="stable")
    kk = min(k, 256)
    assert np.array_equal(oi[:, :kk], o[:, :kk])
    assert np.array_equal(ov[:, :kk], np.take_along_axis(vals, o, 1)[:, :kk])
    assert np.all(oi[:, kk:] == -1) and np.all(np.isposinf(ov[:, kk:]))


# --------------------------------------------------------------------------
# sorting networks (Algorithms 1 and 2)
def _apply(net, X):
    X = X.copy()
    for lo, hi, _ in net:
        a, b = X[:, lo].copy(), X[:, hi].copy()
        X[:, lo] = np.minimum(a, b)
        X[:, hi] = np.maximum(a, b)
    return X


def _steps_disjoint(net):
    by_step = {}
    for lo, hi, s in net:
        used = by_step.setdefault(s, set())
        assert lo not in used and hi not in used
        used.update((lo, hi))
        assert lo < hi


def test_odd_merge_golden_example():
    for lL, lR, steps in _golden_rows("odd_merge_steps.txt"):
        _, s = oracle.odd_merge_network(lL, lR)
        assert s == steps


@pytest.mark.parametrize("lL", range(1, 13))
def test_odd_merge_network_zero_one_principle(lL):
    for lR in range(1, 13):
        net, steps = oracle.odd_merge_network(lL, lR)
        assert steps == math.ceil(math.log2(max(lL, lR))) + 1
        _steps_disjoint(net)
        # every pair of sorted 0/1 inputs
        rows = []
        for zl in range(lL + 1):
            for zr in range(lR + 1):
                rows.append([0] * zl + [1] * (lL - zl) + [0] * zr + [1] * (lR - zr))
        out = _apply(net, np.array(rows, np.int8))
        assert np.all(np.diff(out, axis=1) >= 0)


@pytest.mark.parametrize("l", list(range(1, 21)))
def test_odd_sort_network_zero_one_principle(l):
    net, steps = oracle.odd_sort_network(l)
    c = math.ceil(math.log2(l)) if l > 1 else 0
    assert steps == (c * c + c) // 2
    _steps_disjoint(net)
    allv = ((np.arange(1 << l)[:, None] >> np.arange(l)[None, :]) & 1).astype(np.int8)
    out = _apply(net, allv)
    assert np.all(np.diff(out, axis=1) >= 0)


def test_odd_sort_network_sorts_random_reals():
    g = _rng(10)
    for l in (64, 96, 128, 256, 320):
        net, _ = oracle.odd_sort_network(l)
        X = g.standard_normal((20, l))
        assert np.array_equal(_apply(net, X), np.sort(X, axis=1))


# --------------------------------------------------------------------------
# WarpSelect (Algorithm 3), simulated on the host with invariant checks
@pytest.mark.parametrize("k", [1, 10, 32, 33, 100])
@pytest.mark.parametrize("t", [1, 2, 4, 8])
def test_warpselect_simulation_invariants_and_result(k, t):
    from approximate_nearest_neighbour_gb300 import synthetic
    for kind, n in (("normal", 700), ("reverse", 300), ("ties", 400), ("inf", 350)):
        vals = synthetic.random_rows(1, n, seed=k * 10 + t, kind=kind)[0]
        st, ov, oi, merges = oracle.warpselect_sim(vals, k, t)
        assert st == 0, (kind, st)
        o = np.argsort(vals, kind="stable")[:k]
        assert np.array_equal(oi[: len(o)], o)
        assert np.array_equal(ov[: len(o)], vals[o])


def test_warpselect_simulation_short_input_pads():
    st, ov, oi, _ = oracle.warpselect_sim(np.array([3.0, 1.0, 2.0], np.float32), 5, 2)
    assert st == 0
    assert oi.tolist() == [1, 2, 0, -1, -1]
    assert np.isinf(ov[3:]).all()


# --------------------------------------------------------------------------
# index-building helpers
def test_pq_training_objective_decreases_and_encoding_is_nearest():
    g = _rng(11)
    x = (g.standard_normal((3000, 8)) * 0.2).astype(np.float32)
    init = g.choice(3000, 256, replace=False)
    cb, obj = oracle.pq_train(x, 2, 10, init)
    assert np.all(np.diff(obj) <= 1e-12 * obj[0])
    codes = oracle.pq_encode(x, cb)
    for j in range(2):
        dd = ssd.cdist(x[:, 4 * j:4 * j + 4].astype(np.float64), cb[j].astype(np.float64),
                       "sqeuclidean")
        assert np.array_equal(codes[:, j], dd.argmin(1))
    decoded = cb[np.arange(2), codes].reshape(3000, 8).astype(np.float64)
    err = ((x.astype(np.float64) - decoded) ** 2).sum()
    assert abs(err - obj[-1]) <= 1e-9 * err


def test_one_lloyd_pass_is_the_mean_of_the_nearest_points():
    """Closed form of one Lloyd pass ([BSS] section 6: assignment, then
    update): each codeword becomes the mean of the points whose nearest seed
    it is (brute force, lowest index on ties), a seed nobody chose stays, and
    the first objective is the sum of the squared distances to the nearest
    seed."""
    g = _rng(12)
    m, dsub, n = 2, 3, 2000
    x = g.standard_normal((n, m * dsub)).astype(np.float32)
    init = g.choice(n, 256, replace=False)
    # two seeds on the same point: the higher-indexed one stays empty
    init[7] = init[3]
    cb, obj = oracle.pq_train(x, m, 1, init)
    x64 = x.astype(np.float64)
    total = 0.0
    for j in range(m):
        sub = x64[:, j * dsub:(j + 1) * dsub]
        seeds = sub[init]
        dd = ssd.cdist(sub, seeds, "sqeuclidean")
        a = dd.argmin(1)
        total += dd[np.arange(n), a].sum()
        for c in range(256):
            pts = sub[a == c]
            want = pts.mean(0) if len(pts) else seeds[c]
            assert np.allclose(cb[j, c], want, rtol=1e-6, atol=1e-6), (j, c)
        assert not (a == 7).any()
        assert np.array_equal(cb[j, 7], x[init[7], j * dsub:(j + 1) * dsub])
    assert abs(obj[0] - total) <= 1e-9 * total


def test_recall_definition():
    assert oracle.recall_at_k(np.array([[1, 2, 3]]), np.array([[3, 2, 9]])) == pytest.approx(2 / 3)
