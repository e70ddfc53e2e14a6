"""Index preparation on the GPU against the oracle: residuals against the
nearest centroid, the hint-checked encoder, and an index built from raw
mixture vectors (training, encoding, add) searched against the oracle."""

import numpy as np
import pytest

import oracle
from approximate_nearest_neighbour_gb300 import synthetic as S
from parity import compare_knn

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from approximate_nearest_neighbour_gb300 import binding
    return binding


def _t(x):
    import torch
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def _mixture(seed, nlist, d, n, sigma=0.15):
    g = np.random.default_rng(seed)
    cent = g.standard_normal((nlist, d)).astype(np.float32)
    lab = g.integers(0, nlist, n).astype(np.int32)
    x = (cent[lab] + sigma * g.standard_normal((n, d))).astype(np.float32)
    return cent, lab, x


def _check_codes(x, lists, codes, cent, cb, context):
    """codes equal the oracle's nearest-codeword encoding of the residuals
    (fp64), except where two codewords are equally near to within the fp32
    rounding of the GPU's distances."""
    resid = x.astype(np.float64) - cent[lists].astype(np.float64)
    oc = oracle.pq_encode(resid.astype(np.float32), cb)
    m, dsub = cb.shape[0], cb.shape[2]
    diff = np.argwhere(oc != codes)
    for r, j in diff:
        sub = resid[r, j * dsub:(j + 1) * dsub]
        dg = ((sub - cb[j, codes[r, j]].astype(np.float64)) ** 2).sum()
        do = ((sub - cb[j, oc[r, j]].astype(np.float64)) ** 2).sum()
        assert dg - do <= 1e-5 * max(do, 1e-6), f"{context}: row {r} sub-quantizer {j}"
    return len(diff)


def test_residuals_are_against_the_nearest_centroid(B):
    import torch
    cent, _, x = _mixture(1, 300, 48, 5000)
    lists, resid = B.ivfpq_residuals(_t(cent), _t(x))
    torch.cuda.synchronize()
    ol, _ = oracle.coarse(x, cent, 1)
    assert np.array_equal(lists.cpu().numpy(), ol[:, 0])
    # one fp32 subtraction per element: exactly numpy's
    assert np.array_equal(resid.cpu().numpy(), x - cent[ol[:, 0]])


@pytest.mark.parametrize("kind", ["true", "random", "invalid", "midpoints"])
def test_hinted_encoding_equals_the_full_search(B, kind):
    """Whatever the hints, the lists are the nearest centroids and the codes
    those of ivfpq_encode; hints are taken only where the triangle
    inequality proves them, the rest is searched in full."""
    import torch
    nlist, d, m, n = 300, 48, 16, 6000
    cent, lab, x = _mixture(2, nlist, d, n)
    cent[7] = cent[3]  # a duplicated centroid: its separation is 0
    g = np.random.default_rng(3)
    if kind == "midpoints":
        # rows half-way between two centroids (ties or near-ties)
        a = g.integers(0, nlist, 500)
        b = (a + 1 + g.integers(0, nlist - 1, 500)) % nlist
        x[:500] = (0.5 * (cent[a].astype(np.float64) + cent[b])).astype(np.float32)
        lab[:500] = a
    lab[:20] = 3  # rows near the duplicated pair
    x[:20] = cent[3] + 0.01
    hint = {"true": lab, "random": g.integers(0, nlist, n).astype(np.int32),
            "invalid": np.where(g.random(n) < 0.5, -1, nlist + 5).astype(np.int32),
            "midpoints": lab}[kind]
    cb = (0.15 * g.standard_normal((m, 256, d // m))).astype(np.float32)
    ix = B.ivfpq_index_create(_t(cent), _t(cb))
    hl, hc, searched = B.ivfpq_encode_hinted(ix, _t(x), _t(hint))
    fl, fc = B.ivfpq_encode(ix, _t(x))
    torch.cuda.synchronize()
    hl, hc, fl, fc = (t.cpu().numpy() for t in (hl, hc, fl, fc))
    if kind == "true":
        assert 20 <= searched < n // 10
    elif kind == "invalid":
        assert searched == n
    # nearest centroid: the oracle's (full sort, fp64), up to exact ties
    ol, od = oracle.coarse(x, cent, 2)
    for lists in (hl, fl):
        bad = np.nonzero(lists != ol[:, 0])[0]
        for r in bad:
            dr = ((x[r].astype(np.float64) - cent[lists[r]]) ** 2).sum()
            assert dr - od[r, 0] <= 1e-5 * max(od[r, 0], 1e-6), (kind, r)
    same = hl == fl
    assert same.mean() > 0.99
    assert np.array_equal(hc[same], fc[same])
    _check_codes(x, hl, hc, cent, cb, kind)


def test_index_built_from_raw_vectors_follows_the_oracle(B):
    """A scaled-down large workload (2e5 rows, 512 lists, m = 32) built by
    the library's training, hinted encoding and add: the training objective
    does not increase, the stored codes are the oracle's encoding of the
    drawn rows, and searches match the oracle on the built index."""
    import torch
    from approximate_nearest_neighbour_gb300 import indexing
    w = S.IVFPQ_LARGE
    wi = indexing.workload_index(w, torch.device("cuda"), n=200_000, nlist=512)
    assert np.all(np.diff(wi.objective) <= 1e-6 * wi.objective[0])
    assert wi.index.ntotal == 200_000
    assert wi.searched < 2000
    cb = wi.codebooks.cpu().numpy()
    # the stored encoding of 2,000 rows, against the oracle
    rows = np.random.default_rng(5).choice(200_000, 2000, replace=False)
    x = S.device_points(w.number, wi.cent_dev, wi.labels, w.sigma, 0, 200_000)[
        torch.as_tensor(rows, device="cuda")].cpu().numpy()
    lists = wi.lists.cpu().numpy()[rows]
    codes = wi.codes.cpu().numpy()[rows]
    ol, _ = oracle.coarse(x, wi.cent, 1)
    assert np.array_equal(lists, ol[:, 0])
    _check_codes(x, lists, codes, wi.cent, cb, "built index")
    # search parity over the built index
    q = S.queries(w.number, wi.cent, wi.weights, w.sigma, 64)
    gp, _ = B.ivfpq_search_probes(wi.index, _t(q), 16)
    gd, gi = B.ivfpq_search(wi.index, _t(q), 16, 100)
    torch.cuda.synchronize()
    gp = gp.cpu().numpy()
    codes_h, lists_h, ids_h = indexing.lists_on_host(wi, np.unique(gp))
    off, codes_l, ids_l = oracle.to_lists(codes_h, lists_h, ids_h, 512)
    od, oi, _ = oracle.ivfpq_search(q, wi.cent, cb, off, codes_l, ids_l, 16, 164,
                                    forced_probes=gp)
    compare_knn(gd.cpu().numpy(), gi.cpu().numpy(), od, oi, context="built index")


def test_rows_holding_nan_touch_nothing_outside_the_arguments(B):
    """A row holding NaN has no finite distance to any centroid. With 4,096
    centroids the coarse search takes the filtered plan, which keeps no
    candidate for such a row: its list is -1, its residual NaN and its codes
    zero, and ivfpq_add refuses it; the finite rows are unaffected."""
    import torch
    nlist, d, m = 4096, 32, 8
    cent, _, x = _mixture(6, nlist, d, 3000)
    bad = np.array([5, 77, 2999])
    x[bad] = np.nan
    good = np.setdiff1d(np.arange(3000), bad)
    lists, resid = B.ivfpq_residuals(_t(cent), _t(x))
    torch.cuda.synchronize()
    lists, resid = lists.cpu().numpy(), resid.cpu().numpy()
    assert np.all((lists[bad] >= -1) & (lists[bad] < nlist))
    assert np.all(np.isnan(resid[bad]))
    ol, od = oracle.coarse(x[good], cent, 1)
    for i, r in enumerate(good):
        if lists[r] != ol[i, 0]:
            dr = ((x[r].astype(np.float64) - cent[lists[r]]) ** 2).sum()
            assert dr - od[i, 0] <= 1e-5 * max(od[i, 0], 1e-6), r
    assert np.array_equal(resid[good], x[good] - cent[lists[good]])
    cb = (0.15 * np.random.default_rng(7).standard_normal((m, 256, d // m))).astype(np.float32)
    ix = B.ivfpq_index_create(_t(cent), _t(cb))
    el, ec = B.ivfpq_encode(ix, _t(x))
    torch.cuda.synchronize()
    el, ec = el.cpu().numpy(), ec.cpu().numpy()
    assert np.array_equal(el[good], lists[good])
    assert np.all(ec[bad][el[bad] == -1] == 0)
    _check_codes(x[good], el[good], ec[good], cent, cb, "finite rows")
    if np.any(el == -1):
        with pytest.raises(B.IVFPQError):
            B.ivfpq_add(ix, _t(ec), _t(el), _t(np.arange(3000, dtype=np.int64)))
