"""Index preparation on the GPU (kmeans_lloyd, pq_train, ivfpq_encode)
against the oracle's Lloyd training and encoder (pq_train with m = 1 is plain
k-means with 256 centroids)."""

import numpy as np
import pytest

import oracle
from approximate_nearest_neighbour_gb300 import synthetic as S

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from approximate_nearest_neighbour_gb300 import binding
    return binding


def _t(x):
    import torch
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def _data(n, d, seed):
    rng = np.random.default_rng(seed)
    centres = rng.standard_normal((40, d)).astype(np.float32)
    x = centres[rng.integers(0, 40, n)] + 0.3 * rng.standard_normal((n, d)).astype(np.float32)
    init = rng.choice(n, 256, replace=False).astype(np.int64)
    return x.astype(np.float32), init


def _sq(a, b):
    return ((a.astype(np.float64)[:, None, :] - b.astype(np.float64)[None, :, :]) ** 2).sum(-1)


@pytest.mark.parametrize("m,d", [(1, 16), (4, 32), (8, 24)])
def test_pq_train_follows_the_oracle(B, m, d):
    """Same seeds, same passes: the first objective is the same sum, the
    objective never increases, and after one update the codebooks agree
    (apart from points exactly between two codewords)."""
    import torch
    x, init = _data(12_000, d, 7 + m)
    cb1, obj1 = B.pq_train(_t(x), m, 1, _t(init))
    ocb1, oobj1 = oracle.pq_train(x, m, 1, init)
    torch.cuda.synchronize()
    assert abs(obj1[0] - oobj1[0]) <= 1e-6 * oobj1[0]
    diff = np.abs(cb1.cpu().numpy() - ocb1)
    close = (diff <= 1e-5 * (1 + np.abs(ocb1))).all(axis=-1)
    assert close.mean() >= 0.99, close.mean()
    cb, obj = B.pq_train(_t(x), m, 8, _t(init))
    _, oobj = oracle.pq_train(x, m, 8, init)
    assert np.all(np.diff(obj) <= 1e-6 * obj[0]), obj
    assert abs(obj[-1] - oobj[-1]) <= 1e-3 * oobj[-1]


def test_kmeans_lloyd_is_pq_train_with_one_subspace(B):
    import torch
    x, init = _data(10_000, 20, 3)
    cent, assign, obj = B.kmeans_lloyd(_t(x), _t(init), 5)
    _, oobj = oracle.pq_train(x, 1, 5, init)
    torch.cuda.synchronize()
    assert abs(obj[0] - oobj[0]) <= 1e-6 * oobj[0]
    assert abs(obj[-1] - oobj[-1]) <= 1e-3 * oobj[-1]
    # the returned assignment is the nearest trained centroid
    c = cent.cpu().numpy()
    a = assign.cpu().numpy()
    dd = _sq(x[:2000], c)
    best = dd.min(1)
    got = dd[np.arange(2000), a[:2000]]
    assert np.all(got <= best + 1e-4 * best + 1e-5)
    assert abs(obj[-1] - _sq(x, c).min(1).sum()) <= 1e-4 * obj[-1]


def test_kmeans_empty_cluster_keeps_its_centroid(B):
    """Two seeds on the same point: in the first pass all its points go to
    one of them (ties), so after one update the other, empty cluster still
    holds its seed."""
    import torch
    x, _ = _data(3000, 8, 11)
    init = np.array([5, 5, 17, 400, 999], np.int64)
    _, a0, _ = B.kmeans_lloyd(_t(x), _t(init), 0)
    cent, _, _ = B.kmeans_lloyd(_t(x), _t(init), 1)
    torch.cuda.synchronize()
    counts = np.bincount(a0.cpu().numpy(), minlength=5)
    assert (counts[0] == 0) != (counts[1] == 0), counts
    empty = 0 if counts[0] == 0 else 1
    assert np.array_equal(cent.cpu().numpy()[empty], x[5])


def test_bad_seed_index_is_rejected(B):
    x, _ = _data(1000, 8, 1)
    with pytest.raises(B.IVFPQError) as e:
        B.kmeans_lloyd(_t(x), _t(np.array([0, 1000], np.int64)), 1)
    assert e.value.status == B.IVFPQ_ERR_INVALID_ARG


def test_encode_then_add_then_search(B):
    """Tiny workload: the GPU encoder's lists and codes equal the oracle's
    nearest centroid and nearest codewords (up to exact ties), and an index
    filled from them searches like the oracle."""
    import torch
    from parity import compare_knn
    w = S.IVFPQ_TINY
    cent, x, init = S.tiny_raw(w)
    a_all, _ = oracle.coarse(x, cent, 1)
    cb, _ = oracle.pq_train(x - cent[a_all[:, 0]], w.m, 4, init)
    x = x[:20_000]
    assign = a_all[:20_000]
    ix = B.ivfpq_index_create(_t(cent), _t(cb))
    lists, codes = B.ivfpq_encode(ix, _t(x))
    torch.cuda.synchronize()
    gl, gc = lists.cpu().numpy(), codes.cpu().numpy()
    dc = _sq(x, cent)
    rows = np.arange(x.shape[0])
    assert np.all(dc[rows, gl] <= dc[rows, assign[:, 0]] * (1 + 1e-5) + 1e-6)
    same = gl == assign[:, 0]
    oc = oracle.pq_encode(x[same] - cent[gl[same]], cb)
    r = (x[same] - cent[gl[same]]).reshape(-1, w.m, w.d // w.m).astype(np.float64)
    dg = ((r - cb[np.arange(w.m), gc[same]]) ** 2).sum(-1)
    do = ((r - cb[np.arange(w.m), oc]) ** 2).sum(-1)
    assert np.all(dg <= do * (1 + 1e-5) + 1e-6)
    assert (gc[same] == oc).mean() > 0.999
    ids = np.arange(x.shape[0], dtype=np.int64)
    B.ivfpq_add(ix, codes, lists, _t(ids))
    q = S.queries(w.number, cent, S.component_weights(w.nlist, False), w.sigma, 30)
    gd, gi = B.ivfpq_search(ix, _t(q), 8, 10)
    torch.cuda.synchronize()
    off, cl, il = oracle.to_lists(gc, gl, ids, w.nlist)
    gp, _ = B.ivfpq_search_probes(ix, _t(q), 8)
    od, oi, _ = oracle.ivfpq_search(q, cent, cb, off, cl, il, 8, 10 + 64,
                                    forced_probes=gp.cpu().numpy())
    compare_knn(gd.cpu().numpy(), gi.cpu().numpy(), od, oi, context="encode round trip")
