"""knn_merge (the final k-selection over shards' results) and sharded search
simulated on one GPU: S shards searched one after another, their results
stacked and merged, against the oracle over the whole database."""

import numpy as np
import pytest

import oracle
from approximate_nearest_neighbour_gb300 import sharding
from approximate_nearest_neighbour_gb300 import synthetic as S
from parity import compare_knn, tol

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from approximate_nearest_neighbour_gb300 import binding
    return binding


def _t(x):
    import torch
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


@pytest.mark.parametrize("nshards,nq,kin,k", [(1, 5, 10, 10), (3, 40, 100, 100), (8, 7, 33, 50),
                                              (2, 3, 10, 30), (4, 100, 256, 1024)])
def test_knn_merge_equals_a_sort_of_all_candidates(B, nshards, nq, kin, k):
    """Random shard results with repeated values, +inf padding and -1 ids:
    the merged distances equal the k smallest of all candidates exactly, and
    every returned id belongs to a candidate with that distance."""
    import torch
    rng = np.random.default_rng(nshards * 1000 + k)
    d = rng.integers(0, 50, (nshards, nq, kin)).astype(np.float32) / 4
    ids = rng.integers(0, 1 << 40, (nshards, nq, kin)).astype(np.int64)
    pad = rng.random((nshards, nq, kin)) < 0.1
    d[pad] = np.inf
    ids[pad] = -1
    gd, gi = B.knn_merge(_t(d), _t(ids), k)
    torch.cuda.synchronize()
    gd, gi = gd.cpu().numpy(), gi.cpu().numpy()
    allc = d.transpose(1, 0, 2).reshape(nq, -1)
    alli = ids.transpose(1, 0, 2).reshape(nq, -1)
    for r in range(nq):
        want = np.sort(allc[r])[:k]
        got = gd[r]
        assert np.array_equal(got[:len(want)], want)
        assert np.all(np.isinf(got[len(want):])) and np.all(gi[r, len(want):] == -1)
        pairs = set(zip(allc[r].tolist(), alli[r].tolist()))
        for v, i in zip(got[:len(want)].tolist(), gi[r, :len(want)].tolist()):
            assert (v, i) in pairs
        real = gi[r][gi[r] >= 0]
        assert len(real) == len(set(real.tolist())), "a candidate returned twice"


def test_knn_merge_rejects_bad_arguments(B):
    import torch
    d = torch.zeros((2, 3, 4), device="cuda")
    i = torch.zeros((2, 3, 4), dtype=torch.int64, device="cuda")
    with pytest.raises(B.IVFPQError):
        B.knn_merge(d, i, 0)
    with pytest.raises(B.IVFPQError):
        B.knn_merge(d, i, 4096)


@pytest.mark.parametrize("nshards,k", [(3, 100), (4, 1), (2, 1024)])
def test_sharded_flat_knn_equals_the_whole_database(B, nshards, k):
    import torch
    db, q = S.flat_database(S.FLAT_1M, n=30_000, nq=50)
    ds, is_ = [], []
    for s in range(nshards):
        a, b = sharding.shard_range(db.shape[0], nshards, s)
        d, i = B.flat_knn(_t(db[a:b]), _t(q), k)
        ds.append(d)
        is_.append(sharding.globalize_ids(i, a))
    gd, gi = sharding.merge_results(torch.stack(ds), torch.stack(is_), k)
    torch.cuda.synchronize()
    od, oi = oracle.flat_knn(db, q, k + 64)
    compare_knn(gd.cpu().numpy(), gi.cpu().numpy(), od, oi, context="sharded flat")


def test_sharded_ivfpq_equals_the_unsharded_index(B):
    """The vectors split over 3 indexes with the same centroids and
    codebooks: each shard probes the same lists, so the merged result is the
    unsharded one (compared with the oracle on the GPU's probes)."""
    import torch
    w = S.IVFPQWorkload("t", 77, 30_000, 32, 64, 8, 0.15, False, 20, (8,), (25,), ("fp32",))
    data = S.compressed_index(w)
    q = S.queries(w.number, data.cent, data.weights, w.sigma, w.nq)
    n = data.codes.shape[0]
    nprobe, k = 8, 25
    ds, is_ = [], []
    probes = None
    for s in range(3):
        a, b = sharding.shard_range(n, 3, s)
        ix = B.ivfpq_index_create(_t(data.cent), _t(data.cb))
        B.ivfpq_add(ix, _t(data.codes[a:b]), _t(data.list_ids[a:b]), _t(data.ids[a:b]))
        if probes is None:
            probes, _ = B.ivfpq_search_probes(ix, _t(q), nprobe)
        d, i = B.ivfpq_search(ix, _t(q), nprobe, k)
        ds.append(d)
        is_.append(i)
    gd, gi = sharding.merge_results(torch.stack(ds), torch.stack(is_), k)
    torch.cuda.synchronize()
    off, codes_l, ids_l = oracle.to_lists(data.codes, data.list_ids, data.ids, w.nlist)
    od, oi, _ = oracle.ivfpq_search(q, data.cent, data.cb, off, codes_l, ids_l, nprobe, k + 64,
                                    forced_probes=probes.cpu().numpy())
    compare_knn(gd.cpu().numpy(), gi.cpu().numpy(), od, oi, context="sharded ivfpq")
