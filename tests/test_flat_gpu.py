"""flat_knn against the oracle's exact search."""

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


def _flat(B, db, q, k):
    import torch
    gd, gi = B.flat_knn(torch.from_numpy(db).cuda(), torch.from_numpy(q).cuda(), k)
    torch.cuda.synchronize()
    return gd.cpu().numpy(), gi.cpu().numpy()


@pytest.mark.parametrize("n,d,nq,k", [(1000, 128, 37, 1), (5000, 128, 64, 100), (3001, 96, 5, 1024),
                                      (257, 64, 130, 300), (100, 16, 3, 2048), (20_000, 128, 300, 10)])
def test_flat_small(B, n, d, nq, k):
    db, q = S.flat_database(S.FLAT_1M, n=n, nq=nq)
    db = db[:, :d].copy()
    q = q[:, :d].copy()
    gd, gi = _flat(B, db, q, k)
    od, oi = oracle.flat_knn(db, q, min(k + 64, max(n, 1)) if k < n else k)
    compare_knn(gd, gi, od, oi, context="flat")


@pytest.mark.parametrize("k", [1, 100, 1024])
def test_flat_full_size_sampled(B, k):
    """The 1M x 128 database with all 10,000 queries on the GPU; a seeded
    sample of queries is checked against the oracle."""
    import torch
    db, q = S.flat_database(S.FLAT_1M)
    gd, gi = _flat(B, db, q, k)
    rows = np.random.default_rng(k).choice(q.shape[0], 6, replace=False)
    od, oi = oracle.flat_knn(db, q[rows], k + 64)
    compare_knn(gd[rows], gi[rows], od, oi, context=f"flat full k={k}")
