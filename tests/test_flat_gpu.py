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
                                      (257, 64, 130, 300), (100, 16, 3, 2048), (20_000, 128, 300, 10),
                                      (40_000, 64, 200, 700), (70_000, 32, 20, 2048),
                                      (2_500, 96, 150, 20)])
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
    rows = np.random.default_rng(k).choice(q.shape[0], 64, replace=False)
    od, oi = oracle.flat_knn(db, q[rows], k + 64)
    compare_knn(gd[rows], gi[rows], od, oi, context=f"flat full k={k}")


@pytest.mark.parametrize("k", [10, 64, 300])
def test_flat_filtered_plan_overflow_rows(B, k):
    """The first 4,096 database rows (more than the first pass of the
    filtered plan looks at) lie far from every query, so the bound it takes
    keeps the whole rest of the database: every candidate segment overflows
    and each row is selected over exact distances instead."""
    rng = np.random.default_rng(31 + k)
    n, d, nq = 24_000, 64, 1024
    db = rng.standard_normal((n, d)).astype(np.float32)
    db[:4096] += 40.0
    q = rng.standard_normal((nq, d)).astype(np.float32)
    gd, gi = _flat(B, db, q, k)
    od, oi = oracle.flat_knn(db, q, k + 64)
    compare_knn(gd, gi, od, oi, context="flat overflow")


def test_flat_filtered_plan_some_rows_overflow(B):
    """Half of the queries sit next to a dense cloud of 10,000 points beyond
    the first pass's columns (their candidate segments overflow), the other
    half do not."""
    rng = np.random.default_rng(77)
    n, d, nq, k = 30_000, 32, 1024, 16
    db = rng.standard_normal((n, d)).astype(np.float32) * 3
    db[12_000:22_000] = 0.01 * rng.standard_normal((10_000, d)).astype(np.float32)
    q = rng.standard_normal((nq, d)).astype(np.float32) * 3
    q[::2] = 0.05 * rng.standard_normal((nq // 2, d)).astype(np.float32) + 0.3
    gd, gi = _flat(B, db, q, k)
    od, oi = oracle.flat_knn(db, q, k + 64)
    compare_knn(gd, gi, od, oi, context="flat partial overflow")


def test_flat_all_rows_equal(B):
    """Every database row is the same vector: all distances tie, any k ids
    are a valid answer, and each returned distance is the common value."""
    n, d, nq, k = 20_000, 64, 8, 20
    rng = np.random.default_rng(5)
    v = rng.standard_normal(d).astype(np.float32)
    db = np.tile(v, (n, 1))
    q = rng.standard_normal((nq, d)).astype(np.float32)
    gd, gi = _flat(B, db, q, k)
    od, _ = oracle.flat_knn(db[:1], q, 1)
    assert np.all(np.abs(gd - od[:, :1]) <= 1e-4 * np.abs(od[:, :1]))
    for r in range(nq):
        assert len(set(gi[r].tolist())) == k and gi[r].min() >= 0 and gi[r].max() < n


def test_expired_wait_is_reported_and_the_context_stays_usable(B):
    """A block waits, with a short iteration limit, on a barrier phase that
    nothing completes; device_check reports the expiry once, and the device
    keeps working."""
    import torch
    B.device_check()
    B.selftest_wait_timeout(256)
    with pytest.raises(B.IVFPQError) as e:
        B.device_check()
    assert e.value.status == B.IVFPQ_ERR_TIMEOUT
    B.device_check()  # cleared
    db, q = S.flat_database(S.FLAT_1M, n=2000, nq=4)
    gd, gi = _flat(B, db, q, 5)
    od, oi = oracle.flat_knn(db, q, 5 + 64)
    compare_knn(gd, gi, od, oi, context="after timeout")
    B.device_check()


@pytest.mark.parametrize("k", [300, 1024])
def test_flat_ties_beyond_the_selection_buffer(B, k):
    """2,000 copies of one vector sit next to every query, spread over the
    database: the k nearest all tie, more entries than the radix selection's
    buffer fall under its bound, and those rows are selected again by the
    full-length kernel. Any k of the copies is a valid answer."""
    rng = np.random.default_rng(k)
    n, d, nq = 30_000, 32, 64
    db = 3 * rng.standard_normal((n, d)).astype(np.float32)
    v = rng.standard_normal(d).astype(np.float32)
    db[::15] = v
    q = (v + 0.01 * rng.standard_normal((nq, d))).astype(np.float32)
    gd, gi = _flat(B, db, q, k)
    od, oi = oracle.flat_knn(db, q, 2000 + 64)  # every tied copy is a valid answer
    compare_knn(gd, gi, od, oi, context="flat ties")
    copies = set(range(0, n, 15))
    for r in range(nq):
        assert len(set(gi[r].tolist())) == k and set(gi[r].tolist()) <= copies
