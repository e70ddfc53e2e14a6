"""Host side of sharded search: the row split, the id translation, and the
exchange of the shards' results between two gloo ranks on the CPU. The merge
of the exchanged results is checked here with a plain sort of the gathered
candidates (the device merge, knn_merge, is checked in test_merge_gpu.py)."""

import os
import socket

import numpy as np
import pytest

import oracle
from approximate_nearest_neighbour_gb300 import sharding


@pytest.mark.parametrize("n,S", [(0, 1), (1, 3), (10, 3), (1000, 7), (12, 4)])
def test_shard_range_partitions_the_rows(n, S):
    ranges = [sharding.shard_range(n, S, s) for s in range(S)]
    assert ranges[0][0] == 0 and ranges[-1][1] == n
    for (a0, a1), (b0, b1) in zip(ranges, ranges[1:]):
        assert a1 == b0
    sizes = [b - a for a, b in ranges]
    assert max(sizes) - min(sizes) <= 1 and sum(sizes) == n


def test_shard_range_rejects_bad_arguments():
    with pytest.raises(ValueError):
        sharding.shard_range(10, 0, 0)
    with pytest.raises(ValueError):
        sharding.shard_range(10, 2, 2)


def test_globalize_ids_keeps_missing_entries():
    import torch
    ids = torch.tensor([[0, 5, -1], [2, -1, -1]])
    g = sharding.globalize_ids(ids, 100)
    assert g.tolist() == [[100, 105, -1], [102, -1, -1]]
    assert ids.tolist() == [[0, 5, -1], [2, -1, -1]]


def _merge_cpu(d, i, k):
    """k smallest of [S, nq, k_in] by (distance, id)."""
    S, nq, kin = d.shape
    dd = d.transpose(1, 0, 2).reshape(nq, S * kin)
    ii = i.transpose(1, 0, 2).reshape(nq, S * kin)
    out_d = np.full((nq, k), np.inf)
    out_i = np.full((nq, k), -1, np.int64)
    for r in range(nq):
        order = np.lexsort((ii[r], dd[r]))[:k]
        out_d[r, :len(order)] = dd[r, order]
        out_i[r, :len(order)] = ii[r, order]
    return out_d, out_i


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, db, q, k, outdir):
    import torch
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        start, end = sharding.shard_range(db.shape[0], world, rank)
        d, i = oracle.flat_knn(db[start:end], q, k)
        gi = sharding.globalize_ids(torch.from_numpy(i), start)
        sd, si = sharding.gather_results(torch.from_numpy(d), gi)
        np.save(os.path.join(outdir, f"d{rank}.npy"), sd.numpy())
        np.save(os.path.join(outdir, f"i{rank}.npy"), si.numpy())
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("n,k", [(3001, 10), (50, 40)])
def test_two_gloo_ranks_exchange_and_merge_to_the_full_result(tmp_path, n, k):
    """Two ranks each search half of the database; after the exchange both
    hold the same stacked results, and their merge is the exact result over
    the whole database (including a shard with fewer rows than k)."""
    import torch.multiprocessing as mp
    rng = np.random.default_rng(n)
    db = rng.standard_normal((n, 16)).astype(np.float32)
    q = rng.standard_normal((9, 16)).astype(np.float32)
    world = 2
    mp.spawn(_worker, args=(world, _free_port(), db, q, k, str(tmp_path)), nprocs=world,
             join=True)
    d0, i0 = np.load(tmp_path / "d0.npy"), np.load(tmp_path / "i0.npy")
    d1, i1 = np.load(tmp_path / "d1.npy"), np.load(tmp_path / "i1.npy")
    assert d0.shape == (world, q.shape[0], k)
    assert np.array_equal(d0, d1) and np.array_equal(i0, i1)
    start1, _ = sharding.shard_range(n, world, 1)
    assert np.all(i0[1][i0[1] >= 0] >= start1) and np.all(i0[0] < start1)
    md, mi = _merge_cpu(d0, i0, k)
    od, oi = oracle.flat_knn(db, q, k)
    assert np.array_equal(mi, oi)
    assert np.allclose(md, od, rtol=0, atol=0)
