"""Sharded search across processes: each rank holds a part of the database,
answers every query, and one more k-selection over the ranks' results gives
the answer of the whole database.

Source: multi-GPU sharding ("Billion-scale similarity search with GPUs",
section 5: the database is split across GPUs, each GPU processes all queries,
and the partial results are combined by an additional round of k-selection).

Only the exchange is here (torch.distributed: gloo on CPU tensors, NCCL on
device tensors); the merge itself is the library's knn_merge kernel.
"""

from . import binding


def shard_range(n, nshards, shard):
    """[start, end) of the database rows held by `shard` of `nshards`:
    contiguous, sizes differing by at most one."""
    if nshards < 1 or not 0 <= shard < nshards:
        raise ValueError(f"shard {shard} of {nshards}")
    if n < 0:
        raise ValueError(f"n = {n}")
    base, extra = divmod(n, nshards)
    start = shard * base + min(shard, extra)
    return start, start + base + (1 if shard < extra else 0)


def globalize_ids(ids, start):
    """Row indices local to a shard -> global row indices (missing entries,
    -1, stay -1). Returns a new tensor."""
    return ids.where(ids < 0, ids + start)


def gather_results(dist, ids, group=None):
    """All ranks' [nq, k] results stacked as [world, nq, k] (rank order), on
    every rank. Every rank must pass the same nq and k."""
    import torch
    import torch.distributed as dist_

    world = dist_.get_world_size(group)
    ds = [torch.empty_like(dist) for _ in range(world)]
    is_ = [torch.empty_like(ids) for _ in range(world)]
    dist_.all_gather(ds, dist.contiguous(), group=group)
    dist_.all_gather(is_, ids.contiguous(), group=group)
    return torch.stack(ds), torch.stack(is_)


def merge_results(dists, ids, k, stream=None):
    """k best of [S, nq, k_in] stacked shard results (device tensors):
    ([nq, k] distances ascending, [nq, k] ids)."""
    return binding.knn_merge(dists.contiguous(), ids.contiguous(), k, stream=stream)


def sharded_search(index, queries, nprobe, k, group=None):
    """IVF-PQ search of this rank's index shard (built with global ids) for
    all queries, exchanged with the other ranks and merged: every rank gets
    the result of the whole database."""
    d, i = binding.ivfpq_search(index, queries, nprobe, k)
    sd, si = gather_results(d, i, group)
    return merge_results(sd, si, k)


def sharded_flat_knn(db_shard, start, queries, k, group=None):
    """Exact k-NN over a database split by shard_range: this rank holds rows
    [start, start + len(db_shard)); every rank gets the global result."""
    d, i = binding.flat_knn(db_shard, queries, k)
    sd, si = gather_results(d, globalize_ids(i, start), group)
    return merge_results(sd, si, k)
