"""kselect_noalloc: the k-selection entry point for callers that cannot
allocate device memory during a call (for example when another allocator has
reserved the device memory up front). Its results must match kselect's, and
leftovers from an earlier call in its fixed scratch array must not leak into a
later one, so two different problems are run back to back.

This file is collected last on purpose; it also passes when run on its own in
a fresh process.
"""

import numpy as np
import pytest

from approximate_nearest_neighbour_gb300 import synthetic as S

pytestmark = pytest.mark.gpu


def _compare(vals, k, ref_v, ref_i, got_v, got_i):
    # kselect returns exact input values: compare them exactly; indices must
    # hold their values, be distinct, and agree wherever the value is below the
    # k-th (equal values may come in either order)
    assert np.array_equal(got_v, ref_v)
    for r in range(vals.shape[0]):
        assert np.array_equal(vals[r, got_i[r]], got_v[r])
        assert len(set(got_i[r].tolist())) == k
        kth = ref_v[r, -1]
        assert set(got_i[r][got_v[r] < kth].tolist()) == set(ref_i[r][ref_v[r] < kth].tolist())


def test_kselect_noalloc_matches_kselect_on_two_calls_in_a_row():
    """Two different problems back to back (leftovers of the first in the
    shared array must not reach the second); the library's count of its own
    temporary allocations does not move during the calls, while kselect on
    the same problem does allocate (so the count would show it)."""
    import torch
    from approximate_nearest_neighbour_gb300 import binding as B

    # few long rows: the two-pass plan, whose partials live in the fixed array
    for seed, (rows, cols, k) in enumerate([(3, 1_000_003, 100), (2, 600_000, 1000)]):
        vals = S.random_rows(rows, cols, seed=40 + seed)
        t = torch.from_numpy(vals).cuda()
        a0 = B.workspace_allocations()
        ref_v, ref_i = B.kselect(t, k)
        torch.cuda.synchronize()
        assert B.workspace_allocations() > a0  # kselect takes its partials from the pool
        got_v = torch.empty((rows, k), dtype=torch.float32, device="cuda")
        got_i = torch.empty((rows, k), dtype=torch.int64, device="cuda")
        a1 = B.workspace_allocations()
        B.kselect_noalloc(t, k, got_v, got_i)
        torch.cuda.synchronize()
        assert B.workspace_allocations() == a1  # no allocation
        _compare(vals, k, ref_v.cpu().numpy(), ref_i.cpu().numpy(), got_v.cpu().numpy(),
                 got_i.cpu().numpy())


def test_kselect_noalloc_matches_the_oracle():
    """One case against the oracle's k-selection (a stable full sort)."""
    import torch
    import oracle
    from approximate_nearest_neighbour_gb300 import binding as B

    rows, cols, k = 2, 300_001, 64
    vals = S.random_rows(rows, cols, seed=77)
    t = torch.from_numpy(vals).cuda()
    got_v = torch.empty((rows, k), dtype=torch.float32, device="cuda")
    got_i = torch.empty((rows, k), dtype=torch.int64, device="cuda")
    a0 = B.workspace_allocations()
    B.kselect_noalloc(t, k, got_v, got_i)
    torch.cuda.synchronize()
    assert B.workspace_allocations() == a0
    ref_v, ref_i = oracle.kselect(vals, k)
    _compare(vals, k, ref_v, ref_i, got_v.cpu().numpy(), got_i.cpu().numpy())


def test_kselect_noalloc_rejects_problems_beyond_its_scratch():
    import torch
    from approximate_nearest_neighbour_gb300 import binding as B

    rows, k = 600, 2048  # rows * k > 1,048,576
    t = torch.zeros((rows, 8), dtype=torch.float32, device="cuda")
    ov = torch.empty((rows, k), dtype=torch.float32, device="cuda")
    oi = torch.empty((rows, k), dtype=torch.int64, device="cuda")
    with pytest.raises(B.IVFPQError) as e:
        B.kselect_noalloc(t, k, ov, oi)
    assert e.value.status == B.IVFPQ_ERR_INVALID_ARG
    assert "scratch" in str(e.value)
