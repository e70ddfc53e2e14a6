"""kselect (WarpSelect / BlockSelect) against the oracle's stable full sort."""

import numpy as np
import pytest

import oracle
from approximate_nearest_neighbour_gb300 import synthetic as S
from parity import check_kselect

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    import torch  # noqa: F401
    from approximate_nearest_neighbour_gb300 import binding
    return binding


def _run(B, vals, k):
    import torch
    t = torch.from_numpy(vals).cuda()
    gv, gi = B.kselect(t, k)
    torch.cuda.synchronize()
    return gv.cpu().numpy(), gi.cpu().numpy()


@pytest.mark.parametrize("kind", ["normal", "ties", "equal", "sorted", "reverse", "inf"])
@pytest.mark.parametrize("k", [1, 31, 32, 33, 100, 257, 1000, 1024, 2048])
def test_kselect_kinds(B, kind, k):
    vals = S.random_rows(5, 3000, seed=k, kind=kind)
    gv, gi = _run(B, vals, k)
    ov, oi = oracle.kselect(vals, k)
    check_kselect(vals, k, ov, oi, gv, gi)


@pytest.mark.parametrize("rows,cols,k", [(1, 1, 1), (3, 5, 10), (7, 33, 32), (2, 0, 4),
                                         (1000, 17, 3), (1, 300_001, 100), (3, 1_000_003, 1024),
                                         (2, 200_000, 2048), (700, 4099, 64)])
def test_kselect_shapes(B, rows, cols, k):
    """Ragged widths, k > cols, empty rows, and the two-pass path (few long rows)."""
    vals = S.random_rows(rows, cols, seed=rows + cols + k)
    gv, gi = _run(B, vals, k)
    ov, oi = oracle.kselect(vals, k)
    check_kselect(vals, k, ov, oi, gv, gi)


def test_kselect_unaligned_rows(B):
    """Row width not a multiple of 4 takes the scalar load path."""
    import torch
    vals = S.random_rows(9, 1001, seed=5)
    full = torch.from_numpy(vals).cuda()
    gv, gi = B.kselect(full, 50)
    ov, oi = oracle.kselect(vals, 50)
    check_kselect(vals, 50, ov, oi, gv.cpu().numpy(), gi.cpu().numpy())


@pytest.mark.parametrize("kind", ["normal", "ties", "equal", "sorted", "reverse", "inf"])
@pytest.mark.parametrize("k,cols", [(1, 32768), (100, 33001), (1000, 32768), (2048, 40000)])
def test_kselect_many_long_rows(B, kind, k, cols):
    """Many long rows take the short-queue path: 16 warps per row with queues
    of max(32, K/8), their merge, and the full-queue kernel again for the rows
    a short queue may have cut. Sorted rows put every winner in one warp's
    columns, ties and equal rows make every queue end at the k-th value, so
    those rows go through the repair; an odd width takes the scalar loads."""
    vals = S.random_rows(640, cols, seed=3 * k + cols, kind=kind)
    gv, gi = _run(B, vals, k)
    ov, oi = oracle.kselect(vals, k)
    check_kselect(vals, k, ov, oi, gv, gi)
