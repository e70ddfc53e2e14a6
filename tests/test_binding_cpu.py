"""Host-side checks of the Python binding: the library trusts its pointers,
so caller-given outputs must match the shape, dtype and device a call
writes, and the inputs of one call must share a device."""

import pytest


@pytest.fixture(scope="module")
def B():
    from approximate_nearest_neighbour_gb300 import binding
    return binding


def test_out_allocates_when_none(B):
    import torch
    t = B._out(None, (3, 5), torch.float32, "o", torch.device("cpu"))
    assert t.shape == (3, 5) and t.dtype == torch.float32


def test_out_accepts_an_exact_match(B):
    import torch
    o = torch.empty((3, 5), dtype=torch.int64)
    assert B._out(o, (3, 5), torch.int64, "o", torch.device("cpu")) is o


@pytest.mark.parametrize("bad,exc", [
    ("shape", ValueError), ("rank", ValueError), ("dtype", TypeError),
    ("strided", ValueError), ("type", TypeError),
])
def test_out_rejects_mismatches(B, bad, exc):
    import torch
    cpu = torch.device("cpu")
    o = {"shape": torch.empty((3, 4)), "rank": torch.empty((15,)),
         "dtype": torch.empty((3, 5), dtype=torch.float64),
         "strided": torch.empty((5, 3)).t(), "type": [[0.0] * 5] * 3}[bad]
    with pytest.raises(exc):
        B._out(o, (3, 5), torch.float32, "out", cpu)


def test_out_rejects_another_device(B):
    import torch
    o = torch.empty((2, 2), device="meta")
    with pytest.raises(ValueError):
        B._out(o, (2, 2), torch.float32, "out", torch.device("cpu"))


def test_same_device(B):
    import torch
    a, b = torch.empty(2), torch.empty(2, device="meta")
    B._same_device("f", a, a, None)
    with pytest.raises(ValueError):
        B._same_device("f", a, b)


def test_inputs_must_be_device_tensors(B):
    import torch
    with pytest.raises(ValueError):
        B.kselect(torch.zeros((4, 8)), 2)
    with pytest.raises(TypeError):
        B.kselect(torch.zeros((4, 8), dtype=torch.float64), 2)


@pytest.mark.parametrize("fn", ["ivfpq_search_probes", "ivfpq_search"])
def test_query_width_must_match_the_index(B, fn):
    """The coarse kernel reads d floats per query row: a narrower (or wider)
    query matrix is refused on the host, before anything else is checked."""
    import torch
    ix = B.Index(None, 8, 4, 2)  # a handle is never reached
    q = torch.zeros((3, 5))
    with pytest.raises(ValueError, match="dimension 5 does not match"):
        if fn == "ivfpq_search":
            B.ivfpq_search(ix, q, 2, 1)
        else:
            B.ivfpq_search_probes(ix, q, 2)
