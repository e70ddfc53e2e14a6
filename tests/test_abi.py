"""The C-ABI library loads on a machine without a GPU, exports every entry
point declared in include/ivfpq.h, and rejects bad arguments on the host
before touching the device."""

import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ivfpq.h")


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b([a-z_][a-z0-9_]*)\s*\(", text)) - {"defined"})


@pytest.fixture(scope="module")
def lib():
    from approximate_nearest_neighbour_gb300 import binding, build
    build.build_library()
    return binding.lib()


def test_header_declares_the_boundary():
    names = _declared()
    for n in ("ivfpq_index_create", "ivfpq_add", "ivfpq_search", "flat_knn", "kselect"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in _declared():
        assert hasattr(lib, name), name


def test_binding_signatures_cover_the_header(lib):
    from approximate_nearest_neighbour_gb300 import binding
    assert set(_declared()) == set(binding.SIGNATURES)


def test_host_side_argument_errors(lib):
    from approximate_nearest_neighbour_gb300 import binding as B
    vp = C.c_void_p(16)
    out = C.c_void_p()
    # unsupported product quantizer shapes
    assert lib.ivfpq_index_create(64, 16, 6, 8, vp, vp, C.byref(out)) == B.IVFPQ_ERR_INVALID_ARG
    assert lib.ivfpq_index_create(60, 16, 12, 7, vp, vp, C.byref(out)) == B.IVFPQ_ERR_UNSUPPORTED
    assert lib.ivfpq_index_create(64, 16, 8, 8, None, vp, C.byref(out)) == B.IVFPQ_ERR_INVALID_ARG
    assert b"null" in lib.ivfpq_last_error()
    # k and sizes are checked before any launch
    assert lib.kselect(vp, 4, 10, 0, vp, vp, None) == B.IVFPQ_ERR_INVALID_ARG
    assert lib.kselect(vp, 4, 10, 2049, vp, vp, None) == B.IVFPQ_ERR_INVALID_ARG
    assert lib.kselect(vp, -1, 10, 5, vp, vp, None) == B.IVFPQ_ERR_INVALID_ARG
    assert lib.kselect(vp, 0, 10, 5, vp, vp, None) == B.IVFPQ_OK  # nothing to do
    assert lib.flat_knn(vp, 10, 0, vp, 3, 5, vp, vp, None) == B.IVFPQ_ERR_INVALID_ARG
    assert lib.flat_knn(vp, 10, 8, vp, 3, 5000, vp, vp, None) == B.IVFPQ_ERR_INVALID_ARG
    assert lib.ivfpq_search(None, vp, 1, 1, 1, vp, vp, None) == B.IVFPQ_ERR_INVALID_ARG
    assert lib.ivfpq_set_lut_type(None, 0) == B.IVFPQ_ERR_INVALID_ARG
    assert lib.ivfpq_ntotal(None) == -1
    assert lib.ivfpq_status_string(-3) == b"IVFPQ_ERR_OOM"


def test_host_side_argument_errors_of_the_other_entries(lib):
    """Index preparation, sharded merge, graph and no-alloc selection reject
    bad sizes and null pointers on the host, with a message."""
    from approximate_nearest_neighbour_gb300 import binding as B
    vp = C.c_void_p(16)
    bad = B.IVFPQ_ERR_INVALID_ARG
    cases = [
        # k-means: k > n, k < 1, bad d, null seeds
        lambda: lib.kmeans_lloyd(vp, 10, 4, 11, 1, vp, vp, vp, vp, None),
        lambda: lib.kmeans_lloyd(vp, 10, 4, 0, 1, vp, vp, vp, vp, None),
        lambda: lib.kmeans_lloyd(vp, 10, 0, 3, 1, vp, vp, vp, vp, None),
        lambda: lib.kmeans_lloyd(vp, 10, 4, 3, 1, None, vp, vp, vp, None),
        # PQ training: d not a multiple of m, fewer points than codewords
        lambda: lib.pq_train(vp, 1000, 10, 4, 1, vp, vp, vp, None),
        lambda: lib.pq_train(vp, 100, 16, 4, 1, vp, vp, vp, None),
        # encoder / graph / preassigned search without an index
        lambda: lib.ivfpq_encode(None, vp, 5, vp, vp, None),
        lambda: lib.ivfpq_encode_hinted(None, vp, 5, vp, vp, vp, None, None),
        lambda: lib.ivfpq_repaired_queries(None, None, None),
        # residuals: bad d, no centroids, null outputs
        lambda: lib.ivfpq_residuals(vp, 4, 0, vp, 5, vp, vp, None),
        lambda: lib.ivfpq_residuals(vp, 0, 8, vp, 5, vp, vp, None),
        lambda: lib.ivfpq_residuals(vp, 4, 8, vp, 5, None, vp, None),
        lambda: lib.ivfpq_knn_graph(None, vp, vp, 5, 1, 1, vp, vp, None),
        lambda: lib.ivfpq_search_preassigned(None, vp, 1, 1, vp, 1, vp, vp, None),
        lambda: lib.ivfpq_search_probes(None, vp, 1, 1, vp, vp, None),
        lambda: lib.ivfpq_set_precomputed(None, 0),
        lambda: lib.ivfpq_set_scan_mode(None, 1, 2),
        # merge: k beyond the limit, no shards, null inputs
        lambda: lib.knn_merge(vp, vp, 4, 2, 10, 2049, vp, vp, None),
        lambda: lib.knn_merge(vp, vp, 4, 0, 10, 5, vp, vp, None),
        lambda: lib.knn_merge(None, vp, 4, 2, 10, 5, vp, vp, None),
        # no-alloc selection: k and the fixed workspace limit
        lambda: lib.kselect_noalloc(vp, 4, 10, 0, vp, vp, None),
        lambda: lib.kselect_noalloc(vp, 1 << 20, 1 << 20, 2048, vp, vp, None),
    ]
    for i, call in enumerate(cases):
        rc = call()
        assert rc == bad, (i, rc, lib.ivfpq_last_error())
        assert lib.ivfpq_last_error(), i


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    from approximate_nearest_neighbour_gb300 import binding as B
    monkeypatch.setattr(B, "LIB_PATH", str(tmp_path / "absent.so"))
    monkeypatch.setattr(B, "_lib", None)
    with pytest.raises(B.LibraryMissing):
        B.lib()
