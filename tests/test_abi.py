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


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    from approximate_nearest_neighbour_gb300 import binding as B
    monkeypatch.setattr(B, "LIB_PATH", str(tmp_path / "absent.so"))
    monkeypatch.setattr(B, "_lib", None)
    with pytest.raises(B.LibraryMissing):
        B.lib()
