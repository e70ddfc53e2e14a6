"""Plain CPU oracle for batched IVF-PQ search, exact flat k-NN and k-selection.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package. The product library
(``approximate_nearest_neighbour_gb300``) never imports, links or calls it, and
this package never imports the product library: the two share no code.

The arithmetic lives in ``oracle.cpp`` (C++17, standard library only, IEEE
double). This module compiles it with g++ on first use and marshals numpy
arrays through ctypes. Each function cites, in its C++ docstring, the passage of
the pages it follows:

* "Billion-scale similarity search with GPUs" -- IVFADC tables and the list
  scan (section 5), odd-size merge / sort networks (Algorithms 1-2, Figure 1),
  WarpSelect (Algorithm 3, Figure 2).
* "Custom 8-bit floating point value format for reducing shared memory bank
  conflict in approximate nearest neighbor search" -- IVFPQ build steps 1-4,
  search steps 1-5 and Eq. (1).

Parity unpinned: the absolute recall of IVF-PQ against exact neighbours on the
synthetic mixtures (nothing on the pages fixes it); it is reported, not gated.
"""

from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

NTHREADS = max(1, os.cpu_count() or 1)

LUT_FP32, LUT_FP16, LUT_FP8 = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile oracle.cpp into _build/liboracle.so (skipped when up to date)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    cmd = ["g++", "-O2", "-std=c++17", "-shared", "-fPIC", "-o", tmp, _SRC,
           "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _p(a, ctype):
    return a.ctypes.data_as(C.POINTER(ctype)) if a is not None else None


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = C.CDLL(build())
            i64, i32, f64 = C.c_int64, C.c_int, C.c_double
            P = C.POINTER
            L.oracle_coarse.argtypes = [P(C.c_float), i64, i32, P(C.c_float), i64, i32,
                                        P(C.c_int32), P(f64), i32]
            L.oracle_lut.argtypes = [P(f64), i32, P(C.c_float), i32, P(f64)]
            L.oracle_lut.restype = None
            L.oracle_quantize_lut.argtypes = [P(f64), i32, i32]
            L.oracle_quantize_lut.restype = None
            L.oracle_adc.argtypes = [P(f64), i32, P(C.c_uint8)]
            L.oracle_adc.restype = f64
            L.oracle_f16_encode.argtypes = [f64]
            L.oracle_f16_encode.restype = C.c_uint16
            L.oracle_f16_decode.argtypes = [C.c_uint16]
            L.oracle_f16_decode.restype = f64
            L.oracle_e4m3_encode.argtypes = [f64]
            L.oracle_e4m3_encode.restype = C.c_uint8
            L.oracle_e4m3_decode.argtypes = [C.c_uint8]
            L.oracle_e4m3_decode.restype = f64
            L.oracle_ivfpq_search.argtypes = [
                P(C.c_float), i64, i32, P(C.c_float), i64, P(C.c_float), i32,
                P(C.c_int64), P(C.c_uint8), P(C.c_int64), i32, i32, i32,
                P(C.c_int32), P(f64), P(C.c_int64), P(C.c_int32), i32]
            L.oracle_flat_knn.argtypes = [P(C.c_float), i64, i32, P(C.c_float), i64, i32,
                                          P(f64), P(C.c_int64), i32]
            L.oracle_kselect.argtypes = [P(C.c_float), i64, i64, i32, P(C.c_float),
                                         P(C.c_int64), i32]
            L.oracle_odd_merge_network.argtypes = [i32, i32, P(C.c_int32), i32, P(C.c_int)]
            L.oracle_odd_sort_network.argtypes = [i32, P(C.c_int32), i32, P(C.c_int)]
            L.oracle_warpselect_sim.argtypes = [P(C.c_float), i64, i32, i32, P(C.c_float),
                                                P(C.c_int64), P(C.c_int64)]
            L.oracle_pq_train.argtypes = [P(C.c_float), i64, i32, i32, i32, P(C.c_int64),
                                          P(C.c_float), P(f64), i32]
            L.oracle_pq_encode.argtypes = [P(C.c_float), i64, i32, i32, P(C.c_float),
                                           P(C.c_uint8), i32]
            _lib = L
    return _lib


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what} rejected its arguments (rc={rc})")


# ---------------------------------------------------------------------------
def coarse(q, cent, nprobe, nthreads=NTHREADS):
    """Exact nearest centroids: (lists int32 [nq, nprobe], dist float64)."""
    q, cent = _f32(q), _f32(cent)
    nq, d = q.shape
    lists = np.empty((nq, nprobe), np.int32)
    dist = np.empty((nq, nprobe), np.float64)
    _check(lib().oracle_coarse(_p(q, C.c_float), nq, d, _p(cent, C.c_float), cent.shape[0],
                               nprobe, _p(lists, C.c_int32), _p(dist, C.c_double), nthreads),
           "coarse")
    return lists, dist


def lut(r, cb):
    """ADC table T[j, e] (float64, [m, 256]) for one residual r (length d)."""
    r = np.ascontiguousarray(r, dtype=np.float64)
    cb = _f32(cb)
    m = cb.shape[0]
    T = np.empty((m, 256), np.float64)
    lib().oracle_lut(_p(r, C.c_double), r.shape[0], _p(cb, C.c_float), m, _p(T, C.c_double))
    return T


def quantize_lut(T, lut_type):
    T = np.array(T, dtype=np.float64, order="C", copy=True)
    lib().oracle_quantize_lut(_p(T, C.c_double), T.shape[0], lut_type)
    return T


def adc(T, code):
    T = np.ascontiguousarray(T, dtype=np.float64)
    code = np.ascontiguousarray(code, dtype=np.uint8)
    return lib().oracle_adc(_p(T, C.c_double), T.shape[0], _p(code, C.c_uint8))


def f16_encode(x):
    return int(lib().oracle_f16_encode(float(x)))


def f16_decode(h):
    return float(lib().oracle_f16_decode(int(h)))


def e4m3_encode(x):
    return int(lib().oracle_e4m3_encode(float(x)))


def e4m3_decode(b):
    return float(lib().oracle_e4m3_decode(int(b)))


def to_lists(codes, list_ids, ids, nlist):
    """Group row-major (codes, list_ids, ids) into inverted lists, keeping the
    input order inside each list. Returns (list_off int64 [nlist+1], codes in
    list order, ids in list order)."""
    list_ids = np.asarray(list_ids)
    order = np.argsort(list_ids, kind="stable")
    counts = np.bincount(list_ids, minlength=nlist)
    off = np.zeros(nlist + 1, np.int64)
    np.cumsum(counts, out=off[1:])
    return off, np.ascontiguousarray(codes[order]), np.ascontiguousarray(ids[order], np.int64)


def ivfpq_search(q, cent, cb, list_off, codes, ids, nprobe, k, lut_type=LUT_FP32,
                 forced_probes=None, nthreads=NTHREADS):
    """IVF-PQ search over inverted lists (see oracle.cpp). Returns
    (dist float64 [nq,k], ids int64 [nq,k], probes int32 [nq,nprobe])."""
    q, cent, cb = _f32(q), _f32(cent), _f32(cb)
    nq, d = q.shape
    m = cb.shape[0]
    list_off = np.ascontiguousarray(list_off, np.int64)
    codes = np.ascontiguousarray(codes, np.uint8)
    ids = np.ascontiguousarray(ids, np.int64)
    if forced_probes is not None:
        forced_probes = np.ascontiguousarray(forced_probes, np.int32)
    od = np.empty((nq, k), np.float64)
    oi = np.empty((nq, k), np.int64)
    op = np.empty((nq, nprobe), np.int32)
    _check(lib().oracle_ivfpq_search(
        _p(q, C.c_float), nq, d, _p(cent, C.c_float), cent.shape[0], _p(cb, C.c_float), m,
        _p(list_off, C.c_int64), _p(codes, C.c_uint8), _p(ids, C.c_int64), nprobe, k,
        lut_type, _p(forced_probes, C.c_int32), _p(od, C.c_double), _p(oi, C.c_int64),
        _p(op, C.c_int32), nthreads), "ivfpq_search")
    return od, oi, op


def flat_knn(db, q, k, nthreads=NTHREADS):
    db, q = _f32(db), _f32(q)
    nq, d = q.shape
    od = np.empty((nq, k), np.float64)
    oi = np.empty((nq, k), np.int64)
    _check(lib().oracle_flat_knn(_p(db, C.c_float), db.shape[0], d, _p(q, C.c_float), nq, k,
                                 _p(od, C.c_double), _p(oi, C.c_int64), nthreads), "flat_knn")
    return od, oi


def kselect(vals, k, nthreads=NTHREADS):
    vals = _f32(vals)
    rows, cols = vals.shape
    ov = np.empty((rows, k), np.float32)
    oi = np.empty((rows, k), np.int64)
    _check(lib().oracle_kselect(_p(vals, C.c_float), rows, cols, k, _p(ov, C.c_float),
                                _p(oi, C.c_int64), nthreads), "kselect")
    return ov, oi


def _network(fn, *args):
    cap = 1 << 16
    buf = np.empty(3 * cap, np.int32)
    steps = C.c_int(0)
    n = fn(*args, _p(buf, C.c_int32), cap, C.byref(steps))
    if n < 0:
        raise ValueError("network too large")
    return buf[: 3 * n].reshape(n, 3).copy(), steps.value


def odd_merge_network(lL, lR):
    """Comparators (lo, hi, step) of Algorithm 1 and its number of parallel steps."""
    return _network(lib().oracle_odd_merge_network, lL, lR)


def odd_sort_network(l):
    """Comparators (lo, hi, step) of Algorithm 2 and its number of parallel steps."""
    return _network(lib().oracle_odd_sort_network, l)


def warpselect_sim(vals, k, t):
    """Host simulation of WarpSelect with invariant checks. Returns
    (status, vals [k], idx [k], merges); status 0 = all invariants held."""
    vals = _f32(vals).ravel()
    ov = np.empty(k, np.float32)
    oi = np.empty(k, np.int64)
    merges = C.c_int64(0)
    st = lib().oracle_warpselect_sim(_p(vals, C.c_float), vals.shape[0], k, t,
                                     _p(ov, C.c_float), _p(oi, C.c_int64), C.byref(merges))
    return st, ov, oi, merges.value


def pq_train(x, m, niter, init, nthreads=NTHREADS):
    """Lloyd training of m sub-quantizers x 256 codewords. Returns
    (codebooks float32 [m, 256, d/m], objective per assignment pass)."""
    x = _f32(x)
    n, d = x.shape
    init = np.ascontiguousarray(init, np.int64)
    cb = np.empty((m, 256, d // m), np.float32)
    obj = np.empty(niter + 1, np.float64)
    _check(lib().oracle_pq_train(_p(x, C.c_float), n, d, m, niter, _p(init, C.c_int64),
                                 _p(cb, C.c_float), _p(obj, C.c_double), nthreads), "pq_train")
    return cb, obj


def pq_encode(x, cb, nthreads=NTHREADS):
    x, cb = _f32(x), _f32(cb)
    n, d = x.shape
    m = cb.shape[0]
    codes = np.empty((n, m), np.uint8)
    _check(lib().oracle_pq_encode(_p(x, C.c_float), n, d, m, _p(cb, C.c_float),
                                  _p(codes, C.c_uint8), nthreads), "pq_encode")
    return codes


def recall_at_k(found_ids, true_ids):
    """mean over queries of |found ∩ true| / k (the intersection form used for
    the k-NN graph accuracy in "Billion-scale similarity search with GPUs",
    section 6)."""
    found_ids = np.asarray(found_ids)
    true_ids = np.asarray(true_ids)
    k = true_ids.shape[1]
    hits = 0
    for f, t in zip(found_ids, true_ids):
        hits += len(set(f[f >= 0].tolist()) & set(t[t >= 0].tolist()))
    return hits / (k * true_ids.shape[0])
