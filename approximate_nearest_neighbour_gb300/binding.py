"""Thin ctypes binding of libivfpq_gb300.so (include/ivfpq.h).

Argument marshalling only: every function here checks shapes and dtypes of
torch CUDA tensors, passes their device pointers and the current CUDA stream
to the C entry point of the same name, and raises :class:`IVFPQError` on a
non-zero status. No computation happens in Python and there is no CPU
fallback: if the library has not been built, :class:`LibraryMissing` is
raised.
"""

from __future__ import annotations

import ctypes as C
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libivfpq_gb300.so")

IVFPQ_OK = 0
IVFPQ_ERR_INVALID_ARG = -1
IVFPQ_ERR_UNSUPPORTED = -2
IVFPQ_ERR_OOM = -3
IVFPQ_ERR_CUDA = -4
IVFPQ_ERR_DEVICE_CHECK = -5
IVFPQ_ERR_TIMEOUT = -6

LUT_FP32, LUT_FP16, LUT_FP8 = 0, 1, 2
LUT_TYPES = {"fp32": LUT_FP32, "fp16": LUT_FP16, "fp8": LUT_FP8}
MAX_K = 2048

# name -> (restype, argtypes); mirrors include/ivfpq.h
_VP, _I, _I64 = C.c_void_p, C.c_int, C.c_int64
SIGNATURES = {
    "ivfpq_index_create": (_I, [_I, _I, _I, _I, _VP, _VP, C.POINTER(_VP)]),
    "ivfpq_index_destroy": (_I, [_VP]),
    "ivfpq_set_lut_type": (_I, [_VP, _I]),
    "ivfpq_add": (_I, [_VP, _VP, _VP, _VP, _I64, _VP]),
    "ivfpq_ntotal": (_I64, [_VP]),
    "ivfpq_search": (_I, [_VP, _VP, _I64, _I, _I, _VP, _VP, _VP]),
    "ivfpq_search_probes": (_I, [_VP, _VP, _I64, _I, _VP, _VP, _VP]),
    "ivfpq_search_preassigned": (_I, [_VP, _VP, _I64, _I, _VP, _I, _VP, _VP, _VP]),
    "ivfpq_set_profiling": (_I, [_VP, _I]),
    "ivfpq_stage_times": (_I, [_VP, C.POINTER(C.c_float), C.POINTER(C.c_int)]),
    "ivfpq_last_scan_kernel": (C.c_char_p, [_VP]),
    "ivfpq_set_precomputed": (_I, [_VP, _I]),
    "ivfpq_set_scan_mode": (_I, [_VP, _I, _I]),
    "ivfpq_uses_precomputed": (_I, [_VP]),
    "ivfpq_kernel_launches": (C.c_uint64, []),
    "ivfpq_workspace_allocations": (C.c_uint64, []),
    "flat_knn": (_I, [_VP, _I64, _I, _VP, _I64, _I, _VP, _VP, _VP]),
    "kselect": (_I, [_VP, _I64, _I64, _I, _VP, _VP, _VP]),
    "kselect_noalloc": (_I, [_VP, _I64, _I64, _I, _VP, _VP, _VP]),
    "knn_merge": (_I, [_VP, _VP, _I64, _I, _I, _I, _VP, _VP, _VP]),
    "kmeans_lloyd": (_I, [_VP, _I64, _I, _I, _I, _VP, _VP, _VP, _VP, _VP]),
    "pq_train": (_I, [_VP, _I64, _I, _I, _I, _VP, _VP, _VP, _VP]),
    "ivfpq_encode": (_I, [_VP, _VP, _I64, _VP, _VP, _VP]),
    "ivfpq_residuals": (_I, [_VP, _I, _I, _VP, _I64, _VP, _VP, _VP]),
    "ivfpq_encode_hinted": (_I, [_VP, _VP, _I64, _VP, _VP, _VP, C.POINTER(_I64), _VP]),
    "ivfpq_repaired_queries": (_I, [_VP, C.POINTER(_I64), _VP]),
    "ivfpq_knn_graph": (_I, [_VP, _VP, _VP, _I64, _I, _I, _VP, _VP, _VP]),
    "ivfpq_device_check": (_I, [_VP]),
    "ivfpq_selftest_wait_timeout": (_I, [_I, _VP]),
    "ivfpq_last_error": (C.c_char_p, []),
    "ivfpq_status_string": (C.c_char_p, [_I]),
}


class LibraryMissing(RuntimeError):
    pass


class IVFPQError(RuntimeError):
    def __init__(self, fn, status, msg):
        super().__init__(f"{fn} failed with status {status}: {msg}")
        self.status = status


_lib = None
_lock = threading.Lock()


def lib():
    """The loaded library (raises LibraryMissing if it was never built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise LibraryMissing(
                    f"{LIB_PATH} is missing: build it with "
                    "`python -c 'import __graft_entry__ as g; g.build()'`")
            L = C.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                f = getattr(L, name)
                f.restype = res
                f.argtypes = args
            _lib = L
    return _lib


def _check(fn, status):
    if status != IVFPQ_OK:
        msg = lib().ivfpq_last_error().decode(errors="replace")
        raise IVFPQError(fn, status, msg)


def _torch():
    import torch
    return torch


def _stream(stream=None):
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream()
    return C.c_void_p(stream.cuda_stream)


def _ptr(t):
    return C.c_void_p(t.data_ptr()) if t is not None else None


def _need(t, dtype, name, ndim=None, device=True):
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if device and not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dimensions")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _out(t, shape, dtype, name, device):
    """A caller-given output checked against the shape the call writes
    (the library trusts its pointers), or a new tensor."""
    torch = _torch()
    shape = tuple(int(v) for v in shape)
    if t is None:
        return torch.empty(shape, dtype=dtype, device=device)
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != shape:
        raise ValueError(f"{name} must have shape {shape}, got {tuple(t.shape)}")
    if t.device != torch.device(device):
        raise ValueError(f"{name} must be on {device} (the inputs' device), got {t.device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _same_device(what, *tensors):
    devs = {t.device for t in tensors if t is not None}
    if len(devs) > 1:
        raise ValueError(f"{what}: tensors on several devices {sorted(map(str, devs))}")


# ---------------------------------------------------------------------------
class Index:
    """Owner of an ivfpq_index handle."""

    def __init__(self, handle, d, nlist, m):
        self.handle = handle
        self.d, self.nlist, self.m = d, nlist, m

    def __del__(self):
        try:
            if self.handle:
                lib().ivfpq_index_destroy(self.handle)
                self.handle = None
        except Exception:
            pass

    @property
    def ntotal(self):
        return int(lib().ivfpq_ntotal(self.handle))


def ivfpq_index_create(centroids, codebooks, nbits=8):
    """centroids: fp32 [nlist, d]; codebooks: fp32 [m, 256, d/m] (CUDA)."""
    torch = _torch()
    _need(centroids, torch.float32, "centroids", 2)
    _need(codebooks, torch.float32, "codebooks", 3)
    nlist, d = centroids.shape
    m = codebooks.shape[0]
    if m < 1 or d % m or tuple(codebooks.shape[1:]) != (256, d // m):
        raise ValueError(f"ivfpq_index_create: codebooks must be [m, 256, d/m] with d = {d}, "
                         f"got {tuple(codebooks.shape)}")
    _same_device("ivfpq_index_create", centroids, codebooks)
    h = C.c_void_p()
    _check("ivfpq_index_create",
           lib().ivfpq_index_create(d, nlist, m, nbits, _ptr(centroids), _ptr(codebooks),
                                    C.byref(h)))
    return Index(h, d, nlist, m)


def ivfpq_index_destroy(index):
    if index.handle:
        _check("ivfpq_index_destroy", lib().ivfpq_index_destroy(index.handle))
        index.handle = None


def ivfpq_set_lut_type(index, lut_type):
    if isinstance(lut_type, str):
        lut_type = LUT_TYPES[lut_type]
    _check("ivfpq_set_lut_type", lib().ivfpq_set_lut_type(index.handle, int(lut_type)))


def ivfpq_add(index, codes, list_ids, ids, stream=None):
    """codes: uint8 [n, m]; list_ids: int32 [n]; ids: int64 [n] (CUDA)."""
    torch = _torch()
    _need(codes, torch.uint8, "codes", 2)
    _need(list_ids, torch.int32, "list_ids", 1)
    _need(ids, torch.int64, "ids", 1)
    n = codes.shape[0]
    if codes.shape[1] != index.m or list_ids.shape[0] != n or ids.shape[0] != n:
        raise ValueError("ivfpq_add: inconsistent shapes")
    _same_device("ivfpq_add", codes, list_ids, ids)
    _check("ivfpq_add", lib().ivfpq_add(index.handle, _ptr(codes), _ptr(list_ids), _ptr(ids), n,
                                         _stream(stream)))


def _queries(fn, index, queries):
    """Checks a [nq, d] fp32 query matrix against the index's d (the kernels
    read d floats per row, so a narrower matrix would be read past its end)
    before checking that it is a contiguous CUDA tensor."""
    torch = _torch()
    _need(queries, torch.float32, "queries", 2, device=False)
    if queries.shape[1] != index.d:
        raise ValueError(f"{fn}: query dimension {queries.shape[1]} does not match the "
                         f"index's d = {index.d}")
    _need(queries, torch.float32, "queries", 2)
    return queries.shape[0]


def ivfpq_search(index, queries, nprobe, k, out_dist=None, out_ids=None, stream=None):
    torch = _torch()
    nq = _queries("ivfpq_search", index, queries)
    out_dist = _out(out_dist, (nq, k), torch.float32, "out_dist", queries.device)
    out_ids = _out(out_ids, (nq, k), torch.int64, "out_ids", queries.device)
    _check("ivfpq_search", lib().ivfpq_search(index.handle, _ptr(queries), nq, nprobe, k,
                                               _ptr(out_dist), _ptr(out_ids), _stream(stream)))
    return out_dist, out_ids


def ivfpq_search_probes(index, queries, nprobe, with_dist=True, stream=None):
    torch = _torch()
    nq = _queries("ivfpq_search_probes", index, queries)
    probes = torch.empty((nq, nprobe), dtype=torch.int32, device=queries.device)
    coarse = (torch.empty((nq, nprobe), dtype=torch.float32, device=queries.device)
              if with_dist else None)
    _check("ivfpq_search_probes",
           lib().ivfpq_search_probes(index.handle, _ptr(queries), nq, nprobe, _ptr(probes),
                                     _ptr(coarse), _stream(stream)))
    return probes, coarse


def ivfpq_search_preassigned(index, queries, probes, k, out_dist=None, out_ids=None,
                             stream=None):
    torch = _torch()
    _need(queries, torch.float32, "queries", 2)
    _need(probes, torch.int32, "probes", 2)
    nq, nprobe = probes.shape
    if tuple(queries.shape) != (nq, index.d):
        raise ValueError(f"ivfpq_search_preassigned: queries must be [{nq}, {index.d}] "
                         f"(one row per probe row), got {tuple(queries.shape)}")
    _same_device("ivfpq_search_preassigned", queries, probes)
    out_dist = _out(out_dist, (nq, k), torch.float32, "out_dist", queries.device)
    out_ids = _out(out_ids, (nq, k), torch.int64, "out_ids", queries.device)
    _check("ivfpq_search_preassigned",
           lib().ivfpq_search_preassigned(index.handle, _ptr(queries), nq, nprobe, _ptr(probes), k,
                                          _ptr(out_dist), _ptr(out_ids), _stream(stream)))
    return out_dist, out_ids


def ivfpq_set_profiling(index, enable=True):
    _check("ivfpq_set_profiling", lib().ivfpq_set_profiling(index.handle, int(bool(enable))))


def ivfpq_stage_times(index):
    """([coarse, plan, scan, merge] milliseconds summed over the searches
    recorded since profiling was enabled, number of searches)."""
    buf = (C.c_float * 4)()
    n = C.c_int(0)
    _check("ivfpq_stage_times", lib().ivfpq_stage_times(index.handle, buf, C.byref(n)))
    return list(buf), n.value


def ivfpq_set_precomputed(index, mode):
    """-1 automatic, 0 off, 1 on (where supported) for the precomputed-term
    lookup tables; returns whether searches now use them."""
    _check("ivfpq_set_precomputed", lib().ivfpq_set_precomputed(index.handle, int(mode)))
    return bool(lib().ivfpq_uses_precomputed(index.handle))


def ivfpq_set_scan_mode(index, mode, group=0):
    """-1 automatic, 0 by query, 1 by list (where its shapes apply); group =
    table sets per by-list item (2 or 3, -1 automatic, 0 keeps it)."""
    _check("ivfpq_set_scan_mode", lib().ivfpq_set_scan_mode(index.handle, int(mode), int(group)))


def ivfpq_uses_precomputed(index):
    return bool(lib().ivfpq_uses_precomputed(index.handle))


def last_scan_kernel(index):
    """Name of the list-scan kernel family the index's last search used."""
    r = lib().ivfpq_last_scan_kernel(index.handle)
    return r.decode() if r else None


def kernel_launches():
    """Kernels launched by the library since it was loaded."""
    return int(lib().ivfpq_kernel_launches())


def workspace_allocations():
    """Temporary device allocations the library has made since it was loaded."""
    return int(lib().ivfpq_workspace_allocations())


def device_check(stream=None):
    """Synchronises the stream and raises IVFPQError (IVFPQ_ERR_TIMEOUT) if a
    kernel of the library gave up a bounded wait since the last check."""
    _check("ivfpq_device_check", lib().ivfpq_device_check(_stream(stream)))


def selftest_wait_timeout(spins=1024, stream=None):
    """Launches a block whose bounded wait is bound to expire (nothing
    completes the barrier phase it waits on); device_check() then reports
    it."""
    _check("ivfpq_selftest_wait_timeout",
           lib().ivfpq_selftest_wait_timeout(int(spins), _stream(stream)))


def flat_knn(db, queries, k, out_dist=None, out_ids=None, stream=None):
    torch = _torch()
    _need(db, torch.float32, "db", 2)
    _need(queries, torch.float32, "queries", 2)
    n, d = db.shape
    nq = queries.shape[0]
    if queries.shape[1] != d:
        raise ValueError("flat_knn: dimension mismatch")
    _same_device("flat_knn", db, queries)
    out_dist = _out(out_dist, (nq, k), torch.float32, "out_dist", queries.device)
    out_ids = _out(out_ids, (nq, k), torch.int64, "out_ids", queries.device)
    _check("flat_knn", lib().flat_knn(_ptr(db), n, d, _ptr(queries), nq, k, _ptr(out_dist),
                                       _ptr(out_ids), _stream(stream)))
    return out_dist, out_ids


def kmeans_lloyd(x, init, niter, stream=None):
    """Lloyd k-means on device fp32 x [n, d] seeded from rows init (int64
    [k]): (centroids [k, d], assignment int32 [n], objective per pass as a
    numpy fp64 array of niter + 1)."""
    import numpy as np
    torch = _torch()
    _need(x, torch.float32, "x", 2)
    _need(init, torch.int64, "init", 1)
    n, d = x.shape
    k = init.shape[0]
    _same_device("kmeans_lloyd", x, init)
    cent = torch.empty((k, d), dtype=torch.float32, device=x.device)
    assign = torch.empty((n,), dtype=torch.int32, device=x.device)
    obj = np.zeros(niter + 1, np.float64)
    _check("kmeans_lloyd", lib().kmeans_lloyd(
        _ptr(x), n, d, k, niter, _ptr(init), _ptr(cent), _ptr(assign),
        obj.ctypes.data_as(C.c_void_p), _stream(stream)))
    return cent, assign, obj


def pq_train(x, m, niter, init, stream=None):
    """Product quantizer codebooks [m, 256, d/m] trained on device fp32 x
    [n, d], seeded from rows init (int64 [256]); returns (codebooks,
    objective per pass, numpy fp64 [niter + 1])."""
    import numpy as np
    torch = _torch()
    _need(x, torch.float32, "x", 2)
    _need(init, torch.int64, "init", 1)
    n, d = x.shape
    if init.shape[0] != 256:
        raise ValueError(f"pq_train: init must hold 256 seed rows, got {init.shape[0]}")
    _same_device("pq_train", x, init)
    cb = torch.empty((m, 256, d // m), dtype=torch.float32, device=x.device)
    obj = np.zeros(niter + 1, np.float64)
    _check("pq_train", lib().pq_train(_ptr(x), n, d, m, niter, _ptr(init), _ptr(cb),
                                       obj.ctypes.data_as(C.c_void_p), _stream(stream)))
    return cb, obj


def ivfpq_knn_graph(index, x, self_ids, nprobe, k, stream=None):
    """k approximate neighbours of every row of x among the index's other
    vectors: ([n, k] fp32 distances, [n, k] int64 ids)."""
    torch = _torch()
    _need(x, torch.float32, "x", 2)
    _need(self_ids, torch.int64, "self_ids", 1)
    n = x.shape[0]
    if x.shape[1] != index.d or self_ids.shape[0] != n:
        raise ValueError(f"ivfpq_knn_graph: x must be [n, {index.d}] and self_ids [n], got "
                         f"{tuple(x.shape)} and {tuple(self_ids.shape)}")
    _same_device("ivfpq_knn_graph", x, self_ids)
    d = torch.empty((n, k), dtype=torch.float32, device=x.device)
    i = torch.empty((n, k), dtype=torch.int64, device=x.device)
    _check("ivfpq_knn_graph", lib().ivfpq_knn_graph(index.handle, _ptr(x), _ptr(self_ids), n,
                                                     nprobe, k, _ptr(d), _ptr(i),
                                                     _stream(stream)))
    return d, i


def ivfpq_encode(index, x, stream=None):
    """(list ids int32 [n], codes uint8 [n, m]) of device fp32 x [n, d]."""
    torch = _torch()
    _need(x, torch.float32, "x", 2)
    n = x.shape[0]
    if x.shape[1] != index.d:
        raise ValueError(f"ivfpq_encode: x must be [n, {index.d}], got {tuple(x.shape)}")
    lists = torch.empty((n,), dtype=torch.int32, device=x.device)
    codes = torch.empty((n, index.m), dtype=torch.uint8, device=x.device)
    _check("ivfpq_encode", lib().ivfpq_encode(index.handle, _ptr(x), n, _ptr(lists),
                                               _ptr(codes), _stream(stream)))
    return lists, codes


def ivfpq_residuals(centroids, x, stream=None):
    """(nearest centroid int32 [n], residual x - centroid fp32 [n, d]) of device
    fp32 x [n, d] against device fp32 centroids [nlist, d]."""
    torch = _torch()
    _need(centroids, torch.float32, "centroids", 2)
    _need(x, torch.float32, "x", 2)
    nlist, d = centroids.shape
    n = x.shape[0]
    if x.shape[1] != d:
        raise ValueError(f"ivfpq_residuals: x must be [n, {d}], got {tuple(x.shape)}")
    _same_device("ivfpq_residuals", centroids, x)
    lists = torch.empty((n,), dtype=torch.int32, device=x.device)
    resid = torch.empty((n, d), dtype=torch.float32, device=x.device)
    _check("ivfpq_residuals", lib().ivfpq_residuals(_ptr(centroids), nlist, d, _ptr(x), n,
                                                     _ptr(lists), _ptr(resid), _stream(stream)))
    return lists, resid


def ivfpq_encode_hinted(index, x, hint, list_ids=None, codes=None, stream=None):
    """ivfpq_encode with a candidate list per row (int32 [n]): (list ids,
    codes, rows that needed the full nearest-centroid search)."""
    torch = _torch()
    _need(x, torch.float32, "x", 2)
    _need(hint, torch.int32, "hint", 1)
    n = x.shape[0]
    if x.shape[1] != index.d or hint.shape[0] != n:
        raise ValueError(f"ivfpq_encode_hinted: x must be [n, {index.d}] and hint [n], got "
                         f"{tuple(x.shape)} and {tuple(hint.shape)}")
    _same_device("ivfpq_encode_hinted", x, hint)
    list_ids = _out(list_ids, (n,), torch.int32, "list_ids", x.device)
    codes = _out(codes, (n, index.m), torch.uint8, "codes", x.device)
    searched = C.c_int64(0)
    _check("ivfpq_encode_hinted",
           lib().ivfpq_encode_hinted(index.handle, _ptr(x), n, _ptr(hint), _ptr(list_ids),
                                     _ptr(codes), C.byref(searched), _stream(stream)))
    return list_ids, codes, int(searched.value)


def ivfpq_repaired_queries(index, stream=None):
    """Queries re-scanned with full-length queues since the previous call."""
    n = C.c_int64(0)
    _check("ivfpq_repaired_queries",
           lib().ivfpq_repaired_queries(index.handle, C.byref(n), _stream(stream)))
    return int(n.value)


def knn_merge(dists, ids, k, out_dist=None, out_ids=None, stream=None):
    """k smallest of S shards' results per query. dists fp32 and ids int64,
    both [S, nq, k_in] on the device; returns ([nq, k] fp32, [nq, k] int64)."""
    torch = _torch()
    _need(dists, torch.float32, "dists", 3)
    _need(ids, torch.int64, "ids", 3)
    if tuple(ids.shape) != tuple(dists.shape):
        raise ValueError("knn_merge: dists and ids must have the same shape")
    S, nq, k_in = dists.shape
    _same_device("knn_merge", dists, ids)
    out_dist = _out(out_dist, (nq, k), torch.float32, "out_dist", dists.device)
    out_ids = _out(out_ids, (nq, k), torch.int64, "out_ids", dists.device)
    _check("knn_merge", lib().knn_merge(_ptr(dists), _ptr(ids), nq, S, k_in, k, _ptr(out_dist),
                                         _ptr(out_ids), _stream(stream)))
    return out_dist, out_ids


def kselect(vals, k, out_vals=None, out_idx=None, stream=None):
    torch = _torch()
    _need(vals, torch.float32, "vals", 2)
    rows, cols = vals.shape
    out_vals = _out(out_vals, (rows, k), torch.float32, "out_vals", vals.device)
    out_idx = _out(out_idx, (rows, k), torch.int64, "out_idx", vals.device)
    _check("kselect", lib().kselect(_ptr(vals), rows, cols, k, _ptr(out_vals), _ptr(out_idx),
                                     _stream(stream)))
    return out_vals, out_idx


def kselect_noalloc(vals, k, out_vals, out_idx, stream=None):
    """kselect through the entry point that allocates no device memory; the
    caller provides the outputs (fp32 and int64, [rows, k])."""
    torch = _torch()
    _need(vals, torch.float32, "vals", 2)
    if out_vals is None or out_idx is None:
        raise ValueError("kselect_noalloc: the caller provides out_vals and out_idx")
    rows, cols = vals.shape
    out_vals = _out(out_vals, (rows, k), torch.float32, "out_vals", vals.device)
    out_idx = _out(out_idx, (rows, k), torch.int64, "out_idx", vals.device)
    _check("kselect_noalloc", lib().kselect_noalloc(_ptr(vals), rows, cols, k, _ptr(out_vals),
                                                     _ptr(out_idx), _stream(stream)))
    return out_vals, out_idx
