"""Building an IVF-PQ index from raw vectors with the library's own index
preparation, in the order of the index construction steps on the 8-bit-float
page ("Custom 8-bit floating point value format ...", steps 1-4):

1. coarse centroids (given: the caller's quantizer);
2. residuals of a training sample against its nearest centroid
   (ivfpq_residuals);
3. product-quantizer codebooks, Lloyd iterations on those residuals
   (pq_train);
4. every vector's list (nearest centroid) and code (nearest codeword per
   sub-space, ivfpq_encode / ivfpq_encode_hinted), then ivfpq_add.

Every step runs in the library's kernels; this module only sequences the
calls and moves device tensors. `workload_index` applies it to the seeded
mixture databases of synthetic.py, drawn on the device block by block.
"""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from . import binding as B
from . import synthetic as S

ENCODE_ROWS = 1 << 24  # rows drawn and encoded per step (6.4 GB of fp32 at d = 96)


def train_codebooks(centroids, train_x, m, niter, init):
    """PQ codebooks [m, 256, d/m] (device fp32) trained by `niter` Lloyd
    iterations on the residuals of train_x (device fp32 [n, d]) against their
    nearest centroid, seeded from rows `init` (256 row indices), and the
    objective of each assignment pass."""
    import torch
    _, resid = B.ivfpq_residuals(centroids, train_x)
    init_d = torch.as_tensor(np.asarray(init, np.int64), device=train_x.device)
    cb, obj = B.pq_train(resid, m, niter, init_d)
    return cb, obj


def encode_and_add(index, n, draw, rows=ENCODE_ROWS):
    """Encodes n vectors, produced `rows` at a time by draw(start, count) ->
    (x device fp32 [count, d], hint device int32 [count] or None), and adds
    them with ids 0 .. n-1. Returns (codes uint8 [n, m], list ids int32 [n],
    rows that needed a full nearest-centroid search), all on the device."""
    import torch
    dev = None
    codes = lists = None
    searched = 0
    for a in range(0, n, rows):
        c = min(rows, n - a)
        x, hint = draw(a, c)
        if codes is None:
            dev = x.device
            codes = torch.empty((n, index.m), dtype=torch.uint8, device=dev)
            lists = torch.empty((n,), dtype=torch.int32, device=dev)
        if hint is None:
            lc, cc = B.ivfpq_encode(index, x)
            lists[a:a + c].copy_(lc)
            codes[a:a + c].copy_(cc)
            searched += c
        else:
            _, _, s = B.ivfpq_encode_hinted(index, x, hint, lists[a:a + c], codes[a:a + c])
            searched += s
        del x, hint
    if n == 0:
        return None, None, 0
    ids = torch.arange(n, dtype=torch.int64, device=dev)
    B.ivfpq_add(index, codes, lists, ids)
    del ids
    return codes, lists, searched


@dataclass
class WorkloadIndex:
    """An index built from a workload's raw mixture vectors."""
    index: object
    cent: np.ndarray        # host fp32 [nlist, d] (the mixture centres)
    cent_dev: object        # device copy
    codebooks: object       # device fp32 [m, 256, d/m], trained
    codes: object           # device uint8 [n, m]: row i's code (id i)
    lists: object           # device int32 [n]: row i's list
    labels: object          # device int32 [n]: row i's mixture component
    weights: np.ndarray     # component weights
    objective: np.ndarray   # PQ training objective per pass
    searched: int           # rows whose nearest centroid needed a full search
    n: int


def workload_index(w, device, n=None, nlist=None, niter=10, salt=0):
    """IVF-PQ index of workload w (synthetic.IVFPQWorkload) built from its raw
    vectors: centroids = the mixture centres; codebooks trained by `niter`
    Lloyd iterations on the residuals of the first min(n, 262,144) rows (a
    seeded random sample, the rows being in random order), seeded from 256 of
    them; every row encoded (its mixture component as the list hint, which the
    encoder accepts only where the triangle inequality proves it nearest) and
    added with id = row index. n / nlist override the workload's sizes."""
    import torch
    n = w.n if n is None else n
    nlist = w.nlist if nlist is None else nlist
    cent = S.centres(w.number, nlist, w.d)
    cent_d = torch.from_numpy(cent).to(device)
    weights = S.component_weights(nlist, w.zipf)
    labels = S.device_labels(w.number, n, weights, device, salt=salt)
    ntrain, init = S.training_rows(w.number, n)
    xt = S.device_points(w.number, cent_d, labels, w.sigma, 0, ntrain, salt=salt)
    cb, obj = train_codebooks(cent_d, xt, w.m, niter, init)
    del xt
    ix = B.ivfpq_index_create(cent_d, cb)

    def draw(a, c):
        return (S.device_points(w.number, cent_d, labels, w.sigma, a, c, salt=salt),
                labels[a:a + c])

    codes, lists, searched = encode_and_add(ix, n, draw)
    return WorkloadIndex(ix, cent, cent_d, cb, codes, lists, labels, weights, obj, searched, n)


def lists_on_host(wi, list_set):
    """(codes, list ids, ids) of the rows of a WorkloadIndex whose list is in
    list_set (host numpy arrays, row order), for an oracle run over those
    lists."""
    import torch
    mask = torch.zeros((wi.cent.shape[0],), dtype=torch.bool, device=wi.lists.device)
    mask[torch.as_tensor(np.asarray(list_set, np.int64), device=mask.device)] = True
    sel = mask[wi.lists.long()]
    rows = torch.nonzero(sel).squeeze(1)
    return (wi.codes[rows].cpu().numpy(), wi.lists[rows].cpu().numpy(),
            rows.cpu().numpy().astype(np.int64))
