"""Comparison rules between the CUDA path and the CPU oracle.

Tolerance: a GPU distance g matches an oracle distance D when
|g - D| <= max(1e-4 |D|, 1e-5). The GPU sums at most 64 fp32 table entries
(ADC) or 128 fp32 squares (coarse and flat distances, direct form), each
with a relative rounding error of 2^-24, so its relative error stays near
1e-5; 1e-4 leaves a tenfold margin, and the absolute floor covers
distances that cancel to nearly zero. Result ids
are compared as sets after removing the boundary ties: every id whose oracle
distance is below the k-th oracle distance by more than the tolerance must be
returned, and every returned id must be a genuine candidate whose oracle
distance matches the returned distance.
"""

from __future__ import annotations

import numpy as np

RTOL = 1e-4
ATOL = 1e-5


def tol(d):
    return np.maximum(RTOL * np.abs(d), ATOL)


def compare_knn(gd, gi, od, oi, rtol=RTOL, atol=ATOL, context=""):
    """gd, gi: GPU [nq, k]; od, oi: oracle [nq, k2] with k2 >= k (extra oracle
    entries give the distances of candidates just past the boundary)."""
    gd = np.asarray(gd, np.float64)
    gi = np.asarray(gi)
    od = np.asarray(od, np.float64)
    oi = np.asarray(oi)
    nq, k = gd.shape
    assert od.shape[1] >= k
    for r in range(nq):
        D = od[r, :k]
        g = gd[r]
        fin = np.isfinite(D)
        t = np.maximum(rtol * np.abs(D), atol)
        diff = np.abs(np.where(fin, g, 0.0) - np.where(fin, D, 0.0))
        bad = np.nonzero(fin & ~(diff <= t))[0]
        assert bad.size == 0, f"{context} row {r}: distance mismatch at ranks {bad[:8]}: " \
                              f"gpu {g[bad[:4]]} oracle {D[bad[:4]]}"
        assert np.all(np.isinf(g[~fin])), f"{context} row {r}: missing results must be +inf"
        assert np.all(gi[r][~fin] == -1), f"{context} row {r}: missing results must have id -1"
        # ids
        real = gi[r][gi[r] >= 0]
        assert len(set(real.tolist())) == real.size, f"{context} row {r}: duplicate ids"
        if not fin.any():
            continue
        Dk = D[fin][-1]
        tk = max(rtol * abs(Dk), atol)
        must = set(oi[r, :k][(D < Dk - tk) & fin].tolist())
        got = set(real.tolist())
        missing = must - got
        assert not missing, f"{context} row {r}: ids {sorted(missing)[:8]} missing"
        known = {int(i): float(d) for i, d in zip(oi[r], od[r]) if i >= 0}
        for i, d in zip(gi[r], g):
            if i < 0:
                continue
            assert int(i) in known, f"{context} row {r}: id {i} is not a top candidate"
            dd = known[int(i)]
            assert abs(dd - d) <= max(rtol * abs(dd), atol), \
                f"{context} row {r}: id {i} distance {d} vs oracle {dd}"


def check_probes(gpu_probes, oracle_probes, oracle_dist_all_fn, rtol=RTOL):
    """Per query, the GPU probe set may differ from the oracle's only by lists
    whose oracle coarse distance is within tolerance of the nprobe-th one.
    oracle_dist_all_fn(row) -> exact distances of the query to all centroids."""
    gpu_probes = np.asarray(gpu_probes)
    oracle_probes = np.asarray(oracle_probes)
    nprobe = gpu_probes.shape[1]
    ndiff = 0
    for r in range(gpu_probes.shape[0]):
        a, b = set(gpu_probes[r].tolist()), set(oracle_probes[r].tolist())
        if a == b:
            continue
        ndiff += 1
        dc = oracle_dist_all_fn(r)
        dn = np.sort(dc)[nprobe - 1]
        for l in a ^ b:
            assert abs(dc[l] - dn) <= max(rtol * abs(dn), ATOL), \
                f"row {r}: probe {l} differs but is not a tie ({dc[l]} vs {dn})"
    return ndiff


def check_kselect(vals, k, ov, oi, gv, gi):
    """Exact values (the k smallest, ascending); indices valid and distinct,
    and every index whose value is below the k-th is present."""
    vals = np.asarray(vals)
    rows, cols = vals.shape
    kk = min(k, cols)
    assert np.array_equal(gv[:, :kk], ov[:, :kk]), "kselect values differ"
    assert np.all(np.isposinf(gv[:, kk:])) and np.all(gi[:, kk:] == -1), "kselect padding"
    for r in range(rows):
        idx = gi[r, :kk]
        assert np.all((idx >= 0) & (idx < cols)), f"row {r}: index out of range"
        assert len(set(idx.tolist())) == kk, f"row {r}: duplicate index"
        assert np.array_equal(vals[r, idx], gv[r, :kk]), f"row {r}: index does not hold its value"
        if kk:
            kth = ov[r, kk - 1]
            must = set(oi[r, :kk][ov[r, :kk] < kth].tolist())
            assert must <= set(idx.tolist()), f"row {r}: missing indices"
