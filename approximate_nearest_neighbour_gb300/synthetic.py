"""Seeded synthetic workloads for IVF-PQ search and flat k-NN.

This module only draws random numbers and arranges them; it holds none of the
search method's arithmetic (no distances, no quantization, no selection). Both
the tests (which feed the same arrays to the CPU oracle and to the CUDA path)
and the benchmark use it. It depends on numpy; the device-side draws of large
databases use torch's CUDA generator.

Recipe (stand-in for the pages' Sift1M / Sift1B / Deep1B / Yfcc100M datasets,
which are not available here):

* Gaussian mixture: centres ~ N(0, 1) per dimension; a point of component c is
  centre_c + sigma * N(0, I). Component weights are uniform, or Zipf with
  exponent 0.5 (p_c proportional to (c + 1)^-0.5 in component order).
* Coarse centroids are the true mixture centres (nlist = number of components).
* Large databases as raw vectors, drawn on the device in seeded blocks so
  that any row range can be drawn again: the component of every row
  (`device_labels`), then the rows (`device_points`). The index is built from
  them by the library's own index preparation (indexing.py).
* Large databases in compressed form (`compressed_index`): list sizes from a
  multinomial draw over the component weights, every code byte uniform over
  the 256 reproduction values, and PQ codebooks sampled from the residual
  distribution (codeword = sigma * N(0, I_dsub)); a stored vector is exactly
  centroid + decoded residual.
* Queries are drawn from the same mixture.

Seeds: 20170228 + 1000 * workload number; sub-streams 0 = centres,
1 = database, 2 = queries, 3 = codebooks / training sample.
"""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np

BASE_SEED = 20170228

STREAM_CENTRES, STREAM_DB, STREAM_QUERIES, STREAM_TRAIN = 0, 1, 2, 3


@dataclass(frozen=True)
class IVFPQWorkload:
    """Shape of one IVF-PQ workload."""
    name: str
    number: int
    n: int
    d: int
    nlist: int
    m: int
    sigma: float
    zipf: bool
    nq: int
    nprobe: tuple
    k: tuple
    lut: tuple


@dataclass(frozen=True)
class FlatWorkload:
    name: str
    number: int
    n: int
    d: int
    ncomp: int
    sigma: float
    nq: int
    k: tuple


# The five workloads of the headline benchmark family.
IVFPQ_TINY = IVFPQWorkload("ivfpq_tiny_N1e5_d64_nlist256_m8", 1, 100_000, 64, 256, 8, 0.1,
                           False, 100, (8,), (10,), ("fp32",))
FLAT_1M = FlatWorkload("flat_N1e6_d128", 2, 1_000_000, 128, 1024, 0.2, 10_000, (1, 100, 1024))
IVFPQ_MID = IVFPQWorkload("ivfpq_mid_N1e7_d128_nlist4096_m16", 3, 10_000_000, 128, 4096, 16,
                          0.15, True, 10_000, (16, 64), (100,), ("fp32",))
IVFPQ_LARGE = IVFPQWorkload("ivfpq_large_N2e8_d96_nlist65536_m32", 4, 200_000_000, 96, 65536,
                            32, 0.15, False, 10_000, (64,), (100,), ("fp32", "fp16", "fp8"))
IVFPQ_BILLION = IVFPQWorkload("ivfpq_billion_N1e9_d96_nlist262144_m8", 5, 1_000_000_000, 96,
                              262144, 8, 0.15, True, 10_000, (128,), (1, 100, 1000), ("fp16",))

WORKLOADS = {w.number: w for w in (IVFPQ_TINY, FLAT_1M, IVFPQ_MID, IVFPQ_LARGE, IVFPQ_BILLION)}


def rng(number: int, stream: int, salt: int = 0) -> np.random.Generator:
    seed = BASE_SEED + 1000 * number
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, stream, salt])))


def component_weights(ncomp: int, zipf: bool) -> np.ndarray:
    if not zipf:
        return np.full(ncomp, 1.0 / ncomp)
    w = (np.arange(ncomp, dtype=np.float64) + 1.0) ** -0.5
    return w / w.sum()


def centres(number: int, ncomp: int, d: int) -> np.ndarray:
    return rng(number, STREAM_CENTRES).standard_normal((ncomp, d), dtype=np.float32)


def draw_components(g: np.random.Generator, n: int, weights: np.ndarray) -> np.ndarray:
    """Component of each of n points by inverse-CDF sampling."""
    cdf = np.cumsum(weights)
    cdf[-1] = 1.0
    u = g.random(n)
    return np.searchsorted(cdf, u, side="right").astype(np.int32)


def mixture_points(g: np.random.Generator, cent: np.ndarray, comps: np.ndarray,
                   sigma: float) -> np.ndarray:
    x = g.standard_normal((comps.shape[0], cent.shape[1]), dtype=np.float32)
    x *= np.float32(sigma)
    x += cent[comps]
    return x


def queries(number: int, cent: np.ndarray, weights: np.ndarray, sigma: float, nq: int,
            salt: int = 0) -> np.ndarray:
    g = rng(number, STREAM_QUERIES, salt)
    comps = draw_components(g, nq, weights)
    return mixture_points(g, cent, comps, sigma)


def residual_codebooks(number: int, m: int, dsub: int, sigma: float) -> np.ndarray:
    """Codewords drawn from the residual distribution: [m, 256, dsub] fp32."""
    g = rng(number, STREAM_TRAIN)
    return (g.standard_normal((m, 256, dsub), dtype=np.float32) * np.float32(sigma))


@dataclass
class CompressedIndexData:
    """An IVF-PQ database in compressed form, grouped by list.

    codes[v] (m bytes) and ids[v] belong to list l for
    list_off[l] <= v < list_off[l + 1]; list_ids[v] = l.
    """
    cent: np.ndarray
    cb: np.ndarray
    list_off: np.ndarray
    list_ids: np.ndarray
    codes: np.ndarray
    ids: np.ndarray
    weights: np.ndarray


def compressed_index(w: IVFPQWorkload, n: int | None = None, nlist: int | None = None,
                     salt: int = 0) -> CompressedIndexData:
    """Generate a workload's database directly as codes (see module docstring).
    n / nlist override the workload's sizes for scaled-down cases."""
    n = w.n if n is None else n
    nlist = w.nlist if nlist is None else nlist
    cent = centres(w.number, nlist, w.d)
    cb = residual_codebooks(w.number, w.m, w.d // w.m, w.sigma)
    weights = component_weights(nlist, w.zipf)
    g = rng(w.number, STREAM_DB, salt)
    sizes = g.multinomial(n, weights).astype(np.int64)
    off = np.zeros(nlist + 1, np.int64)
    np.cumsum(sizes, out=off[1:])
    list_ids = np.repeat(np.arange(nlist, dtype=np.int32), sizes)
    codes = np.frombuffer(g.bytes(n * w.m), dtype=np.uint8).reshape(n, w.m)
    ids = np.arange(n, dtype=np.int64)
    return CompressedIndexData(cent, cb, off, list_ids, codes, ids, weights)


def shuffled(data: CompressedIndexData, number: int, salt: int = 7):
    """The same database as row-major arrays in a random order (so that adding
    it exercises the scatter into lists). Returns (codes, list_ids, ids)."""
    g = rng(number, STREAM_DB, salt)
    perm = g.permutation(data.codes.shape[0])
    return (np.ascontiguousarray(data.codes[perm]), np.ascontiguousarray(data.list_ids[perm]),
            np.ascontiguousarray(data.ids[perm]))


def flat_database(w: FlatWorkload, n: int | None = None, nq: int | None = None):
    """(db [n, d], queries [nq, d]) from the workload's Gaussian mixture."""
    n = w.n if n is None else n
    nq = w.nq if nq is None else nq
    cent = centres(w.number, w.ncomp, w.d)
    weights = component_weights(w.ncomp, False)
    g = rng(w.number, STREAM_DB)
    comps = draw_components(g, n, weights)
    db = mixture_points(g, cent, comps, w.sigma)
    q = queries(w.number, cent, weights, w.sigma, nq)
    return db, q


def tiny_raw(w: IVFPQWorkload = IVFPQ_TINY, n: int | None = None):
    """Raw mixture vectors for the tiny workload, whose index is built by
    clustering, residual computation and PQ training (done by the caller).
    Returns (centres, points, train_init_rows)."""
    n = w.n if n is None else n
    cent = centres(w.number, w.nlist, w.d)
    weights = component_weights(w.nlist, w.zipf)
    g = rng(w.number, STREAM_DB)
    comps = draw_components(g, n, weights)
    x = mixture_points(g, cent, comps, w.sigma)
    init = rng(w.number, STREAM_TRAIN).choice(n, size=256, replace=False).astype(np.int64)
    return cent, x, init


# ---------------------------------------------------------------------------
# large databases as raw vectors drawn on the device

NOISE_BLOCK = 1 << 22   # rows per seeded block of device-side noise
LABEL_BLOCK = 1 << 24   # rows per seeded block of device-side labels
TRAIN_ROWS = 262_144    # rows of the product-quantizer training sample


def _block_seed(number: int, role: int, block: int, salt: int) -> int:
    ss = np.random.SeedSequence([BASE_SEED + 1000 * number, STREAM_DB, role + salt, block])
    return int(ss.generate_state(1, np.uint64)[0] >> np.uint64(1))


def device_labels(number: int, n: int, weights: np.ndarray, device, salt: int = 0):
    """Mixture component of each of n database rows (torch int32 [n] on
    `device`), drawn in blocks of LABEL_BLOCK rows from generators seeded by
    (workload, block): uniform integers for uniform weights, else inverse-CDF
    sampling of the weights."""
    import torch
    out = torch.empty((n,), dtype=torch.int32, device=device)
    ncomp = weights.shape[0]
    uniform = bool(np.all(weights == weights[0]))
    cdf = np.cumsum(weights)
    cdf[-1] = 1.0
    cdf_d = torch.from_numpy(cdf).to(device)
    for blk, a in enumerate(range(0, n, LABEL_BLOCK)):
        b = min(n, a + LABEL_BLOCK)
        g = torch.Generator(device=device)
        g.manual_seed(_block_seed(number, 100, blk, salt))
        if uniform:
            out[a:b] = torch.randint(0, ncomp, (b - a,), generator=g, device=device,
                                     dtype=torch.int32)
        else:
            u = torch.rand((b - a,), generator=g, device=device, dtype=torch.float64)
            out[a:b] = torch.searchsorted(cdf_d, u, right=True).clamp_(max=ncomp - 1).int()
    return out


def device_points(number: int, cent, labels_dev, sigma: float, start: int, count: int,
                  salt: int = 0):
    """Rows [start, start + count) of a mixture database, drawn on cent's
    device (torch fp32 [count, d]): the centre of each row's component plus
    sigma * N(0, I). Row i's noise is row i mod NOISE_BLOCK of block
    i // NOISE_BLOCK, which comes from a generator seeded by (workload,
    block), so the same rows come back whatever range they are drawn in."""
    import torch
    d = cent.shape[1]
    dev = cent.device
    out = torch.empty((count, d), dtype=torch.float32, device=dev)
    if count == 0:
        return out
    for blk in range(start // NOISE_BLOCK, (start + count - 1) // NOISE_BLOCK + 1):
        g = torch.Generator(device=dev)
        g.manual_seed(_block_seed(number, 200, blk, salt))
        z = torch.randn((NOISE_BLOCK, d), generator=g, device=dev, dtype=torch.float32)
        lo = max(start, blk * NOISE_BLOCK)
        hi = min(start + count, (blk + 1) * NOISE_BLOCK)
        out[lo - start:hi - start] = z[lo - blk * NOISE_BLOCK:hi - blk * NOISE_BLOCK]
        del z
    out.mul_(sigma)
    out.add_(cent[labels_dev[start:start + count].long()])
    return out


def training_rows(number: int, n: int) -> tuple:
    """(rows used to train the product quantizer, 256 of them that seed its
    codewords). The database rows are in random order, so its first
    min(n, TRAIN_ROWS) rows are a seeded random sample of it; the seeds are
    256 distinct rows of that sample."""
    ntrain = min(n, TRAIN_ROWS)
    init = rng(number, STREAM_TRAIN).choice(ntrain, size=256, replace=False).astype(np.int64)
    return ntrain, init


def random_rows(rows: int, cols: int, seed: int, kind: str = "normal") -> np.ndarray:
    """Rows for k-selection tests: normal values, many ties, sorted,
    reverse-sorted, or with +-inf entries."""
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([BASE_SEED, 99, seed])))
    if kind == "normal":
        return g.standard_normal((rows, cols), dtype=np.float32)
    if kind == "ties":
        return g.integers(0, 8, size=(rows, cols)).astype(np.float32)
    if kind == "equal":
        return np.full((rows, cols), 1.5, np.float32)
    if kind == "sorted":
        return np.sort(g.standard_normal((rows, cols), dtype=np.float32), axis=1)
    if kind == "reverse":
        return np.sort(g.standard_normal((rows, cols), dtype=np.float32), axis=1)[:, ::-1].copy()
    if kind == "inf":
        x = g.standard_normal((rows, cols), dtype=np.float32)
        mask = g.random((rows, cols))
        x[mask < 0.2] = np.inf
        x[mask > 0.95] = -np.inf
        return x
    raise ValueError(kind)
