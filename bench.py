"""Benchmark: batched IVF-PQ search on one GB300 (queries/s), with the list
scan's roofline, the clocks seen during the timed region, an end-to-end figure
through the C ABI with host buffers, and the CPU oracle as a reported baseline.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Workload (default): N = 2e8 vectors, d = 96, nlist = 65,536, PQ m = 32 x 8 bit
(6.4 GB of codes resident in HBM), nq = 10,000 queries per step, nprobe = 64,
k = 100, fp32 lookup tables; seeded synthetic Gaussian mixture (see
approximate_nearest_neighbour_gb300/synthetic.py) drawn on the device, the
index built from it by the library's own index preparation (codebooks trained
by 10 Lloyd iterations on residuals, every vector encoded by nearest centroid
and nearest codeword; see approximate_nearest_neighbour_gb300/indexing.py).
A step is one ivfpq_search call over the whole query batch: coarse quantizer,
table build + list scan + per-chunk selection, and the cross-chunk merge.

With N > 1 (torchrun, one rank per GPU) every rank holds a replica of the index
and searches its own batch of nq queries (queries are independent, so there is
no data-path collective; weak scaling). `value` counts the queries of all
ranks over the slowest rank's time.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from approximate_nearest_neighbour_gb300 import synthetic as S  # noqa: E402

FALLBACK_HBM_GBS = 6800.0
# ncu summary of the scan kernel on the large workload, per kernel family
PROFILE_FILE = os.path.join(ROOT, "profiles", "{kernel}_large.md")
SCAN_SOURCES = ["scan_lm.cuh", "scan2.cuh", "scan.cuh", "select.cuh", "layout.cuh", "common.cuh"]
LOOKUPS_PER_SM_CLOCK = 32  # one 4-byte shared-memory word per bank and clock, 32 banks


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=10)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--lut", default=None, choices=["fp32", "fp16", "fp8"],
                   help="lookup-table storage (default: the workload's stated one: fp32, "
                        "binary16 for billion)")
    p.add_argument("--n", type=int, default=None, help="database size override (development)")
    p.add_argument("--nq", type=int, default=None)
    p.add_argument("--nlist", type=int, default=None, help="list count override (development)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--profile-range", action="store_true",
                   help="bracket the timed calls with cudaProfilerStart/Stop (for "
                        "ncu --profile-from-start off)")
    p.add_argument("--workload", default="large", choices=sorted(WORKLOADS),
                   help="large (default, the headline), mid, billion, flat (exact k-NN) "
                        "or kselect (stand-alone k-selection)")
    p.add_argument("--k", type=int, default=None, help="k override")
    p.add_argument("--nprobe", type=int, default=None,
                   help="nprobe override (IVF-PQ workloads; the mid workload states 16 and 64)")
    p.add_argument("--scan-mode", type=int, default=-1, choices=[-1, 0, 1],
                   help="list scan organisation: -1 automatic, 0 by query, 1 by list")
    return p.parse_args()


# workload -> (shape, nprobe, k); "large" is the configuration the scan target is quoted on
WORKLOADS = {"large": (S.IVFPQ_LARGE, 64, 100), "mid": (S.IVFPQ_MID, 64, 100),
             "billion": (S.IVFPQ_BILLION, 128, 100), "flat": (S.FLAT_1M, 0, 100),
             "kselect": (None, 0, 100)}
KSELECT_ROWS, KSELECT_COLS = 10_000, 65_536  # 2.6 GB of fp32 rows, above L2
WORKLOAD = S.IVFPQ_LARGE
NPROBE, K = 64, 100


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def sm_max_mhz():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            pk = json.load(f)
        if pk.get("sm_max_mhz"):
            return float(pk["sm_max_mhz"])
    return 2070.0


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def scan_source_hash():
    h = hashlib.sha256()
    for name in SCAN_SOURCES:
        with open(os.path.join(ROOT, "approximate_nearest_neighbour_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel):
    """DRAM bytes per scan launch from the committed ncu summary, if it was
    taken on the current scan source; else None."""
    path = PROFILE_FILE.format(kernel=kernel)
    if not os.path.exists(path):
        return None
    vals = {}
    with open(path) as f:
        for line in f:
            if ":" in line and line.strip().startswith("- "):
                k, v = line.strip()[2:].split(":", 1)
                vals[k.strip()] = v.strip().strip("`")
    if vals.get("scan_source_sha256") != scan_source_hash():
        return None
    try:
        return float(vals["dram_bytes_per_full_launch"])
    except (KeyError, ValueError):
        return None


class Clocks:
    """nvidia-smi sampling during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.3)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "samples": len(sm), "reasons": sorted(reasons)}


def make_workload(n=None, nq=None, rank=0, nlist=None):
    """The workload in compressed form (codes drawn directly, list sizes a
    multinomial draw over the component weights): what the oracle is timed
    on. Its per-query work equals that of the encoded index up to the
    sampling noise of the list sizes; the oracle's cost per stored code does
    not depend on the code bytes."""
    w = WORKLOAD
    data = S.compressed_index(w, n=n, nlist=nlist)
    q = S.queries(w.number, data.cent, data.weights, w.sigma, nq or w.nq, salt=rank)
    return data, q


STANDIN_NOTE = ("the workload's shape in compressed form (list sizes drawn from the component "
                "weights, uniform code bytes): the oracle's work per stored code does not "
                "depend on the code bytes")


def cpu_baseline(data, q, lut, target_s=12.0, max_queries=4096):
    """The oracle, as it stands, on this host's cores, on a bounded sample of
    the step's queries, over the workload in compressed form."""
    import oracle
    threads = oracle.NTHREADS
    lut_type = {"fp32": 0, "fp16": 1, "fp8": 2}[lut]
    probe = min(2 * threads, q.shape[0])
    t0 = time.perf_counter()
    oracle.ivfpq_search(q[:probe], data.cent, data.cb, data.list_off, data.codes, data.ids,
                        NPROBE, K, lut_type)
    dt = time.perf_counter() - t0
    n = int(min(max_queries, q.shape[0], max(probe, target_s / max(dt, 1e-6) * probe)))
    t0 = time.perf_counter()
    oracle.ivfpq_search(q[:n], data.cent, data.cb, data.list_off, data.codes, data.ids,
                        NPROBE, K, lut_type)
    dt = time.perf_counter() - t0
    one = min(16, q.shape[0])
    t0 = time.perf_counter()
    oracle.ivfpq_search(q[:one], data.cent, data.cb, data.list_off, data.codes, data.ids,
                        NPROBE, K, lut_type, nthreads=1)
    dt1 = time.perf_counter() - t0
    return {"value": n / dt, "unit": "queries/s", "cores": threads, "kind": "oracle",
            "sample": f"first {n} of the {q.shape[0]} step queries, full-size index "
                      f"({STANDIN_NOTE}), {threads} threads, {dt:.1f} s",
            "per_core": {"value": one / dt1, "unit": "queries/s",
                         "sample": f"first {one} queries, 1 thread, {dt1:.2f} s"},
            "cpu_model": cpu_model()}


L2_BYTES = 129e6  # GB300 L2


def l2_note(nbytes, what):
    """Whether the step's input is larger than L2 (no flush between steps is
    then needed) or would stay cached between steps."""
    where = "larger than L2" if nbytes > L2_BYTES else "fits in L2: timed warm, no flush"
    return f"{what} {nbytes / 1e9:.2f} GB, {where}"


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else platform)."""
    import platform
    import subprocess
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.processor() or platform.machine()


def emit(obj):
    print(json.dumps(obj), flush=True)


# ---------------------------------------------------------------------------
def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    data, q = make_workload(args.n, args.nq, 0, args.nlist)
    threads = oracle.NTHREADS
    per_step = max(1, min(q.shape[0], 4 * threads))
    lut_type = {"fp32": 0, "fp16": 1, "fp8": 2}[args.lut]
    times = []
    for i in range(args.warmup + args.steps):
        sl = slice((i * per_step) % q.shape[0], (i * per_step) % q.shape[0] + per_step)
        t0 = time.perf_counter()
        oracle.ivfpq_search(q[sl], data.cent, data.cb, data.list_off, data.codes, data.ids,
                            NPROBE, K, lut_type)
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    total = sum(times)
    value = per_step * args.steps / total
    emit({"impl": "reference", "metric": f"IVF-PQ queries/s (k={K}, nprobe={NPROBE})",
          "value": value, "unit": "queries/s", "n_gpus": args.gpus, "steps": args.steps,
          "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
          "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
          "data": "synthetic",
          "config": config_dict(args, data.codes.shape[0], data.cent.shape[0]),
          "cpu_baseline": {"value": value, "unit": "queries/s", "cores": threads,
                           "kind": "oracle",
                           "sample": f"{per_step} queries per step (of {q.shape[0]}), "
                                     f"full-size index ({STANDIN_NOTE})"},
          "e2e": {"value": value, "unit": "queries/s", "h2d_bytes_per_step": 0,
                  "d2h_bytes_per_step": 0}})


def config_dict(args, n, nlist):
    w = WORKLOAD
    scaled = args.n is not None or args.nlist is not None
    return {"workload": w.name if not scaled else f"{w.name}(N={n},nlist={nlist})", "n": n,
            "d": w.d, "nlist": nlist, "m": w.m, "nq_per_gpu": args.nq or w.nq, "nprobe": NPROBE, "k": K,
            "lut": args.lut, "scan_mode": {-1: "automatic", 0: "by query", 1: "by list"}[
                args.scan_mode], "parallelism": f"replicas x{args.gpus}",
            "index": "centroids = mixture centres; PQ codebooks trained by 10 Lloyd iterations "
                     "on the residuals of 262,144 rows; every vector encoded by nearest centroid "
                     "and nearest codeword on the GPU",
            "l2": l2_note(n * w.m, "PQ codes")}


def run_ours(args):
    import torch
    import torch.distributed as dist
    from approximate_nearest_neighbour_gb300 import binding as B

    from approximate_nearest_neighbour_gb300 import indexing

    world, rank, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = WORKLOAD
    t_build = time.perf_counter()
    wi = indexing.workload_index(w, dev, n=args.n, nlist=args.nlist)
    torch.cuda.synchronize()
    t_build = time.perf_counter() - t_build
    ix = wi.index
    n, nlist = wi.n, wi.cent.shape[0]
    lens = torch.bincount(wi.lists.long(), minlength=nlist).cpu().numpy()
    lists_are_components = bool(torch.equal(wi.lists, wi.labels))
    searched = wi.searched
    del wi.codes, wi.lists, wi.labels
    torch.cuda.empty_cache()
    q = S.queries(w.number, wi.cent, wi.weights, w.sigma, args.nq or w.nq, salt=rank)
    nq = q.shape[0]
    B.ivfpq_set_lut_type(ix, args.lut)
    B.ivfpq_set_scan_mode(ix, args.scan_mode)
    qd = torch.from_numpy(q).to(dev)
    out_d = torch.empty((nq, K), dtype=torch.float32, device=dev)
    out_i = torch.empty((nq, K), dtype=torch.int64, device=dev)
    stream = torch.cuda.current_stream(dev)

    # algorithmic bytes of one scan launch: the codes of every probed list
    probes, _ = B.ivfpq_search_probes(ix, qd, NPROBE, with_dist=False)
    scan_bytes = float(lens[probes.cpu().numpy()].sum()) * WORKLOAD.m
    scanned_codes = scan_bytes / WORKLOAD.m

    for _ in range(args.warmup):
        B.ivfpq_search(ix, qd, NPROBE, K, out_d, out_i)
    torch.cuda.synchronize()
    B.ivfpq_repaired_queries(ix)

    clocks = Clocks(local)
    B.ivfpq_set_profiling(ix, True)
    launches0 = B.kernel_launches()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    if args.profile_range:
        torch.cuda.profiler.start()
    ev0.record(stream)
    for _ in range(args.steps):
        B.ivfpq_search(ix, qd, NPROBE, K, out_d, out_i)
    ev1.record(stream)
    torch.cuda.synchronize()
    if args.profile_range:
        torch.cuda.profiler.stop()
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    launches = B.kernel_launches() - launches0
    repaired = B.ivfpq_repaired_queries(ix)
    scan_kernel = B.last_scan_kernel(ix)
    elapsed = ev0.elapsed_time(ev1) / 1e3
    sums, count = B.ivfpq_stage_times(ix)
    B.ivfpq_set_profiling(ix, False)
    if world > 1:
        t = torch.tensor([elapsed], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        elapsed = float(t.item())

    # end to end through the C ABI: pinned host queries in, host results out
    qh = torch.from_numpy(q).pin_memory()
    hd = torch.empty((nq, K), dtype=torch.float32).pin_memory()
    hi = torch.empty((nq, K), dtype=torch.int64).pin_memory()
    qbuf = torch.empty_like(qd)
    for _ in range(2):
        qbuf.copy_(qh, non_blocking=True)
        B.ivfpq_search(ix, qbuf, NPROBE, K, out_d, out_i)
        hd.copy_(out_d, non_blocking=True)
        hi.copy_(out_i, non_blocking=True)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        qbuf.copy_(qh, non_blocking=True)
        B.ivfpq_search(ix, qbuf, NPROBE, K, out_d, out_i)
        hd.copy_(out_d, non_blocking=True)
        hi.copy_(out_i, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_elapsed = e0.elapsed_time(e1) / 1e3
    if world > 1:
        t = torch.tensor([e2e_elapsed], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        e2e_elapsed = float(t.item())

    if rank == 0:
        peak, peak_kind = peaks()
        scan_ms = sums[2] / max(count, 1)
        achieved = scan_bytes / (scan_ms / 1e3) / 1e9
        traffic = profiled_traffic(scan_kernel)
        # the look-up bound: one 4-byte shared-memory word per code byte and
        # query, or per two / four queries where the by-list scan packs two
        # binary16 / four E4M3 entries into a word
        nsm = torch.cuda.get_device_properties(dev).multi_processor_count
        sm_mhz = sm_max_mhz()
        per_word = ({"fp16": 2, "fp8": 4}.get(args.lut, 1)
                    if scan_kernel == "ivfpq_scan_lm_kernel" else 1)
        lookup_peak = nsm * LOOKUPS_PER_SM_CLOCK * per_word * sm_mhz * 1e6
        lookups_per_s = scan_bytes / (scan_ms / 1e3)
        if traffic is not None and (args.n is not None or args.nlist is not None
                                    or args.workload != "large" or args.lut != "fp32"
                                    or args.nprobe is not None or args.k is not None):
            traffic = None
        total_q = nq * world * args.steps
        line = {
            "metric": f"IVF-PQ queries/s (k={K}, nprobe={NPROBE})",
            "value": total_q / elapsed, "unit": "queries/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * elapsed / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": config_dict(args, n, nlist),
            "index_build": {"seconds": t_build, "rows_searched_in_full": searched,
                            "lists_equal_components": lists_are_components},
            "repaired_queries_per_step": repaired / args.steps,
            "roofline": {"bound": "hbm", "kernel": scan_kernel, "achieved": achieved,
                         "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                         "peak_source": f"{peak_kind} hbm_gbs (copy)",
                         "traffic": traffic, "algorithmic_bytes_per_launch": scan_bytes,
                         "launch_ms": scan_ms},
            "lookup_roofline": {"bound": "shared-memory look-ups", "kernel": scan_kernel,
                                "achieved": lookups_per_s / 1e12, "unit": "Tlookups/s",
                                "peak": lookup_peak / 1e12, "frac": lookups_per_s / lookup_peak,
                                "peak_source": f"{nsm} SMs x {LOOKUPS_PER_SM_CLOCK} banks x "
                                               f"{per_word} entries per word x "
                                               f"{sm_mhz:.0f} MHz"},
            "stage_ms": {"coarse": sums[0] / max(count, 1), "plan": sums[1] / max(count, 1),
                         "scan": scan_ms, "merge": sums[3] / max(count, 1)},
            "scanned_codes_per_s": scanned_codes / (scan_ms / 1e3) * world,
            "e2e": {"value": total_q / e2e_elapsed, "unit": "queries/s",
                    "h2d_bytes_per_step": int(q.nbytes),
                    "d2h_bytes_per_step": int(hd.numel() * 4 + hi.numel() * 8)},
            "gpu_launches": launches,
            "clocks": clk,
        }
        if not args.no_cpu_baseline:
            data, _ = make_workload(args.n, args.nq, rank, args.nlist)
            line["cpu_baseline"] = cpu_baseline(data, q, args.lut)
        emit(line)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


# ---------------------------------------------------------------------------
# exact k-NN (flat) workload: 1e6 x 128 database, 10,000 queries
FALLBACK_BF16_TFLOPS = 1900.0
TF32_PER_BF16 = 1.1 / 2.25  # nominal dense TF32 / bf16 ratio


def tf32_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            pk = json.load(f)
        return float(pk["bf16_tflops"]) * TF32_PER_BF16, "measured bf16_tflops x 1.1/2.25"
    return FALLBACK_BF16_TFLOPS * TF32_PER_BF16, "fallback bf16 x 1.1/2.25"


def flat_config(args, n, nq, d):
    return {"workload": WORKLOAD.name if args.n is None else f"{WORKLOAD.name}(N={n})", "n": n,
            "d": d, "nq_per_gpu": nq, "k": K, "parallelism": f"replicas x{args.gpus}",
            "l2": l2_note(n * d * 4 + 2 * n * 128 * 4, "fp32 database + tensor-core operands")}


def run_flat(args):
    import torch
    import torch.distributed as dist
    from approximate_nearest_neighbour_gb300 import binding as B

    world, rank, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    db, q = S.flat_database(WORKLOAD, n=args.n, nq=args.nq)
    n, d = db.shape
    nq = q.shape[0]
    dbd = torch.from_numpy(db).to(dev)
    qd = torch.from_numpy(q).to(dev)
    out_d = torch.empty((nq, K), dtype=torch.float32, device=dev)
    out_i = torch.empty((nq, K), dtype=torch.int64, device=dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(args.warmup):
        B.flat_knn(dbd, qd, K, out_d, out_i)
    torch.cuda.synchronize()
    clocks = Clocks(local)
    launches0 = B.kernel_launches()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    if args.profile_range:
        torch.cuda.profiler.start()
    ev0.record(stream)
    for _ in range(args.steps):
        B.flat_knn(dbd, qd, K, out_d, out_i)
    ev1.record(stream)
    torch.cuda.synchronize()
    if args.profile_range:
        torch.cuda.profiler.stop()
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    launches = B.kernel_launches() - launches0
    elapsed = ev0.elapsed_time(ev1) / 1e3
    if world > 1:
        t = torch.tensor([elapsed], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        elapsed = float(t.item())
    # end to end: pinned host queries in, host results out (database resident)
    qh = torch.from_numpy(q).pin_memory()
    hd = torch.empty((nq, K), dtype=torch.float32).pin_memory()
    hi = torch.empty((nq, K), dtype=torch.int64).pin_memory()
    qbuf = torch.empty_like(qd)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        qbuf.copy_(qh, non_blocking=True)
        B.flat_knn(dbd, qbuf, K, out_d, out_i)
        hd.copy_(out_d, non_blocking=True)
        hi.copy_(out_i, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e = e0.elapsed_time(e1) / 1e3
    if rank == 0:
        peak, src = tf32_peak()
        call_s = elapsed / args.steps
        # 3xTF32: three TF32 products of 2 * d flops per (query, database row)
        flops = 3.0 * 2.0 * d * n * nq
        achieved = flops / call_s / 1e12
        line = {
            "metric": f"flat k-NN queries/s (k={K})", "value": nq * world * args.steps / elapsed,
            "unit": "queries/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * call_s, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32 (3xTF32 products)", "data": "synthetic",
            "config": flat_config(args, n, nq, d),
            "roofline": {"bound": "tensor", "kernel": "flat_knn (all kernels of one call)",
                         "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                         "frac": achieved / peak, "peak_source": src, "traffic": None,
                         "algorithmic_flops_per_call": flops},
            "e2e": {"value": nq * world * args.steps / e2e, "unit": "queries/s",
                    "h2d_bytes_per_step": int(q.nbytes),
                    "d2h_bytes_per_step": int(hd.numel() * 4 + hi.numel() * 8)},
            "gpu_launches": launches, "clocks": clk,
        }
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = flat_cpu_baseline(db, q)
        emit(line)


def flat_cpu_baseline(db, q, target_s=10.0):
    import oracle
    threads = oracle.NTHREADS
    m = min(2 * threads, q.shape[0])
    t0 = time.perf_counter()
    oracle.flat_knn(db, q[:m], K)
    dt = time.perf_counter() - t0
    nsel = int(min(q.shape[0], max(m, target_s / max(dt, 1e-6) * m)))
    t0 = time.perf_counter()
    oracle.flat_knn(db, q[:nsel], K)
    dt = time.perf_counter() - t0
    one = min(4, q.shape[0])
    t0 = time.perf_counter()
    oracle.flat_knn(db, q[:one], K, nthreads=1)
    dt1 = time.perf_counter() - t0
    return {"value": nsel / dt, "unit": "queries/s", "cores": threads, "kind": "oracle",
            "sample": f"first {nsel} of the {q.shape[0]} queries, full database, "
                      f"{threads} threads, {dt:.1f} s",
            "per_core": {"value": one / dt1, "unit": "queries/s",
                         "sample": f"first {one} queries, 1 thread, {dt1:.2f} s"},
            "cpu_model": cpu_model()}


def run_flat_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    db, q = S.flat_database(WORKLOAD, n=args.n, nq=args.nq)
    b = flat_cpu_baseline(db, q, target_s=max(1.0, 10.0 / max(args.steps, 1)))
    emit({"impl": "reference", "metric": f"flat k-NN queries/s (k={K})", "value": b["value"],
          "unit": "queries/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
          # the step's queries at the sample's rate
          "ms_per_step": 1e3 * q.shape[0] / b["value"], "higher_is_better": True, "scaling": "weak",
          "vs_baseline": None, "dtype": "f64", "data": "synthetic",
          "config": flat_config(args, db.shape[0], q.shape[0], db.shape[1]), "cpu_baseline": b,
          "e2e": {"value": b["value"], "unit": "queries/s", "h2d_bytes_per_step": 0,
                  "d2h_bytes_per_step": 0}})


# ---------------------------------------------------------------------------
# stand-alone row-wise k-selection: 10,000 rows x 65,536 fp32 values
def run_kselect(args):
    import numpy as np
    import torch
    from approximate_nearest_neighbour_gb300 import binding as B

    world, rank, local = dist_env()
    if args.impl == "reference" and rank != 0:
        return
    rows, cols = args.nq or KSELECT_ROWS, args.n or KSELECT_COLS
    x = S.random_rows(rows, cols, seed=20260)
    if args.impl == "reference":
        run_kselect_reference(args, x)
        return
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    vals = torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(dev)
    out_v = torch.empty((rows, K), dtype=torch.float32, device=dev)
    out_i = torch.empty((rows, K), dtype=torch.int64, device=dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(args.warmup):
        B.kselect(vals, K, out_v, out_i)
    torch.cuda.synchronize()
    clocks = Clocks(local)
    launches0 = B.kernel_launches()
    clocks.start()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    if args.profile_range:
        torch.cuda.profiler.start()
    e0.record(stream)
    for _ in range(args.steps):
        B.kselect(vals, K, out_v, out_i)
    e1.record(stream)
    torch.cuda.synchronize()
    if args.profile_range:
        torch.cuda.profiler.stop()
    clk = clocks.stop()
    launches = B.kernel_launches() - launches0
    call_s = e0.elapsed_time(e1) / 1e3 / args.steps
    # end to end: host rows in, host results out
    xh = torch.from_numpy(np.ascontiguousarray(x, np.float32)).pin_memory()
    hv = torch.empty((rows, K), dtype=torch.float32).pin_memory()
    hi = torch.empty((rows, K), dtype=torch.int64).pin_memory()
    buf = torch.empty_like(vals)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(args.steps):
        buf.copy_(xh, non_blocking=True)
        B.kselect(buf, K, out_v, out_i)
        hv.copy_(out_v, non_blocking=True)
        hi.copy_(out_i, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_s = e0.elapsed_time(e1) / 1e3 / args.steps
    peak, kind = peaks()
    nbytes = 4.0 * rows * cols
    line = {"metric": f"kselect rows/s (k={K}, {cols} columns)", "value": rows / call_s,
            "unit": "rows/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * call_s, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": f"kselect_{rows}x{cols}", "rows": rows, "cols": cols, "k": K,
                       "l2": l2_note(nbytes, "fp32 input")},
            "roofline": {"bound": "hbm", "kernel": "kselect (all kernels of one call)", "achieved": nbytes / call_s / 1e9,
                         "peak": peak, "unit": "GB/s", "frac": nbytes / call_s / 1e9 / peak,
                         "peak_source": f"{kind} hbm_gbs (copy)", "traffic": None,
                         "algorithmic_bytes_per_call": nbytes},
            "e2e": {"value": rows / e2e_s, "unit": "rows/s", "h2d_bytes_per_step": int(nbytes),
                    "d2h_bytes_per_step": int(rows * K * 12)},
            "gpu_launches": launches, "clocks": clk}
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = kselect_cpu_baseline(x)
    emit(line)


def kselect_cpu_baseline(x, target_s=10.0):
    import oracle
    threads = oracle.NTHREADS
    m = min(x.shape[0], 2 * threads)
    t0 = time.perf_counter()
    oracle.kselect(x[:m], K)
    dt = time.perf_counter() - t0
    m = int(min(x.shape[0], max(m, target_s / max(dt, 1e-6) * m)))
    t0 = time.perf_counter()
    oracle.kselect(x[:m], K)
    dt = time.perf_counter() - t0
    one = min(16, x.shape[0])
    t0 = time.perf_counter()
    oracle.kselect(x[:one], K, nthreads=1)
    dt1 = time.perf_counter() - t0
    return {"value": m / dt, "unit": "rows/s", "cores": threads, "kind": "oracle",
            "sample": f"first {m} of the {x.shape[0]} rows, {threads} threads, {dt:.1f} s",
            "per_core": {"value": one / dt1, "unit": "rows/s",
                         "sample": f"first {one} rows, 1 thread, {dt1:.2f} s"},
            "cpu_model": cpu_model()}


def run_kselect_reference(args, x):
    rows, cols = x.shape
    b = kselect_cpu_baseline(x, target_s=max(1.0, 10.0 / max(args.steps, 1)))
    emit({"impl": "reference", "metric": f"kselect rows/s (k={K}, {cols} columns)",
          "value": b["value"], "unit": "rows/s", "n_gpus": args.gpus, "steps": args.steps,
          "warmup": args.warmup, "ms_per_step": 1e3 * rows / b["value"],
          "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
          "data": "synthetic",
          "config": {"workload": f"kselect_{rows}x{cols}", "rows": rows, "cols": cols, "k": K},
          "cpu_baseline": b,
          "e2e": {"value": b["value"], "unit": "rows/s", "h2d_bytes_per_step": 0,
                  "d2h_bytes_per_step": 0}})


def main():
    global WORKLOAD, NPROBE, K
    args = parse()
    WORKLOAD, NPROBE, K = WORKLOADS[args.workload]
    if args.lut is None:
        # the billion workload states binary16 tables; the others fp32 (the
        # large workload's fp16 / E4M3 variants are recall-gated in the tests)
        args.lut = "fp16" if args.workload == "billion" else "fp32"
    if args.k is not None:
        K = args.k
    if args.nprobe is not None:
        NPROBE = args.nprobe
    if args.workload == "kselect":
        run_kselect(args)
    elif args.workload == "flat":
        if args.impl == "reference":
            run_flat_reference(args)
        else:
            run_flat(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
