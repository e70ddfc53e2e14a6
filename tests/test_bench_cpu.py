"""bench.py's reference arm (the oracle on the host cores) at small sizes:
one JSON line with the keys every bench line carries, and nothing from a
rank other than 0."""

import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

COMMON = {"metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
          "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
          "cpu_baseline", "e2e", "impl"}


def _run(args, env_extra=None):
    env = dict(os.environ)
    env.update(env_extra or {})
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args],
                       capture_output=True, text=True, timeout=600, cwd=ROOT, env=env)
    assert p.returncode == 0, p.stderr[-2000:]
    return [ln for ln in p.stdout.splitlines() if ln.startswith("{")]


@pytest.mark.parametrize("extra", [
    ["--n", "20000", "--nlist", "64", "--nq", "16"],
    ["--workload", "flat", "--n", "3000", "--nq", "16"],
    ["--workload", "kselect", "--n", "4096", "--nq", "32", "--k", "50"],
])
def test_reference_arm_prints_one_contract_line(extra):
    lines = _run(["--impl", "reference", "--steps", "3", "--warmup", "3", *extra])
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert COMMON <= set(d), COMMON - set(d)
    assert d["impl"] == "reference" and d["value"] > 0 and d["ms_per_step"] > 0
    assert d["steps"] == 3 and d["warmup"] == 3 and d["higher_is_better"] is True
    assert d["vs_baseline"] is None and d["data"] == "synthetic"
    assert "workload" in d["config"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    assert cb["unit"] == d["unit"] and "sample" in cb
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0


@pytest.mark.parametrize("workload", ["large", "flat", "kselect"])
def test_reference_arm_other_ranks_print_nothing(workload):
    lines = _run(["--impl", "reference", "--workload", workload, "--steps", "3", "--warmup", "3",
                  "--n", "4096", "--nq", "16", "--nlist", "64"],
                 {"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert lines == []


def test_reference_arm_takes_the_nprobe_override():
    """--nprobe reaches the timed configuration: the metric and the config
    name it (the mid workload states nprobe 16 and 64)."""
    lines = _run(["--impl", "reference", "--workload", "mid", "--nprobe", "16", "--steps", "3",
                  "--warmup", "3", "--n", "20000", "--nlist", "64", "--nq", "16"])
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert "nprobe=16" in d["metric"]
    assert d["config"]["nprobe"] == 16
