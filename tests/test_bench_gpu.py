"""bench.py end to end on small workloads: the JSON line's contract keys, the
end-to-end leg, the graph and one-call paths (a quick run, not a timing)."""
from __future__ import annotations

import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench(*args: str) -> dict:
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                         capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, out.stdout[-2000:]
    return json.loads(lines[0])


def _contract(d: dict) -> None:
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "roofline", "clocks", "gpu_launches"):
        assert key in d, key
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["gpu_launches"] > 0
    r = d["roofline"]
    assert r["bound"] == "hbm" and r["peak"] > 0 and r["achieved"] > 0
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-3


def test_bench_stand_with_the_end_to_end_leg():
    d = _bench("--workload", "stand", "--steps", "2", "--warmup", "3", "--e2e-steps", "1",
               "--no-cpu-baseline")
    _contract(d)
    e = d["e2e"]
    assert e["value"] > 0 and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0


def test_bench_pythia_one_call_rounds_in_a_graph():
    d = _bench("--workload", "pythia14m", "--api", "round", "--graph", "--steps", "3",
               "--warmup", "3", "--e2e-steps", "0", "--no-cpu-baseline")
    _contract(d)
    assert d["config"]["api"] == "round" and d["config"]["cuda_graph"] is True
