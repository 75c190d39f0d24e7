"""Host-side pieces of bench.py: the CPU oracle legs split over host threads."""
from concurrent.futures import ThreadPoolExecutor

import numpy as np

import bench
import oracle
from checkpoint_averaging_gb300 import workloads as W


def _arrays(n, k, seed):
    rng = np.random.default_rng(seed)
    theta = (rng.standard_normal(n) * 0.02).astype(np.float32)
    xs = [(theta + rng.standard_normal(n).astype(np.float32) * 1e-3).astype(np.float32)
          for _ in range(k)]
    m = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    return theta, xs, m, theta.copy()


def test_split_oracle_equals_one_call_bitwise():
    n, tokens = 10_007, [120_000, 101_313, 149_999]
    theta, xs, m, e = _arrays(n, len(tokens), 7)
    t1, m1, e1 = theta.copy(), m.copy(), e.copy()
    oracle.merge_tensor(xs, t1, mode=oracle.DELTA_NESTEROV, tokens=tokens, lr=0.7, mu=0.9,
                        m=m1, e=e1, beta=0.9)

    def one(lo, hi):
        oracle.merge_tensor([x[lo:hi] for x in xs], theta[lo:hi], mode=oracle.DELTA_NESTEROV,
                            tokens=tokens, lr=0.7, mu=0.9, m=m[lo:hi], e=e[lo:hi], beta=0.9)

    with ThreadPoolExecutor(max_workers=4) as pool:
        bench.run_split(one, n, 4, pool)
    for a, b in ((theta, t1), (m, m1), (e, e1)):
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_split_covers_every_element_once():
    seen = np.zeros(1001, np.int32)

    def mark(lo, hi):
        seen[lo:hi] += 1

    with ThreadPoolExecutor(max_workers=3) as pool:
        for threads in (1, 2, 3, 7, 2000):
            seen[:] = 0
            bench.run_split(mark, seen.size, threads, pool)
            assert (seen == 1).all()


def test_threaded_sample_rate_runs_on_a_small_workload():
    wl = W.workload("pythia14m")
    gbs, secs, n, desc = bench.oracle_sample_rate(wl, 0.2, max_elems=1 << 18,
                                                  pool_elems=1 << 16, threads=2)
    assert gbs > 0 and secs > 0 and n == 1 << 18
    assert "2 host threads" in desc


def test_other_configs_records_each_child_line_or_its_error(monkeypatch):
    """A default run's other_configs: one record per configuration, with the
    child's figures, or the child's last error line when it failed."""
    import json
    import subprocess
    import types

    good = {"metric": "m", "value": 123.4, "unit": "GB/s", "ms_per_step": 1.5,
            "config": {"workload": "w"}, "gpu_launches": 3,
            "roofline": {"frac": 0.9, "bound": "hbm", "kernel": "k", "traffic": None},
            "clocks": {"sm_mhz": 2070.0, "reasons": []}}
    calls = []

    def fake_run(cmd, capture_output, text, timeout):
        calls.append(cmd)
        if len(calls) == 2:
            return types.SimpleNamespace(returncode=1, stdout="", stderr="a\nboom\n")
        return types.SimpleNamespace(returncode=0, stdout="noise\n" + json.dumps(good) + "\n",
                                     stderr="")

    monkeypatch.setattr(subprocess, "run", fake_run)
    out = bench.other_configs(bench.parse([]))
    assert len(out) == len(bench.OTHER_CONFIGS) == len(calls)
    assert all("--no-configs" in c and "--no-cpu-baseline" in c for c in calls)
    assert out[0]["value"] == 123.4 and out[0]["frac"] == 0.9 and out[0]["unit"] == "GB/s"
    assert out[1]["error"] == "boom" and "value" not in out[1]
    assert out[0]["workload"] == bench.OTHER_CONFIGS[0][0]
