"""Benchmark of the DiLoCo outer merge on GB300.

A step is one merge round over the workload (every round of the workload's
round list, the in-flight ones committed together on separate streams) with
its inputs resident in HBM. The default workload is the 1.08B-parameter
DiffuRefill-1B tensor list: K = 5 fp32 worker checkpoints, plain mean in
arrival order, plain replacement, EMA beta 0.9 (34.43 GB of algorithmic
traffic per round, far larger than the 129 MB L2, so no flush is needed).

Prints one JSON line: whole-job algorithmic HBM GB/s (value), ms per round,
the roofline of the fused merge kernel against the measured HBM copy
bandwidth, SM clocks sampled during the timed region, an end-to-end figure
through the public API with inputs in pinned host memory, and the CPU oracle
timed on a bounded sample of the same workload. A default run (one GPU, the
default workload) then measures the other configurations of the metric, each
in a short child run, and adds their figures to the line (other_configs;
--no-configs skips them).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload diffurefill1b|diffurefill1b_bf16|stand|pythia14m|sweep:T,N,K]
Under torchrun (N > 1) each rank merges its own replica on its own GPU; no data
crosses GPUs (the merge has no exchange step on one box), and the reported
value is every rank's bytes over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "merge round ms and achieved HBM GB/s (% of GB300 peak) at 1.08B params"
DEFAULT_WORKLOAD = "diffurefill1b"
KERNEL_SRCS = [os.path.join(ROOT, "checkpoint_averaging_gb300", "csrc", f)
               for f in ("merge_fused.cuh", "merge_fused_f32.cu", "merge_fused_bf16.cu",
                         "merge_staged.cuh", "merge_staged_f32.cu", "merge_staged_bf16.cu",
                         "merge_device.cuh", "norm_device.cuh", "cam_internal.h")]
PROFILES = os.path.join(ROOT, "profiles")
FALLBACK_HBM_GBS = 6800.0


# ---- byte model ----------------------------------------------------------------

def round_bytes(wl, frag: int, k_incl: int) -> int:
    """Algorithmic HBM bytes of one round: each included worker element read
    once, theta read (token-weighted mode or norms) and written once, momentum
    read+written (Nesterov), EMA read+written."""
    b_in = 2 if wl.ckpt_dtype == "bf16" else 4
    per = k_incl * b_in + 4
    if wl.mode == "delta" or wl.norms:
        per += 4
    if wl.mode == "delta":
        per += 8
    if wl.ema_beta is not None:
        per += 8
    if wl.swa:
        per += 8
    return per * wl.fragment_numel(frag)


def measured_peaks() -> dict:
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f)
    except (OSError, ValueError):
        return {}


def _code_only(text: str) -> str:
    """C++ source without comments and blank lines, each line right-stripped:
    what the compiler sees, so a reworded comment does not retire a profile."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    out = []
    for line in text.splitlines():
        q = line.find("//")
        if q >= 0 and line.count('"', 0, q) % 2 == 0:
            line = line[:q]
        line = line.rstrip()
        if line:
            out.append(line)
    return "\n".join(out)


def kernel_sha() -> str:
    """Hash of the code (comments aside) of the sources the merge pass is
    compiled from."""
    h = hashlib.sha256()
    for path in KERNEL_SRCS:
        with open(path, encoding="utf-8") as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def stored_traffic(workload: str, kernel: str = "merge_staged"):
    """dram bytes per launch from the committed ncu summary of this workload's
    merge kernel, or None if absent or taken on a different kernel source."""
    path = os.path.join(PROFILES, f"{kernel}_{workload}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    sha = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]+)", text)
    val = re.search(r"dram_bytes_per_launch:\s*([0-9]+)", text)
    if not sha or not val or sha.group(1) != kernel_sha():
        return None
    return int(val.group(1))


# ---- clocks ----------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self) -> dict:
        sm, mx, reasons = [], None, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for name, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---- distributed plumbing ------------------------------------------------------------

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(value: float, ws: int, device=None) -> float:
    if ws == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(ws: int) -> None:
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def aggregate(per_rank_bytes: int, steps: int, elapsed_s: float, ws: int, device=None) -> dict:
    """Whole-job figure: every rank's bytes over the slowest rank's time."""
    t = max_over_ranks(elapsed_s, ws, device)
    return {"seconds": t, "gbs": per_rank_bytes * steps * ws / t / 1e9,
            "ms_per_step": t / steps * 1e3}


# ---- CPU oracle timing ---------------------------------------------------------------

def host_threads() -> int:
    """Host cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def run_split(fn, n: int, threads: int, pool) -> None:
    """Calls fn(lo, hi) on `threads` contiguous element ranges of [0, n) at once.
    The oracle is elementwise, so each range's results equal those of one call
    over the whole span; its ctypes calls release the GIL, so the ranges run on
    separate cores."""
    if threads <= 1 or pool is None:
        fn(0, n)
        return
    step = (n + threads - 1) // threads
    futs = [pool.submit(fn, lo, min(n, lo + step)) for lo in range(0, n, step)]
    for f in futs:
        f.result()


def oracle_sample_rate(wl, max_seconds: float, seed: int = 0, max_elems: int | None = None,
                       pool_elems: int = 1 << 24, threads: int = 1):
    """Times the CPU oracle over the workload's first round, tensor by tensor in
    list order, until max_seconds of wall time (or max_elems elements) are
    spent. Inputs follow the same recipe but are drawn once into a pool of
    pool_elems values per array and reused slice by slice (the oracle is
    elementwise, so its time does not depend on which values it sees). With
    threads > 1 every slice is split into that many element ranges, each run
    by the unchanged oracle on its own host thread.
    Returns (GB/s, seconds, elements, description)."""
    from concurrent.futures import ThreadPoolExecutor

    import numpy as np
    import torch

    import oracle
    from checkpoint_averaging_gb300 import workloads as W

    rnd, frag = wl.rounds[0]
    draw = W.draw_round(wl, 0, seed)
    k_incl = len(draw.included)
    tensors = [t for t, s in enumerate(wl.specs) if frag == -1 or s.fragment == frag]
    gen = torch.Generator().manual_seed(W.subseed(seed, wl.name, "cpu-sample"))
    P = pool_elems
    theta = (torch.randn(P, generator=gen) * wl.global_std).numpy()
    xs = []
    for _ in range(k_incl):
        x = torch.from_numpy(theta) + torch.randn(P, generator=gen) * wl.noise_std
        if wl.ckpt_dtype == "bf16":
            xs.append(x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16))
        else:
            xs.append(x.numpy().astype(np.float32))
    m = np.zeros(P, np.float32) if wl.mode == "delta" else None
    e = theta.copy() if wl.ema_beta is not None else None
    mode = oracle.DELTA_NESTEROV if wl.mode == "delta" else oracle.MEAN_REPLACE
    tokens = [draw.tokens[k] for k in draw.included] if wl.mode == "delta" else None
    beta = wl.ema_beta if wl.ema_beta is not None else 0.9
    b_per = round_bytes(wl, frag, k_incl) / max(1, wl.fragment_numel(frag))
    def one(lo: int, hi: int) -> None:
        oracle.merge_tensor([x[lo:hi] for x in xs], theta[lo:hi], mode=mode, tokens=tokens,
                            lr=wl.lr, mu=wl.mu, m=None if m is None else m[lo:hi],
                            e=None if e is None else e[lo:hi], beta=beta)

    pool = ThreadPoolExecutor(max_workers=threads) if threads > 1 else None
    spent, elems, used = 0.0, 0, 0
    try:
        for t in tensors:
            n = wl.specs[t].numel
            if max_elems is not None:
                n = min(n, max_elems - elems)
            for s0 in range(0, n, P):
                c = min(P, n - s0)
                t0 = time.perf_counter()
                run_split(one, c, threads, pool)
                spent += time.perf_counter() - t0
                elems += c
            used += 1
            if spent >= max_seconds or (max_elems is not None and elems >= max_elems):
                break
    finally:
        if pool is not None:
            pool.shutdown()
    how = "single-threaded C oracle" if threads <= 1 else \
        f"C oracle on {threads} host threads, each slice split into {threads} element ranges"
    desc = (f"first {used} of the round's {len(tensors)} tensors ({elems:,} of "
            f"{wl.fragment_numel(frag):,} elements), same recipe, {how}")
    return elems * b_per / spent / 1e9, spent, elems, desc


def cpu_threads(args) -> int:
    return args.cpu_threads if args.cpu_threads > 0 else host_threads()


def cpu_baseline(wl, args) -> dict:
    """The oracle on the host: once split over every core (the reported value)
    and once on one thread, each for about args.cpu_seconds of wall time."""
    nt = cpu_threads(args)
    g1, s1, n1, d1 = oracle_sample_rate(wl, args.cpu_seconds)
    out = {"value": round(g1, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
           "sample": d1 + f"; {s1:.1f} s"}
    if nt > 1:
        gn, sn, nn, dn = oracle_sample_rate(wl, args.cpu_seconds, threads=nt)
        out = {"value": round(gn, 4), "unit": "GB/s", "cores": nt, "kind": "oracle",
               "sample": dn + f"; {sn:.1f} s",
               "single_thread": {"value": round(g1, 4), "sample": d1 + f"; {s1:.1f} s"}}
    return out


# ---- the two arms ----------------------------------------------------------------------

def run_reference(args, wl, ws, rank) -> int:
    if rank != 0:
        return 0
    # each step times a bounded sample so that warmup + steps end within minutes
    nt = cpu_threads(args)
    rates, secs = [], []
    for i in range(args.warmup + args.steps):
        gbs, s, n, desc = oracle_sample_rate(wl, max_seconds=args.ref_seconds_per_step,
                                             pool_elems=1 << 22, threads=nt)
        if i >= args.warmup:
            rates.append(gbs)
            secs.append(s)
    gbs = statistics.median(rates)
    bytes_full = sum(round_bytes(wl, f, wl.K - wl.n_masked) for _, f in wl.rounds)
    ms_full = bytes_full / (gbs * 1e9) * 1e3
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_full, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": wl.name, "n_params": wl.n_params, "K": wl.K,
                   "sample_per_step": desc,
                   "ms_per_step_note": "extrapolated from the sample's rate to the full round"},
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": nt, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


# The other configurations of the same metric, run after the headline one:
# (workload, extra arguments). Each is one short run of this script in a
# child process, the parent idle meanwhile, so their lines are recorded with
# the headline's.
OTHER_CONFIGS = [
    ("pythia14m", ["--graph", "--steps", "200", "--warmup", "5"]),
    ("pythia14m", ["--api", "round", "--steps", "100", "--warmup", "5"]),
    ("stand", ["--steps", "10", "--warmup", "3"]),
    ("diffurefill1b_bf16", ["--steps", "10", "--warmup", "3"]),
    ("diffurefill1b_bf16_wnorms", ["--steps", "10", "--warmup", "3"]),
    ("sweep:64,16000000,4", ["--steps", "10", "--warmup", "3"]),
    ("sweep:128,256000000,4", ["--steps", "10", "--warmup", "3"]),
    ("sweep:256,1000000000,4", ["--steps", "10", "--warmup", "3"]),
    (DEFAULT_WORKLOAD, ["--op", "fold", "--fold-last", "--steps", "3", "--warmup", "3"]),
    (DEFAULT_WORKLOAD, ["--op", "adopt", "--steps", "5", "--warmup", "3"]),
    (DEFAULT_WORKLOAD, ["--op", "ortho", "--ortho-precision", "bf16", "--steps", "3",
                        "--warmup", "3"]),
    (DEFAULT_WORKLOAD, ["--op", "ortho", "--steps", "3", "--warmup", "3"]),
]


def other_configs(args) -> list:
    out = []
    for name, extra in OTHER_CONFIGS:
        cmd = [sys.executable, os.path.abspath(__file__), "--workload", name, *extra,
               "--no-cpu-baseline", "--e2e-steps", "0", "--no-configs"]
        rec = {"workload": name, "args": " ".join(extra)}
        try:
            r = subprocess.run(cmd, capture_output=True, text=True, timeout=900)
            lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
            if r.returncode != 0 or len(lines) != 1:
                rec["error"] = (r.stderr.strip().splitlines() or ["no output"])[-1][:300]
            else:
                d = json.loads(lines[0])
                roof, clk = d.get("roofline") or {}, d.get("clocks") or {}
                rec.update({"name": (d.get("config") or {}).get("workload"),
                            "metric": d.get("metric"), "value": d.get("value"),
                            "unit": d.get("unit"), "ms_per_step": d.get("ms_per_step"),
                            "frac": roof.get("frac"), "bound": roof.get("bound"),
                            "kernel": roof.get("kernel"), "traffic": roof.get("traffic"),
                            "gpu_launches": d.get("gpu_launches"),
                            "sm_mhz": clk.get("sm_mhz"), "clock_reasons": clk.get("reasons")})
        except (subprocess.TimeoutExpired, OSError, ValueError, KeyError, TypeError) as exc:
            rec["error"] = f"{type(exc).__name__}: {exc}"[:300]
        out.append(rec)
    return out


def run_ours(args, wl, ws, rank, local) -> int:
    import torch

    import __graft_entry__
    from checkpoint_averaging_gb300 import binding as B
    from checkpoint_averaging_gb300 import workloads as W

    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device; the merge runs only on the GPU")
    if rank == 0:
        __graft_entry__.build()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        barrier(ws)
        __graft_entry__.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    seed = args.seed + rank

    # inputs resident in HBM: the global, the state, K workers per round
    g = W.make_global(wl, seed, dev)
    theta = W.empty_arena(g.numels, torch.float32, dev)
    theta.flat.copy_(g.flat)
    m = W.empty_arena(g.numels, torch.float32, dev) if wl.mode == "delta" else None
    e = None
    if wl.ema_beta is not None:
        e = W.empty_arena(g.numels, torch.float32, dev)
        e.flat.copy_(g.flat)
    swa = W.empty_arena(g.numels, torch.float32, dev) if wl.swa else None
    draws = [W.draw_round(wl, i, seed) for i in range(len(wl.rounds))]
    workers = [[W.make_worker(wl, g, rnd, k, seed, dev) for k in range(wl.K)]
               for rnd, _ in wl.rounds]
    del g
    mg = B.Merger(theta.views, momentum=None if m is None else m.views,
                  ema=None if e is None else e.views, fragment_of=wl.fragment_of,
                  n_fragments=wl.n_fragments, quorum=wl.quorum,
                  swa=None if swa is None else swa.views, staging=not args.no_staging,
                  fused_finish=not args.no_fused_finish, share_sms=args.share_sms or wl.share_sms)
    n_streams = max(1, wl.in_flight)
    # with --graph the step is captured into a CUDA graph: it runs on a stream
    # of its own, which the capture can take
    main_stream = torch.cuda.Stream(dev) if args.graph else torch.cuda.current_stream(dev)
    main_stream.wait_stream(torch.cuda.current_stream(dev))
    streams = [main_stream] + [torch.cuda.Stream(dev) for _ in range(n_streams - 1)]
    norm_out = [(torch.zeros(len(mg.fragment_tensors(f)) or 1, dtype=torch.float64, device=dev),
                 torch.zeros(1, dtype=torch.float64, device=dev)) for _, f in wl.rounds]
    wnorm_out = [(torch.zeros(wl.K * max(1, len(mg.fragment_tensors(f))), dtype=torch.float64,
                              device=dev), torch.zeros(wl.K, dtype=torch.float64, device=dev))
                 for _, f in wl.rounds]
    mode = B.DELTA_NESTEROV if wl.mode == "delta" else B.MEAN_REPLACE
    round_no = [0]
    ev_pairs = []
    prepared = [{k: mg.checkpoint(w[k].views, frag) for k in d.included}
                for (_, frag), w, d in zip(wl.rounds, workers, draws)]

    group_pairs = []
    # Rounds on disjoint fragments go to the stream with the fewest bytes so far
    # (largest round first), so a long round runs beside the short ones.
    rb = [round_bytes(wl, f, len(d.included)) for (_, f), d in zip(wl.rounds, draws)]
    load = [0] * n_streams
    stream_of = [0] * len(wl.rounds)
    for i in sorted(range(len(wl.rounds)), key=lambda i: -rb[i]):
        stream_of[i] = min(range(n_streams), key=lambda j: load[j])
        load[stream_of[i]] += rb[i]

    many = max(0, args.many if args.many is not None else wl.commit_many)
    one_call = args.api == "round"
    if one_call and (many >= 2 or wl.swa or wl.worker_norms):
        raise SystemExit("bench.py: --api round takes rounds without SWA, per-worker drift or "
                         "--many")
    round_ckpts = [[prepared[i][k] for k in d.included] for i, d in enumerate(draws)]
    round_tokens = [[d.tokens[k] for k in d.included] if wl.mode == "delta" else None
                    for d in draws]
    # CUDA events for the timed region, made (and their CUDA events created by
    # a first record) before it, so that making them is not timed
    ev_pool = []

    def new_event():
        return ev_pool.pop() if ev_pool else torch.cuda.Event(enable_timing=True)

    def step_many(timed: bool) -> None:
        # the step's rounds opened, then committed in groups of `many` rounds
        # by one call each (cam_merge_commit_many), all on the main stream
        main = streams[0]
        if timed:
            a, b = new_event(), new_event()
            a.record(main)
        for g0 in range(0, len(wl.rounds), many):
            opened = []
            for i in range(g0, min(len(wl.rounds), g0 + many)):
                (_, frag), d = wl.rounds[i], draws[i]
                rd = mg.begin(round_no[0], frag)
                round_no[0] += 1
                for k in d.included:
                    rd.accumulate(prepared[i][k], d.tokens[k])
                rd.finalize(mode, wl.lr, wl.mu)
                if wl.ema_beta is not None:
                    rd.ema_update(wl.ema_beta)
                if wl.swa:
                    rd.swa_update()
                if wl.norms:
                    rd.drift_norm(*norm_out[i])
                if wl.worker_norms:
                    rd.worker_drift_norm(*wnorm_out[i])
                opened.append(rd)
            mg.commit_many(opened, main)
        if timed:
            b.record(main)
            group_pairs.append((a, b))

    def step(timed: bool) -> None:
        if many >= 2:
            step_many(timed)
            return
        main = streams[0]
        if timed and n_streams > 1:
            ga = new_event()
            ga.record(main)
        for s in streams[1:]:
            s.wait_stream(main)
        for i, ((_, frag), w, d) in enumerate(zip(wl.rounds, workers, draws)):
            s = streams[stream_of[i]]
            if one_call:  # the whole round through cam_merge_round
                if timed:
                    a, b = new_event(), new_event()
                    a.record(s)
                mg.merge(round_no[0], round_ckpts[i], round_tokens[i], fragment=frag, mode=mode,
                         lr=wl.lr, mu=wl.mu, ema_beta=wl.ema_beta,
                         norms=norm_out[i] if wl.norms else None, stream=s)
                round_no[0] += 1
                if timed:
                    b.record(s)
                    ev_pairs.append((a, b))
                continue
            rd = mg.begin(round_no[0], frag)
            round_no[0] += 1
            for k in d.included:
                rd.accumulate(prepared[i][k], d.tokens[k])
            rd.finalize(mode, wl.lr, wl.mu)
            if wl.ema_beta is not None:
                rd.ema_update(wl.ema_beta)
            if wl.swa:
                rd.swa_update()
            if wl.norms:
                rd.drift_norm(*norm_out[i])
            if wl.worker_norms:
                rd.worker_drift_norm(*wnorm_out[i])
            if timed:
                a, b = new_event(), new_event()
                a.record(s)
            rd.commit(s)
            if timed:
                b.record(s)
                ev_pairs.append((a, b))
        for s in streams[1:]:
            main.wait_stream(s)
        if timed and n_streams > 1:
            gb = new_event()
            gb.record(main)
            group_pairs.append((ga, gb))

    for _ in range(args.warmup):
        step(False)
    torch.cuda.synchronize(dev)
    graph = None
    if args.graph:  # one step captured; the timed region replays it
        l_cap, st_cap = mg.launch_count, mg.staged_count
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=streams[0]):
            step(False)
        per_replay, staged_per_replay = mg.launch_count - l_cap, mg.staged_count - st_cap
        with torch.cuda.stream(streams[0]):
            graph.replay()  # its first replay uploads it
        torch.cuda.synchronize(dev)
    launches0, staged0 = mg.launch_count, mg.staged_count
    ev_pool.extend(torch.cuda.Event(enable_timing=True)
                   for _ in range(args.steps * (2 * len(wl.rounds) + 2)))
    for ev in ev_pool:
        ev.record(streams[0])
    barrier(ws)
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clocks:
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(streams[0])
        for _ in range(args.steps):
            if graph is None:
                step(True)
                continue
            with torch.cuda.stream(streams[0]):
                a, b = new_event(), new_event()
                a.record(streams[0])
                graph.replay()
                b.record(streams[0])
                group_pairs.append((a, b))
        t1.record(streams[0])
        torch.cuda.synchronize(dev)
    elapsed = t0.elapsed_time(t1) / 1e3
    barrier(ws)
    launches = mg.launch_count - launches0
    # which form of the merge pass the library chose for these rounds
    staged_launches = mg.staged_count - staged0
    if graph is not None:  # replays do not pass through the library's counters
        launches, staged_launches = per_replay * args.steps, staged_per_replay * args.steps
    kernel = "merge_staged" if staged_launches > 0 else "merge_fused"
    k_incl = [len(d.included) for d in draws]
    step_bytes = sum(round_bytes(wl, f, k) for (_, f), k in zip(wl.rounds, k_incl))
    agg = aggregate(step_bytes, args.steps, elapsed, ws, dev)

    # roofline of the dominant launch: the merge pass of the biggest round.
    # Rounds committed together on several streams share HBM, so their
    # launches are timed as one group from the fork to the join.
    per_round = [round_bytes(wl, f, k) for (_, f), k in zip(wl.rounds, k_incl)]
    big = max(range(len(per_round)), key=per_round.__getitem__)
    if many >= 2 and launches > 0 and launches <= (len(wl.rounds) + many - 1) // many * args.steps:
        kernel = "merge_multi"
    if graph is not None:
        launch_s = [a.elapsed_time(b) / 1e3 for a, b in group_pairs]
        kern_s = statistics.mean(launch_s)
        launch_bytes = step_bytes
        kernel_desc = f"{kernel} x{len(wl.rounds)} rounds, one CUDA graph replay per step"
    elif many >= 2:
        launch_s = [a.elapsed_time(b) / 1e3 for a, b in group_pairs]
        kern_s = statistics.mean(launch_s)
        launch_bytes = step_bytes
        kernel_desc = f"{kernel}: {len(wl.rounds)} rounds, {many} per call"
    elif n_streams > 1:
        launch_s = [a.elapsed_time(b) / 1e3 for a, b in group_pairs]
        kern_s = statistics.mean(launch_s)
        launch_bytes = step_bytes
        kernel_desc = f"{kernel} x{len(wl.rounds)} concurrent on {n_streams} streams"
    else:
        launch_s = [a.elapsed_time(b) / 1e3 for i, (a, b) in enumerate(ev_pairs)
                    if i % len(wl.rounds) == big]
        kern_s = statistics.mean(launch_s)
        launch_bytes = per_round[big]
        kernel_desc = kernel
    peaks = measured_peaks()
    peak = peaks.get("hbm_gbs")
    peak_src = "measured"
    if not peak:
        peak, peak_src = FALLBACK_HBM_GBS, "fallback"
    achieved = launch_bytes / kern_s / 1e9
    traffic = stored_traffic(wl.name, kernel)

    # end to end through the public API: worker inputs start in pinned host
    # memory and are copied in every step; the new global and EMA are read back.
    e2e = None
    if args.e2e_steps > 0 and ws == 1:
        e2e = run_e2e(args, wl, mg, workers, draws, theta, e, streams[0], mode, round_no)

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(wl, args)

    ck = clocks.summary()
    mg.close()
    others = None
    if rank == 0 and ws == 1 and args.op == "merge" and not args.no_configs and \
            args.workload == DEFAULT_WORKLOAD and not args.graph and args.many is None:
        others = other_configs(args)
    if rank == 0:
        line = {
            "metric": METRIC, "value": round(agg["gbs"], 2), "unit": "GB/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(agg["ms_per_step"], 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": "f32" if wl.ckpt_dtype == "f32" else "bf16->f32",
            "data": "synthetic",
            "config": {"workload": wl.name, "n_params": wl.n_params, "K": wl.K,
                       "included": k_incl, "mode": wl.mode, "ema": wl.ema_beta is not None,
                       "swa": wl.swa, "worker_norms": wl.worker_norms,
                       "norms": wl.norms, "rounds_per_step": len(wl.rounds),
                       "streams": 1 if many >= 2 else n_streams, "commit_many": many,
                       "bytes_per_step": step_bytes,
                       "l2": "inputs larger than L2 (no flush needed)",
                       "parallelism": f"replicas{ws}", "cuda_graph": bool(args.graph), "api": args.api,
                       "fused_finish": not args.no_fused_finish,
                       "share_sms": args.share_sms or wl.share_sms},
            "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak,
                         "unit": "GB/s", "frac": round(achieved / peak, 4),
                         "peak_source": peak_src, "traffic": traffic,
                         "kernel": kernel_desc, "kernel_ms": round(kern_s * 1e3, 4),
                         "kernel_ms_median": round(statistics.median(launch_s) * 1e3, 4),
                         "kernel_ms_best": round(min(launch_s) * 1e3, 4),
                         "algorithmic_bytes_per_launch": launch_bytes},
            "clocks": ck,
            "e2e": e2e,
            "gpu_launches": launches,
            "cpu_baseline": cpu,
        }
        if others is not None:
            line["other_configs"] = others
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def run_e2e(args, wl, mg, workers, draws, theta, e, stream, mode, round_no) -> dict:
    """The round through the public API with the inputs in pinned host memory
    and the result read back to pinned host memory, every step.

    stream (default): the fused pass reads the included workers straight from
      host memory (cam_merge_accumulate_host) and writes the new global and
      EMA into host buffers in the same pass (cam_merge_publish).
    copy: the workers are copied host->device with the copy engine, merged,
      and the new global and EMA copied device->host afterwards.
    fold: as stream, but each worker except the last is folded into the
      running sum as it arrives (cam_merge_fold); the last arrival is
      accumulated, and the commit's final pass folds it, finishes and
      publishes in one pass (its reads and the published writes share the
      host link at once).

    In stream and fold mode, post_arrival_ms is the time from the last
    worker's arrival (its accumulate or fold call) to the new global in host
    memory: what remains of a round once its quorum is in."""
    import torch

    from checkpoint_averaging_gb300 import workloads as W

    dev = theta.flat.device
    pinned = [[None] * wl.K for _ in wl.rounds]
    h2d = d2h = 0
    x_size = 2 if wl.ckpt_dtype == "bf16" else 4
    for i, ((_, frag), d) in enumerate(zip(wl.rounds, draws)):
        for k in d.included:
            h = torch.empty(workers[i][k].flat.numel(), dtype=workers[i][k].flat.dtype,
                            pin_memory=True)
            h.copy_(workers[i][k].flat)
            pinned[i][k] = W.Arena(h, workers[i][k].offsets, workers[i][k].numels)
            # stream/fold read only the round's fragment; copy moves whole arenas
            h2d += (h.numel() * h.element_size() if args.e2e_mode == "copy"
                    else wl.fragment_numel(frag) * x_size)
        if args.e2e_mode != "copy":  # the published global (and EMA) of the fragment
            d2h += wl.fragment_numel(frag) * 4 * (2 if e is not None else 1)
    out_theta = W.Arena(torch.empty(theta.flat.numel(), pin_memory=True), theta.offsets,
                        theta.numels)
    out_e = None
    if e is not None:
        out_e = W.Arena(torch.empty(e.flat.numel(), pin_memory=True), e.offsets, e.numels)
    if args.e2e_mode == "copy":
        d2h = out_theta.flat.numel() * 4 + (out_e.flat.numel() * 4 if out_e is not None else 0)

    host_src = args.e2e_mode in ("stream", "fold")
    src = [{k: mg.checkpoint((pinned[i][k] if host_src else w[k]).views, frag)
            for k in d.included} for i, ((_, frag), w, d) in enumerate(zip(wl.rounds, workers, draws))]
    lat_pairs = []

    def step(timed=False):
        with torch.cuda.stream(stream):
            for i, ((_, frag), w, d) in enumerate(zip(wl.rounds, workers, draws)):
                if args.e2e_mode == "copy":
                    for k in d.included:
                        w[k].flat.copy_(pinned[i][k].flat, non_blocking=True)
                rd = mg.begin(round_no[0], frag)
                round_no[0] += 1
                ev_a = ev_b = None
                if timed and host_src:
                    ev_a = torch.cuda.Event(enable_timing=True)
                    ev_b = torch.cuda.Event(enable_timing=True)
                for j, k in enumerate(d.included):
                    last = j == len(d.included) - 1
                    if ev_a is not None and last:
                        ev_a.record(stream)  # the last worker arrives
                    if args.e2e_mode == "fold" and not last:
                        rd.fold(src[i][k], d.tokens[k], mode, stream=stream)
                    else:
                        rd.accumulate(src[i][k], d.tokens[k])
                rd.finalize(mode, wl.lr, wl.mu)
                if wl.ema_beta is not None:
                    rd.ema_update(wl.ema_beta)
                if wl.swa:
                    rd.swa_update()
                if host_src:
                    ids = mg.fragment_tensors(frag)
                    rd.publish([out_theta.views[t] for t in ids],
                               None if out_e is None else [out_e.views[t] for t in ids])
                rd.commit(stream)
                if ev_b is not None:
                    ev_b.record(stream)
                    lat_pairs.append((ev_a, ev_b))
            if args.e2e_mode == "copy":
                out_theta.flat.copy_(theta.flat, non_blocking=True)
                if out_e is not None:
                    out_e.flat.copy_(e.flat, non_blocking=True)
        stream.synchronize()

    step()
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for _ in range(args.e2e_steps):
        step(timed=True)
    el = time.perf_counter() - t0
    step_bytes = sum(round_bytes(wl, f, len(d.included)) for (_, f), d in zip(wl.rounds, draws))
    post = (round(statistics.mean(a.elapsed_time(b) for a, b in lat_pairs), 3)
            if lat_pairs else None)
    return {"value": round(step_bytes * args.e2e_steps / el / 1e9, 2), "unit": "GB/s",
            "ms_per_step": round(el / args.e2e_steps * 1e3, 3),
            "post_arrival_ms": post,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "steps": args.e2e_steps, "mode": args.e2e_mode,
            "note": "algorithmic merge bytes per wall second; each step moves the included "
                    "workers host->device and the new global and EMA device->host"}


def run_adopt(args, wl, ws, rank, local) -> int:
    """Times keep-drift adoption, theta_w += g - theta_pushed, over the workload's
    tensor list (technical report, section 5.1): 16 B/element with fp32 pushed
    copies (theta_w read and written, g and the pushed copy read), 14 with bf16."""
    import torch

    import __graft_entry__
    from checkpoint_averaging_gb300 import binding as B
    from checkpoint_averaging_gb300 import workloads as W

    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device")
    __graft_entry__.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    g = W.make_global(wl, args.seed, dev)
    pushed = W.make_worker(wl, g, 0, 0, args.seed, dev)
    local_w = W.make_worker(W.Workload(wl.name, wl.specs, 1, K=1, n_masked=0, quorum=1,
                                       ckpt_dtype="f32", mode="mean"), g, 1, 1, args.seed, dev)
    b_in = 2 if wl.ckpt_dtype == "bf16" else 4
    step_bytes = (12 + b_in) * wl.n_params
    s = torch.cuda.current_stream(dev)
    for _ in range(args.warmup):
        B.adopt_keep_drift(local_w.views, g.views, pushed.views, s)
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clocks:
        evs = []
        for _ in range(args.steps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(s)
            B.adopt_keep_drift(local_w.views, g.views, pushed.views, s)
            b.record(s)
            evs.append((a, b))
        torch.cuda.synchronize(dev)
    t = statistics.mean(a.elapsed_time(b) for a, b in evs) / 1e3
    peak = measured_peaks().get("hbm_gbs") or FALLBACK_HBM_GBS
    gbs = step_bytes / t / 1e9
    print(json.dumps({
        "metric": "keep-drift adoption HBM GB/s", "value": round(gbs, 2), "unit": "GB/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(t * 1e3, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": wl.name, "op": "adopt_keep_drift", "n_params": wl.n_params,
                   "pushed_dtype": wl.ckpt_dtype, "bytes_per_step": step_bytes},
        "roofline": {"bound": "hbm", "achieved": round(gbs, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(gbs / peak, 4), "traffic": None,
                     "kernel": "adopt_keep_drift"},
        "clocks": clocks.summary(), "gpu_launches": args.steps}), flush=True)
    return 0


def run_fold(args, wl, ws, rank, local) -> int:
    """Times eagerly folded rounds with device-resident workers: per step,
    every round of the workload folds its included workers as they "arrive"
    (cam_merge_fold), then commits (the final pass from the running sums).
    Bytes are the eager path's algorithmic traffic:

    - per fold: the worker (4 or 2 B), the sum written (4 B) and, after the
      first, read (4 B), and theta (4 B) in delta mode;
    - the final pass: the sum (4 B) plus the state bytes of the round, plus
      the last worker (4 or 2 B) with --fold-last, where the last arrival is
      accumulated and the final pass folds it.

    The roofline takes the fold kernel alone, from CUDA events around each
    fold. post_arrival_ms is the device time from the last arrival (its fold,
    or with --fold-last its accumulate) to the end of the commit."""
    import torch

    import __graft_entry__
    from checkpoint_averaging_gb300 import binding as B
    from checkpoint_averaging_gb300 import workloads as W

    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device")
    __graft_entry__.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    g = W.make_global(wl, args.seed, dev)
    theta = W.empty_arena(g.numels, torch.float32, dev)
    theta.flat.copy_(g.flat)
    delta = wl.mode == "delta"
    m = W.empty_arena(g.numels, torch.float32, dev) if delta else None
    e = None
    if wl.ema_beta is not None:
        e = W.empty_arena(g.numels, torch.float32, dev)
        e.flat.copy_(g.flat)
    draws = [W.draw_round(wl, i, args.seed) for i in range(len(wl.rounds))]
    workers = [[W.make_worker(wl, g, rnd, k, args.seed, dev) for k in range(wl.K)]
               for rnd, _ in wl.rounds]
    del g
    mg = B.Merger(theta.views, momentum=None if m is None else m.views,
                  ema=None if e is None else e.views, fragment_of=wl.fragment_of,
                  n_fragments=wl.n_fragments, quorum=wl.quorum)
    code = B.DELTA_NESTEROV if delta else B.MEAN_REPLACE
    ck = [{k: mg.checkpoint(w[k].views, frag) for k in d.included}
          for (_, frag), w, d in zip(wl.rounds, workers, draws)]
    x_size = 2 if wl.ckpt_dtype == "bf16" else 4
    fold_bytes, step_bytes = [], 0
    last_acc = args.fold_last
    for (_, frag), d in zip(wl.rounds, draws):
        n = wl.fragment_numel(frag)
        n_fold = len(d.included) - (1 if last_acc else 0)
        for j in range(n_fold):
            b = n * (x_size + 4 + (4 if j > 0 else 0) + (4 if delta else 0))
            fold_bytes.append(b)
            step_bytes += b
        step_bytes += n * (4 + 4 + (4 if delta or wl.norms else 0) + (8 if delta else 0)
                           + (8 if e is not None else 0) + (x_size if last_acc else 0))
    s = torch.cuda.current_stream(dev)
    rnd_no = [0]
    fold_ev, post_ev = [], []

    def step(timed):
        i_fold = 0
        for (_, frag), d, c in zip(wl.rounds, draws, ck):
            rd = mg.begin(rnd_no[0], frag)
            rnd_no[0] += 1
            for j, k in enumerate(d.included):
                last = j == len(d.included) - 1
                if timed and last:
                    p0 = torch.cuda.Event(enable_timing=True)
                    p0.record(s)
                if last and last_acc:
                    rd.accumulate(c[k], d.tokens[k])
                    continue
                if timed:
                    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    a.record(s)
                rd.fold(c[k], d.tokens[k], code, stream=s)
                if timed:
                    b.record(s)
                    fold_ev.append((a, b, fold_bytes[i_fold]))
                i_fold += 1
            rd.finalize(code, wl.lr, wl.mu)
            if e is not None:
                rd.ema_update(wl.ema_beta)
            rd.commit(s)
            if timed:
                p1 = torch.cuda.Event(enable_timing=True)
                p1.record(s)
                post_ev.append((p0, p1))

    for _ in range(args.warmup):
        step(False)
    torch.cuda.synchronize(dev)
    l0 = mg.launch_count
    with ClockSampler(local) as clocks:
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(s)
        for _ in range(args.steps):
            step(True)
        t1.record(s)
        torch.cuda.synchronize(dev)
    t = t0.elapsed_time(t1) / 1e3 / args.steps
    launches = mg.launch_count - l0
    # the fold kernel: bytes over time of the largest folds (a full worker)
    big = max(b for _, _, b in fold_ev)
    fold_gbs = statistics.mean(b / (x.elapsed_time(y) / 1e3) / 1e9 for x, y, b in fold_ev
                               if b == big)
    peak = measured_peaks().get("hbm_gbs") or FALLBACK_HBM_GBS
    gbs = step_bytes / t / 1e9
    mg.close()
    print(json.dumps({
        "metric": "eagerly folded merge round HBM GB/s", "value": round(gbs, 2), "unit": "GB/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(t * 1e3, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32" if wl.ckpt_dtype == "f32" else "bf16->f32",
        "data": "synthetic",
        "config": {"workload": wl.name, "op": "fold", "n_params": wl.n_params, "K": wl.K,
                   "bytes_per_step": step_bytes, "last_arrival_folded_at_commit": last_acc,
                   "post_arrival_ms": round(statistics.mean(x.elapsed_time(y) for x, y in post_ev), 4),
                   "l2": "inputs larger than L2 (no flush needed)"},
        "roofline": {"bound": "hbm", "achieved": round(fold_gbs, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(fold_gbs / peak, 4), "traffic": None,
                     "kernel": "fold_worker (non-first folds)"},
        "clocks": clocks.summary(), "gpu_launches": launches}), flush=True)
    return 0


def ortho_executed_flops(shape, its, short):
    """Flops the library's GEMM kernels execute for one matrix: each side
    padded to a multiple of 128; the Gram matrix only in the tiles (128 rows x
    256 or 128 columns) that reach its upper triangle; the update in full.
    The short-side form adds its r x r products (CUDA cores, fp32)."""
    pad = lambda v: -(-v // 128) * 128
    r, big = min(shape), max(shape)
    rp, lp = pad(r), pad(big)
    if short:  # Gram of X_0, three r x r products per step, the final product
        return 2 * rp * rp * lp + its * 6 * rp ** 3 + 2 * rp * lp * rp
    bn = 256 if rp % 256 == 0 else 128
    tri = sum(min(rp // 128, (bn * cb + bn - 1) // 128 + 1) for cb in range(rp // bn))
    return its * (tri * 2 * 128 * bn * lp + 2 * lp * rp * rp)


def run_ortho(args, wl, ws, rank, local) -> int:
    """Times an orthogonalised plain-mean round (technical report, section 5.3)
    over the workload's tensor list: every matrix's averaged update replaced by
    its polar factor with `--ortho-iterations` Newton-Schulz steps, each two
    GEMMs of this library (tcgen05 tensor cores for bf16 and tf32, CUDA cores
    for fp32). The figure is GEMM TFLOP/s on the plain count: each step of an
    m x n matrix costs 4 max(m,n) min(m,n)^2 flops (Gram matrix, then its
    product with X). The roofline's `achieved` uses the flops the kernels
    execute instead (padding to 128, the Gram matrix's upper-triangle tiles
    only)."""
    import torch

    import __graft_entry__
    from checkpoint_averaging_gb300 import binding as B
    from checkpoint_averaging_gb300 import workloads as W

    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device")
    __graft_entry__.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    g = W.make_global(wl, args.seed, dev)
    th = W.empty_arena(g.numels, torch.float32, dev)
    th.flat.copy_(g.flat)
    e = W.empty_arena(g.numels, torch.float32, dev)
    e.flat.copy_(g.flat)
    rows = [sp.shape[0] if len(sp.shape) == 2 else 0 for sp in wl.specs]
    workers = [W.make_worker(wl, g, 0, k, args.seed, dev) for k in range(wl.K)]
    mg = B.Merger(th.views, ema=e.views, quorum=wl.K, rows=rows)
    ck = [mg.checkpoint(w.views) for w in workers]
    prec = {"fp32": B.ORTHO_FP32, "tf32": B.ORTHO_TF32, "bf16": B.ORTHO_BF16}[args.ortho_precision]
    its = args.ortho_iterations

    def short(shape):  # takes the short-side form of the iteration
        return args.ortho_short_side and max(shape) >= 4 * min(shape)

    def mat_flops(shape):
        big, r = max(shape), min(shape)
        if short(shape):  # Gram matrix, 3 r x r products per step, the final product
            return 2 * big * r * r + its * 6 * r ** 3 + 2 * big * r * r
        return 4 * big * r * r * its
    flops = sum(mat_flops(sp.shape) for sp in wl.specs if len(sp.shape) == 2)
    executed = sum(ortho_executed_flops(sp.shape, args.ortho_iterations, short(sp.shape))
                   for sp in wl.specs if len(sp.shape) == 2)
    flag = B.ORTHO_SHORT_SIDE if args.ortho_short_side else 0
    s = torch.cuda.current_stream(dev)
    rnd = [0]

    def step():
        rd = mg.begin(rnd[0])
        rnd[0] += 1
        for c in ck:
            rd.accumulate(c, 0)
        rd.finalize(B.MEAN_REPLACE)
        rd.ema_update(0.9)
        rd.orthogonalize(0.01, B.ORTHO_SCALE_MATCH_NORM, prec | flag, its)
        rd.commit(s)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    l0 = mg.launch_count
    with ClockSampler(local) as clocks:
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(s)
        for _ in range(args.steps):
            step()
        b.record(s)
        torch.cuda.synchronize(dev)
    t = a.elapsed_time(b) / 1e3 / args.steps
    own_launches = mg.launch_count - l0
    n_mat = sum(1 for sp in wl.specs if len(sp.shape) == 2)
    peaks = measured_peaks()
    bf16 = peaks.get("bf16_tflops_sustained") or 1700.0
    # fp32 on the CUDA cores: 152 SMs x 128 fp32 lanes x 2 flops (an FMA) x
    # the 2,070 MHz maximum SM clock
    fp32_alu = 152 * 128 * 2 * 2.07e9 / 1e12
    peak = {B.ORTHO_TF32: bf16 * (1.1 / 2.25), B.ORTHO_BF16: bf16,
            B.ORTHO_FP32: fp32_alu}[prec]
    tflops = flops / t / 1e12
    exec_tflops = executed / t / 1e12
    mg.close()
    print(json.dumps({
        "metric": "orthogonalised merge round GEMM TFLOP/s", "value": round(tflops, 2),
        "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(t * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": args.ortho_precision, "data": "synthetic",
        "config": {"workload": wl.name, "op": "orthogonalize", "iterations": its,
                   "n_params": wl.n_params, "K": wl.K, "flops_per_step": flops,
                   "executed_flops_per_step": executed,
                   "matrices": n_mat, "short_side": bool(args.ortho_short_side)},
        "roofline": {"bound": "alu" if prec == B.ORTHO_FP32 else "tensor",
                     "achieved": round(exec_tflops, 2),
                     "peak": round(peak, 1), "unit": "TFLOP/s",
                     "frac": round(exec_tflops / peak, 4),
                     "achieved_from": "executed flops (padded, Gram upper-triangle tiles) over "
                                      "the whole round's time, streaming kernels included",
                     "peak_source": ("measured bf16 sustained" if prec == B.ORTHO_BF16 else
                                     "152 SMs x 128 fp32 lanes x 2 flops x 2.07 GHz (nominal)"
                                     if prec == B.ORTHO_FP32 else
                                     "measured bf16 sustained x nominal tf32/bf16 (1.1/2.25)")
                     + ("; the short-side form runs its r x r products in fp32"
                        if args.ortho_short_side else ""),
                     "traffic": None,
                     "kernel": ("nt_gemm_simt (fp32 CUDA cores)" if prec == B.ORTHO_FP32 else
                                "nt_gemm_tc (tcgen05, TMA, TMEM)") + " + ortho kernels"},
        "clocks": clocks.summary(), "gpu_launches": own_launches}), flush=True)
    return 0


def run_hostcost(args, wl, ws, rank, local) -> int:
    """Host time the C ABI spends per round: the workload's rounds (begin,
    accumulate for each included worker, finalize, optional EMA and drift
    norms, commit) issued in a loop through ctypes with every argument made
    ahead of time, each call timed with perf_counter_ns. ctypes' own cost per
    call, taken from a call that does nothing (cam_ctx_launch_count), is
    reported beside it and subtracted in `library_us_per_round`. The same
    rounds through the binding's Merger/Round give `binding_us_per_round`,
    and through Merger.merge and a bare cam_merge_round call (one host call
    per round) `one_call`.
    The device is synchronised between batches of rounds, outside the timed
    calls, so no call waits for a full launch queue."""
    import ctypes
    import time

    import torch

    import __graft_entry__
    from checkpoint_averaging_gb300 import binding as B
    from checkpoint_averaging_gb300 import workloads as W

    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device")
    __graft_entry__.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    seed = args.seed
    g = W.make_global(wl, seed, dev)
    theta = W.empty_arena(g.numels, torch.float32, dev)
    theta.flat.copy_(g.flat)
    m = W.empty_arena(g.numels, torch.float32, dev) if wl.mode == "delta" else None
    e = None
    if wl.ema_beta is not None:
        e = W.empty_arena(g.numels, torch.float32, dev)
        e.flat.copy_(g.flat)
    draws = [W.draw_round(wl, i, seed) for i in range(len(wl.rounds))]
    workers = [[W.make_worker(wl, g, rnd, k, seed, dev) for k in range(wl.K)]
               for rnd, _ in wl.rounds]
    mg = B.Merger(theta.views, momentum=None if m is None else m.views,
                  ema=None if e is None else e.views, fragment_of=wl.fragment_of,
                  n_fragments=wl.n_fragments, quorum=wl.quorum)
    mode = B.DELTA_NESTEROV if wl.mode == "delta" else B.MEAN_REPLACE
    L = B.lib()
    s = torch.cuda.current_stream(dev)
    sp = ctypes.c_void_p(int(s.cuda_stream))
    prepared = [{k: mg.checkpoint(w[k].views, frag) for k in d.included}
                for (_, frag), w, d in zip(wl.rounds, workers, draws)]
    norm_out = [(torch.zeros(max(1, len(mg.fragment_tensors(f))), dtype=torch.float64, device=dev),
                 torch.zeros(1, dtype=torch.float64, device=dev)) for _, f in wl.rounds]
    calls = ["begin", "accumulate", "finalize", "ema_update", "drift_norm", "commit"]
    tot = dict.fromkeys(calls, 0)
    cnt = dict.fromkeys(calls, 0)
    rnd = [0]
    ns = time.perf_counter_ns

    def raw_round(i):
        (_, frag), d = wl.rounds[i], draws[i]
        h = ctypes.c_void_p()
        t = ns(); rc = L.cam_merge_begin(mg.ctx, rnd[0], frag, ctypes.byref(h)); tot["begin"] += ns() - t
        cnt["begin"] += 1
        rnd[0] += 1
        if rc != 0:
            raise RuntimeError(B.last_error())
        for k in d.included:
            c = prepared[i][k]
            t = ns(); L.cam_merge_accumulate(h, c.ptr_array, c.dtype_code, d.tokens[k])
            tot["accumulate"] += ns() - t
            cnt["accumulate"] += 1
        t = ns(); L.cam_merge_finalize(h, mode, wl.lr, wl.mu); tot["finalize"] += ns() - t
        cnt["finalize"] += 1
        if wl.ema_beta is not None:
            t = ns(); L.cam_ema_update(h, wl.ema_beta); tot["ema_update"] += ns() - t
            cnt["ema_update"] += 1
        if wl.norms:
            pt, pf = norm_out[i]
            a, b = ctypes.c_void_p(pt.data_ptr()), ctypes.c_void_p(pf.data_ptr())
            t = ns(); L.cam_drift_norm(h, a, b); tot["drift_norm"] += ns() - t
            cnt["drift_norm"] += 1
        t = ns(); rc = L.cam_merge_commit(h, sp); tot["commit"] += ns() - t
        cnt["commit"] += 1
        if rc != 0:
            raise RuntimeError(B.last_error())

    def binding_round(i):
        (_, frag), d = wl.rounds[i], draws[i]
        rd = mg.begin(rnd[0], frag)
        rnd[0] += 1
        for k in d.included:
            rd.accumulate(prepared[i][k], d.tokens[k])
        rd.finalize(mode, wl.lr, wl.mu)
        if wl.ema_beta is not None:
            rd.ema_update(wl.ema_beta)
        if wl.norms:
            rd.drift_norm(*norm_out[i])
        rd.commit(s)

    round_ck = [[prepared[i][k] for k in d.included] for i, d in enumerate(draws)]
    round_tok = [[d.tokens[k] for k in d.included] if wl.mode == "delta" else None for d in draws]

    def one_call_round(i):
        mg.merge(rnd[0], round_ck[i], round_tok[i], fragment=wl.rounds[i][1], mode=mode,
                 lr=wl.lr, mu=wl.mu, ema_beta=wl.ema_beta,
                 norms=norm_out[i] if wl.norms else None, stream=s)
        rnd[0] += 1

    # the same call through ctypes alone, its arguments made ahead of time
    raw_args = []
    for i, ((_, frag), d) in enumerate(zip(wl.rounds, draws)):
        arr = (ctypes.POINTER(ctypes.c_void_p) * len(round_ck[i]))(*[c.ptr_array for c in round_ck[i]])
        tok = None if round_tok[i] is None else (ctypes.c_int64 * len(round_tok[i]))(*round_tok[i])
        pt, pf = norm_out[i]
        raw_args.append((frag, len(round_ck[i]), arr, round_ck[i][0].dtype_code, tok,
                         ctypes.c_void_p(pt.data_ptr()) if wl.norms else None,
                         ctypes.c_void_p(pf.data_ptr()) if wl.norms else None))
    raw_one_ns = [0]

    def raw_one_call(i):
        frag, n, arr, dt, tok, pt, pf = raw_args[i]
        t = ns()
        rc = L.cam_merge_round(mg.ctx, rnd[0], frag, n, arr, dt, tok, mode, wl.lr, wl.mu,
                               0 if wl.ema_beta is None else 1,
                               0.0 if wl.ema_beta is None else wl.ema_beta, pt, pf, sp)
        raw_one_ns[0] += ns() - t
        rnd[0] += 1
        if rc != 0:
            raise RuntimeError(B.last_error())

    n_rounds, batch = 600, 30
    for i in range(len(wl.rounds) * 3):  # warm-up
        raw_round(i % len(wl.rounds))
    torch.cuda.synchronize(dev)
    tot = dict.fromkeys(calls, 0)
    cnt = dict.fromkeys(calls, 0)
    for j in range(n_rounds):
        raw_round(j % len(wl.rounds))
        if (j + 1) % batch == 0:
            torch.cuda.synchronize(dev)
    torch.cuda.synchronize(dev)
    out = ctypes.c_int64()
    t = ns()
    for _ in range(20000):
        L.cam_ctx_launch_count(mg.ctx, ctypes.byref(out))
    noop_us = (ns() - t) / 20000 / 1e3
    per_call = {c: tot[c] / cnt[c] / 1e3 for c in calls if cnt[c]}
    calls_per_round = sum(cnt.values()) / n_rounds
    raw_us = sum(tot.values()) / n_rounds / 1e3
    bind_ns = 0
    for j in range(n_rounds):
        t = ns()
        binding_round(j % len(wl.rounds))
        bind_ns += ns() - t
        if (j + 1) % batch == 0:
            torch.cuda.synchronize(dev)
    torch.cuda.synchronize(dev)
    one_ns = 0
    for j in range(n_rounds):
        t = ns()
        one_call_round(j % len(wl.rounds))
        one_ns += ns() - t
        if (j + 1) % batch == 0:
            torch.cuda.synchronize(dev)
    torch.cuda.synchronize(dev)
    for j in range(n_rounds):
        raw_one_call(j % len(wl.rounds))
        if (j + 1) % batch == 0:
            torch.cuda.synchronize(dev)
    torch.cuda.synchronize(dev)
    mg.close()
    print(json.dumps({
        "metric": "host us per round (C ABI)", "value": round(raw_us - calls_per_round * noop_us, 2),
        "unit": "us", "n_gpus": 1, "steps": n_rounds, "warmup": 3 * len(wl.rounds),
        "higher_is_better": False, "data": "synthetic",
        "config": {"workload": wl.name, "op": "hostcost", "calls_per_round": calls_per_round},
        "library_us_per_round": round(raw_us - calls_per_round * noop_us, 2),
        "ctypes_us_per_round": round(raw_us, 2), "ctypes_noop_us_per_call": round(noop_us, 3),
        "per_call_us_with_ctypes": {c: round(v, 2) for c, v in per_call.items()},
        "binding_us_per_round": round(bind_ns / n_rounds / 1e3, 2),
        "one_call": {"binding_us_per_round": round(one_ns / n_rounds / 1e3, 2),
                     "library_us_per_round": round(raw_one_ns[0] / n_rounds / 1e3 - noop_us, 2),
                     "note": "Merger.merge / cam_merge_round: the same round in one call"}}),
          flush=True)
    return 0


def parse(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", choices=("ours", "reference"), default="ours")
    p.add_argument("--workload", default=DEFAULT_WORKLOAD)
    p.add_argument("--op", choices=("merge", "adopt", "ortho", "fold", "hostcost"), default="merge")
    p.add_argument("--ortho-iterations", type=int, default=30)
    p.add_argument("--ortho-precision", choices=("tf32", "fp32", "bf16"), default="tf32")
    p.add_argument("--ortho-short-side", action="store_true",
                   help="iterate in the short side's space for matrices of aspect ratio >= 4")
    p.add_argument("--seed", type=int, default=0)
    p.add_argument("--e2e-steps", type=int, default=3)
    p.add_argument("--e2e-mode", choices=("stream", "copy", "fold"), default="stream")
    p.add_argument("--many", type=int, default=None,
                   help="commit the step's rounds in groups of this many by one call "
                        "(cam_merge_commit_many); 0: one commit per round (default: the workload's)")
    p.add_argument("--no-configs", action="store_true",
                   help="skip the other configurations that a default run measures after the "
                        "headline one (other_configs in its line)")
    p.add_argument("--api", choices=("steps", "round"), default="steps",
                   help="merge op: each round through begin/accumulate/finalize/.../commit "
                        "(steps) or through one cam_merge_round call (round)")
    p.add_argument("--graph", action="store_true",
                   help="capture one step of the merge op into a CUDA graph and time its replays")
    p.add_argument("--fold-last", action="store_true",
                   help="--op fold: accumulate the last arrival; the commit's final pass folds it")
    p.add_argument("--cpu-seconds", type=float, default=8.0)
    p.add_argument("--cpu-threads", type=int, default=0,
                   help="host threads for the CPU oracle legs (0: every core this process may use)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-staging", action="store_true",
                   help="merge passes in the register form instead of the staged (bulk-copy) form")
    p.add_argument("--share-sms", action="store_true",
                   help="merge passes take at most three quarters of the register form's block "
                        "slots, so rounds in flight on other streams start beside them "
                        "(CAM_SHARE_SMS)")
    p.add_argument("--no-fused-finish", action="store_true",
                   help="drift norms always finished by the separate norm pass (small rounds "
                        "otherwise finish them in a register-form merge pass)")
    p.add_argument("--ref-seconds-per-step", type=float, default=1.5)
    return p.parse_args(argv)


def main(argv=None) -> int:
    args = parse(argv)
    args.warmup = max(3, args.warmup)  # timing rule: at least 3 untimed warm-up steps
    from checkpoint_averaging_gb300 import workloads as W
    wl = W.workload(args.workload)
    ws, rank, local = dist_env()
    if args.impl == "reference":
        return run_reference(args, wl, ws, rank)
    if args.op == "adopt":
        return run_adopt(args, wl, ws, rank, local)
    if args.op == "ortho":
        return run_ortho(args, wl, ws, rank, local)
    if args.op == "hostcost":
        return run_hostcost(args, wl, ws, rank, local)
    if args.op == "fold":
        return run_fold(args, wl, ws, rank, local)
    return run_ours(args, wl, ws, rank, local)


if __name__ == "__main__":
    sys.exit(main())
