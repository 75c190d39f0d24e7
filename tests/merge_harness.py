"""Runs a seeded workload through libcam (via the C ABI binding) and through the
CPU oracle on identical inputs, and compares the results.

Full comparison: every element of theta, m, e and every drift norm.
Sampled comparison (for the 1.08B and larger lists): for each tensor a set of
element indices (both ends, the ragged tail, chunk-boundary neighbourhoods and
random positions) is gathered before and after the GPU round; the oracle runs
the round on the gathered inputs, which is exact because the merge is
elementwise. Drift norms at full size are checked on the whole of a few
tensors, and the fragment norm against the per-tensor norms.

The tolerance is the one fixed for this path: per fp32 element
|gpu - oracle| <= 1e-7 + 2e-6 |oracle|; norms within 1e-5 relative.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np
import torch

import oracle
from checkpoint_averaging_gb300 import binding as B
from checkpoint_averaging_gb300 import workloads as W

ATOL, RTOL = 1e-7, 2e-6
NORM_RTOL = 1e-5


def to_np(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.detach().cpu().numpy()


def close(got: np.ndarray, want: np.ndarray) -> np.ndarray:
    """Boolean mask of elements outside the tolerance (NaN-aware)."""
    got = np.asarray(got, np.float32)
    want = np.asarray(want, np.float32)
    bad = np.abs(got.astype(np.float64) - want) > ATOL + RTOL * np.abs(want.astype(np.float64))
    bad |= np.isnan(got) != np.isnan(want)
    return bad


def assert_close(got, want, what: str) -> None:
    bad = close(got, want)
    if bad.any():
        i = int(np.flatnonzero(bad)[0])
        raise AssertionError(f"{what}: {int(bad.sum())}/{bad.size} elements outside "
                             f"tolerance; first at {i}: gpu={got.ravel()[i]!r} "
                             f"oracle={want.ravel()[i]!r}")


def bitwise_equal(a, b) -> bool:
    return (np.asarray(a, np.float32).view(np.uint32) == np.asarray(b, np.float32).view(np.uint32)).all()


@dataclass
class GpuState:
    theta: W.Arena
    m: W.Arena | None
    e: W.Arena | None
    merger: B.Merger
    swa: W.Arena | None = None


def make_gpu_state(wl: W.Workload, g: W.Arena, dev, quorum=None, staging=True,
                   fused_finish=True, test_stall_staged=False, share_sms=False,
                   test_bad_chunk=False, test_bad_tag=False) -> GpuState:
    theta = W.empty_arena(g.numels, torch.float32, dev)
    theta.flat.copy_(g.flat)
    m = W.empty_arena(g.numels, torch.float32, dev) if wl.mode == "delta" else None
    e = None
    if wl.ema_beta is not None:
        e = W.empty_arena(g.numels, torch.float32, dev)
        e.flat.copy_(g.flat)  # EMA starts at the first global
    swa = W.empty_arena(g.numels, torch.float32, dev) if wl.swa else None
    mg = B.Merger(theta.views, momentum=None if m is None else m.views,
                  ema=None if e is None else e.views, fragment_of=wl.fragment_of,
                  n_fragments=wl.n_fragments, quorum=wl.quorum if quorum is None else quorum,
                  swa=None if swa is None else swa.views, staging=staging,
                  fused_finish=fused_finish, test_stall_staged=test_stall_staged,
                  share_sms=share_sms, test_bad_chunk=test_bad_chunk, test_bad_tag=test_bad_tag)
    return GpuState(theta, m, e, mg, swa)


def gpu_round(st: GpuState, wl: W.Workload, rnd: int, frag: int, workers, draw,
              stream=None, norms=None, fold=False):
    """Opens, fills and commits one round on the GPU, its workers accumulated
    or (fold=True) folded as they arrive, or (fold="last") folded except the
    last arrival, which is accumulated and folded by the commit. Returns
    (per_tensor, per_fragment) device tensors when norms are requested."""
    rd = st.merger.begin(rnd, frag)
    code = B.DELTA_NESTEROV if wl.mode == "delta" else B.MEAN_REPLACE
    for i, k in enumerate(draw.included):
        if fold and not (fold == "last" and i == len(draw.included) - 1):
            rd.fold(workers[k].views, draw.tokens[k], code, stream=stream)
        else:
            rd.accumulate(workers[k].views, draw.tokens[k])
    rd.finalize(B.DELTA_NESTEROV if wl.mode == "delta" else B.MEAN_REPLACE, wl.lr, wl.mu)
    if wl.ema_beta is not None:
        rd.ema_update(wl.ema_beta)
    if wl.swa:
        rd.swa_update()
    out = None
    if wl.norms if norms is None else norms:
        dev = st.theta.flat.device
        pt = torch.full((max(1, len(rd.tensors)),), -1.0, dtype=torch.float64, device=dev)
        pf = torch.full((1,), -1.0, dtype=torch.float64, device=dev)
        rd.drift_norm(pt, pf)
        out = (pt, pf)
    rd.commit(stream)
    return out


def oracle_state_from(g: W.Arena, wl: W.Workload) -> oracle.OracleState:
    th = [to_np(v).copy() for v in g.views]
    return oracle.OracleState(
        theta=th,
        m=[np.zeros(n, np.float32) for n in g.numels] if wl.mode == "delta" else None,
        e=[t.copy() for t in th] if wl.ema_beta is not None else None,
        fragment_of=wl.fragment_of,
        swa=[np.zeros(n, np.float32) for n in g.numels] if wl.swa else None,
        swa_count=[0] * len(g.numels) if wl.swa else None)


def oracle_round(ost: oracle.OracleState, wl: W.Workload, rnd: int, frag: int, workers,
                 draw, quorum=None):
    ck = [[to_np(v) for v in w.views] for w in workers]
    return oracle.merge_round(
        ost, round=rnd, fragment=frag, ckpts=ck, included=draw.included,
        tokens=draw.tokens if wl.mode == "delta" else None,
        mode=oracle.DELTA_NESTEROV if wl.mode == "delta" else oracle.MEAN_REPLACE,
        lr=wl.lr, mu=wl.mu, quorum=wl.quorum if quorum is None else quorum,
        ema_beta=wl.ema_beta, swa_update=wl.swa)


def compare_full(st: GpuState, ost: oracle.OracleState, what: str, bitwise=False) -> None:
    torch.cuda.synchronize()
    for t in range(len(ost.theta)):
        pairs = [("theta", st.theta, ost.theta)]
        if st.m is not None:
            pairs.append(("m", st.m, ost.m))
        if st.e is not None:
            pairs.append(("e", st.e, ost.e))
        if st.swa is not None:
            pairs.append(("swa", st.swa, ost.swa))
        for name, arena, ref in pairs:
            got = to_np(arena.views[t])
            assert_close(got, ref[t], f"{what}: {name}[{t}]")
            if bitwise:
                assert bitwise_equal(got, ref[t]), f"{what}: {name}[{t}] not bitwise equal"


def compare_norms(gpu_norms, ora_norms, what: str) -> None:
    pt, pf = gpu_norms
    torch.cuda.synchronize()
    per_t, frag = ora_norms
    got = pt.cpu().numpy()[:len(per_t)]
    want = np.asarray(per_t)
    assert np.all(np.abs(got - want) <= NORM_RTOL * np.abs(want) + 1e-300), \
        f"{what}: per-tensor drift norms differ: {got[:4]} vs {want[:4]}"
    assert abs(pf.item() - frag) <= NORM_RTOL * abs(frag) + 1e-300, \
        f"{what}: fragment drift norm {pf.item()} vs {frag}"


def run_full(wl: W.Workload, seed: int = 0, dev="cuda", bitwise=False, share_sms=False):
    """Every round of the workload, full element-by-element comparison."""
    g = W.make_global(wl, seed, dev)
    st = make_gpu_state(wl, g, dev, share_sms=share_sms)
    ost = oracle_state_from(g, wl)
    for idx, (rnd, frag) in enumerate(wl.rounds):
        draw = W.draw_round(wl, idx, seed)
        base = g
        if wl.workers_track_global:  # workers start from the oracle's current global
            base = W.empty_arena(g.numels, torch.float32, dev)
            for v, h in zip(base.views, ost.theta):
                v.copy_(torch.from_numpy(h))
        workers = [W.make_worker(wl, base, rnd, k, seed, dev) for k in range(wl.K)]
        gn = gpu_round(st, wl, rnd, frag, workers, draw)
        on = oracle_round(ost, wl, rnd, frag, workers, draw)
        compare_full(st, ost, f"{wl.name} round {rnd}", bitwise=bitwise)
        if gn is not None:
            compare_norms(gn, on, f"{wl.name} round {rnd}")
        del workers
    assert st.merger.status() == 0, "a merge pass gave up waiting on a barrier"
    st.merger.close()
    return st, ost


# ---- sampled comparison at full size ------------------------------------------------

def sample_indices(n: int, per_tensor: int, rng: np.random.Generator) -> np.ndarray:
    if n <= per_tensor:
        return np.arange(n, dtype=np.int64)
    fixed = [0, 1, 7, 8, n - 1, n - 2, n - 8, n - 9]
    for q in (2048, 16384):  # neighbourhoods of chunk boundaries
        for b in range(q, n, max(q, (n // 16) // q * q)):
            fixed += [b - 1, b]
    idx = np.concatenate([np.array(fixed, np.int64), rng.integers(0, n, per_tensor)])
    return np.unique(np.clip(idx, 0, n - 1))


def gather(arena: W.Arena, tensors, idxs) -> list[np.ndarray]:
    return [to_np(arena.views[t][torch.from_numpy(i).to(arena.flat.device)])
            for t, i in zip(tensors, idxs)]


def sampled_round_check(wl, st: GpuState, frag, workers, draw, idxs, before, what):
    """`before` holds the gathered (theta, m, e) ahead of the GPU round."""
    tensors = [t for t in range(len(wl.specs)) if frag == -1 or wl.specs[t].fragment == frag]
    xs = [gather(workers[k], tensors, idxs) for k in draw.included]
    th_b, m_b, e_b = before
    th_a = gather(st.theta, tensors, idxs)
    m_a = gather(st.m, tensors, idxs) if st.m is not None else None
    e_a = gather(st.e, tensors, idxs) if st.e is not None else None
    for j, t in enumerate(tensors):
        th = th_b[j].copy()
        m = m_b[j].copy() if m_b is not None else None
        e = e_b[j].copy() if e_b is not None else None
        oracle.merge_tensor([x[j] for x in xs], th,
                            mode=oracle.DELTA_NESTEROV if wl.mode == "delta" else oracle.MEAN_REPLACE,
                            tokens=[draw.tokens[k] for k in draw.included] if wl.mode == "delta" else None,
                            lr=wl.lr, mu=wl.mu, m=m, e=e,
                            beta=wl.ema_beta if wl.ema_beta is not None else 0.9)
        assert_close(th_a[j], th, f"{what}: theta[{t}] (sampled)")
        if m is not None:
            assert_close(m_a[j], m, f"{what}: m[{t}] (sampled)")
        if e is not None:
            assert_close(e_a[j], e, f"{what}: e[{t}] (sampled)")


def gather_state(st: GpuState, tensors, idxs):
    return (gather(st.theta, tensors, idxs),
            gather(st.m, tensors, idxs) if st.m is not None else None,
            gather(st.e, tensors, idxs) if st.e is not None else None)


def sliced_tensor_norm(wl, workers, draw, theta_before, t: int, step: int = 1 << 27) -> float:
    """Oracle drift norm of one tensor too large to copy to the host at once
    (theta_before: its state before, on the device): the oracle's fp64 sum of
    squared drift slice by slice, the slice sums added in fp64."""
    xs = [workers[k].views[t] for k in draw.included]
    n = theta_before.numel()
    s = 0.0
    for a in range(0, n, step):
        b = min(n, a + step)
        th = to_np(theta_before[a:b]).copy()
        m = np.zeros_like(th) if wl.mode == "delta" else None
        s += oracle.merge_tensor(
            [to_np(x[a:b]) for x in xs], th,
            mode=oracle.DELTA_NESTEROV if wl.mode == "delta" else oracle.MEAN_REPLACE,
            tokens=[draw.tokens[k] for k in draw.included] if wl.mode == "delta" else None,
            lr=wl.lr, mu=wl.mu, m=m)
    return math.sqrt(s)


def full_tensor_norm(wl, workers, draw, theta_before: np.ndarray, t: int) -> float:
    """Oracle drift norm of one whole tensor (theta_before: its state before)."""
    xs = [to_np(workers[k].views[t]) for k in draw.included]
    th = theta_before.copy()
    m = np.zeros_like(th) if wl.mode == "delta" else None
    s = oracle.merge_tensor(xs, th, mode=oracle.DELTA_NESTEROV if wl.mode == "delta" else oracle.MEAN_REPLACE,
                            tokens=[draw.tokens[k] for k in draw.included] if wl.mode == "delta" else None,
                            lr=wl.lr, mu=wl.mu, m=m)
    return math.sqrt(s)
