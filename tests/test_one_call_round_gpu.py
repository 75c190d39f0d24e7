"""cam_merge_round (Merger.merge): one whole round in one host call.

The bar is the step-by-step round's, bit for bit: the same rounds run through
begin / accumulate / finalize / ema_update / drift_norm / commit give the same
theta, m, e and drift norms, and both agree with the oracle within the fixed
tolerance. A round that fails a check before the commit's launches is dropped
with the failing step's error, launches nothing and leaves its fragment free.
"""
from __future__ import annotations

import pytest
import torch

from checkpoint_averaging_gb300 import binding as B
from checkpoint_averaging_gb300 import workloads as W
from merge_harness import (compare_full, compare_norms, make_gpu_state, oracle_round,
                           oracle_state_from)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _bitwise(a: torch.Tensor, b: torch.Tensor) -> bool:
    return torch.equal(a.contiguous().view(torch.int32), b.contiguous().view(torch.int32))


def _norm_out(mg, frag):
    n = max(1, len(mg.fragment_tensors(frag)))
    return (torch.full((n,), -1.0, dtype=torch.float64, device=DEV),
            torch.full((1,), -1.0, dtype=torch.float64, device=DEV))


def _code(wl):
    return B.DELTA_NESTEROV if wl.mode == "delta" else B.MEAN_REPLACE


def _steps(st, wl, rnd, frag, workers, draw):
    rd = st.merger.begin(rnd, frag)
    for k in draw.included:
        rd.accumulate(workers[k].views, draw.tokens[k])
    rd.finalize(_code(wl), wl.lr, wl.mu)
    if wl.ema_beta is not None:
        rd.ema_update(wl.ema_beta)
    out = None
    if wl.norms:
        out = _norm_out(st.merger, frag)
        rd.drift_norm(*out)
    rd.commit()
    return out


def _one_call(st, wl, rnd, frag, workers, draw, prepared=None):
    ck = prepared if prepared is not None else \
        [st.merger.checkpoint(workers[k].views, frag) for k in draw.included]
    out = _norm_out(st.merger, frag) if wl.norms else None
    st.merger.merge(rnd, ck, [draw.tokens[k] for k in draw.included] if wl.mode == "delta" else None,
                    fragment=frag, mode=_code(wl), lr=wl.lr, mu=wl.mu, ema_beta=wl.ema_beta,
                    norms=out)
    return out


def _states_equal(x, y):
    for name in ("theta", "m", "e"):
        ax, ay = getattr(x, name), getattr(y, name)
        if ax is not None:
            assert _bitwise(ax.flat, ay.flat), name


@pytest.mark.parametrize("name", ["pythia14m", "stand", "sweep:16,2000000,3,norms-ema"])
def test_one_call_round_matches_step_by_step_and_oracle(name):
    wl = W.workload(name)
    seed = 5
    g = W.make_global(wl, seed, DEV)
    one = make_gpu_state(wl, g, DEV)
    seq = make_gpu_state(wl, g, DEV)
    ost = oracle_state_from(g, wl)
    for idx, (rnd, frag) in enumerate(wl.rounds[:4]):
        draw = W.draw_round(wl, idx, seed)
        workers = [W.make_worker(wl, g, rnd, k, seed, DEV) for k in range(wl.K)]
        n0 = one.merger.launch_count
        o1 = _one_call(one, wl, rnd, frag, workers, draw)
        assert one.merger.launch_count - n0 >= 1
        o2 = _steps(seq, wl, rnd, frag, workers, draw)
        torch.cuda.synchronize()
        _states_equal(one, seq)
        if o1 is not None:
            assert _bitwise(o1[0], o2[0]) and _bitwise(o1[1], o2[1])
        on = oracle_round(ost, wl, rnd, frag, workers, draw)
        compare_full(one, ost, f"{wl.name} round {rnd} in one call")
        if o1 is not None:
            compare_norms(o1, on, f"{wl.name} round {rnd} in one call")
    assert one.merger.status() == 0
    one.merger.close()
    seq.merger.close()


def test_one_call_round_reuses_marshalled_checkpoints_across_rounds():
    # the same prepared Checkpoints and tokens on every round: the cached
    # argument arrays must still name this round's buffers and counts
    wl = W.workload("pythia14m")
    seed = 8
    g = W.make_global(wl, seed, DEV)
    one = make_gpu_state(wl, g, DEV)
    seq = make_gpu_state(wl, g, DEV)
    frag = wl.rounds[0][1]
    draw = W.draw_round(wl, 0, seed)
    workers = [W.make_worker(wl, g, 0, k, seed, DEV) for k in range(wl.K)]
    prepared = [one.merger.checkpoint(workers[k].views, frag) for k in draw.included]
    for r in range(3):
        for k in draw.included:  # new worker values in the same buffers
            workers[k].flat.mul_(1.0 + 0.25 * (r + 1))
        _one_call(one, wl, r, frag, workers, draw, prepared=prepared)
        _steps(seq, wl, r, frag, workers, draw)
        torch.cuda.synchronize()
        _states_equal(one, seq)
    one.merger.close()
    seq.merger.close()


def test_one_call_round_errors_drop_the_round():
    wl = W.workload("pythia14m")
    seed = 2
    g = W.make_global(wl, seed, DEV)
    st = make_gpu_state(wl, g, DEV)
    mg = st.merger
    frag = wl.rounds[0][1]
    workers = [W.make_worker(wl, g, 0, k, seed, DEV) for k in range(wl.K)]
    ck = [mg.checkpoint(w.views, frag) for w in workers]
    before = st.theta.flat.clone()
    n0 = mg.launch_count
    # below the quorum: nothing launched, the fragment stays free
    with pytest.raises(B.QuorumError):
        mg.merge(1, ck[:wl.quorum - 1], [100] * (wl.quorum - 1), fragment=frag,
                 mode=B.DELTA_NESTEROV, lr=wl.lr, mu=wl.mu)
    # no tokens in delta mode
    with pytest.raises(B.ArgError):
        mg.merge(2, ck[:wl.quorum], [0] * wl.quorum, fragment=frag, mode=B.DELTA_NESTEROV,
                 lr=wl.lr, mu=wl.mu)
    # a round number not above those used (the failed rounds' numbers count as used)
    with pytest.raises(B.StaleRoundError):
        mg.merge(2, ck[:wl.quorum], [100] * wl.quorum, fragment=frag, mode=B.DELTA_NESTEROV,
                 lr=wl.lr, mu=wl.mu)
    assert mg.launch_count == n0
    torch.cuda.synchronize()
    assert _bitwise(st.theta.flat, before)
    # the fragment takes a round again
    mg.merge(3, ck[:wl.quorum], [100] * wl.quorum, fragment=frag, mode=B.DELTA_NESTEROV,
             lr=wl.lr, mu=wl.mu)
    torch.cuda.synchronize()
    assert mg.launch_count > n0
    assert mg.status() == 0
    mg.close()


def test_one_call_rounds_captured_in_a_cuda_graph_replay_bit_for_bit():
    wl = W.workload("pythia14m")
    seed = 4
    g = W.make_global(wl, seed, DEV)
    cap = make_gpu_state(wl, g, DEV)
    ref = make_gpu_state(wl, g, DEV)
    draws = [W.draw_round(wl, i, seed) for i in range(len(wl.rounds))]
    workers = [[W.make_worker(wl, g, rnd, k, seed, DEV) for k in range(wl.K)]
               for rnd, _ in wl.rounds]
    prepared = [[cap.merger.checkpoint(w[k].views, f) for k in d.included]
                for (_, f), w, d in zip(wl.rounds, workers, draws)]
    outs = [_norm_out(cap.merger, f) for _, f in wl.rounds]
    rno = [0]

    def step():
        for i, (_, frag) in enumerate(wl.rounds):
            d = draws[i]
            cap.merger.merge(rno[0], prepared[i], [d.tokens[k] for k in d.included],
                             fragment=frag, mode=B.DELTA_NESTEROV, lr=wl.lr, mu=wl.mu,
                             norms=outs[i])
            rno[0] += 1

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        step()
    for rep in range(3):
        graph.replay()
        for i, ((_, frag), w, d) in enumerate(zip(wl.rounds, workers, draws)):
            o = _steps(ref, wl, 100 + 10 * rep + i, frag, w, d)
            torch.cuda.synchronize()
            assert _bitwise(o[0], outs[i][0]) and _bitwise(o[1], outs[i][1])
        _states_equal(cap, ref)
    cap.merger.close()
    ref.merger.close()
