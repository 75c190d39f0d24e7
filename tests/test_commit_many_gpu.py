"""cam_merge_commit_many: rounds on disjoint fragments committed by one call.

The bar is the single-round path's, bit for bit: the same rounds committed one
after another (cam_merge_commit, already held to the oracle element by element)
give the same theta, m, e, published copies and drift norms; and the oracle,
run round by round, agrees within the fixed tolerance. Rounds of one
register-form variant share one merge pass (one launch); others fall back to
one commit after another.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from checkpoint_averaging_gb300 import binding as B
from checkpoint_averaging_gb300 import workloads as W
from merge_harness import (NORM_RTOL, compare_full, compare_norms, make_gpu_state, oracle_round,
                           oracle_state_from, to_np)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _custom(sizes, frags, *, K=4, mode="delta", dtype="f32", ema=False, n_masked=1,
            norms=True, n_fragments=None):
    specs = tuple(W.TensorSpec(f"t{i}", (n,), f) for i, (n, f) in enumerate(zip(sizes, frags)))
    nf = n_fragments or (max(frags) + 1)
    rounds = tuple((r, f) for r, f in enumerate(sorted(set(frags))))
    return W.Workload("many", specs, nf, K=K, n_masked=n_masked, quorum=K - n_masked,
                      ckpt_dtype=dtype, mode=mode, lr=0.7 if mode == "delta" else 1.0,
                      mu=0.9 if mode == "delta" else 0.0, ema_beta=0.9 if ema else None,
                      rounds=rounds, tokens=(200_000, 600_000) if mode == "delta" else None,
                      norms=norms)


def _open(st, wl, idx, workers, draw, norms, round_no=None, publish=None):
    rnd, frag = wl.rounds[idx]
    rd = st.merger.begin(rnd if round_no is None else round_no, frag)
    for k in draw.included:
        rd.accumulate(workers[k].views, draw.tokens[k])
    rd.finalize(B.DELTA_NESTEROV if wl.mode == "delta" else B.MEAN_REPLACE, wl.lr, wl.mu)
    if wl.ema_beta is not None:
        rd.ema_update(wl.ema_beta)
    out = None
    if norms:
        n_t = max(1, len(rd.tensors))
        out = (torch.full((n_t,), -1.0, dtype=torch.float64, device=DEV),
               torch.full((1,), -1.0, dtype=torch.float64, device=DEV))
        rd.drift_norm(*out)
    if publish is not None:
        rd.publish(*publish)
    return rd, out


def _bitwise(a: torch.Tensor, b: torch.Tensor) -> bool:
    return torch.equal(a.contiguous().view(torch.int32), b.contiguous().view(torch.int32))


def _states_equal(x, y):
    for name in ("theta", "m", "e"):
        ax, ay = getattr(x, name), getattr(y, name)
        if ax is not None:
            assert _bitwise(ax.flat, ay.flat), name


def _run(wl, seed=0, norms=True, publish=False, rounds=None, expect_one_pass=True):
    """The workload's rounds (or those listed) committed by one call and one
    after another; both against each other bit for bit, the first against
    the oracle."""
    rounds = list(range(len(wl.rounds))) if rounds is None else rounds
    g = W.make_global(wl, seed, DEV)
    many = make_gpu_state(wl, g, DEV)
    seq = make_gpu_state(wl, g, DEV)
    ost = oracle_state_from(g, wl)
    draws = [W.draw_round(wl, i, seed) for i in rounds]
    workers = [[W.make_worker(wl, g, wl.rounds[i][0], k, seed, DEV) for k in range(wl.K)]
               for i in rounds]
    pubs = {}
    opened, outs_many = [], []
    for j, i in enumerate(rounds):
        pub = None
        if publish:
            frag = wl.rounds[i][1]
            ts = many.merger.fragment_tensors(frag)
            pub = ([torch.full((many.merger.numel[t],), -7.0, device=DEV) for t in ts],
                   [torch.full((many.merger.numel[t],), -7.0, device=DEV) for t in ts]
                   if wl.ema_beta is not None else None)
            pubs[i] = pub
        rd, out = _open(many, wl, i, workers[j], draws[j], norms, publish=pub)
        opened.append(rd)
        outs_many.append(out)
    n0 = many.merger.launch_count
    many.merger.commit_many(opened)
    launches = many.merger.launch_count - n0
    outs_seq = []
    for j, i in enumerate(rounds):
        rd, out = _open(seq, wl, i, workers[j], draws[j], norms)
        rd.commit()
        outs_seq.append(out)
    torch.cuda.synchronize()
    _states_equal(many, seq)
    for om, osq in zip(outs_many, outs_seq):
        if om is not None:
            assert _bitwise(om[0], osq[0]) and _bitwise(om[1], osq[1])
    if expect_one_pass:
        assert launches == 1, launches
    else:
        assert launches > 1, launches
    for j, i in enumerate(rounds):
        rnd, frag = wl.rounds[i]
        on = oracle_round(ost, wl, rnd, frag, workers[j], draws[j])
        if outs_many[j] is not None:
            compare_norms(outs_many[j], on, f"round {rnd}")
    compare_full(many, ost, "rounds committed together")
    for i, (pt, pe) in pubs.items():
        frag = wl.rounds[i][1]
        for t, buf in zip(many.merger.fragment_tensors(frag), pt):
            assert _bitwise(buf, many.theta.views[t])
        if pe is not None:
            for t, buf in zip(many.merger.fragment_tensors(frag), pe):
                assert _bitwise(buf, many.e.views[t])
    assert many.merger.status() == 0 and seq.merger.status() == 0
    many.merger.close()
    seq.merger.close()


def test_pythia14m_three_fragment_rounds_in_one_pass():
    _run(W.workload("pythia14m"))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_ragged_fragments_mean_ema_published_in_one_pass(dtype):
    sizes = [1, 2049, 7, 100_003, 0, 16385, 3, 65536, 2047]
    frags = [0, 0, 1, 1, 1, 2, 2, 3, 3]
    wl = _custom(sizes, frags, mode="mean", dtype=dtype, ema=True, n_masked=0, K=3)
    _run(wl, publish=True)


def test_rounds_without_norms_in_one_pass():
    sizes = [300_000, 5, 70_000, 2049, 131_072]
    frags = [0, 0, 1, 1, 2]
    _run(_custom(sizes, frags, dtype="bf16"), norms=False)


def test_two_of_three_rounds_in_one_pass():
    _run(W.workload("pythia14m"), rounds=[0, 2])


def test_rounds_of_different_variants_commit_one_after_another():
    wl = W.workload("pythia14m")
    g = W.make_global(wl, 0, DEV)
    many = make_gpu_state(wl, g, DEV)
    seq = make_gpu_state(wl, g, DEV)
    draws = [W.draw_round(wl, i, 0) for i in range(3)]
    workers = [[W.make_worker(wl, g, wl.rounds[i][0], k, 0, DEV) for k in range(wl.K)]
               for i in range(3)]
    norms = [True, False, True]  # one round without drift norms: another variant
    opened, outs = [], []
    for i in range(3):
        rd, out = _open(many, wl, i, workers[i], draws[i], norms[i])
        opened.append(rd)
        outs.append(out)
    n0 = many.merger.launch_count
    many.merger.commit_many(opened)
    assert many.merger.launch_count - n0 == 3
    for i in range(3):
        rd, out = _open(seq, wl, i, workers[i], draws[i], norms[i])
        rd.commit()
        if out is not None:
            torch.cuda.synchronize()
            assert _bitwise(out[0], outs[i][0]) and _bitwise(out[1], outs[i][1])
    torch.cuda.synchronize()
    _states_equal(many, seq)
    many.merger.close()
    seq.merger.close()


def test_commit_many_refusals_leave_every_round_open():
    wl = W.workload("pythia14m")
    g = W.make_global(wl, 0, DEV)
    st = make_gpu_state(wl, g, DEV)
    draws = [W.draw_round(wl, i, 0) for i in range(2)]
    workers = [[W.make_worker(wl, g, wl.rounds[i][0], k, 0, DEV) for k in range(wl.K)]
               for i in range(2)]
    rd0, _ = _open(st, wl, 0, workers[0], draws[0], True)
    rd1 = st.merger.begin(1, wl.rounds[1][1])  # not finalized
    for k in draws[1].included:
        rd1.accumulate(workers[1][k].views, draws[1].tokens[k])
    n0 = st.merger.launch_count
    with pytest.raises(B.StateError):
        st.merger.commit_many([rd0, rd1])
    with pytest.raises(B.ArgError):
        B.merge_commit_many([rd0.handle, rd0.handle])
    assert st.merger.launch_count == n0  # nothing ran; both rounds still open
    rd1.finalize(B.DELTA_NESTEROV, wl.lr, wl.mu)
    rd1.drift_norm(torch.zeros(len(rd1.tensors), dtype=torch.float64, device=DEV),
                   torch.zeros(1, dtype=torch.float64, device=DEV))  # the same variant as rd0
    st.merger.commit_many([rd0, rd1])
    torch.cuda.synchronize()
    assert st.merger.launch_count - n0 == 1
    assert st.merger.status() == 0
    st.merger.close()


def test_commit_many_captured_in_a_cuda_graph_replays_bit_for_bit():
    wl = W.workload("pythia14m")
    g = W.make_global(wl, 0, DEV)
    many = make_gpu_state(wl, g, DEV)
    seq = make_gpu_state(wl, g, DEV)
    draws = [W.draw_round(wl, i, 0) for i in range(3)]
    workers = [[W.make_worker(wl, g, wl.rounds[i][0], k, 0, DEV) for k in range(wl.K)]
               for i in range(3)]
    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    outs = []
    with torch.cuda.graph(graph, stream=s):
        opened = []
        for i in range(3):
            rd, out = _open(many, wl, i, workers[i], draws[i], True, round_no=i)
            opened.append(rd)
            outs.append(out)
        many.merger.commit_many(opened, stream=s)
    for rep in range(2):
        with torch.cuda.stream(s):
            graph.replay()
        torch.cuda.synchronize()
        for i in range(3):
            rd, out = _open(seq, wl, i, workers[i], draws[i], True, round_no=3 * rep + i)
            rd.commit()
            torch.cuda.synchronize()
            assert _bitwise(out[0], outs[i][0]) and _bitwise(out[1], outs[i][1]), (rep, i)
        _states_equal(many, seq)
    assert many.merger.status() == 0
    many.merger.close()
    seq.merger.close()


def test_corrupted_chunks_are_skipped_in_a_shared_pass():
    """CAM_TEST_BAD_CHUNK with rounds on two fragments in one pass: each
    fragment's first tensor's last chunk runs 2,048 elements past its end (the
    arena's next tensor of the same fragment is there). The shared pass skips
    both chunks, reports CAM_STATUS_BAD_CHUNK, and equals, bit for bit, the same
    rounds committed one after another with the same tables (whose skipping
    the single-round tests hold to the oracle)."""
    sizes = [300_000, 70_000, 200_000, 50_000]
    frags = [0, 0, 1, 1]
    wl = _custom(sizes, frags)
    g = W.make_global(wl, 0, DEV)
    for t in (0, 2):
        assert g.offsets[t + 1] + g.numels[t + 1] >= g.offsets[t] + g.numels[t] + 2048
    many = make_gpu_state(wl, g, DEV, test_bad_chunk=True)
    seq = make_gpu_state(wl, g, DEV, test_bad_chunk=True)
    draws = [W.draw_round(wl, i, 0) for i in range(2)]
    workers = [[W.make_worker(wl, g, wl.rounds[i][0], k, 0, DEV) for k in range(wl.K)]
               for i in range(2)]
    opened, outs = [], []
    for i in range(2):
        rd, out = _open(many, wl, i, workers[i], draws[i], True)
        opened.append(rd)
        outs.append(out)
    many.merger.commit_many(opened)
    for i in range(2):
        rd, out = _open(seq, wl, i, workers[i], draws[i], True)
        rd.commit()
        torch.cuda.synchronize()
        assert _bitwise(out[0], outs[i][0]) and _bitwise(out[1], outs[i][1])
    torch.cuda.synchronize()
    _states_equal(many, seq)
    for t in (0, 2):  # the skipped chunks kept their bits
        th, g0 = to_np(many.theta.views[t]), to_np(g.views[t])
        assert (th[-1:].view(np.uint32) == g0[-1:].view(np.uint32)).all()
    assert many.merger.status() == B.STATUS_BAD_CHUNK
    many.merger.close()
    seq.merger.close()
