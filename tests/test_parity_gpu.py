"""GPU parity: libcam's fused merge pass against the CPU oracle, through the C ABI.

Workloads are the five synthetic configurations (Pythia-14M fragments with a
quorum and Nesterov; the 63M stand with plain mean + EMA over 10 rounds; the
1.08B list in fp32 with plain mean + EMA; the 1.08B list with bf16 workers,
fragments, quorum, Nesterov, norms and two rounds in flight; ragged sweeps up
to 4e9 parameters) plus edge cases: ragged and empty tensors, misaligned
views, K = 1 and K = KMAX, many tensors per round, the round state machine.
Tolerance per fp32 element: |gpu - oracle| <= 1e-7 + 2e-6 |oracle|; drift
norms within 1e-5 relative.
"""
import dataclasses
import gc
import math

import numpy as np
import pytest
import torch

import oracle
from checkpoint_averaging_gb300 import binding as B
from checkpoint_averaging_gb300 import workloads as W

from merge_harness import (assert_close, bitwise_equal, compare_full, gather_state,
                           gpu_round, make_gpu_state, oracle_round, oracle_state_from,
                           run_full, sample_indices, sampled_round_check, to_np,
                           full_tensor_norm, sliced_tensor_norm, NORM_RTOL)

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(autouse=True)
def _cuda_cleanup():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    yield
    gc.collect()
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


# ---- the five workloads ----------------------------------------------------------

def test_pythia14m_fragments_quorum_nesterov_full():
    run_full(W.workload("pythia14m"))


def test_stand_mean_ema_ten_rounds_full():
    run_full(W.workload("stand"))


def test_rounds_sharing_the_sms_equal_the_oracle_bitwise():
    """CAM_SHARE_SMS (each pass takes at most three quarters of the register
    form's block slots, so rounds in flight run side by side) changes only the launch shape: the Pythia-14M rounds still
    equal the oracle bit for bit, norms within their tolerance."""
    run_full(W.workload("pythia14m"), seed=9, bitwise=True, share_sms=True)


def test_small_workloads_bitwise_equal_to_oracle():
    # The fixed op sequence makes GPU and oracle agree bit for bit, not only
    # within tolerance.
    run_full(W.workload("pythia14m"), seed=3, bitwise=True)
    wl = W.workload("stand")
    run_full(W.Workload(wl.name, wl.specs, 1, K=5, n_masked=0, quorum=5, ckpt_dtype="f32",
                        mode="mean", ema_beta=0.9, rounds=((0, -1), (1, -1)), noise_std=2e-3,
                        workers_track_global=True), seed=4, bitwise=True)


def _sampled_workload(wl, seed=0, per_tensor=4096, norm_tensors=(), fold=False):
    g = W.make_global(wl, seed, DEV)
    st = make_gpu_state(wl, g, DEV)
    rng = np.random.default_rng(seed)
    for idx, (rnd, frag) in enumerate(wl.rounds):
        draw = W.draw_round(wl, idx, seed)
        workers = [W.make_worker(wl, g, rnd, k, seed, DEV) for k in range(wl.K)]
        tensors = [t for t in range(len(wl.specs)) if frag == -1 or wl.specs[t].fragment == frag]
        idxs = [sample_indices(wl.specs[t].numel, per_tensor, rng) for t in tensors]
        before = gather_state(st, tensors, idxs)
        full_before = {t: to_np(st.theta.views[t]).copy() for t in norm_tensors if t in tensors}
        gn = gpu_round(st, wl, rnd, frag, workers, draw, fold=fold)
        torch.cuda.synchronize()
        sampled_round_check(wl, st, frag, workers, draw, idxs, before, f"{wl.name} round {rnd}")
        if gn is not None:
            pt = gn[0].cpu().numpy()[:len(tensors)]
            pf = gn[1].item()
            assert (pt >= 0).all()
            assert abs(math.sqrt(float(np.sum(pt.astype(np.float64) ** 2))) - pf) <= 1e-9 * pf
            for t, th0 in full_before.items():
                want = full_tensor_norm(wl, workers, draw, th0, t)
                got = pt[tensors.index(t)]
                assert abs(got - want) <= NORM_RTOL * want, f"norm of tensor {t}: {got} vs {want}"
        del workers
    st.merger.close()


def test_diffurefill1b_f32_mean_ema_sampled():
    _sampled_workload(W.workload("diffurefill1b"))


def test_diffurefill1b_f32_mean_ema_folded_sampled():
    # the 1.08B round with its five workers folded as they arrive
    _sampled_workload(W.workload("diffurefill1b"), seed=1, fold=True)


def test_diffurefill1b_bf16_fragments_folded_sampled():
    _sampled_workload(W.workload("diffurefill1b_bf16"), seed=2, norm_tensors=(0, 9), fold=True)


def test_diffurefill1b_bf16_fragments_last_arrival_folded_at_commit_sampled():
    _sampled_workload(W.workload("diffurefill1b_bf16"), seed=3, norm_tensors=(0, 9), fold="last")


def test_diffurefill1b_bf16_fragments_nesterov_norms_sampled():
    # last fragment includes the final norm; tensor 0 is the 151M embedding
    _sampled_workload(W.workload("diffurefill1b_bf16"), norm_tensors=(0, 8, 9, 10, 18))


def test_diffurefill1b_bf16_two_rounds_in_flight_equal_sequential():
    """Rounds 0 and 1 (fragments 0 and 1) committed on two streams before any
    synchronisation give the same bits as committing them one after another,
    and match the oracle on sampled elements."""
    wl = W.workload("diffurefill1b_bf16")
    g = W.make_global(wl, 0, DEV)
    draws = [W.draw_round(wl, i, 0) for i in range(2)]
    workers = [[W.make_worker(wl, g, rnd, k, 0, DEV) for k in range(wl.K)]
               for rnd, _ in wl.rounds]
    rng = np.random.default_rng(5)
    frag_tensors = [[t for t in range(len(wl.specs)) if wl.specs[t].fragment == f]
                    for _, f in wl.rounds]
    idxs = [[sample_indices(wl.specs[t].numel, 2048, rng) for t in ts] for ts in frag_tensors]

    par = make_gpu_state(wl, g, DEV)
    befores = [gather_state(par, ts, ix) for ts, ix in zip(frag_tensors, idxs)]
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    cur = torch.cuda.current_stream()
    s1.wait_stream(cur)
    s2.wait_stream(cur)
    norms_par = []
    for (rnd, frag), w, d, s in zip(wl.rounds, workers, draws, (s1, s2)):
        with torch.cuda.stream(s):
            norms_par.append(gpu_round(par, wl, rnd, frag, w, d, stream=s))
    cur.wait_stream(s1)
    cur.wait_stream(s2)
    torch.cuda.synchronize()
    for (rnd, frag), w, d, ix, bf in zip(wl.rounds, workers, draws, idxs, befores):
        sampled_round_check(wl, par, frag, w, d, ix, bf, f"in flight round {rnd}")

    seq = make_gpu_state(wl, g, DEV)
    norms_seq = [gpu_round(seq, wl, rnd, frag, w, d)
                 for (rnd, frag), w, d in zip(wl.rounds, workers, draws)]
    torch.cuda.synchronize()
    assert torch.equal(par.theta.flat.view(torch.int32), seq.theta.flat.view(torch.int32))
    assert torch.equal(par.m.flat.view(torch.int32), seq.m.flat.view(torch.int32))
    for a, b in zip(norms_par, norms_seq):
        assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    par.merger.close()
    seq.merger.close()


@pytest.mark.parametrize("K", [2, 4, 8])
def test_sweep_16m_full(K):
    run_full(W.sweep_workload(64, 16_000_000, K))


@pytest.mark.parametrize("t,n,K", [(128, 256_000_000, 4), (256, 1_000_000_000, 4),
                                   (512, 4_000_000_000, 8)])
def test_sweep_large_sampled(t, n, K):
    _sampled_workload(W.sweep_workload(t, n, K), per_tensor=1024)


# ---- edge cases ------------------------------------------------------------------

RAGGED = [1, 2, 7, 8, 9, 15, 0, 2047, 2048, 2049, 16383, 16384, 16385, 100_003, 3]


def _custom(sizes, *, K, mode="delta", dtype="f32", ema=True, frags=None, n_fragments=1,
            rounds=((0, -1),), n_masked=0, quorum=None, tokens=(100_000, 150_000), norms=True):
    frags = frags or [0] * len(sizes)
    specs = tuple(W.TensorSpec(f"t{i}", (n,), f) for i, (n, f) in enumerate(zip(sizes, frags)))
    return W.Workload("custom", specs, n_fragments, K=K, n_masked=n_masked,
                      quorum=quorum or (K - n_masked), ckpt_dtype=dtype, mode=mode,
                      lr=0.7 if mode == "delta" else 1.0, mu=0.9 if mode == "delta" else 0.0,
                      ema_beta=0.9 if ema else None, rounds=rounds,
                      tokens=tokens if mode == "delta" else None, norms=norms)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("mode", ["mean", "delta"])
def test_ragged_and_empty_tensors(dtype, mode):
    run_full(_custom(RAGGED, K=3, mode=mode, dtype=dtype), seed=7)


@pytest.mark.parametrize("mode,fold", [("mean", False), ("mean", True), ("delta", False)])
def test_tensor_of_more_than_2_pow_31_elements(mode, fold):
    """One tensor of 2^31 + 13 elements (and a small one after it): 64-bit
    element offsets in every form. Plain mean + EMA takes the staged form,
    Nesterov + EMA the register form, fold=True the fold and final passes.
    Sampled elements, 2^31 and 2^32 neighbourhoods included, match the
    oracle; the big tensor's drift norm matches the oracle's, summed slice by
    slice in fp64."""
    n = (1 << 31) + 13
    wl = _custom([n, 2049], K=2, mode=mode, dtype="bf16", ema=True, norms=True)
    g = W.make_global(wl, 17, DEV)
    st = make_gpu_state(wl, g, DEV)
    draw = W.draw_round(wl, 0, 17)
    workers = [W.make_worker(wl, g, 0, k, 17, DEV) for k in range(wl.K)]
    rng = np.random.default_rng(17)
    edge = [(1 << 31) + o for o in (-9, -8, -1, 0, 1, 7, 8, 12)]
    idxs = [np.unique(np.concatenate([sample_indices(n, 2048, rng), np.array(edge, np.int64)])),
            sample_indices(2049, 2048, rng)]
    before = gather_state(st, [0, 1], idxs)
    th0 = st.theta.views[0].clone()
    pt, pf = gpu_round(st, wl, 0, -1, workers, draw, fold=fold)
    torch.cuda.synchronize()
    sampled_round_check(wl, st, -1, workers, draw, idxs, before, f"2^31+13 elements, {mode}")
    want = sliced_tensor_norm(wl, workers, draw, th0, 0)
    got = pt[0].item()
    assert abs(got - want) <= NORM_RTOL * want, (got, want)
    assert abs(pf.item() - math.sqrt(got ** 2 + pt[1].item() ** 2)) <= 1e-9 * pf.item()
    assert st.merger.status() == 0
    st.merger.close()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_k1_replacement_returns_input_bitwise(dtype):
    wl = _custom([4099, 65536], K=1, mode="mean", dtype=dtype, ema=False, norms=False)
    g = W.make_global(wl, 0, DEV)
    st = make_gpu_state(wl, g, DEV)
    w = [W.make_worker(wl, g, 0, 0, 0, DEV)]
    gpu_round(st, wl, 0, -1, w, W.RoundDraw(0, -1, [0], [0]))
    torch.cuda.synchronize()
    for t in range(2):
        assert torch.equal(st.theta.views[t].view(torch.int32),
                           w[0].views[t].float().view(torch.int32))
    st.merger.close()


def test_kmax_workers_and_one_more_rejected():
    wl = _custom([5000, 33], K=8)
    run_full(wl, seed=8)
    g = W.make_global(wl, 0, DEV)
    st = make_gpu_state(wl, g, DEV)
    w = W.make_worker(wl, g, 0, 0, 0, DEV)
    rd = st.merger.begin(0)
    for _ in range(8):
        rd.accumulate(w.views, 1)
    with pytest.raises(B.KmaxError):
        rd.accumulate(w.views, 1)
    rd.abort()
    st.merger.close()


@pytest.mark.parametrize("mode,ema", [("delta", True), ("delta", False), ("mean", True)])
def test_many_tensors_split_over_launches(mode, ema):
    # 1000 tensors with K = 8 exceed one launch's pointer block (3520 pointers);
    # the last two cases write two state arrays and take the staged form
    sizes = [(i * 37) % 300 + 1 for i in range(1000)]
    run_full(_custom(sizes, K=8, mode=mode, dtype="bf16", ema=ema), seed=9)


def test_empty_fragment_and_zero_size_tensors():
    sizes = [0, 0, 5000, 0]
    frags = [0, 0, 1, 2]   # fragment 0 has only empty tensors, fragment 3 has none
    wl = _custom(sizes, K=2, frags=frags, n_fragments=4,
                 rounds=((0, 0), (1, 3), (2, 1), (3, 2)))
    run_full(wl, seed=10)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_misaligned_views_take_the_scalar_path(dtype):
    """Tensors viewed at odd element offsets (not 16/32-byte aligned)."""
    sizes = [1001, 4096, 77]
    wl = _custom(sizes, K=3, dtype=dtype)
    dt = torch.bfloat16 if dtype == "bf16" else torch.float32
    g = W.make_global(wl, 0, DEV)

    def shifted(src_views, dtype_):
        views = []
        for v in src_views:
            buf = torch.empty(v.numel() + 1, dtype=dtype_, device=DEV)
            buf[1:].copy_(v)
            views.append(buf[1:])
        return views

    theta = shifted(g.views, torch.float32)
    m = shifted([torch.zeros_like(v) for v in g.views], torch.float32)
    e = shifted(g.views, torch.float32)
    mg = B.Merger(theta, momentum=m, ema=e, quorum=3)
    ost = oracle_state_from(g, wl)
    draw = W.draw_round(wl, 0, 0)
    workers = [W.make_worker(wl, g, 0, k, 0, DEV) for k in range(3)]
    xw = [shifted(w.views, dt) for w in workers]
    rd = mg.begin(0)
    for k in draw.included:
        rd.accumulate(xw[k], draw.tokens[k])
    rd.finalize(B.DELTA_NESTEROV, 0.7, 0.9)
    rd.ema_update(0.9)
    rd.commit()
    oracle_round(ost, wl, 0, -1, workers, draw)
    torch.cuda.synchronize()
    for t in range(3):
        assert_close(to_np(theta[t]), ost.theta[t], f"theta[{t}]")
        assert_close(to_np(m[t]), ost.m[t], f"m[{t}]")
        assert_close(to_np(e[t]), ost.e[t], f"e[{t}]")
    mg.close()


def test_large_token_counts_round_like_the_oracle():
    # counts above 2**24 are not exact in fp32: both sides round them the same way
    wl = _custom([3000, 129], K=3, tokens=(2**24 + 1, 2**26 + 7))
    run_full(wl, seed=11, bitwise=True)


def test_lr1_mu0_delta_is_token_weighted_mean():
    wl = _custom([4096, 999], K=4, ema=False)
    wl = W.Workload(wl.name, wl.specs, 1, K=4, n_masked=0, quorum=4, ckpt_dtype="f32",
                    mode="delta", lr=1.0, mu=0.0, tokens=(100_000, 150_000))
    g = W.make_global(wl, 0, DEV)
    st = make_gpu_state(wl, g, DEV)
    draw = W.draw_round(wl, 0, 0)
    workers = [W.make_worker(wl, g, 0, k, 0, DEV) for k in range(4)]
    gpu_round(st, wl, 0, -1, workers, draw)
    torch.cuda.synchronize()
    Wt = sum(draw.tokens[k] for k in draw.included)
    u = 2.0 ** -24
    for t in range(2):
        th0 = g.views[t].double()
        want = sum(draw.tokens[k] * workers[k].views[t].double() for k in draw.included) / Wt
        dmag = torch.stack([(workers[k].views[t].double() - th0).abs()
                            for k in draw.included]).max(0).values
        got = st.theta.views[t].double()
        # fp32 error bound of theta - 1*(-Delta) with Delta a 4-term weighted sum
        assert ((got - want).abs() <= 4 * u * (th0.abs() + 8 * dmag) + 1e-12).all()
    st.merger.close()


def test_determinism_repeat_is_bitwise_identical():
    wl = W.workload("pythia14m")
    runs = []
    for _ in range(2):
        g = W.make_global(wl, 0, DEV)
        st = make_gpu_state(wl, g, DEV)
        norms = []
        for idx, (rnd, frag) in enumerate(wl.rounds):
            draw = W.draw_round(wl, idx, 0)
            workers = [W.make_worker(wl, g, rnd, k, 0, DEV) for k in range(wl.K)]
            pt, pf = gpu_round(st, wl, rnd, frag, workers, draw)
            norms.append((pt.clone(), pf.clone()))
        torch.cuda.synchronize()
        runs.append((st.theta.flat.clone(), st.m.flat.clone(), norms))
        st.merger.close()
    (a_th, a_m, a_n), (b_th, b_m, b_n) = runs
    assert torch.equal(a_th.view(torch.int32), b_th.view(torch.int32))
    assert torch.equal(a_m.view(torch.int32), b_m.view(torch.int32))
    for (x1, y1), (x2, y2) in zip(a_n, b_n):
        assert torch.equal(x1, x2) and torch.equal(y1, y2)


def test_masked_worker_is_never_read():
    wl = _custom([3000, 17], K=4, n_masked=1, quorum=3)
    g = W.make_global(wl, 0, DEV)
    st = make_gpu_state(wl, g, DEV)
    draw = W.draw_round(wl, 0, 0)
    masked = [k for k in range(4) if k not in draw.included][0]
    workers = [W.make_worker(wl, g, 0, k, 0, DEV) for k in range(4)]
    workers[masked].flat.fill_(float("nan"))
    gpu_round(st, wl, 0, -1, workers, draw)
    torch.cuda.synchronize()
    assert torch.isfinite(st.theta.flat).all() and torch.isfinite(st.e.flat).all()
    st.merger.close()


# ---- the round state machine -----------------------------------------------------

def _tiny_merger(n_fragments=2, quorum=2):
    th = [torch.zeros(100, device=DEV), torch.zeros(50, device=DEV)]
    m = [torch.zeros_like(t) for t in th]
    e = [torch.zeros_like(t) for t in th]
    return B.Merger(th, momentum=m, ema=e, fragment_of=[0, n_fragments - 1],
                    n_fragments=n_fragments, quorum=quorum), th


def test_quorum_stale_busy_and_order_errors():
    mg, th = _tiny_merger()
    x = [torch.ones(100, device=DEV)]
    rd = mg.begin(5, 0)
    with pytest.raises(B.BusyError):
        mg.begin(6, 0)            # same fragment open
    with pytest.raises(B.BusyError):
        mg.begin(6, -1)           # "all" overlaps
    rd2 = mg.begin(7, 1)          # disjoint fragment: fine (two rounds in flight)
    with pytest.raises(B.StaleRoundError):
        B.merge_begin(mg.ctx, 6, 1)   # not newer than round 7
    rd.accumulate(x, 10)
    with pytest.raises(B.StateError):
        rd.commit()               # not finalized
    rd.finalize(B.DELTA_NESTEROV, 0.7, 0.9)
    with pytest.raises(B.StateError):
        rd.finalize(B.DELTA_NESTEROV, 0.7, 0.9)
    with pytest.raises(B.StateError):
        rd.accumulate(x, 10)      # after finalize
    with pytest.raises(B.QuorumError):
        rd.commit()               # 1 < quorum 2; round stays open
    assert torch.count_nonzero(th[0]) == 0
    rd2.abort()
    rd.abort()
    rd = mg.begin(8, 0)
    rd.accumulate(x, 10)
    rd.accumulate(x, 30)
    rd.finalize(B.DELTA_NESTEROV, 1.0, 0.0)
    rd.commit()
    torch.cuda.synchronize()
    assert torch.allclose(th[0], torch.ones(100, device=DEV))
    assert mg.last_round == 8
    with pytest.raises(B.StaleRoundError):
        mg.last_round = 3
    mg.last_round = 20
    with pytest.raises(B.StaleRoundError):
        mg.begin(20, 0)
    mg.close()


def test_argument_errors():
    mg, th = _tiny_merger()
    rd = mg.begin(0, 0)
    with pytest.raises(ValueError):
        rd.accumulate([torch.ones(99, device=DEV)], 1)            # wrong size
    rd.accumulate([torch.ones(100, device=DEV)], 1)
    with pytest.raises(ValueError):
        rd.accumulate([torch.ones(100, device=DEV, dtype=torch.bfloat16)], 1)
    with pytest.raises(B.ArgError):                               # mixed dtype at the ABI
        B.merge_accumulate(rd.handle, [torch.ones(100, device=DEV, dtype=torch.bfloat16).data_ptr()], B.BF16, 1)
    with pytest.raises(B.ArgError):
        B.merge_accumulate(rd.handle, [0], B.F32, 1)              # null pointer
    with pytest.raises(B.ArgError):
        rd.accumulate([torch.ones(100, device=DEV)], -5)          # negative tokens
    with pytest.raises(B.ArgError):
        rd.finalize(B.DELTA_NESTEROV, float("nan"), 0.9)
    with pytest.raises(B.ArgError):
        rd.ema_update(float("inf"))
    rd.accumulate([torch.ones(100, device=DEV)], 0)
    rd.finalize(B.DELTA_NESTEROV, 0.7, 0.9)
    rd.abort()
    rd = mg.begin(1, 0)
    rd.accumulate([torch.ones(100, device=DEV)], 0)
    rd.accumulate([torch.ones(100, device=DEV)], 0)
    rd.finalize(B.DELTA_NESTEROV, 0.7, 0.9)
    with pytest.raises(B.ArgError):
        rd.commit()                                               # zero total weight
    rd.abort()
    with pytest.raises(B.ArgError):
        mg.begin(2, 5)                                            # no such fragment
    mg.close()


def test_resume_after_restart_is_bitwise_identical():
    """A merger killed between rounds and restarted from its saved theta, m, e
    and round counter continues exactly as an uninterrupted one."""
    wl = W.workload("pythia14m")
    g = W.make_global(wl, 0, DEV)
    draws = [W.draw_round(wl, i, 0) for i in range(3)]
    workers = [[W.make_worker(wl, g, rnd, k, 0, DEV) for k in range(wl.K)] for rnd, _ in wl.rounds]
    a = make_gpu_state(wl, g, DEV)
    for (rnd, frag), w, d in zip(wl.rounds, workers, draws):
        gpu_round(a, wl, rnd, frag, w, d)
    b = make_gpu_state(wl, g, DEV)
    gpu_round(b, wl, 0, 0, workers[0], draws[0])
    torch.cuda.synchronize()
    saved = (b.theta.flat.cpu(), b.m.flat.cpu(), b.merger.last_round)
    b.merger.close()
    c = make_gpu_state(wl, g, DEV)          # "restarted process"
    c.theta.flat.copy_(saved[0])
    c.m.flat.copy_(saved[1])
    c.merger.last_round = saved[2]
    with pytest.raises(B.StaleRoundError):
        c.merger.begin(0, 0)                # the old round number is refused
    for (rnd, frag), w, d in list(zip(wl.rounds, workers, draws))[1:]:
        gpu_round(c, wl, rnd, frag, w, d)
    torch.cuda.synchronize()
    assert torch.equal(a.theta.flat.view(torch.int32), c.theta.flat.view(torch.int32))
    assert torch.equal(a.m.flat.view(torch.int32), c.m.flat.view(torch.int32))
    a.merger.close()
    c.merger.close()


# ---- host-resident checkpoints and published copies ------------------------------------

def _host_copy(arena, pinned=True):
    h = torch.empty(arena.flat.numel(), dtype=arena.flat.dtype, pin_memory=pinned)
    h.copy_(arena.flat)
    return W.Arena(h, arena.offsets, arena.numels)


@pytest.mark.parametrize("where", ["pinned", "pageable", "mixed"])
def test_host_resident_checkpoints_match_oracle(where):
    """Workers left in host memory are streamed by the fused pass itself."""
    wl = _custom(RAGGED, K=3, mode="delta", dtype="bf16", rounds=((0, -1), (1, -1)))
    g = W.make_global(wl, 0, DEV)
    st = make_gpu_state(wl, g, DEV)
    ost = oracle_state_from(g, wl)
    for idx, (rnd, frag) in enumerate(wl.rounds):
        draw = W.draw_round(wl, idx, 0)
        workers = [W.make_worker(wl, g, rnd, k, 0, DEV) for k in range(wl.K)]
        if where == "mixed":
            used = [_host_copy(w) if k % 2 == 0 else w for k, w in enumerate(workers)]
        else:
            used = [_host_copy(w, pinned=where == "pinned") for w in workers]
        try:
            gn = gpu_round(st, wl, rnd, frag, used, draw)
        except B.ArgError as ex:
            assert where == "pageable" and "cannot read" in str(ex)
            pytest.skip("this GPU does not read pageable host memory")
        on = oracle_round(ost, wl, rnd, frag, workers, draw)
        compare_full(st, ost, f"host workers ({where}) round {rnd}", bitwise=True)
        from merge_harness import compare_norms
        compare_norms(gn, on, f"host workers ({where}) round {rnd}")
    st.merger.close()


@pytest.mark.parametrize("dest", ["pinned", "device"])
@pytest.mark.parametrize("mode", ["delta", "mean"])  # mean + EMA takes the staged form
def test_publish_writes_copies_of_theta_and_ema(dest, mode):
    wl = _custom(RAGGED, K=3, mode=mode, dtype="f32")
    g = W.make_global(wl, 0, DEV)
    st = make_gpu_state(wl, g, DEV)
    draw = W.draw_round(wl, 0, 0)
    workers = [W.make_worker(wl, g, 0, k, 0, DEV) for k in range(3)]
    if dest == "pinned":
        pth = W.Arena(torch.full((st.theta.flat.numel(),), float("nan")).pin_memory(),
                      st.theta.offsets, st.theta.numels)
        pe = W.Arena(torch.full((st.e.flat.numel(),), float("nan")).pin_memory(),
                     st.e.offsets, st.e.numels)
    else:
        pth = W.empty_arena(st.theta.numels, torch.float32, DEV)
        pe = W.empty_arena(st.e.numels, torch.float32, DEV)
    rd = st.merger.begin(0)
    for k in draw.included:
        rd.accumulate(workers[k].views, draw.tokens[k])
    rd.finalize(B.DELTA_NESTEROV if mode == "delta" else B.MEAN_REPLACE, wl.lr, wl.mu)
    rd.ema_update(0.9)
    rd.publish(pth.views, pe.views)
    rd.commit()
    torch.cuda.synchronize()
    for t, n in enumerate(RAGGED):
        assert torch.equal(pth.views[t].cpu().view(torch.int32), st.theta.views[t].cpu().view(torch.int32))
        assert torch.equal(pe.views[t].cpu().view(torch.int32), st.e.views[t].cpu().view(torch.int32))
    st.merger.close()


def test_publish_ema_needs_an_ema_update():
    mg, th = _tiny_merger(n_fragments=1, quorum=1)
    x = [torch.ones(100, device=DEV), torch.ones(50, device=DEV)]
    out = [torch.empty(100, device=DEV), torch.empty(50, device=DEV)]
    rd = mg.begin(0)
    rd.accumulate(x, 1)
    rd.finalize(B.MEAN_REPLACE)
    rd.publish(out, [torch.empty(100, device=DEV), torch.empty(50, device=DEV)])
    with pytest.raises(B.StateError):
        rd.commit()
    rd.ema_update(0.9)
    rd.commit()
    torch.cuda.synchronize()
    assert torch.equal(out[0], th[0]) and torch.equal(out[1], th[1])
    mg.close()


# ---- uniform average of the globals (SWA) and snapshot averages --------------------

def _swa_workload(rounds, mode="delta", dtype="bf16"):
    wl = _custom(RAGGED, K=3, mode=mode, dtype=dtype, frags=[i % 2 for i in range(len(RAGGED))],
                 n_fragments=2, rounds=rounds)
    return W.Workload(wl.name, wl.specs, wl.n_fragments, K=wl.K, n_masked=0, quorum=3,
                      ckpt_dtype=dtype, mode=mode, lr=wl.lr, mu=wl.mu, ema_beta=0.9,
                      rounds=rounds, tokens=wl.tokens, norms=True, swa=True)


@pytest.mark.parametrize("mode,dtype", [("delta", "bf16"), ("mean", "f32")])
def test_swa_over_fragment_rounds_matches_oracle(mode, dtype):
    wl = _swa_workload(((0, 0), (1, 1), (2, 0), (3, 1), (4, -1)), mode, dtype)
    st, ost = run_full(wl, seed=12, bitwise=True)
    assert ost.swa_count == [3] * len(RAGGED)


def test_swa_counts_must_agree_within_a_round():
    wl = _swa_workload(((0, 0),))
    g = W.make_global(wl, 0, DEV)
    st = make_gpu_state(wl, g, DEV)
    draw = W.draw_round(wl, 0, 0)
    workers = [W.make_worker(wl, g, 0, k, 0, DEV) for k in range(3)]
    gpu_round(st, wl, 0, 0, workers, draw)          # fragment 0 now holds one global
    rd = st.merger.begin(1, -1)
    for k in draw.included:
        rd.accumulate(workers[k].views, draw.tokens[k])
    rd.finalize(B.DELTA_NESTEROV, 0.7, 0.9)
    rd.swa_update()
    with pytest.raises(B.StateError, match="different"):
        rd.commit()
    rd.abort()
    counts = st.merger.swa_counts
    assert [counts[t] for t in range(len(RAGGED)) if t % 2 == 0 and RAGGED[t]] == \
        [1] * sum(1 for t in range(0, len(RAGGED), 2) if RAGGED[t])
    st.merger.swa_reset(0)
    assert all(c == 0 for c in st.merger.swa_counts)
    torch.cuda.synchronize()
    assert torch.count_nonzero(st.swa.flat) == 0
    st.merger.swa_counts = [5] * len(RAGGED)       # resume from saved counts
    assert st.merger.swa_counts == [5] * len(RAGGED)
    rd = st.merger.begin(2, 1)
    with pytest.raises(B.BusyError):
        st.merger.swa_reset(-1)
    with pytest.raises(B.StateError):
        st.merger.swa_counts = [0] * len(RAGGED)
    rd.abort()
    st.merger.close()


def test_swa_on_the_1b_list_two_rounds_sampled():
    wl = W.workload("diffurefill1b_swa")
    g = W.make_global(wl, 0, DEV)
    st = make_gpu_state(wl, g, DEV)
    rng = np.random.default_rng(3)
    draw = W.draw_round(wl, 0, 0)
    idxs = [sample_indices(s.numel, 1024, rng) for s in wl.specs]
    tensors = list(range(len(wl.specs)))
    for rnd in (0, 1):
        workers = [W.make_worker(wl, g, rnd, k, 0, DEV) for k in range(wl.K)]
        before = gather_state(st, tensors, idxs)
        swa_before = [to_np(st.swa.views[t][torch.from_numpy(i).to(DEV)]) for t, i in zip(tensors, idxs)]
        gpu_round(st, wl, rnd, -1, workers, draw)
        torch.cuda.synchronize()
        sampled_round_check(wl, st, -1, workers, draw, idxs, before, f"swa round {rnd}")
        th_after = [to_np(st.theta.views[t][torch.from_numpy(i).to(DEV)]) for t, i in zip(tensors, idxs)]
        for t, i in zip(tensors, idxs):
            want = swa_before[t].copy()
            oracle.swa(th_after[t], rnd + 1, want)
            assert_close(to_np(st.swa.views[t][torch.from_numpy(i).to(DEV)]), want, f"swa[{t}]")
        del workers
    st.merger.close()


@pytest.mark.parametrize("window,dtype", [(3, "f32"), (5, "f32"), (5, "bf16")])
def test_average_of_the_last_snapshots_matches_oracle(window, dtype):
    specs = tuple(W.TensorSpec(f"t{i}", (n,), 0) for i, n in enumerate(RAGGED))
    wl = W.Workload("snap", specs, 1, K=window, n_masked=0, quorum=window, ckpt_dtype=dtype,
                    mode="mean")
    g = W.make_global(wl, 1, DEV)
    snaps = [W.make_worker(wl, g, 0, j, 1, DEV) for j in range(window)]
    out = W.empty_arena(g.numels, torch.float32, DEV)
    B.average_snapshots(out.views, [s.views for s in snaps])
    torch.cuda.synchronize()
    for t in range(len(RAGGED)):
        want = oracle.plain_average([to_np(s.views[t]) for s in snaps])
        assert bitwise_equal(to_np(out.views[t]), want)


# ---- per-worker drift (technical report, section 5.1) ------------------------------

def _worker_norm_check(wl, seed, with_round_norms, swa=False):
    g = W.make_global(wl, seed, DEV)
    st = make_gpu_state(wl, g, DEV)
    for idx, (rnd, frag) in enumerate(wl.rounds):
        draw = W.draw_round(wl, idx, seed)
        workers = [W.make_worker(wl, g, rnd, k, seed, DEV) for k in range(wl.K)]
        tensors = [t for t in range(len(wl.specs)) if frag == -1 or wl.specs[t].fragment == frag]
        th_before = {t: to_np(st.theta.views[t]).copy() for t in tensors}
        K = len(draw.included)
        pwt = torch.full((K * len(tensors),), -1.0, dtype=torch.float64, device=DEV)
        pw = torch.full((K,), -1.0, dtype=torch.float64, device=DEV)
        rd = st.merger.begin(rnd, frag)
        for k in draw.included:
            rd.accumulate(workers[k].views, draw.tokens[k])
        rd.finalize(B.DELTA_NESTEROV if wl.mode == "delta" else B.MEAN_REPLACE, wl.lr, wl.mu)
        if wl.ema_beta is not None:
            rd.ema_update(wl.ema_beta)
        if swa:
            rd.swa_update()
        if with_round_norms:
            rd.drift_norm(torch.zeros(len(tensors), dtype=torch.float64, device=DEV), None)
        rd.worker_drift_norm(pwt, pw)
        rd.commit()
        torch.cuda.synchronize()
        got = pwt.cpu().numpy().reshape(K, len(tensors))
        tot = np.zeros(K)
        for j, t in enumerate(tensors):
            want = oracle.worker_drift([to_np(workers[k].views[t]) for k in draw.included],
                                       th_before[t])
            tot += np.asarray(want)
            for k in range(K):
                w = math.sqrt(want[k])
                assert abs(got[k, j] - w) <= NORM_RTOL * w + 1e-300, (t, k, got[k, j], w)
        for k in range(K):
            w = math.sqrt(tot[k])
            assert abs(pw[k].item() - w) <= NORM_RTOL * w + 1e-300
        del workers
    st.merger.close()


@pytest.mark.parametrize("mode,dtype,round_norms", [("delta", "bf16", True), ("mean", "f32", False),
                                                    ("delta", "f32", False), ("mean", "bf16", True)])
def test_worker_drift_matches_oracle(mode, dtype, round_norms):
    wl = _custom(RAGGED, K=4, mode=mode, dtype=dtype, n_masked=1, quorum=3,
                 rounds=((0, -1), (1, -1)))
    _worker_norm_check(wl, 13, round_norms)


def test_worker_drift_with_ema_and_swa_fp32():
    wl = _swa_workload(((0, -1), (1, -1)), "delta", "f32")
    _worker_norm_check(wl, 14, True, swa=True)


def test_worker_drift_on_the_1b_bf16_fragment_whole_tensors():
    wl = W.workload("diffurefill1b_bf16")
    g = W.make_global(wl, 0, DEV)
    st = make_gpu_state(wl, g, DEV)
    draw = W.draw_round(wl, 0, 0)
    rnd, frag = wl.rounds[0]
    workers = [W.make_worker(wl, g, rnd, k, 0, DEV) for k in range(wl.K)]
    tensors = [t for t in range(len(wl.specs)) if wl.specs[t].fragment == frag]
    K = len(draw.included)
    pwt = torch.zeros(K * len(tensors), dtype=torch.float64, device=DEV)
    pw = torch.zeros(K, dtype=torch.float64, device=DEV)
    th0 = {t: to_np(st.theta.views[t]).copy() for t in tensors}
    rd = st.merger.begin(rnd, frag)
    for k in draw.included:
        rd.accumulate(workers[k].views, draw.tokens[k])
    rd.finalize(B.DELTA_NESTEROV, wl.lr, wl.mu)
    rd.worker_drift_norm(pwt, pw)
    rd.commit()
    torch.cuda.synchronize()
    got = pwt.cpu().numpy().reshape(K, len(tensors))
    for j, t in enumerate(tensors):   # fragment 0: the 151M-element embedding
        want = oracle.worker_drift([to_np(workers[k].views[t]) for k in draw.included], th0[t])
        for k in range(K):
            assert abs(got[k, j] - math.sqrt(want[k])) <= NORM_RTOL * math.sqrt(want[k])
    st.merger.close()


# ---- keep-drift adoption (technical report, section 5.1) ----------------------------

@pytest.mark.parametrize("dtype,misaligned", [("f32", False), ("bf16", False), ("f32", True)])
def test_keep_drift_adoption_matches_oracle(dtype, misaligned):
    wl = _custom(RAGGED + [300_001], K=3, mode="mean", dtype=dtype)
    g = W.make_global(wl, 21, DEV)
    pushed = W.make_worker(wl, g, 0, 0, 21, DEV)       # the checkpoint as pushed
    local = W.make_worker(wl, g, 1, 1, 21, DEV)        # the worker kept training
    newg = W.make_worker(wl, g, 2, 2, 21, DEV)          # the merged global
    th = [v.float().clone() for v in local.views]
    gl = [v.float().clone() for v in newg.views]
    if misaligned:  # odd element offsets: the scalar path
        def shift(ts):
            out = []
            for t in ts:
                buf = torch.empty(t.numel() + 1, dtype=t.dtype, device=DEV)
                buf[1:].copy_(t)
                out.append(buf[1:])
            return out
        th, gl = shift(th), shift(gl)
    want = [to_np(t).copy() for t in th]
    for w, gg, p in zip(want, gl, pushed.views):
        oracle.adopt_keep_drift(w, to_np(gg), to_np(p))
    B.adopt_keep_drift(th, gl, pushed.views)
    torch.cuda.synchronize()
    for t, w in enumerate(want):
        assert bitwise_equal(to_np(th[t]), w), f"tensor {t}"


def test_keep_drift_adoption_of_an_unmoved_worker_lands_near_the_global():
    n = 1 << 20
    p = torch.randn(n, device=DEV) * 0.02
    g = p + torch.randn(n, device=DEV) * 1e-3
    th = p.clone()
    B.adopt_keep_drift([th], [g], [p])
    torch.cuda.synchronize()
    assert ((th - g).abs() <= 2 * 2 ** -24 * (p.abs() + g.abs()) + 1e-30).all()


# ---- outer orthogonalisation (technical report, section 5.3) -----------------------

ORTHO_SHAPES = [(96, 40), (40, 96), (64, 64), (333, 0), (50, 7), (1, 0)]
# Error of the applied step relative to its largest element, by GEMM precision.
# TF32 rounds GEMM inputs to 11 significant bits (u = 2^-11 = 4.9e-4); the
# Newton-Schulz fixed point absorbs each step's rounding, and the measured
# error stays at 1.4-1.8 u (2048x2048 to 96x40 after 40 steps): the bound is
# 8 u. With fp32 GEMMs the measured error is 0.6-2e-6; the bound is 1e-5.
# A bf16 iterate is rounded to 8 significant bits (u = 2^-8) on every step;
# the same rule gives 8 u.
ORTHO_TOL = {B.ORTHO_FP32: 1e-5, B.ORTHO_TF32: 8 * 2.0 ** -11, B.ORTHO_BF16: 8 * 2.0 ** -8}


def _ortho_round(shapes, dtype, precision, mode, lr, iterations=40, seed=31, K=3):
    sizes = [r * c if c else r for r, c in shapes]
    rows = [r if c else 0 for r, c in shapes]
    wl = _custom(sizes, K=K, mode="mean", dtype=dtype)
    g = W.make_global(wl, seed, DEV)
    th = W.empty_arena(g.numels, torch.float32, DEV)
    th.flat.copy_(g.flat)
    e = W.empty_arena(g.numels, torch.float32, DEV)
    e.flat.copy_(g.flat)
    mg = B.Merger(th.views, ema=e.views, quorum=K, rows=rows)
    workers = [W.make_worker(wl, g, 0, k, seed, DEV) for k in range(K)]
    rd = mg.begin(0)
    for k in range(K):
        rd.accumulate(workers[k].views, 0)
    rd.finalize(B.MEAN_REPLACE)
    rd.ema_update(0.9)
    rd.orthogonalize(lr, mode, precision, iterations)
    rd.commit()
    torch.cuda.synchronize()
    out = []
    for t, (r, c) in enumerate(shapes):
        xs = [to_np(w.views[t]) for w in workers]
        th0 = to_np(g.views[t]).copy()
        got = to_np(th.views[t])
        if c:
            want, delta = oracle.orthogonal_update(xs, th0, r, lr=lr, scale_mode=mode)
            out.append(("matrix", t, r, c, th0, got, want, delta, to_np(e.views[t])))
        else:
            want = th0.copy()
            oracle.merge_tensor(xs, want, mode=oracle.MEAN_REPLACE)
            out.append(("vector", t, r, c, th0, got, want, None, to_np(e.views[t])))
    mg.close()
    return out


@pytest.mark.parametrize("precision", [B.ORTHO_FP32, B.ORTHO_TF32, B.ORTHO_BF16])
@pytest.mark.parametrize("mode", [B.ORTHO_SCALE_FIXED, B.ORTHO_SCALE_MATCH_NORM])
def test_orthogonalised_round_matches_the_polar_factor(precision, mode):
    lr = 0.01 if mode == B.ORTHO_SCALE_FIXED else 0.7
    for kind, t, r, c, th0, got, want, delta, e in _ortho_round(ORTHO_SHAPES, "f32", precision,
                                                                 mode, lr):
        if kind == "vector":   # non-matrix tensors take plain replacement, bit for bit
            assert bitwise_equal(got, want.astype(np.float32)), t
            continue
        step_want = want - th0.astype(np.float64)
        scale = np.abs(step_want).max()
        err = np.abs(got.astype(np.float64) - want).max()
        print(f"ortho precision={precision} mode={mode} {r}x{c}: max err / max step = {err / scale:.3e}")
        # the fp32 rounding of theta' itself adds at most one ulp of |theta'|
        assert err <= ORTHO_TOL[precision] * scale + 2 * np.spacing(np.float32(np.abs(want).max()))
        # the applied step is semi-orthogonal up to the same tolerance
        o = (got.astype(np.float64) - th0).reshape(r, c)
        o *= np.sqrt(min(r, c)) / np.linalg.norm(o)   # singular values ~1 if semi-orthogonal
        gram = o.T @ o if r >= c else o @ o.T
        # to first order O^T O - I = Q^T E + E^T Q for O = Q + E: twice the
        # step's error (measured 1e-6, 7e-4 and 2.7e-3 for fp32, tf32, bf16)
        assert np.abs(gram - np.eye(min(r, c))).max() <= 4 * ORTHO_TOL[precision]
        # EMA of the new global, from the GPU's theta'
        e_want = 0.9 * th0.astype(np.float64) + np.float64(np.float32(1) - np.float32(0.9)) * got
        assert np.abs(e.astype(np.float64) - e_want).max() <= 4 * np.spacing(np.float32(np.abs(e_want).max()))


def test_orthogonalised_round_bf16_workers():
    for kind, t, r, c, th0, got, want, delta, e in _ortho_round(ORTHO_SHAPES[:3], "bf16",
                                                                 B.ORTHO_FP32, B.ORTHO_SCALE_FIXED,
                                                                 0.01, seed=32):
        scale = np.abs(want - th0).max()
        assert np.abs(got - want).max() <= ORTHO_TOL[B.ORTHO_FP32] * scale + 1e-9


@pytest.mark.parametrize("precision", [B.ORTHO_TF32, B.ORTHO_BF16])
def test_orthogonalised_round_on_1b_block_shapes(precision):
    shapes = [(2048, 2048), (5632, 2048), (2048, 5632), (2048, 0)]
    for kind, t, r, c, th0, got, want, delta, e in _ortho_round(shapes, "f32", precision,
                                                                 B.ORTHO_SCALE_MATCH_NORM, 0.7,
                                                                 iterations=40, seed=33):
        if kind == "vector":
            continue
        scale = np.abs(want - th0).max()
        err = np.abs(got.astype(np.float64) - want).max()
        print(f"1b block precision={precision} {r}x{c}: max err / max step = {err / scale:.3e}")
        assert err <= ORTHO_TOL[precision] * scale + 2 * np.spacing(np.float32(np.abs(want).max()))


def test_orthogonalisation_of_a_zero_update_leaves_theta():
    th = [torch.randn(64 * 32, device=DEV) * 0.02]
    orig = th[0].clone()
    mg = B.Merger(th, quorum=2, rows=[64])
    rd = mg.begin(0)
    rd.accumulate([orig.clone()], 0)
    rd.accumulate([orig.clone()], 0)
    rd.finalize(B.MEAN_REPLACE)
    rd.orthogonalize(1.0)
    rd.commit()
    torch.cuda.synchronize()
    assert torch.equal(th[0], orig)
    mg.close()


def test_orthogonalisation_takes_only_plain_mean_with_ema():
    th = [torch.zeros(16 * 8, device=DEV)]
    m = [torch.zeros_like(th[0])]
    mg = B.Merger(th, momentum=m, quorum=1, rows=[16])
    x = [torch.ones(16 * 8, device=DEV)]
    rd = mg.begin(0)
    rd.accumulate(x, 5)
    rd.finalize(B.DELTA_NESTEROV, 0.7, 0.9)
    rd.orthogonalize(1.0)
    with pytest.raises(B.StateError, match="plain-mean"):
        rd.commit()
    rd.abort()
    rd = mg.begin(1)
    rd.accumulate(x, 5)
    rd.finalize(B.MEAN_REPLACE)
    for bad in ((7, 0, 10), (0, 9, 10), (0, 0, 0)):   # scale mode, precision, iterations
        with pytest.raises(B.ArgError):
            B.merge_orthogonalize(rd.handle, 1.0, *bad)
    rd.orthogonalize(1.0)
    with pytest.raises(B.StateError, match="twice"):
        rd.orthogonalize(1.0)
    rd.drift_norm(torch.zeros(1, dtype=torch.float64, device=DEV), None)
    with pytest.raises(B.StateError, match="only an EMA"):
        rd.commit()
    rd.abort()
    mg.close()


def test_orthogonalisation_batches_equal_shapes_each_with_its_own_norm():
    # interleaved shapes: the three 48x20 and two 20x48 matrices are each
    # orthogonalised in one strided batch, every matrix with its own |Delta|
    shapes = [(48, 20), (20, 48), (7, 0), (48, 20), (20, 48), (48, 20), (33, 3)]
    for precision in (B.ORTHO_FP32, B.ORTHO_TF32):
        for kind, t, r, c, th0, got, want, delta, e in _ortho_round(
                shapes, "f32", precision, B.ORTHO_SCALE_MATCH_NORM, 0.5, seed=34):
            if kind == "vector":
                assert bitwise_equal(got, want.astype(np.float32))
                continue
            scale = np.abs(want - th0).max()
            assert np.abs(got.astype(np.float64) - want).max() <= ORTHO_TOL[precision] * scale + 1e-9, \
                (precision, t)


def test_orthogonalised_fragment_round_with_pinned_host_workers():
    """Only the round's fragment changes; its workers stream from host memory."""
    shapes = [(40, 24), (24, 40), (100, 0), (40, 24)]
    frags = [0, 1, 1, 0]
    sizes = [r * c if c else r for r, c in shapes]
    rows = [r if c else 0 for r, c in shapes]
    wl = _custom(sizes, K=3, mode="mean", dtype="bf16", frags=frags, n_fragments=2)
    g = W.make_global(wl, 35, DEV)
    th = W.empty_arena(g.numels, torch.float32, DEV)
    th.flat.copy_(g.flat)
    mg = B.Merger(th.views, fragment_of=frags, n_fragments=2, quorum=3, rows=rows)
    workers = [W.make_worker(wl, g, 0, k, 35, DEV) for k in range(3)]
    host = [_host_copy(w) for w in workers]
    rd = mg.begin(0, 1)
    for h in host:
        rd.accumulate(h.views, 0)
    rd.finalize(B.MEAN_REPLACE)
    rd.orthogonalize(0.02, B.ORTHO_SCALE_FIXED, B.ORTHO_FP32, 40)
    rd.commit()
    torch.cuda.synchronize()
    for t, (r, c) in enumerate(shapes):
        got, th0 = to_np(th.views[t]), to_np(g.views[t])
        if frags[t] != 1:
            assert bitwise_equal(got, th0), t           # other fragment untouched
            continue
        xs = [to_np(w.views[t]) for w in workers]
        if c:
            want, _ = oracle.orthogonal_update(xs, th0, r, lr=0.02)
            assert np.abs(got - want).max() <= ORTHO_TOL[B.ORTHO_FP32] * np.abs(want - th0).max() + 1e-9
        else:
            want = th0.copy()
            oracle.merge_tensor(xs, want, mode=oracle.MEAN_REPLACE)
            assert bitwise_equal(got, want)
    mg.close()


# ---- the staged and register forms of the merge pass ------------------------------

STAGED_SIZES = [1, 7, 8, 9, 2047, 2048, 2049, 6000, 16385, 100_003, 0, 3, 1 << 20, 4100]


def _ab_round(st, wl, rnd, workers, draw, *, worker_norms, publish):
    rd = st.merger.begin(rnd, -1)
    for k in draw.included:
        rd.accumulate(workers[k].views, draw.tokens[k])
    rd.finalize(B.DELTA_NESTEROV if wl.mode == "delta" else B.MEAN_REPLACE, wl.lr, wl.mu)
    if wl.ema_beta is not None:
        rd.ema_update(wl.ema_beta)
    if wl.swa:
        rd.swa_update()
    T = len(rd.tensors)
    out = {}
    if wl.norms:
        out["pt"] = torch.full((T,), -1.0, dtype=torch.float64, device=DEV)
        out["pf"] = torch.full((1,), -1.0, dtype=torch.float64, device=DEV)
        rd.drift_norm(out["pt"], out["pf"])
    if worker_norms:
        out["pwt"] = torch.full((len(draw.included) * T,), -1.0, dtype=torch.float64, device=DEV)
        out["pw"] = torch.full((len(draw.included),), -1.0, dtype=torch.float64, device=DEV)
        rd.worker_drift_norm(out["pwt"], out["pw"])
    if publish:
        out["th_pub"] = [torch.full_like(v, float("nan")) for v in st.theta.views]
        out["e_pub"] = ([torch.full_like(v, float("nan")) for v in st.e.views]
                        if st.e is not None else None)
        rd.publish(out["th_pub"], out["e_pub"])
    rd.commit()
    return out


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("mode,ema,norms,swa,K,worker_norms,publish", [
    ("mean", True, False, False, 5, False, False),   # the 1.08B round's variant
    ("mean", False, True, False, 1, False, False),
    ("delta", False, True, False, 3, False, False),  # the bf16 in-flight rounds' variant
    ("delta", False, True, False, 8, True, True),    # K = CAM_KMAX, worker norms, publish
    ("mean", False, False, True, 2, False, True),    # running average, publish
    ("mean", True, True, False, 3, True, True),
    # three state arrays written: both sides take the register form
    ("delta", True, True, True, 8, True, False),
    ("mean", True, False, True, 2, False, True),
])
def test_staged_and_register_forms_agree_bitwise(dtype, mode, ema, norms, swa, K,
                                                 worker_norms, publish):
    """Same seeded rounds through both forms of the pass: theta, m, e, the running
    average and the published copies agree bit for bit; drift norms (whose fp32
    per-thread grouping differs between the forms) agree within the norm
    tolerance; the oracle checks the staged form's values."""
    wl = dataclasses.replace(_custom(STAGED_SIZES, K=K, mode=mode, dtype=dtype, ema=ema,
                                     norms=norms, rounds=((0, -1), (1, -1))), swa=swa)
    g = W.make_global(wl, 3, DEV)
    # the separate norm pass on both sides, so small rounds keep each form
    states = [make_gpu_state(wl, g, DEV, staging=sg, fused_finish=False) for sg in (True, False)]
    ost = oracle_state_from(g, wl)
    for idx, (rnd, frag) in enumerate(wl.rounds):
        draw = W.draw_round(wl, idx, 3)
        workers = [W.make_worker(wl, g, rnd, k, 3, DEV) for k in range(wl.K)]
        outs = [_ab_round(st, wl, rnd, workers, draw, worker_norms=worker_norms, publish=publish)
                for st in states]
        oracle_round(ost, wl, rnd, frag, workers, draw)
        torch.cuda.synchronize()
        a, b = states
        for name in ("theta", "m", "e", "swa"):
            x, y = getattr(a, name), getattr(b, name)
            if x is not None:
                assert torch.equal(x.flat.view(torch.int32), y.flat.view(torch.int32)), \
                    f"round {rnd}: {name} differs between the staged and register forms"
        compare_full(a, ost, f"staged round {rnd}")
        if publish:
            for t, v in enumerate(a.theta.views):
                assert torch.equal(outs[0]["th_pub"][t].view(torch.int32), v.view(torch.int32))
                if a.e is not None:
                    assert torch.equal(outs[0]["e_pub"][t].view(torch.int32),
                                       a.e.views[t].view(torch.int32))
        for key in ("pt", "pf", "pwt", "pw"):
            if key in outs[0]:
                x, y = outs[0][key].cpu().numpy(), outs[1][key].cpu().numpy()
                assert (x >= 0).all(), f"{key}: norm not written"
                assert np.all(np.abs(x - y) <= NORM_RTOL * np.abs(y) + 1e-300), f"{key}: {x} vs {y}"
    for st in states:
        assert st.merger.status() == 0
        st.merger.close()


@pytest.mark.parametrize("fused", [False, True])
def test_staged_form_is_used_and_reproducible(fused):
    """Two identical runs agree bit for bit, norms included, and a round of
    device workers launches exactly one merge pass plus the norm finish, or
    one pass alone when it finishes its norms itself (a small round)."""
    wl = _custom([1 << 20, 3, 2049, 5_000_000], K=4, mode="delta", dtype="bf16", ema=True)
    g = W.make_global(wl, 0, DEV)
    res = []
    for _ in range(2):
        st = make_gpu_state(wl, g, DEV, fused_finish=fused)
        draw = W.draw_round(wl, 0, 0)
        workers = [W.make_worker(wl, g, 0, k, 0, DEV) for k in range(wl.K)]
        n0 = st.merger.launch_count
        pt, pf = gpu_round(st, wl, 0, -1, workers, draw)
        assert st.merger.launch_count - n0 == (1 if fused else 2)
        torch.cuda.synchronize()
        res.append((st.theta.flat.clone(), st.m.flat.clone(), st.e.flat.clone(), pt.clone(), pf.clone()))
        assert st.merger.status() == 0
        st.merger.close()
    for x, y in zip(*res):
        assert torch.equal(x, y)


@pytest.mark.parametrize("mode,dtype,ema,publish,host", [
    ("delta", "f32", False, False, False),   # the Pythia rounds' variant
    ("mean", "bf16", True, False, False),    # a staged round without the fusion
    ("delta", "bf16", True, True, False),
    ("mean", "f32", False, False, True),     # pinned host workers
])
def test_fused_norm_finish_equals_the_norm_pass(mode, dtype, ema, publish, host):
    """Small rounds whose merge pass finishes the drift norms itself give the
    bits of the same rounds with the separate norm pass: theta, m, e, the
    published copies and the norms, over several rounds and fragments (the
    per-plan block counter is reset by every launch)."""
    wl = _custom(RAGGED + [300_001], K=3, mode=mode, dtype=dtype, ema=ema, norms=True,
                 frags=[i % 2 for i in range(len(RAGGED) + 1)], n_fragments=2,
                 rounds=((0, 0), (1, 1), (2, -1), (3, 0)))
    g = W.make_global(wl, 18, DEV)
    # the fused pass is the register form: compare with that form's norm pass
    states = [make_gpu_state(wl, g, DEV), make_gpu_state(wl, g, DEV, staging=False, fused_finish=False)]
    for idx, (rnd, frag) in enumerate(wl.rounds):
        draw = W.draw_round(wl, idx, 18)
        workers = [W.make_worker(wl, g, rnd, k, 18, DEV) for k in range(wl.K)]
        if host:
            workers = [W.Arena(w.flat.cpu().pin_memory(), w.offsets, w.numels) for w in workers]
        outs, launches = [], []
        for st in states:
            rd = st.merger.begin(rnd, frag)
            for k in draw.included:
                rd.accumulate(workers[k].views, draw.tokens[k])
            code = B.DELTA_NESTEROV if mode == "delta" else B.MEAN_REPLACE
            rd.finalize(code, wl.lr, wl.mu)
            if ema:
                rd.ema_update(0.9)
            pt = torch.full((max(1, len(rd.tensors)),), -1.0, dtype=torch.float64, device=DEV)
            pf = torch.full((1,), -1.0, dtype=torch.float64, device=DEV)
            rd.drift_norm(pt, pf)
            pub = None
            if publish:
                pub = [torch.full((st.merger.numel[t],), float("nan"), device=DEV)
                       for t in rd.tensors]
                rd.publish(pub)
            n0 = st.merger.launch_count
            rd.commit()
            launches.append(st.merger.launch_count - n0)
            outs.append((pt, pf, pub))
        torch.cuda.synchronize()
        fused, plain = states
        for name in ("theta", "m", "e"):
            x, y = getattr(fused, name), getattr(plain, name)
            if x is not None:
                assert torch.equal(x.flat.view(torch.int32), y.flat.view(torch.int32)), (rnd, name)
        assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1]), rnd
        assert (outs[0][0] >= 0).all() and outs[0][1].item() >= 0
        if publish:
            for a, b in zip(outs[0][2], outs[1][2]):
                assert torch.equal(a.view(torch.int32), b.view(torch.int32))
        assert launches[0] == launches[1] - 1, launches   # the norm pass is not launched
    for st in states:
        assert st.merger.status() == 0
        st.merger.close()


@pytest.mark.parametrize("mode,norms", [("mean", False), ("delta", True)])
def test_staged_wait_that_runs_out_is_reported_and_the_device_recovers(mode, norms):
    """The staged pass's bounded waits, driven to their limit on purpose: with
    CAM_TEST_STALL_STAGED every staged pass withholds its first tile, so its
    consumers' waits (and, with norms, the reducer's) give up after about 1 ms.
    The pass returns with CAM_STATUS_WAIT_TIMEOUT in the context's status word
    and no copy in flight; nothing faults or hangs. A fresh context on the
    same device then runs the round and matches the oracle."""
    wl = _custom([300_000, 70_000, 2049], K=2, mode=mode, ema=mode == "mean", norms=norms)
    g = W.make_global(wl, 0, DEV)
    draw = W.draw_round(wl, 0, 0)
    workers = [W.make_worker(wl, g, 0, k, 0, DEV) for k in range(wl.K)]
    # the norm pass stays separate, so a round with norms takes the staged form too
    st = make_gpu_state(wl, g, DEV, fused_finish=False, test_stall_staged=True)
    n0 = st.merger.staged_count
    gpu_round(st, wl, 0, -1, workers, draw)
    torch.cuda.synchronize()
    assert st.merger.staged_count - n0 > 0
    assert st.merger.status() & B.STATUS_WAIT_TIMEOUT
    st.merger.close()
    fresh = make_gpu_state(wl, g, DEV, fused_finish=False)
    gn = gpu_round(fresh, wl, 0, -1, workers, draw)
    torch.cuda.synchronize()
    assert fresh.merger.staged_count > 0
    ost = oracle_state_from(g, wl)
    norms_want = oracle_round(ost, wl, 0, -1, workers, draw)
    compare_full(fresh, ost, f"after a stalled pass: {mode}")
    if norms:
        pt, _ = norms_want
        got = gn[0].cpu().numpy()[:len(pt)]
        assert np.all(np.abs(got - np.asarray(pt)) <= NORM_RTOL * np.abs(np.asarray(pt)))
    assert fresh.merger.status() == 0
    fresh.merger.close()


@pytest.mark.parametrize("form", ["register_fin", "register", "staged", "fold"])
def test_corrupted_chunk_is_skipped_and_reported(form):
    """The passes' own chunk checks, met on purpose: with CAM_TEST_BAD_CHUNK
    the device copy of the chunk table has the first tensor's last chunk reach
    2,048 elements past that tensor's end. The arena puts the next tensor
    there, so even an unchecked pass would stay inside the allocations (and
    show up as wrong values in that tensor). Every form -- the register pass
    with and without its fused norm finish, the staged pass and the eager
    folds with their final pass -- must skip the chunk: its elements keep
    their values, its drift counts as 0, CAM_STATUS_BAD_CHUNK is set, and
    everything else equals the oracle run on the list without that chunk."""
    wl = _custom([300_000, 70_000, 2049], K=2, mode="delta", ema=False, norms=True)
    g = W.make_global(wl, 0, DEV)
    assert g.offsets[1] + g.numels[1] >= g.numels[0] + 2048  # room for the overrun
    draw = W.draw_round(wl, 0, 0)
    workers = [W.make_worker(wl, g, 0, k, 0, DEV) for k in range(wl.K)]
    st = make_gpu_state(wl, g, DEV, staging=form == "staged",
                        fused_finish=form == "register_fin", test_bad_chunk=True)
    n0 = st.merger.staged_count
    pt, pf = gpu_round(st, wl, 0, -1, workers, draw, fold=form == "fold")
    torch.cuda.synchronize()
    assert (st.merger.staged_count - n0 > 0) == (form == "staged")
    assert st.merger.status() == B.STATUS_BAD_CHUNK
    # the skipped chunk: the trailing run of tensor 0 that kept its bits
    g0 = to_np(g.views[0])
    th0 = to_np(st.theta.views[0])
    same = th0.view(np.uint32) == g0.view(np.uint32)
    s = len(same) - int(np.argmin(same[::-1])) if not same.all() else 0
    assert 0 < s < len(g0) and s % 2048 == 0, s
    assert not same[:s].any()
    assert (to_np(st.m.views[0])[s:] == 0).all()
    # what lies between tensor 0's end and tensor 1 kept its bits
    gap = slice(g.numels[0], g.offsets[1])
    assert torch.equal(st.theta.flat[gap].view(torch.int32), g.flat[gap].view(torch.int32))
    assert (st.m.flat[gap] == 0).all()
    # the oracle on the list without the skipped chunk
    ost = oracle.OracleState(
        theta=[g0[:s].copy()] + [to_np(v).copy() for v in g.views[1:]],
        m=[np.zeros(s, np.float32)] + [np.zeros(n, np.float32) for n in g.numels[1:]],
        fragment_of=wl.fragment_of)
    ck = [[to_np(w.views[0])[:s]] + [to_np(v) for v in w.views[1:]] for w in workers]
    pt_want, pf_want = oracle.merge_round(
        ost, round=0, fragment=-1, ckpts=ck, included=draw.included, tokens=draw.tokens,
        mode=oracle.DELTA_NESTEROV, lr=wl.lr, mu=wl.mu, quorum=wl.quorum, ema_beta=None,
        swa_update=False)
    assert_close(th0[:s], ost.theta[0], "theta, tensor 0 before the skipped chunk")
    assert_close(to_np(st.m.views[0])[:s], ost.m[0], "m, tensor 0 before the skipped chunk")
    for t in (1, 2):
        assert_close(to_np(st.theta.views[t]), ost.theta[t], f"theta, tensor {t}")
        assert_close(to_np(st.m.views[t]), ost.m[t], f"m, tensor {t}")
    got = pt.cpu().numpy()
    want = np.asarray(pt_want)
    assert np.all(np.abs(got - want) <= NORM_RTOL * np.abs(want)), (got, want)
    assert abs(pf.item() - pf_want) <= NORM_RTOL * abs(pf_want)
    st.merger.close()


@pytest.mark.parametrize("mode,norms", [("mean", False), ("delta", True)])
def test_staged_stage_out_of_sequence_is_reported(mode, norms):
    """The staged pass's protocol check, met on purpose: with CAM_TEST_BAD_TAG
    every staged pass labels its end marker with a wrong fill number. The
    consumers find that it does not match the number of stages they took, set
    CAM_STATUS_PROTOCOL and stop without releasing it; the producer's wait for
    that release then gives up after about 1 ms, with every copy landed.
    Nothing faults or hangs, and a fresh context on the same device runs the
    round like the oracle."""
    wl = _custom([300_000, 70_000, 2049], K=2, mode=mode, ema=mode == "mean", norms=norms)
    g = W.make_global(wl, 0, DEV)
    draw = W.draw_round(wl, 0, 0)
    workers = [W.make_worker(wl, g, 0, k, 0, DEV) for k in range(wl.K)]
    st = make_gpu_state(wl, g, DEV, fused_finish=False, test_bad_tag=True)
    n0 = st.merger.staged_count
    gpu_round(st, wl, 0, -1, workers, draw)
    torch.cuda.synchronize()
    assert st.merger.staged_count - n0 > 0
    assert st.merger.status() & B.STATUS_PROTOCOL
    st.merger.close()
    fresh = make_gpu_state(wl, g, DEV, fused_finish=False)
    gpu_round(fresh, wl, 0, -1, workers, draw)
    ost = oracle_state_from(g, wl)
    oracle_round(ost, wl, 0, -1, workers, draw)
    compare_full(fresh, ost, f"after a pass stopped on its protocol check: {mode}")
    assert fresh.merger.status() == 0
    fresh.merger.close()


@pytest.mark.parametrize("mode,ema,swa,host,staging,want_staged", [
    ("mean", True, False, False, True, True),     # theta, e written
    ("delta", False, False, False, True, True),   # theta, m written
    ("delta", True, False, False, True, False),   # theta, m, e: register form
    ("mean", True, True, False, True, False),     # theta, e, swa: register form
    ("mean", True, False, True, True, False),     # host-resident workers
    ("mean", True, False, False, False, False),   # CAM_NO_STAGING
])
def test_form_of_the_merge_pass(mode, ema, swa, host, staging, want_staged):
    wl = dataclasses.replace(_custom([70_000, 2049], K=2, mode=mode, ema=ema, norms=False),
                             swa=swa)
    g = W.make_global(wl, 0, DEV)
    st = make_gpu_state(wl, g, DEV, staging=staging)
    draw = W.draw_round(wl, 0, 0)
    workers = [W.make_worker(wl, g, 0, k, 0, DEV) for k in range(wl.K)]
    if host:
        workers = [W.Arena(w.flat.cpu().pin_memory(), w.offsets, w.numels) for w in workers]
    n0 = st.merger.staged_count
    gpu_round(st, wl, 0, -1, workers, draw)
    torch.cuda.synchronize()
    assert (st.merger.staged_count - n0 > 0) == want_staged
    ost = oracle_state_from(g, wl)
    oracle_round(ost, wl, 0, -1, workers, draw)
    compare_full(st, ost, f"form test {mode} ema={ema} swa={swa} host={host}")
    assert st.merger.status() == 0
    st.merger.close()


# tall and wide enough (long side >= 4 x short side) for the short-side form,
# plus shapes below that ratio, which keep the plain iteration in the same round
SHORT_SIDE_SHAPES = [(512, 64), (1000, 100), (48, 400), (96, 40), (64, 64), (333, 0)]


@pytest.mark.parametrize("precision", [B.ORTHO_FP32, B.ORTHO_TF32])
@pytest.mark.parametrize("mode", [B.ORTHO_SCALE_FIXED, B.ORTHO_SCALE_MATCH_NORM])
def test_short_side_iteration_matches_the_polar_factor(precision, mode):
    lr = 0.01 if mode == B.ORTHO_SCALE_FIXED else 0.7
    for kind, t, r, c, th0, got, want, delta, e in _ortho_round(
            SHORT_SIDE_SHAPES, "f32", precision | B.ORTHO_SHORT_SIDE, mode, lr, seed=35):
        if kind == "vector":
            assert bitwise_equal(got, want.astype(np.float32)), t
            continue
        scale = np.abs(want - th0.astype(np.float64)).max()
        err = np.abs(got.astype(np.float64) - want).max()
        print(f"short side precision={precision} mode={mode} {r}x{c}: "
              f"max err / max step = {err / scale:.3e}")
        assert err <= ORTHO_TOL[precision] * scale + 2 * np.spacing(np.float32(np.abs(want).max()))
        o = (got.astype(np.float64) - th0).reshape(r, c)
        o *= np.sqrt(min(r, c)) / np.linalg.norm(o)
        gram = o.T @ o if r >= c else o @ o.T
        assert np.abs(gram - np.eye(min(r, c))).max() <= 30 * ORTHO_TOL[precision]


def test_short_side_flag_is_validated():
    th = [torch.zeros(64, device=DEV)]
    e = [torch.zeros(64, device=DEV)]
    mg = B.Merger(th, ema=e, quorum=1, rows=[8])
    rd = mg.begin(0)
    for bad in (3, B.ORTHO_BF16 | B.ORTHO_SHORT_SIDE, 7, 8, 11):
        with pytest.raises(B.ArgError):
            rd.orthogonalize(0.1, B.ORTHO_SCALE_FIXED, bad, 10)
    rd.orthogonalize(0.1, B.ORTHO_SCALE_FIXED, B.ORTHO_FP32 | B.ORTHO_SHORT_SIDE, 10)
    rd.abort()
    mg.close()


# ---- eagerly folded rounds (cam_merge_fold) ----------------------------------------

def _fold_round(st, wl, rnd, workers, draw, *, norms, wnorms, publish, streams=None,
                pub_host=False, accumulate_last=0):
    rd = st.merger.begin(rnd, -1)
    code = B.DELTA_NESTEROV if wl.mode == "delta" else B.MEAN_REPLACE
    T = len(rd.tensors)
    out = {}
    if wnorms:
        out["pwt"] = torch.full((len(draw.included) * T,), -1.0, dtype=torch.float64, device=DEV)
        out["pw"] = torch.full((len(draw.included),), -1.0, dtype=torch.float64, device=DEV)
        rd.worker_drift_norm(out["pwt"], out["pw"])
    n_inc = len(draw.included)
    for i, k in enumerate(draw.included):
        s = None if streams is None else streams[i % len(streams)]
        if streams is None or i >= n_inc - accumulate_last:  # the last ones: folded at commit
            rd.accumulate(workers[k].views, draw.tokens[k])
        else:
            rd.fold(workers[k].views, draw.tokens[k], code, stream=s)
    rd.finalize(code, wl.lr, wl.mu)
    if wl.ema_beta is not None:
        rd.ema_update(wl.ema_beta)
    if wl.swa:
        rd.swa_update()
    if norms:
        out["pt"] = torch.full((T,), -1.0, dtype=torch.float64, device=DEV)
        out["pf"] = torch.full((1,), -1.0, dtype=torch.float64, device=DEV)
        rd.drift_norm(out["pt"], out["pf"])
    if publish:
        def buf(v):
            t = torch.full_like(v, float("nan"))
            return t.cpu().pin_memory() if pub_host else t
        out["th_pub"] = [buf(v) for v in st.theta.views]
        out["e_pub"] = [buf(v) for v in st.e.views] if st.e is not None else None
        rd.publish(out["th_pub"], out["e_pub"])
    rd.commit()
    return out


@pytest.mark.parametrize("mode,dtype,ema,swa,norms,wnorms,publish,host", [
    ("mean", "f32", True, False, False, False, False, False),
    ("mean", "bf16", True, True, True, True, True, False),
    ("delta", "bf16", False, False, True, True, False, False),
    ("delta", "f32", True, False, True, False, True, True),   # pinned host workers
    ("mean", "f32", False, True, True, False, False, True),
])
def test_folded_round_equals_accumulated_round_bitwise(mode, dtype, ema, swa, norms, wnorms,
                                                       publish, host):
    wl = dataclasses.replace(
        _custom(STAGED_SIZES, K=4, mode=mode, dtype=dtype, ema=ema, norms=norms, n_masked=1,
                rounds=((0, -1), (1, -1))), swa=swa)
    g = W.make_global(wl, 4, DEV)
    acc, fold = make_gpu_state(wl, g, DEV), make_gpu_state(wl, g, DEV)
    ost = oracle_state_from(g, wl)
    for idx, (rnd, _) in enumerate(wl.rounds):
        draw = W.draw_round(wl, idx, 4)
        workers = [W.make_worker(wl, g, rnd, k, 4, DEV) for k in range(wl.K)]
        if host:
            workers = [W.Arena(w.flat.cpu().pin_memory(), w.offsets, w.numels) for w in workers]
        oa = _fold_round(acc, wl, rnd, workers, draw, norms=norms, wnorms=wnorms, publish=publish)
        of = _fold_round(fold, wl, rnd, workers, draw, norms=norms, wnorms=wnorms, publish=publish,
                         streams=[torch.cuda.current_stream()], pub_host=host)
        oracle_round(ost, wl, rnd, -1, workers, draw)
        torch.cuda.synchronize()
        for name in ("theta", "m", "e", "swa"):
            x, y = getattr(acc, name), getattr(fold, name)
            if x is not None:
                assert torch.equal(x.flat.view(torch.int32), y.flat.view(torch.int32)), \
                    f"round {rnd}: {name} differs between folded and accumulated"
        compare_full(fold, ost, f"folded round {rnd}")
        if publish:
            for t, v in enumerate(fold.theta.views):
                assert torch.equal(of["th_pub"][t].cpu().view(torch.int32), v.cpu().view(torch.int32))
                if fold.e is not None:
                    assert torch.equal(of["e_pub"][t].cpu().view(torch.int32),
                                       fold.e.views[t].cpu().view(torch.int32))
        for key in ("pt", "pf", "pwt", "pw"):
            if key in oa:
                x, y = of[key].cpu().numpy(), oa[key].cpu().numpy()
                assert (x >= 0).all(), f"{key}: norm not written"
                assert np.all(np.abs(x - y) <= NORM_RTOL * np.abs(y) + 1e-300), f"{key}: {x} vs {y}"
    for st in (acc, fold):
        assert st.merger.status() == 0
        st.merger.close()


@pytest.mark.parametrize("mode,dtype,ema,swa,norms,wnorms,publish,host,last", [
    ("mean", "f32", True, False, True, False, True, True, 1),   # the e2e pattern: pinned host in and out
    ("delta", "bf16", True, False, True, True, True, False, 1),
    ("delta", "f32", False, True, False, False, False, True, 2),
    ("mean", "f32", True, False, True, True, False, True, 2),
    ("mean", "bf16", False, True, True, True, False, False, 3),  # every included worker accumulated
])
def test_folded_round_with_its_last_arrivals_accumulated(mode, dtype, ema, swa, norms, wnorms,
                                                         publish, host, last):
    """Folding the first arrivals and accumulating the last ones (folded by the
    commit's final pass) gives the bits of a round whose workers are all
    accumulated, published copies included; each worker's drift equals, bit
    for bit, what a fold of that worker reports."""
    wl = dataclasses.replace(
        _custom(STAGED_SIZES, K=4, mode=mode, dtype=dtype, ema=ema, norms=norms, n_masked=1,
                rounds=((0, -1), (1, -1))), swa=swa)
    g = W.make_global(wl, 14, DEV)
    acc, mixed, folded = (make_gpu_state(wl, g, DEV), make_gpu_state(wl, g, DEV),
                          make_gpu_state(wl, g, DEV))
    ost = oracle_state_from(g, wl)
    for idx, (rnd, _) in enumerate(wl.rounds):
        draw = W.draw_round(wl, idx, 14)
        workers = [W.make_worker(wl, g, rnd, k, 14, DEV) for k in range(wl.K)]
        if host:
            workers = [W.Arena(w.flat.cpu().pin_memory(), w.offsets, w.numels) for w in workers]
        oa = _fold_round(acc, wl, rnd, workers, draw, norms=norms, wnorms=wnorms, publish=publish)
        om = _fold_round(mixed, wl, rnd, workers, draw, norms=norms, wnorms=wnorms, publish=publish,
                         streams=[torch.cuda.current_stream()], pub_host=host, accumulate_last=last)
        of = _fold_round(folded, wl, rnd, workers, draw, norms=norms, wnorms=wnorms, publish=False,
                         streams=[torch.cuda.current_stream()])
        oracle_round(ost, wl, rnd, -1, workers, draw)
        torch.cuda.synchronize()
        for name in ("theta", "m", "e", "swa"):
            x, y = getattr(acc, name), getattr(mixed, name)
            if x is not None:
                assert torch.equal(x.flat.view(torch.int32), y.flat.view(torch.int32)), \
                    f"round {rnd}: {name} differs from the accumulated round"
        compare_full(mixed, ost, f"round {rnd} with its last {last} arrivals accumulated")
        if publish:
            for t, v in enumerate(mixed.theta.views):
                assert torch.equal(om["th_pub"][t].cpu().view(torch.int32), v.cpu().view(torch.int32))
                if mixed.e is not None:
                    assert torch.equal(om["e_pub"][t].cpu().view(torch.int32),
                                       mixed.e.views[t].cpu().view(torch.int32))
        for key in ("pt", "pf", "pwt", "pw"):
            if key in oa:
                x, y = om[key].cpu().numpy(), oa[key].cpu().numpy()
                assert (x >= 0).all(), f"{key}: norm not written"
                assert np.all(np.abs(x - y) <= NORM_RTOL * np.abs(y) + 1e-300), f"{key}: {x} vs {y}"
        if last < len(draw.included):  # at least one fold: the commit takes the final pass
            assert mixed.merger.last_commit()["form"] == B.FORM_FOLDED
            for key in ("pwt", "pw"):   # the same per-worker sums as the folds compute
                if key in of:
                    assert torch.equal(om[key], of[key]), key
    for st in (acc, mixed, folded):
        assert st.merger.status() == 0
        st.merger.close()


def test_folds_on_several_streams_are_ordered():
    wl = _custom([1 << 20, 4097, 33], K=5, mode="delta", dtype="bf16", ema=True)
    g = W.make_global(wl, 6, DEV)
    draw = W.draw_round(wl, 0, 6)
    workers = [W.make_worker(wl, g, 0, k, 6, DEV) for k in range(wl.K)]
    seq, par = make_gpu_state(wl, g, DEV), make_gpu_state(wl, g, DEV)
    streams = [torch.cuda.Stream() for _ in range(3)]
    for s in streams:
        s.wait_stream(torch.cuda.current_stream())
    _fold_round(seq, wl, 0, workers, draw, norms=True, wnorms=False, publish=False,
                streams=[torch.cuda.current_stream()])
    _fold_round(par, wl, 0, workers, draw, norms=True, wnorms=False, publish=False, streams=streams)
    torch.cuda.synchronize()
    for name in ("theta", "m", "e"):
        assert torch.equal(getattr(seq, name).flat.view(torch.int32), getattr(par, name).flat.view(torch.int32))
    seq.merger.close()
    par.merger.close()


@pytest.mark.filterwarnings("ignore:The CUDA Graph is empty")  # the refused capture records nothing
def test_rounds_captured_in_a_cuda_graph_replay_bit_for_bit():
    """The Pythia-14M step (three fragment rounds, Nesterov + drift norms)
    captured once into a CUDA graph and replayed gives, replay after replay,
    the bits of the same rounds committed one by one; the graph reads the
    workers' buffers afresh at every replay."""
    wl = W.workload("pythia14m")
    g = W.make_global(wl, 21, DEV)
    draws = [W.draw_round(wl, i, 21) for i in range(len(wl.rounds))]
    workers = [[W.make_worker(wl, g, rnd, k, 21, DEV) for k in range(wl.K)] for rnd, _ in wl.rounds]
    eager, graphed = make_gpu_state(wl, g, DEV), make_gpu_state(wl, g, DEV)
    norms = {}

    def step(st, rnd0, key):
        for i, ((_, frag), w, d) in enumerate(zip(wl.rounds, workers, draws)):
            rd = st.merger.begin(rnd0 + i, frag)
            for k in d.included:
                rd.accumulate(w[k].views, d.tokens[k])
            rd.finalize(B.DELTA_NESTEROV, wl.lr, wl.mu)
            if (key, i) not in norms:
                norms[key, i] = (torch.zeros(len(rd.tensors), dtype=torch.float64, device=DEV),
                                 torch.zeros(1, dtype=torch.float64, device=DEV))
            rd.drift_norm(*norms[key, i])
            rd.commit()

    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(graph, stream=side):
        step(graphed, 0, "graph")
    torch.cuda.synchronize()
    assert torch.equal(graphed.theta.flat, g.flat)  # capturing ran nothing
    for rep in range(3):
        if rep == 1:  # the replay reads the buffers as they are now
            for w in workers:
                for x in w:
                    x.flat.mul_(1.001)
        step(eager, 100 + 10 * rep, "eager")
        graph.replay()
        torch.cuda.synchronize()
        for name in ("theta", "m"):
            assert torch.equal(getattr(eager, name).flat.view(torch.int32),
                               getattr(graphed, name).flat.view(torch.int32)), (rep, name)
        for i in range(len(wl.rounds)):
            a, b = norms["eager", i], norms["graph", i]
            assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    assert graphed.merger.status() == 0
    # what cannot be replayed faithfully is refused inside a capture
    th = [torch.zeros(4096, device=DEV)]
    sw = [torch.zeros(4096, device=DEV)]
    mg = B.Merger(th, swa=sw, quorum=1)
    x = [torch.ones(4096, device=DEV)]
    g2 = torch.cuda.CUDAGraph()
    with pytest.raises(B.StateError):
        with torch.cuda.graph(g2, stream=side):
            rd = mg.begin(0)
            rd.accumulate(x, 1)
            rd.finalize(B.MEAN_REPLACE)
            rd.swa_update()
            rd.commit()
    rd.abort()
    mg.close()
    eager.merger.close()
    graphed.merger.close()


def test_folded_and_orthogonalised_rounds_captured_in_a_cuda_graph():
    """Once a context has made its running-sum buffer and its Newton-Schulz
    workspace (outside any capture), a folded round (last arrival folded by the
    commit) and an orthogonalised round can be captured and replayed; each
    replay equals the same round committed directly."""
    shapes = [(256, 192), (333, 0), (96, 40)]
    sizes = [r * c if c else r for r, c in shapes]
    rows = [r if c else 0 for r, c in shapes]
    wl = _custom(sizes, K=3, mode="mean", dtype="f32", norms=False)
    g = W.make_global(wl, 16, DEV)
    workers = [W.make_worker(wl, g, 0, k, 16, DEV) for k in range(wl.K)]
    side = torch.cuda.Stream()

    def state():
        th = W.empty_arena(g.numels, torch.float32, DEV)
        th.flat.copy_(g.flat)
        e = W.empty_arena(g.numels, torch.float32, DEV)
        e.flat.copy_(g.flat)
        return th, e, B.Merger(th.views, ema=e.views, quorum=wl.K, rows=rows)

    def folded(mg, rnd, stream=None):
        rd = mg.begin(rnd)
        for k in range(wl.K - 1):
            rd.fold(workers[k].views, 0, B.MEAN_REPLACE, stream=stream)
        rd.accumulate(workers[wl.K - 1].views, 0)
        rd.finalize(B.MEAN_REPLACE)
        rd.ema_update(0.9)
        rd.commit(stream)

    def ortho(mg, rnd, stream=None):
        rd = mg.begin(rnd)
        for k in range(wl.K):
            rd.accumulate(workers[k].views, 0)
        rd.finalize(B.MEAN_REPLACE)
        rd.ema_update(0.9)
        rd.orthogonalize(0.05, B.ORTHO_SCALE_MATCH_NORM, B.ORTHO_FP32, 20)
        rd.commit(stream)

    for body in (folded, ortho):
        th_d, e_d, mg_d = state()
        th_g, e_g, mg_g = state()
        body(mg_g, 0)                  # allocates outside the capture
        body(mg_d, 0)
        side.wait_stream(torch.cuda.current_stream())
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=side):
            body(mg_g, 1, side)
        for rep in range(2):
            body(mg_d, 2 + rep)
            graph.replay()
            torch.cuda.synchronize()
            assert torch.equal(th_d.flat.view(torch.int32), th_g.flat.view(torch.int32)), (body, rep)
            assert torch.equal(e_d.flat.view(torch.int32), e_g.flat.view(torch.int32)), (body, rep)
        mg_d.close()
        mg_g.close()


def test_quorum_lowered_for_the_leftovers():
    """A merger whose fleet shrank lowers the quorum without a new context and
    merges the single remaining worker (plain replacement returns it)."""
    th = [torch.zeros(5000, device=DEV)]
    mg = B.Merger(th, quorum=3)
    x = [torch.randn(5000, device=DEV)]
    rd = mg.begin(0)
    rd.accumulate(x, 1)
    rd.finalize(B.MEAN_REPLACE)
    with pytest.raises(B.QuorumError):
        rd.commit()
    assert mg.quorum == 3
    mg.quorum = 1                       # applies to the open round too
    rd.commit()
    torch.cuda.synchronize()
    assert torch.equal(th[0], x[0])
    for bad in (0, 9):
        with pytest.raises(B.ArgError):
            mg.quorum = bad
    assert mg.quorum == 1
    mg.close()


def test_dropped_and_orphaned_round_handles():
    """A round dropped while open is aborted (its fragment takes a new round);
    closing the merger with a round open invalidates that round's handle, so
    dropping it afterwards touches nothing."""
    import gc
    th = [torch.zeros(4096, device=DEV)]
    mg = B.Merger(th, quorum=1)
    rd = mg.begin(0)
    rd.accumulate([torch.ones(4096, device=DEV)], 0)
    del rd
    gc.collect()
    rd = mg.begin(1)  # no BusyError: the dropped round was aborted
    rd.accumulate([torch.ones(4096, device=DEV)], 0)
    mg.close()
    assert rd.handle is None
    del rd
    gc.collect()
    mg2 = B.Merger(th, quorum=1)
    rd = mg2.begin(0)
    rd.accumulate([torch.full((4096,), 2.0, device=DEV)], 0)
    rd.finalize(B.MEAN_REPLACE)
    rd.commit()
    torch.cuda.synchronize()
    assert torch.equal(th[0], torch.full((4096,), 2.0, device=DEV))
    mg2.close()


def test_rounds_on_shared_tensors_run_in_call_order_across_streams():
    """Rounds that share tensors, each committed on another stream with no
    synchronisation between them, give the bits of the same rounds on one
    stream: the library orders work on shared tensors in call order (a
    whole-list round before a fragment round and back), while the two
    fragments' rounds may overlap."""
    wl = _custom([3 << 20, 1 << 20, 4097], K=4, mode="delta", dtype="bf16", frags=[0, 1, 1],
                 n_fragments=2, rounds=((0, -1), (1, 0), (2, 1), (3, -1), (4, 0)))
    g = W.make_global(wl, 11, DEV)
    draws = [W.draw_round(wl, i, 11) for i in range(len(wl.rounds))]
    workers = [[W.make_worker(wl, g, rnd, k, 11, DEV) for k in range(wl.K)] for rnd, _ in wl.rounds]
    seq, par = make_gpu_state(wl, g, DEV), make_gpu_state(wl, g, DEV)
    cur = torch.cuda.current_stream()
    streams = [torch.cuda.Stream() for _ in range(3)]
    for s in streams:
        s.wait_stream(cur)
    norms_par = []
    for i, ((rnd, frag), w, d) in enumerate(zip(wl.rounds, workers, draws)):
        s = streams[i % len(streams)]
        with torch.cuda.stream(s):
            norms_par.append(gpu_round(par, wl, rnd, frag, w, d, stream=s))
    for s in streams:
        cur.wait_stream(s)
    norms_seq = [gpu_round(seq, wl, rnd, frag, w, d)
                 for (rnd, frag), w, d in zip(wl.rounds, workers, draws)]
    torch.cuda.synchronize()
    for name in ("theta", "m", "e"):
        assert torch.equal(getattr(seq, name).flat.view(torch.int32),
                           getattr(par, name).flat.view(torch.int32)), name
    for a, b in zip(norms_par, norms_seq):
        assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    seq.merger.close()
    par.merger.close()


def test_random_round_sequences_on_random_streams_equal_one_stream():
    """Randomised: twelve rounds over three fragments and the whole list, each
    accumulated, folded, or folded with its last arrival left to the commit,
    each on one of three streams (folds on streams of their own), with no
    synchronisation in between, end with the bits of the same calls issued on
    one stream."""
    rng = np.random.default_rng(77)
    rounds = tuple((i, int(f)) for i, f in enumerate(rng.choice([-1, 0, 1, 2], size=12)))
    wl = _custom([1 << 20, 300_001, 4097, 65_536, 9, 2_000_000], K=4, mode="delta", dtype="bf16",
                 frags=[0, 0, 1, 1, 2, 2], n_fragments=3, rounds=rounds, n_masked=1)
    g = W.make_global(wl, 15, DEV)
    draws = [W.draw_round(wl, i, 15) for i in range(len(rounds))]
    how = rng.choice(["accumulate", "fold", "fold_last"], size=len(rounds))
    which = rng.integers(0, 3, size=(len(rounds), wl.K + 1))
    workers = [[W.make_worker(wl, g, rnd, k, 15, DEV) for k in range(wl.K)] for rnd, _ in rounds]
    code = B.DELTA_NESTEROV

    def run(streams):
        st = make_gpu_state(wl, g, DEV)
        cur = torch.cuda.current_stream()
        for s in streams:
            s.wait_stream(cur)
        outs = []
        for i, ((rnd, frag), d) in enumerate(zip(rounds, draws)):
            cs = streams[which[i, -1] % len(streams)]
            with torch.cuda.stream(cs):
                rd = st.merger.begin(rnd, frag)
                for j, k in enumerate(d.included):
                    fold = how[i] == "fold" or (how[i] == "fold_last" and j < len(d.included) - 1)
                    if fold:
                        rd.fold(workers[i][k].views, d.tokens[k], code,
                                stream=streams[which[i, j] % len(streams)])
                    else:
                        rd.accumulate(workers[i][k].views, d.tokens[k])
                rd.finalize(code, wl.lr, wl.mu)
                rd.ema_update(0.9)
                pt = torch.zeros(len(rd.tensors) or 1, dtype=torch.float64, device=DEV)
                pf = torch.zeros(1, dtype=torch.float64, device=DEV)
                rd.drift_norm(pt, pf)
                rd.commit(cs)
                outs.append((pt, pf))
        for s in streams:
            cur.wait_stream(s)
        torch.cuda.synchronize()
        return st, outs

    par, norms_par = run([torch.cuda.Stream() for _ in range(3)])
    seq, norms_seq = run([torch.cuda.current_stream()])
    for name in ("theta", "m", "e"):
        assert torch.equal(getattr(seq, name).flat.view(torch.int32),
                           getattr(par, name).flat.view(torch.int32)), name
    for a, b in zip(norms_par, norms_seq):
        assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    for st in (par, seq):
        assert st.merger.status() == 0
        st.merger.close()


def test_orthogonalised_rounds_on_two_streams_take_the_workspace_in_turn():
    """Orthogonalised rounds on disjoint fragments, committed on two streams
    at once, share the context's Newton-Schulz workspace one after the other
    and give the bits of the same rounds on one stream."""
    shapes = [(256, 192), (96, 40), (333, 0), (256, 192), (40, 96)]
    sizes = [r * c if c else r for r, c in shapes]
    rows = [r if c else 0 for r, c in shapes]
    wl = _custom(sizes, K=3, mode="mean", dtype="f32", frags=[0, 0, 0, 1, 1], n_fragments=2,
                 rounds=((0, 0), (1, 1)), norms=False)
    g = W.make_global(wl, 12, DEV)
    workers = [[W.make_worker(wl, g, rnd, k, 12, DEV) for k in range(wl.K)] for rnd, _ in wl.rounds]

    def run(streams):
        th = W.empty_arena(g.numels, torch.float32, DEV)
        th.flat.copy_(g.flat)
        e = W.empty_arena(g.numels, torch.float32, DEV)
        e.flat.copy_(g.flat)
        mg = B.Merger(th.views, ema=e.views, fragment_of=wl.fragment_of, n_fragments=2,
                      quorum=wl.K, rows=rows)
        cur = torch.cuda.current_stream()
        for s in streams:
            s.wait_stream(cur)
        for i, (rnd, frag) in enumerate(wl.rounds):
            s = streams[i % len(streams)]
            with torch.cuda.stream(s):
                rd = mg.begin(rnd, frag)
                for k in range(wl.K):
                    rd.accumulate(workers[i][k].views, 0)
                rd.finalize(B.MEAN_REPLACE)
                rd.ema_update(0.9)
                rd.orthogonalize(0.05, B.ORTHO_SCALE_MATCH_NORM, B.ORTHO_FP32, 30)
                rd.commit(s)
        for s in streams:
            cur.wait_stream(s)
        torch.cuda.synchronize()
        mg.close()
        return th, e

    th_par, e_par = run([torch.cuda.Stream(), torch.cuda.Stream()])
    th_seq, e_seq = run([torch.cuda.current_stream()])
    assert torch.equal(th_par.flat.view(torch.int32), th_seq.flat.view(torch.int32))
    assert torch.equal(e_par.flat.view(torch.int32), e_seq.flat.view(torch.int32))
    assert not torch.equal(th_seq.flat, g.flat)  # the rounds did move theta


def test_worker_buffers_are_free_once_their_fold_has_run():
    wl = _custom([100_003, 2048], K=3, mode="mean", dtype="f32", ema=True, norms=False)
    g = W.make_global(wl, 8, DEV)
    draw = W.draw_round(wl, 0, 8)
    workers = [W.make_worker(wl, g, 0, k, 8, DEV) for k in range(wl.K)]
    want = oracle_state_from(g, wl)
    oracle_round(want, wl, 0, -1, workers, draw)
    st = make_gpu_state(wl, g, DEV)
    rd = st.merger.begin(0)
    for k in draw.included:
        rd.fold(workers[k].views, 0, B.MEAN_REPLACE)
        torch.cuda.synchronize()
        workers[k].flat.fill_(float("nan"))  # the fold has read it: the buffer may be reused
    rd.finalize(B.MEAN_REPLACE)
    rd.ema_update(0.9)
    rd.commit()
    compare_full(st, want, "folded round with reused worker buffers", bitwise=True)
    st.merger.close()


def test_fold_rules():
    th = [torch.zeros(4096, device=DEV)]
    m = [torch.zeros(4096, device=DEV)]
    mg = B.Merger(th, momentum=m, quorum=1)
    x = [torch.ones(4096, device=DEV)]
    rd = mg.begin(0)
    rd.accumulate(x, 1)
    with pytest.raises(B.StateError):          # accumulated, then folded
        rd.fold(x, 1, B.MEAN_REPLACE)
    rd.abort()
    rd = mg.begin(1)
    rd.fold(x, 1, B.DELTA_NESTEROV)
    with pytest.raises(B.ArgError):            # another mode than the earlier folds
        rd.fold(x, 1, B.MEAN_REPLACE)
    with pytest.raises(B.StateError):          # per-worker drift after the first fold
        rd.worker_drift_norm(torch.zeros(1, dtype=torch.float64, device=DEV), None)
    with pytest.raises(B.StateError):          # orthogonalisation needs the workers at commit
        rd.orthogonalize(0.1)
    rd.accumulate(x, 1)                        # folded, then accumulated: the commit folds it
    with pytest.raises(B.StateError):          # a fold after an accumulated worker
        rd.fold(x, 1, B.DELTA_NESTEROV)
    with pytest.raises(B.StateError):          # finalize with another mode
        rd.finalize(B.MEAN_REPLACE)
    rd.finalize(B.DELTA_NESTEROV, 0.7, 0.9)
    with pytest.raises(B.StateError):          # fold after finalize
        rd.fold(x, 1, B.DELTA_NESTEROV)
    rd.commit()
    torch.cuda.synchronize()
    # two workers at 1 from theta 0, equal weights: Delta 1, m' = -1, step -1.9, theta' = 1.33
    want = np.float32(0) - np.float32(0.7) * (np.float32(-1) + np.float32(0.9) * np.float32(-1))
    assert torch.equal(th[0], torch.full((4096,), float(want), device=DEV))
    rd = mg.begin(2)
    pw = torch.full((2,), -1.0, dtype=torch.float64, device=DEV)
    rd.worker_drift_norm(None, pw)
    rd.fold(x, 1, B.DELTA_NESTEROV)
    rd.accumulate(x, 1)                        # its drift comes from the commit's final pass
    rd.finalize(B.DELTA_NESTEROV, 0.7, 0.9)
    rd.commit()
    torch.cuda.synchronize()
    d = abs(1.0 - float(want))                 # both workers sit at 1, theta was at `want`
    assert torch.equal(pw[0], pw[1])
    assert abs(pw[0].item() - 64.0 * d) <= 1e-6 * 64.0 * d
    assert mg.status() == 0
    mg.close()


def test_abort_after_folds_then_a_fresh_round():
    wl = _custom([50_000, 7], K=3, mode="mean", dtype="bf16", ema=False, norms=True)
    g = W.make_global(wl, 12, DEV)
    st = make_gpu_state(wl, g, DEV)
    junk = [W.make_worker(wl, g, 9, k, 99, DEV) for k in range(2)]
    rd = st.merger.begin(0)
    for w in junk:
        rd.fold(w.views, 0, B.MEAN_REPLACE)
    rd.abort()
    draw = W.draw_round(wl, 0, 12)
    workers = [W.make_worker(wl, g, 1, k, 12, DEV) for k in range(wl.K)]
    want = oracle_state_from(g, wl)
    oracle_round(want, wl, 1, -1, workers, draw)
    _fold_round(st, wl, 1, workers, draw, norms=False, wnorms=False, publish=False,
                streams=[torch.cuda.current_stream()])
    compare_full(st, want, "fresh folded round after an abort", bitwise=True)
    st.merger.close()


def test_commit_record():
    sizes = [70_001, 2048, 5]
    n = sum(sizes)
    th = [torch.randn(k, device=DEV) * 0.02 for k in sizes]
    m = [torch.zeros(k, device=DEV) for k in sizes]
    e = [t.clone() for t in th]
    sw = [torch.zeros(k, device=DEV) for k in sizes]
    mg = B.Merger(th, momentum=m, ema=e, swa=sw, quorum=1, time_commits=True)
    xs = [[(t + 1e-3 * torch.randn_like(t)).to(torch.bfloat16) for t in th] for _ in range(3)]

    rd = mg.begin(0)                    # Nesterov + norms, a small round: the register pass
    for x in xs:                        # finishes the norms itself, one launch
        rd.accumulate(x, 1000)
    rd.finalize(B.DELTA_NESTEROV, 0.7, 0.9)
    rd.drift_norm(torch.zeros(3, dtype=torch.float64, device=DEV), None)
    rd.commit()
    rec = mg.last_commit()
    assert (rec["round"], rec["fragment"], rec["K"], rec["mode"]) == (0, -1, 3, B.DELTA_NESTEROV)
    assert rec["form"] == B.FORM_REGISTER and rec["elements"] == n
    assert rec["bytes"] == (3 * 2 + 4 + 4 + 8) * n and rec["launches"] == 1 and rec["ms"] > 0

    rd = mg.begin(1)                    # the same, folded
    for x in xs:
        rd.fold(x, 1000, B.DELTA_NESTEROV)
    rd.finalize(B.DELTA_NESTEROV, 0.7, 0.9)
    rd.commit()
    rec = mg.last_commit()
    assert rec["form"] == B.FORM_FOLDED and rec["bytes"] == (4 + 4 + 4 + 8) * n
    assert rec["launches"] == 1 and rec["ms"] > 0

    rd = mg.begin(2)                    # mean + EMA + running average: three arrays written
    for x in xs:
        rd.accumulate(x)
    rd.finalize(B.MEAN_REPLACE)
    rd.ema_update(0.9)
    rd.swa_update()
    rd.commit()
    rec = mg.last_commit()
    assert rec["form"] == B.FORM_REGISTER and rec["bytes"] == (3 * 2 + 4 + 8 + 8) * n

    rd = mg.begin(3)                    # Nesterov, no norms: theta, m written -> staged
    for x in xs:
        rd.accumulate(x, 1000)
    rd.finalize(B.DELTA_NESTEROV, 0.7, 0.9)
    rd.commit()
    rec = mg.last_commit()
    assert rec["form"] == B.FORM_STAGED and rec["bytes"] == (3 * 2 + 4 + 4 + 8) * n
    assert rec["launches"] == 1 and rec["ms"] > 0
    assert mg.status() == 0
    mg.close()
