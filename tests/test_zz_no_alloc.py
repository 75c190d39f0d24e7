"""The no-allocation entry point, cam_merge_round_noalloc, against the context path.

Some callers cannot allocate device memory. Examples are code embedded in a
framework whose pool has already reserved the GPU's memory, and merges issued
where the device-wide synchronisation of cudaMalloc/cudaFree would stall other
work. For them the library offers one call that runs a whole round on
caller-owned buffers, with its scratch in a fixed array inside the library.
These tests call it through the C ABI twice in a row and compare every output
with the existing context entry points on identical inputs, and with the CPU
oracle, within the tolerance of the other parity tests. Rounds beyond its
fixed scratch are refused on the host before any CUDA call (tested without a
GPU in test_abi_host.py). The file is named so that pytest collects it last.
"""
import numpy as np
import pytest
import torch

import oracle
from checkpoint_averaging_gb300 import binding as B
from checkpoint_averaging_gb300 import workloads as W

from merge_harness import NORM_RTOL, assert_close, to_np

pytestmark = pytest.mark.gpu

DEV = "cuda"
SIZES = [50_000, 1, 7, 0, 2049, 16_385, 100_003, 33]


@pytest.fixture(autouse=True)
def _needs_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    yield
    torch.cuda.synchronize()


def _state(wl, g):
    th = W.empty_arena(g.numels, torch.float32, DEV)
    th.flat.copy_(g.flat)
    m = W.empty_arena(g.numels, torch.float32, DEV)
    e = W.empty_arena(g.numels, torch.float32, DEV)
    e.flat.copy_(g.flat)
    return th, m, e


@pytest.mark.parametrize("dtype,mode", [("bf16", "delta"), ("f32", "mean")])
def test_two_calls_in_a_row_match_the_context_path(dtype, mode):
    specs = tuple(W.TensorSpec(f"t{i}", (n,), 0) for i, n in enumerate(SIZES))
    wl = W.Workload("noalloc", specs, 1, K=4, n_masked=1, quorum=3, ckpt_dtype=dtype, mode=mode,
                    lr=0.7 if mode == "delta" else 1.0, mu=0.9 if mode == "delta" else 0.0,
                    ema_beta=0.9, rounds=((0, -1), (1, -1)), tokens=(100_000, 150_000))
    g = W.make_global(wl, 0, DEV)
    ref_th, ref_m, ref_e = _state(wl, g)   # existing entry points (context path)
    na_th, na_m, na_e = _state(wl, g)      # no-allocation entry point
    mg = B.Merger(ref_th.views, momentum=ref_m.views, ema=ref_e.views, quorum=3)
    code = B.DELTA_NESTEROV if mode == "delta" else B.MEAN_REPLACE
    dt = B.BF16 if dtype == "bf16" else B.F32
    T = len(SIZES)
    for idx, (rnd, _) in enumerate(wl.rounds):
        draw = W.draw_round(wl, idx, 0)
        workers = [W.make_worker(wl, g, rnd, k, 0, DEV) for k in range(wl.K)]
        ref_pt = torch.full((T,), -1.0, dtype=torch.float64, device=DEV)
        ref_pf = torch.full((1,), -1.0, dtype=torch.float64, device=DEV)
        rd = mg.begin(rnd)
        for k in draw.included:
            rd.accumulate(workers[k].views, draw.tokens[k])
        rd.finalize(code, wl.lr, wl.mu)
        rd.ema_update(0.9)
        rd.drift_norm(ref_pt, ref_pf)
        rd.commit()

        na_pt = torch.full((T,), -1.0, dtype=torch.float64, device=DEV)
        na_pf = torch.full((1,), -1.0, dtype=torch.float64, device=DEV)
        B.merge_round_noalloc(
            [t.numel() for t in na_th.views], [t.data_ptr() for t in na_th.views],
            [[t.data_ptr() for t in workers[k].views] for k in draw.included], dt, code,
            tokens=[draw.tokens[k] for k in draw.included], lr=wl.lr, mu=wl.mu,
            momentum=[t.data_ptr() for t in na_m.views], ema=[t.data_ptr() for t in na_e.views],
            beta=0.9, per_tensor=na_pt.data_ptr(), per_round=na_pf.data_ptr(),
            stream=torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize()
        for t in range(T):
            assert_close(to_np(na_th.views[t]), to_np(ref_th.views[t]), f"call {idx}: theta[{t}]")
            assert_close(to_np(na_e.views[t]), to_np(ref_e.views[t]), f"call {idx}: e[{t}]")
            if mode == "delta":
                assert_close(to_np(na_m.views[t]), to_np(ref_m.views[t]), f"call {idx}: m[{t}]")
        got, want = na_pt.cpu().numpy(), ref_pt.cpu().numpy()
        assert np.all(np.abs(got - want) <= NORM_RTOL * np.abs(want)), (got, want)
        assert abs(na_pf.item() - ref_pf.item()) <= NORM_RTOL * abs(ref_pf.item())
    mg.close()


def test_second_call_takes_no_device_memory():
    n = 1 << 20
    th = torch.zeros(n, device=DEV)
    xs = [torch.randn(n, device=DEV) for _ in range(2)]
    pf = torch.zeros(1, dtype=torch.float64, device=DEV)

    def call():
        B.merge_round_noalloc([n], [th.data_ptr()], [[x.data_ptr()] for x in xs], B.F32,
                              B.MEAN_REPLACE, per_round=pf.data_ptr(),
                              stream=torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize()

    call()  # the first call on the device looks up the scratch address
    free_before, _ = torch.cuda.mem_get_info()
    reserved_before = torch.cuda.memory_reserved()
    call()
    free_after, _ = torch.cuda.mem_get_info()
    assert free_after == free_before
    assert torch.cuda.memory_reserved() == reserved_before
    assert torch.allclose(th, (xs[0] + xs[1]) / 2)


def _np_worker(t):
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


@pytest.mark.parametrize("dtype,mode", [("bf16", "delta"), ("f32", "mean")])
def test_more_tensors_than_one_launch_match_the_oracle(dtype, mode):
    """300 ragged tensors, some empty: more than one launch's worth (256), so
    the call runs two launches whose drift partials sit at different offsets of
    the fixed scratch. Two calls in a row, each checked element by element
    against the CPU oracle and against the context path, drift norms against
    the oracle's fp64 sums."""
    rng = np.random.default_rng(5)
    sizes = [int(v) for v in rng.integers(1, 40_000, 300)]
    for i in range(0, 300, 23):
        sizes[i] = 0
    for i in range(5, 300, 31):
        sizes[i] = int(rng.integers(1, 9))
    specs = tuple(W.TensorSpec(f"t{i}", (n,), 0) for i, n in enumerate(sizes))
    wl = W.Workload("noalloc300", specs, 1, K=3, n_masked=0, quorum=3, ckpt_dtype=dtype,
                    mode=mode, lr=0.7 if mode == "delta" else 1.0,
                    mu=0.9 if mode == "delta" else 0.0, ema_beta=0.9,
                    rounds=((0, -1), (1, -1)), tokens=(100_000, 150_000))
    g = W.make_global(wl, 1, DEV)
    ref_th, ref_m, ref_e = _state(wl, g)
    na_th, na_m, na_e = _state(wl, g)
    o_th = [to_np(v).copy() for v in g.views]
    o_m = [np.zeros(n, np.float32) for n in sizes]
    o_e = [to_np(v).copy() for v in g.views]
    mg = B.Merger(ref_th.views, momentum=ref_m.views, ema=ref_e.views, quorum=3)
    code = B.DELTA_NESTEROV if mode == "delta" else B.MEAN_REPLACE
    ocode = oracle.DELTA_NESTEROV if mode == "delta" else oracle.MEAN_REPLACE
    dt = B.BF16 if dtype == "bf16" else B.F32
    T = len(sizes)
    for idx, (rnd, _) in enumerate(wl.rounds):
        draw = W.draw_round(wl, idx, 1)
        workers = [W.make_worker(wl, g, rnd, k, 1, DEV) for k in range(wl.K)]
        tokens = [draw.tokens[k] for k in draw.included] if mode == "delta" else None
        ref_pt = torch.full((T,), -1.0, dtype=torch.float64, device=DEV)
        rd = mg.begin(rnd)
        for k in draw.included:
            rd.accumulate(workers[k].views, draw.tokens[k])
        rd.finalize(code, wl.lr, wl.mu)
        rd.ema_update(0.9)
        rd.drift_norm(ref_pt, None)
        rd.commit()
        na_pt = torch.full((T,), -1.0, dtype=torch.float64, device=DEV)
        na_pf = torch.full((1,), -1.0, dtype=torch.float64, device=DEV)
        B.merge_round_noalloc(
            sizes, [t.data_ptr() for t in na_th.views],
            [[t.data_ptr() for t in workers[k].views] for k in draw.included], dt, code,
            tokens=[draw.tokens[k] for k in draw.included], lr=wl.lr, mu=wl.mu,
            momentum=[t.data_ptr() for t in na_m.views], ema=[t.data_ptr() for t in na_e.views],
            beta=0.9, per_tensor=na_pt.data_ptr(), per_round=na_pf.data_ptr(),
            stream=torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize()
        sumsq = []
        for t in range(T):
            xs = [_np_worker(workers[k].views[t]) for k in draw.included]
            sumsq.append(oracle.merge_tensor(xs, o_th[t], mode=ocode, tokens=tokens, lr=wl.lr,
                                             mu=wl.mu, m=o_m[t] if mode == "delta" else None,
                                             e=o_e[t], beta=0.9))
            where = f"call {idx}: tensor {t} ({sizes[t]} elements)"
            assert_close(to_np(na_th.views[t]), o_th[t], "theta " + where)
            assert_close(to_np(na_e.views[t]), o_e[t], "e " + where)
            assert_close(to_np(na_th.views[t]), to_np(ref_th.views[t]), "theta vs context " + where)
            if mode == "delta":
                assert_close(to_np(na_m.views[t]), o_m[t], "m " + where)
        want = np.sqrt(np.array(sumsq))
        got = na_pt.cpu().numpy()
        assert np.all(np.abs(got - want) <= NORM_RTOL * want), (got, want)
        ref = ref_pt.cpu().numpy()
        assert np.all(np.abs(got - ref) <= NORM_RTOL * ref), (got, ref)
        whole = np.sqrt(np.sum(sumsq))
        assert abs(na_pf.item() - whole) <= NORM_RTOL * whole
    mg.close()
