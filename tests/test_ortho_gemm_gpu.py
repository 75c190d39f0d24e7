"""GPU: the Newton-Schulz GEMMs of the outer orthogonalisation ("DiffuRefill-1B"
technical report, section 5.3), one step at a time, through the C ABI.

With `iterations = 1` an orthogonalised round applies
theta' = theta + lr X1 with X1 = 1.5 X0 - 0.5 (X0 X0^T) X0 (Gram matrix on the
short side) and X0 = Delta / |Delta|_F; the library forms it as X1 = H X0 (wide
orientation) with H = 1.5 I - 0.5 X0 X0^T, or, with TF32 inputs, as
1.5 X0 - 0.5 G X0 with X0 read in fp32. The reference here restates that one
step in fp64 from the round's Delta (the oracle's plain mean minus theta) and
reproduces the roundings the library's storage makes: X0 rounded once to the
iterate's type, H (or G) stored in it. What remains between the two is fp32
accumulation against fp64, TF32 inputs, and the final rounding of X1, so the
bound is a few units of the storage type's rounding, far below what a wrong
index, a dropped term or a transposed operand would leave.

The shapes cover every path of the GEMM kernels: tiles 128 and 256 wide, more
than one tile each way, sides that are not multiples of 128 (zero padding),
tall and wide matrices, batches of equal shapes, and a Gram matrix whose long
side is split over several K ranges (fp32 partials summed by a second kernel).
"""
import gc

import numpy as np
import pytest
import torch

import oracle
from checkpoint_averaging_gb300 import binding as B
from checkpoint_averaging_gb300 import workloads as W

pytestmark = pytest.mark.gpu

DEV = "cuda"

# Bound on |X1_gpu - X1_ref| relative to max |X1|, in units of the storage
# type's unit roundoff (bf16 2^-8, tf32 inputs 2^-11, fp32 2^-24 with a floor
# for fp32 accumulation over long sides).
STEP_TOL = {B.ORTHO_BF16: 3 * 2.0 ** -8, B.ORTHO_TF32: 4 * 2.0 ** -11, B.ORTHO_FP32: 2e-6}

# (rows, cols): wide 300 x 700 (padded 384 x 768, 128-wide tiles), tall
# 1100 x 256 (256-wide tiles), a long wide matrix whose Gram product is split,
# a batch of three equal shapes, a square, a small odd one.
STEP_SHAPES = [(300, 700), (1100, 256), (256, 8192), (200, 520), (520, 200), (200, 520),
               (200, 520), (128, 128), (33, 5)]


@pytest.fixture(autouse=True)
def _cuda_cleanup():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    yield
    gc.collect()
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def _to_bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16).float().numpy()


def newton_schulz_step(delta, precision):
    """One Newton-Schulz step from Delta, in fp64, with the library's storage
    roundings: X0 = fp32(Delta * fp32(1/|Delta|_F)), rounded to bf16 for a bf16
    iterate; H = 1.5 I - 0.5 W W^T rounded to the iterate's type."""
    m, n = delta.shape
    d64 = delta.astype(np.float64)
    inv = np.float32(1.0 / np.sqrt(np.sum(d64 * d64)))
    x0 = (delta * inv).astype(np.float32)
    if precision == B.ORTHO_BF16:
        x0 = _to_bf16(x0)
    w = x0.T.astype(np.float64) if m >= n else x0.astype(np.float64)  # r x L
    if precision == B.ORTHO_TF32:  # X1 = 1.5 X0 - 0.5 G X0, X0 exact in the epilogue
        g = (w @ w.T).astype(np.float32).astype(np.float64)
        x1 = 1.5 * w - 0.5 * (g @ w)
    else:                          # X1 = H X0, H stored in the iterate's type
        h = (1.5 * np.eye(w.shape[0]) - 0.5 * (w @ w.T)).astype(np.float32)
        if precision == B.ORTHO_BF16:
            h = _to_bf16(h)
        x1 = h.astype(np.float64) @ w
    return x1.T if m >= n else x1


def _one_step_round(shapes, precision, iterations=1, seed=41, K=2):
    sizes = [r * c for r, c in shapes]
    specs = tuple(W.TensorSpec(f"t{i}", (n,), 0) for i, n in enumerate(sizes))
    wl = W.Workload("ns_step", specs, 1, K=K, n_masked=0, quorum=K, ckpt_dtype="f32",
                    mode="mean", ema_beta=0.9, rounds=((0, -1),))
    g = W.make_global(wl, seed, DEV)
    th = W.empty_arena(g.numels, torch.float32, DEV)
    th.flat.copy_(g.flat)
    e = W.empty_arena(g.numels, torch.float32, DEV)
    e.flat.copy_(g.flat)
    mg = B.Merger(th.views, ema=e.views, quorum=K, rows=[r for r, _ in shapes])
    workers = [W.make_worker(wl, g, 0, k, seed, DEV) for k in range(K)]
    rd = mg.begin(0)
    for k in range(K):
        rd.accumulate(workers[k].views, 0)
    rd.finalize(B.MEAN_REPLACE)
    rd.ema_update(0.9)
    rd.orthogonalize(1.0, B.ORTHO_SCALE_FIXED, precision, iterations)
    rd.commit()
    torch.cuda.synchronize()
    out = []
    for t, (r, c) in enumerate(shapes):
        xs = [w.views[t].cpu().numpy() for w in workers]
        th0 = g.views[t].cpu().numpy().copy()
        delta = (oracle.plain_mean(xs) - th0).reshape(r, c)
        step = th.views[t].cpu().numpy().astype(np.float64) - th0.astype(np.float64)
        out.append((r, c, delta, step.reshape(r, c)))
    assert mg.status() == 0
    mg.close()
    return out


@pytest.mark.parametrize("precision", [B.ORTHO_BF16, B.ORTHO_TF32, B.ORTHO_FP32])
def test_one_newton_schulz_step(precision):
    for r, c, delta, got in _one_step_round(STEP_SHAPES, precision):
        want = newton_schulz_step(delta, precision)
        scale = np.abs(want).max()
        err = np.abs(got - want).max()
        print(f"one step precision={precision} {r}x{c}: max err / max |X1| = {err / scale:.3e}")
        assert err <= STEP_TOL[precision] * scale, (r, c)


@pytest.mark.parametrize("precision", [B.ORTHO_TF32, B.ORTHO_FP32])
def test_one_short_side_step(precision):
    """In the short-side form one step is P1 = 1.5 I - 0.5 G0 and X1 = P1 X0:
    the same matrix as the plain step, through different products."""
    shapes = [(1100, 256), (256, 8192), (520, 100), (64, 300)]
    for r, c, delta, got in _one_step_round(shapes, precision | B.ORTHO_SHORT_SIDE):
        want = newton_schulz_step(delta, B.ORTHO_FP32)
        scale = np.abs(want).max()
        err = np.abs(got - want).max()
        print(f"short-side step precision={precision} {r}x{c}: max err / max |X1| = {err / scale:.3e}")
        assert err <= STEP_TOL[precision] * scale, (r, c)


# The polar factor after 40 steps, relative to the largest element of the step
# (the bounds the other orthogonalisation tests use: 8 units of the storage's
# rounding).
POLAR_TOL = {B.ORTHO_BF16: 8 * 2.0 ** -8, B.ORTHO_TF32: 8 * 2.0 ** -11}


@pytest.mark.parametrize("precision", [B.ORTHO_BF16, B.ORTHO_TF32])
def test_polar_factor_on_full_operand_boxes(precision):
    """After one step the Gram product's share of the step is small (X0 has
    unit Frobenius norm, so its singular values are about 1/sqrt(r)); after 40
    it decides the result. These shapes fill every 128-byte operand box along
    the short side (r = 256, 384, 512: no zero padding there), tall and wide,
    with 256- and 128-wide tiles, so a wrong operand layout in any box shows
    here against the oracle's polar factor (fp64 SVD)."""
    shapes = [(640, 256), (256, 1000), (384, 1152), (1536, 512)]
    sizes = [r * c for r, c in shapes]
    specs = tuple(W.TensorSpec(f"t{i}", (n,), 0) for i, n in enumerate(sizes))
    wl = W.Workload("ns_polar", specs, 1, K=2, n_masked=0, quorum=2, ckpt_dtype="f32",
                    mode="mean", ema_beta=0.9, rounds=((0, -1),))
    g = W.make_global(wl, 47, DEV)
    th = W.empty_arena(g.numels, torch.float32, DEV)
    th.flat.copy_(g.flat)
    e = W.empty_arena(g.numels, torch.float32, DEV)
    e.flat.copy_(g.flat)
    mg = B.Merger(th.views, ema=e.views, quorum=2, rows=[r for r, _ in shapes])
    workers = [W.make_worker(wl, g, 0, k, 47, DEV) for k in range(2)]
    rd = mg.begin(0)
    for k in range(2):
        rd.accumulate(workers[k].views, 0)
    rd.finalize(B.MEAN_REPLACE)
    rd.ema_update(0.9)
    rd.orthogonalize(0.7, B.ORTHO_SCALE_MATCH_NORM, precision, 40)
    rd.commit()
    torch.cuda.synchronize()
    for t, (r, c) in enumerate(shapes):
        xs = [w.views[t].cpu().numpy() for w in workers]
        th0 = g.views[t].cpu().numpy().copy()
        want, _ = oracle.orthogonal_update(xs, th0, r, lr=0.7, scale_mode=oracle.ORTHO_SCALE_MATCH_NORM)
        got = th.views[t].cpu().numpy().astype(np.float64)
        scale = np.abs(want - th0.astype(np.float64)).max()
        err = np.abs(got - want).max()
        print(f"polar precision={precision} {r}x{c}: max err / max step = {err / scale:.3e}")
        assert err <= POLAR_TOL[precision] * scale + 2 * np.spacing(np.float32(np.abs(want).max())), (r, c)
    assert mg.status() == 0
    mg.close()


@pytest.mark.parametrize("precision", [B.ORTHO_BF16, B.ORTHO_TF32])
def test_polar_factor_of_a_tied_embedding(precision):
    """The width-512 stand's tied embedding (73,760 x 512) with a q/k/v/o-sized
    matrix beside it, 30 steps, against the oracle's polar factor: the Gram
    product of the long matrix is split over many K ranges (fp32 partials
    summed by the reduce kernel) and shares its launches with the small one."""
    shapes = [(73760, 512), (512, 512)]
    sizes = [r * c for r, c in shapes]
    specs = tuple(W.TensorSpec(f"t{i}", (n,), 0) for i, n in enumerate(sizes))
    wl = W.Workload("ns_embed", specs, 1, K=2, n_masked=0, quorum=2, ckpt_dtype="f32",
                    mode="mean", ema_beta=0.9, rounds=((0, -1),))
    g = W.make_global(wl, 53, DEV)
    th = W.empty_arena(g.numels, torch.float32, DEV)
    th.flat.copy_(g.flat)
    e = W.empty_arena(g.numels, torch.float32, DEV)
    e.flat.copy_(g.flat)
    mg = B.Merger(th.views, ema=e.views, quorum=2, rows=[r for r, _ in shapes])
    workers = [W.make_worker(wl, g, 0, k, 53, DEV) for k in range(2)]
    rd = mg.begin(0)
    for k in range(2):
        rd.accumulate(workers[k].views, 0)
    rd.finalize(B.MEAN_REPLACE)
    rd.ema_update(0.9)
    rd.orthogonalize(0.7, B.ORTHO_SCALE_MATCH_NORM, precision, 30)
    rd.commit()
    torch.cuda.synchronize()
    for t, (r, c) in enumerate(shapes):
        xs = [w.views[t].cpu().numpy() for w in workers]
        th0 = g.views[t].cpu().numpy().copy()
        want, _ = oracle.orthogonal_update(xs, th0, r, lr=0.7, scale_mode=oracle.ORTHO_SCALE_MATCH_NORM)
        got = th.views[t].cpu().numpy().astype(np.float64)
        scale = np.abs(want - th0.astype(np.float64)).max()
        err = np.abs(got - want).max()
        print(f"embedding polar precision={precision} {r}x{c}: max err / max step = {err / scale:.3e}")
        assert err <= POLAR_TOL[precision] * scale + 2 * np.spacing(np.float32(np.abs(want).max())), (r, c)
    assert mg.status() == 0
    mg.close()


@pytest.mark.parametrize("precision", [B.ORTHO_BF16, B.ORTHO_TF32])
def test_orthogonalised_rounds_repeat_bit_for_bit(precision):
    """The GEMMs sum in a fixed order (no atomics; split partials summed in
    range order), so the same round gives the same bits."""
    shapes = [(256, 8192), (300, 700)]
    a = _one_step_round(shapes, precision, iterations=3, seed=43)
    b = _one_step_round(shapes, precision, iterations=3, seed=43)
    for (_, _, _, x), (_, _, _, y) in zip(a, b):
        assert np.array_equal(x, y)
