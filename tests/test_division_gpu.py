"""The merge's one division -- s / K in plain-mean mode, s / W (the token
total) in delta mode -- is the correctly rounded binary32 quotient, the value
IEEE division gives.

The passes form it from the round's correctly rounded reciprocal with two
corrections (Markstein's) wherever that is exact, and take the division
instruction sequence for the other dividends: zeros' signs, subnormals, the
ends of the exponent range, infinities and NaN, and divisors outside the
range the corrections cover. A wrong range or a wrong correction shows as a
quotient one unit off, or a wrong zero sign, for some dividends, so these
tests take, against numpy's binary32 division:

- every binary32 dividend (all 2^32 bit patterns) for one divisor of each
  mode: K = 3, and W = 2^24 - 1, whose significand is all ones;
- for more divisors and through every merge path (staged and register forms,
  the eagerly folded round's final pass, the no-allocation entry point, the
  multi-round pass), random dividends of every exponent plus every power of
  two with its neighbours, zeros, subnormals, infinities and NaN.

The rounds are set up so that the stored result is the quotient itself:
plain mean over K workers of which one carries the dividends and the others
zeros (theta' = (x + 0 + ... + 0) / K); delta mode with two workers, the
dividends at token count 1 and zeros at token count W - 1, theta = 0, m = 0,
lr = 1, mu = 0, so theta' = -(g + 0 * m'), g = -(x / W), m' = 0 * 0 + g. The
expected values run those binary32 operations in numpy.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

from checkpoint_averaging_gb300 import binding as B

pytestmark = pytest.mark.gpu
DEV = "cuda"
F32 = np.float32


def _expected(x: np.ndarray, mode: str, d: int):
    """theta' (and m' in delta mode) of the rounds above, in numpy binary32."""
    with np.errstate(all="ignore"):
        zero = F32(0.0)
        if mode == "mean":
            s = zero + x
            for _ in range(d - 1):
                s = s + zero
            return s / F32(d), None
        s = zero + F32(1.0) * (x - zero)
        s = s + F32(d - 1) * (zero - zero)
        q = s / F32(d)
        g = -q
        m_new = zero * zero + g
        step = g + zero * m_new
        return zero - F32(1.0) * step, m_new


def _same(got: np.ndarray, want: np.ndarray) -> np.ndarray:
    """Elements whose bits agree, or that are NaN on both sides."""
    return (got.view(np.uint32) == want.view(np.uint32)) | (np.isnan(got) & np.isnan(want))


def _check(got: np.ndarray, x: np.ndarray, mode: str, d: int, what: str, m_got=None) -> None:
    want, m_want = _expected(x, mode, d)
    ok = _same(got, want)
    if m_got is not None:
        ok &= _same(m_got, m_want)
    if not ok.all():
        i = int(np.flatnonzero(~ok)[0])
        raise AssertionError(
            f"{what}: {int((~ok).sum())} of {ok.size} quotients differ; first: dividend "
            f"{x[i]!r} (0x{int(x.view(np.uint32)[i]):08x}) / {d}: got {got[i]!r} "
            f"(0x{int(got.view(np.uint32)[i]):08x}), want {want[i]!r} "
            f"(0x{int(want.view(np.uint32)[i]):08x})")


def _workers(x: torch.Tensor, zeros: torch.Tensor, mode: str, d: int):
    """(tensor, tokens) per worker in arrival order."""
    if mode == "mean":
        return [(x, 0)] + [(zeros, 0)] * (d - 1)
    return [(x, 1), (zeros, d - 1)]


def _code(mode: str) -> int:
    return B.MEAN_REPLACE if mode == "mean" else B.DELTA_NESTEROV


class _Runner:
    """One merger over a single tensor of n elements, rounds run one after
    another with theta and m set to zero before each."""

    def __init__(self, n: int, mode: str, staging: bool):
        self.mode = mode
        self.theta = torch.zeros(n, dtype=torch.float32, device=DEV)
        self.m = torch.zeros_like(self.theta) if mode == "delta" else None
        self.zeros = torch.zeros_like(self.theta)
        self.mg = B.Merger([self.theta], momentum=None if self.m is None else [self.m],
                           staging=staging)
        self.rnd = 0

    def run(self, x: torch.Tensor, d: int, fold: bool = False):
        self.theta.zero_()
        if self.m is not None:
            self.m.zero_()
        rd = self.mg.begin(self.rnd)
        self.rnd += 1
        for i, (t, tok) in enumerate(_workers(x, self.zeros, self.mode, d)):
            if fold and i == 0:
                rd.fold([t], tok, _code(self.mode))
            else:
                rd.accumulate([t], tok)
        rd.finalize(_code(self.mode), 1.0, 0.0)
        rd.commit()
        torch.cuda.synchronize()
        return (self.theta.cpu().numpy(),
                None if self.m is None else self.m.cpu().numpy())

    def close(self):
        self.mg.close()


def _edge_dividends() -> np.ndarray:
    """Every power of two from the smallest subnormal to 2^127 with its two
    neighbours, both signs, plus zeros, the largest finite value, the
    infinities and a NaN."""
    pows = np.array([np.ldexp(F32(1.0), e) for e in range(-149, 128)], dtype=F32)
    up = np.nextafter(pows, F32(np.inf))
    dn = np.nextafter(pows, F32(0.0))
    v = np.concatenate([pows, up, dn, [F32(0.0), np.finfo(F32).max, F32(np.inf), F32(np.nan)]])
    return np.concatenate([v, -v]).astype(F32)


def _sample(n_random: int, seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    r = rng.integers(0, 1 << 32, size=n_random, dtype=np.uint64).astype(np.uint32).view(F32)
    return np.concatenate([_edge_dividends(), r]).astype(F32)


# ---- every binary32 dividend ---------------------------------------------------

@pytest.mark.parametrize("mode,d", [("mean", 3), ("delta", (1 << 24) - 1)])
def test_division_every_dividend(mode, d):
    n = 1 << 28
    run = _Runner(n, mode, staging=True)
    workers = min(16, os.cpu_count() or 1)
    try:
        with ThreadPoolExecutor(workers) as pool:
            for base in range(0, 1 << 32, n):
                x = np.arange(base, base + n, dtype=np.int64).astype(np.uint32).view(F32)
                got, m_got = run.run(torch.from_numpy(x).to(DEV), d)
                step = n // workers

                def part(i, x=x, got=got, m_got=m_got):
                    sl = slice(i * step, (i + 1) * step)
                    _check(got[sl], x[sl], mode, d, f"dividends 0x{base + i * step:08x}..",
                           None if m_got is None else m_got[sl])

                for f in [pool.submit(part, i) for i in range(workers)]:
                    f.result()
    finally:
        run.close()


# ---- sampled dividends, every path ---------------------------------------------

ALL_DIVISORS = [("mean", 3), ("mean", 5), ("mean", 6), ("mean", 7),
                ("delta", 3), ("delta", 10), ("delta", 1000), ("delta", 123_457),
                ("delta", (1 << 24) - 1), ("delta", (1 << 24) + 2), ("delta", 999_999_999),
                ("delta", (1 << 31) - 1), ("delta", 3 * (1 << 40) + 12_345), ("delta", 1 << 56)]


@pytest.mark.parametrize("mode,d", ALL_DIVISORS)
def test_division_sampled_staged(mode, d):
    x = _sample((1 << 22) + 1_731, seed=d)
    run = _Runner(x.size, mode, staging=True)
    try:
        n0 = run.mg.staged_count
        got, m_got = run.run(torch.from_numpy(x).to(DEV), d)
        assert run.mg.staged_count > n0
        _check(got, x, mode, d, "staged form", m_got)
    finally:
        run.close()


PATH_DIVISORS = [("mean", 3), ("mean", 7), ("delta", (1 << 24) - 1), ("delta", 999_999_999),
                 ("delta", 1 << 56)]


@pytest.mark.parametrize("mode,d", PATH_DIVISORS)
@pytest.mark.parametrize("path", ["register", "fold"])
def test_division_sampled_register_and_fold(path, mode, d):
    x = _sample((1 << 21) + 13, seed=7 * d + 1)
    run = _Runner(x.size, mode, staging=False)
    try:
        got, m_got = run.run(torch.from_numpy(x).to(DEV), d, fold=(path == "fold"))
        _check(got, x, mode, d, path, m_got)
    finally:
        run.close()


@pytest.mark.parametrize("mode,d", PATH_DIVISORS)
def test_division_sampled_noalloc(mode, d):
    x = _sample((1 << 21) + 29, seed=11 * d + 3)
    xd = torch.from_numpy(x).to(DEV)
    theta = torch.zeros_like(xd)
    m = torch.zeros_like(xd) if mode == "delta" else None
    zeros = torch.zeros_like(xd)
    ws = _workers(xd, zeros, mode, d)
    B.merge_round_noalloc([x.size], [theta.data_ptr()], [[t.data_ptr()] for t, _ in ws], B.F32,
                          _code(mode), tokens=[tok for _, tok in ws] if mode == "delta" else None,
                          lr=1.0, mu=0.0, momentum=None if m is None else [m.data_ptr()])
    torch.cuda.synchronize()
    _check(theta.cpu().numpy(), x, mode, d, "no-allocation entry point",
           None if m is None else m.cpu().numpy())


@pytest.mark.parametrize("mode,d", PATH_DIVISORS)
def test_division_sampled_commit_many(mode, d):
    x = _sample((1 << 21) + 4_096, seed=13 * d + 5)
    h = (x.size // 2) & ~7
    parts = [x[:h], x[h:]]
    theta = [torch.zeros(p.size, dtype=torch.float32, device=DEV) for p in parts]
    m = [torch.zeros_like(t) for t in theta] if mode == "delta" else None
    zeros = [torch.zeros_like(t) for t in theta]
    xs = [torch.from_numpy(p).to(DEV) for p in parts]
    mg = B.Merger(theta, momentum=m, fragment_of=[0, 1], n_fragments=2, staging=False)
    try:
        rds = []
        for f in range(2):
            rd = mg.begin(f, f)
            for t, tok in _workers(xs[f], zeros[f], mode, d):
                rd.accumulate([t], tok)
            rd.finalize(_code(mode), 1.0, 0.0)
            rds.append(rd)
        n0 = mg.launch_count
        mg.commit_many(rds)
        torch.cuda.synchronize()
        assert mg.launch_count - n0 == 1  # one multi-round pass
        for f in range(2):
            _check(theta[f].cpu().numpy(), parts[f], mode, d, f"multi-round pass, round {f}",
                   None if m is None else m[f].cpu().numpy())
    finally:
        mg.close()
