"""CPU oracle for the DiLoCo outer merge -- TEST INFRASTRUCTURE.

Only the test suite, the package smoke check and the benchmark's CPU-baseline
and reference arms may import this package. It wraps the plain C loops in
``merge_oracle.c`` (built by ``oracle/build.py``) and adds the round-level
selection: which tensors a round touches (its fragment) and which workers it
includes (its quorum subset).

Sources (page title, section):
  * "DiffuRefill-1B" model card, "How it is trained": plain mean folded into a
    running fp32 sum as checkpoints arrive; EMA of the globals, beta 0.9.
  * "DiffuRefill-1B: Pretraining a Masked Diffusion Language Model on Free,
    Preemptible Notebook GPUs", section 3, Table 2: plain replacement (outer
    learning rate 1, no momentum); merger waits for N fresh checkpoints of the
    current round tag; section 3 "Failure handling" (iii): a rollback gets a
    new round number.
  * "Pythia-14M on four rented GPUs and a bucket", "Getting updates through
    the bucket": fragments=4, quorum_size=3, token-weighted mean of the deltas,
    outer Nesterov (lr 0.7, momentum 0.9), two rounds in flight.

All arrays are numpy; floating point is fp32 as the pages fix it (the running
sum is kept in fp32), drift sums are fp64.
"""
from __future__ import annotations

import ctypes
import math
from dataclasses import dataclass, field
from typing import Sequence

import numpy as np

from . import build as _build

F32 = 0
BF16 = 1
MEAN_REPLACE = 0
DELTA_NESTEROV = 1

_lib = None


def lib():
    """Load (building first if needed) the C oracle."""
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        i64, i32, f32 = ctypes.c_int64, ctypes.c_int, ctypes.c_float
        vp, vpp = ctypes.c_void_p, ctypes.POINTER(ctypes.c_void_p)
        L.ora_widen_bf16.argtypes = [i64, vp, vp]
        L.ora_plain_mean.argtypes = [i64, i32, vpp, i32, vp]
        L.ora_weighted_delta.argtypes = [i64, i32, vpp, i32, vp, vp, vp]
        L.ora_outer_nesterov.argtypes = [i64, vp, f32, f32, vp, vp]
        L.ora_ema.argtypes = [i64, vp, f32, vp]
        L.ora_swa.argtypes = [i64, vp, i64, vp]
        L.ora_worker_drift.argtypes = [i64, i32, vpp, i32, vp, vp]
        L.ora_adopt_keep_drift.argtypes = [i64, vp, vp, vp, i32]
        L.ora_merge_tensor.argtypes = [i64, i32, vpp, i32, vp, i32, f32, f32,
                                       i32, f32, vp, vp, vp,
                                       ctypes.POINTER(ctypes.c_double)]
        for fn in (L.ora_widen_bf16, L.ora_plain_mean, L.ora_weighted_delta,
                   L.ora_outer_nesterov, L.ora_ema, L.ora_swa, L.ora_merge_tensor,
                   L.ora_worker_drift, L.ora_adopt_keep_drift):
            fn.restype = ctypes.c_int
        _lib = L
    return _lib


class OracleError(ValueError):
    pass


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise OracleError(f"{what}: oracle rejected its arguments (rc={rc})")


def _ptr(a: np.ndarray | None):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:  # bf16 bit patterns
        return BF16
    raise OracleError(f"unsupported checkpoint storage {a.dtype}")


def _ptr_array(xs: Sequence[np.ndarray]):
    arr = (ctypes.c_void_p * len(xs))(*[x.ctypes.data for x in xs])
    return ctypes.cast(arr, ctypes.POINTER(ctypes.c_void_p)), arr


def _contig(a: np.ndarray, dtype) -> np.ndarray:
    if a.dtype != dtype:
        raise OracleError(f"expected {dtype}, got {a.dtype}")
    return np.ascontiguousarray(a)


# ---- single steps ---------------------------------------------------------

def widen_bf16(bits: np.ndarray) -> np.ndarray:
    bits = _contig(bits, np.uint16)
    out = np.empty(bits.shape, np.float32)
    _check(lib().ora_widen_bf16(bits.size, _ptr(bits), _ptr(out)), "widen_bf16")
    return out


def plain_mean(xs: Sequence[np.ndarray]) -> np.ndarray:
    xs = [np.ascontiguousarray(x) for x in xs]
    dt = _dtype_code(xs[0])
    pp, keep = _ptr_array(xs)
    out = np.empty(xs[0].shape, np.float32)
    _check(lib().ora_plain_mean(xs[0].size, len(xs), pp, dt, _ptr(out)), "plain_mean")
    return out


def weighted_delta(xs: Sequence[np.ndarray], tokens: Sequence[int],
                   theta: np.ndarray) -> np.ndarray:
    xs = [np.ascontiguousarray(x) for x in xs]
    dt = _dtype_code(xs[0])
    theta = _contig(theta, np.float32)
    tok = np.ascontiguousarray(np.asarray(tokens, dtype=np.int64))
    pp, keep = _ptr_array(xs)
    out = np.empty(theta.shape, np.float32)
    _check(lib().ora_weighted_delta(theta.size, len(xs), pp, dt, _ptr(tok),
                                    _ptr(theta), _ptr(out)), "weighted_delta")
    return out


def outer_nesterov(delta: np.ndarray, lr: float, mu: float, theta: np.ndarray,
                   m: np.ndarray) -> None:
    """In place on theta and m."""
    delta = _contig(delta, np.float32)
    assert theta.flags.c_contiguous and m.flags.c_contiguous
    _check(lib().ora_outer_nesterov(delta.size, _ptr(delta), lr, mu, _ptr(theta),
                                    _ptr(m)), "outer_nesterov")


def ema(theta_new: np.ndarray, beta: float, e: np.ndarray) -> None:
    """In place on e."""
    theta_new = _contig(theta_new, np.float32)
    assert e.flags.c_contiguous and e.dtype == np.float32
    _check(lib().ora_ema(theta_new.size, _ptr(theta_new), beta, _ptr(e)), "ema")


def swa(theta_new: np.ndarray, count: int, mu: np.ndarray) -> None:
    """In place on mu: fold one more global into the uniform running average;
    count (>= 1) is the number of globals in the average after this one."""
    theta_new = _contig(theta_new, np.float32)
    assert mu.flags.c_contiguous and mu.dtype == np.float32
    _check(lib().ora_swa(theta_new.size, _ptr(theta_new), int(count), _ptr(mu)), "swa")


def worker_drift(xs: Sequence[np.ndarray], theta: np.ndarray) -> list[float]:
    """Per worker, the fp64 sum of (x_k - theta)^2 over the tensor (theta is
    the global before the round)."""
    xs = [np.ascontiguousarray(x) for x in xs]
    dt = _dtype_code(xs[0])
    theta = _contig(theta, np.float32)
    pp, keep = _ptr_array(xs)
    out = np.zeros(len(xs), np.float64)
    _check(lib().ora_worker_drift(theta.size, len(xs), pp, dt, _ptr(theta), _ptr(out)),
           "worker_drift")
    return [float(v) for v in out]


def adopt_keep_drift(theta_w: np.ndarray, g: np.ndarray, pushed: np.ndarray) -> None:
    """In place on theta_w: theta_w + (g - pushed)."""
    assert theta_w.dtype == np.float32 and theta_w.flags.c_contiguous
    g = _contig(g, np.float32)
    pushed = np.ascontiguousarray(pushed)
    _check(lib().ora_adopt_keep_drift(theta_w.size, _ptr(theta_w), _ptr(g), _ptr(pushed),
                                      _dtype_code(pushed)), "adopt_keep_drift")


ORTHO_SCALE_FIXED = 0       # update = lr * polar(Delta)
ORTHO_SCALE_MATCH_NORM = 1  # update = lr * |Delta|_F / sqrt(r) * polar(Delta)


def polar(delta: np.ndarray) -> np.ndarray:
    """The polar factor U V^T of a 2-D array (thin SVD in fp64): the
    semi-orthogonal matrix nearest to it ("DiffuRefill-1B" technical report,
    section 5.3: outer orthogonalisation replaces the averaged update by its
    polar factor)."""
    u, _, vt = np.linalg.svd(np.asarray(delta, np.float64), full_matrices=False)
    return u @ vt


def orthogonal_update(xs: Sequence[np.ndarray], theta: np.ndarray, rows: int, *,
                      lr: float, scale_mode: int = ORTHO_SCALE_FIXED):
    """One orthogonalised plain-mean round on one 2-D tensor (row-major, `rows`
    rows). The averaged update Delta = mean_k(x_k) - theta is formed in fp32
    exactly as in a plain-mean round, then replaced by its polar factor:
    theta' = theta + s * polar(Delta), s = lr (fixed) or lr * |Delta|_F /
    sqrt(min(m, n)) (the update keeps Delta's Frobenius norm, the RMS-matched
    form of the same report's section 5.3). Returns (theta' in fp64, Delta)."""
    mean = plain_mean(xs)
    delta = (mean - np.asarray(theta, np.float32)).astype(np.float32)  # one fp32 op
    m = int(rows)
    d2 = delta.reshape(m, -1)
    o = polar(d2)
    s = float(lr)
    if scale_mode == ORTHO_SCALE_MATCH_NORM:
        s = s * math.sqrt(float(np.sum(d2.astype(np.float64) ** 2))) / math.sqrt(min(d2.shape))
    out = np.asarray(theta, np.float64).reshape(d2.shape) + s * o
    return out.reshape(np.shape(theta)), delta


def plain_average(snapshots: Sequence[np.ndarray]) -> np.ndarray:
    """Average of stored snapshots (the last-n snapshot averages of the
    technical report's Table 5): their plain mean in the given order."""
    return plain_mean(snapshots)


def merge_tensor(xs: Sequence[np.ndarray], theta: np.ndarray, *, mode: int,
                 tokens: Sequence[int] | None = None, lr: float = 1.0,
                 mu: float = 0.0, m: np.ndarray | None = None,
                 e: np.ndarray | None = None, beta: float = 0.9) -> float:
    """One round on one tensor, in place on theta (and m, e). Returns the
    fp64 sum of squared drift over the tensor's elements."""
    xs = [np.ascontiguousarray(x) for x in xs]
    dt = _dtype_code(xs[0])
    for x in xs:
        if x.size != theta.size or _dtype_code(x) != dt:
            raise OracleError("checkpoint shape/dtype mismatch")
    assert theta.dtype == np.float32 and theta.flags.c_contiguous
    for a in (m, e):
        assert a is None or (a.dtype == np.float32 and a.flags.c_contiguous
                             and a.size == theta.size)
    tok = None
    if tokens is not None:
        tok = np.ascontiguousarray(np.asarray(tokens, dtype=np.int64))
    pp, keep = _ptr_array(xs)
    sumsq = ctypes.c_double(0.0)
    rc = lib().ora_merge_tensor(theta.size, len(xs), pp, dt, _ptr(tok), mode,
                                lr, mu, int(e is not None), beta, _ptr(theta),
                                _ptr(m), _ptr(e), ctypes.byref(sumsq))
    _check(rc, "merge_tensor")
    return sumsq.value


# ---- one round over a tensor list -----------------------------------------

class QuorumError(OracleError):
    pass


class StaleRoundError(OracleError):
    pass


@dataclass
class OracleState:
    """The merger's state: fp32 master theta, momentum m and EMA e per tensor,
    plus the last round number it accepted."""
    theta: list
    m: list | None = None
    e: list | None = None
    fragment_of: list = field(default_factory=list)
    last_round: int = -1
    swa: list | None = None            # running uniform average of the globals
    swa_count: list | None = None      # globals folded into it, per tensor


def fragment_tensors(fragment_of: Sequence[int], fragment: int) -> list[int]:
    """Tensor indices a round on `fragment` touches, in tensor-list order;
    fragment -1 means every tensor."""
    return [t for t, f in enumerate(fragment_of) if fragment == -1 or f == fragment]


def merge_round(state: OracleState, *, round: int, fragment: int,
                ckpts: Sequence[Sequence[np.ndarray]], included: Sequence[int],
                tokens: Sequence[int] | None, mode: int, lr: float = 1.0,
                mu: float = 0.0, quorum: int = 1, ema_beta: float | None = None,
                swa_update: bool = False):
    """Apply one merge round in place on `state`.

    ckpts[k][t] is worker k's copy of tensor t (full tensor list; only the
    fragment's tensors are read). `included` lists the workers that made the
    round, in arrival order; the others are never read. Returns
    (per_tensor_drift_norms, fragment_drift_norm).
    """
    if round <= state.last_round:
        raise StaleRoundError(f"round {round} is not newer than {state.last_round}")
    if len(included) < max(1, quorum):
        raise QuorumError(f"{len(included)} participants < quorum {quorum}")
    if mode == DELTA_NESTEROV and state.m is None:
        raise OracleError("momentum buffers required")
    if ema_beta is not None and state.e is None:
        raise OracleError("EMA buffers required")
    if swa_update and state.swa is None:
        raise OracleError("SWA buffers required")
    tlist = fragment_tensors(state.fragment_of, fragment)
    w = None if tokens is None else [int(tokens[k]) for k in included]
    sumsqs = []
    for t in tlist:
        xs = [ckpts[k][t] for k in included]
        s = merge_tensor(xs, state.theta[t], mode=mode, tokens=w, lr=lr, mu=mu,
                         m=None if state.m is None else state.m[t],
                         e=None if ema_beta is None else state.e[t],
                         beta=0.9 if ema_beta is None else ema_beta)
        if swa_update:
            state.swa_count[t] += 1
            swa(state.theta[t], state.swa_count[t], state.swa[t])
        sumsqs.append(s)
    total = 0.0
    for s in sumsqs:
        total += s
    state.last_round = round
    return [math.sqrt(s) for s in sumsqs], math.sqrt(total)
