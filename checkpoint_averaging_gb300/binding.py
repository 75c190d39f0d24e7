"""ctypes binding of libcam (C ABI in include/cam.h): argument marshalling only.

The functions here carry the C ABI's names without the ``cam_`` prefix and
turn error codes into exceptions. ``Merger`` / ``Round`` are a thin layer
for torch users: they check that tensors live on the right CUDA device with
the right dtype and layout, pass ``data_ptr()`` values and the current CUDA
stream, and keep borrowed checkpoint tensors alive on the commit stream.
Every step of a merge runs in libcam's CUDA kernels; there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import weakref
from typing import Sequence

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libcam.so")

KMAX = 8
MAX_OPEN_ROUNDS = 8

F32, BF16 = 0, 1
MEAN_REPLACE, DELTA_NESTEROV = 0, 1
INIT_EMA_FROM_MASTER, INIT_ZERO_MOMENTUM, INIT_ZERO_SWA = 1, 2, 4
NO_STAGING = 8
TIME_COMMITS = 16
NO_FUSED_FINISH = 32
TEST_STALL_STAGED = 64  # test hook: staged passes withhold their first tile and time out
SHARE_SMS = 128  # merge passes leave block slots for rounds in flight beside them
TEST_BAD_CHUNK = 256  # test hook: the first tensor's last chunk runs past its end on the device
TEST_BAD_TAG = 512  # test hook: staged passes mislabel their end marker and stop
FORM_REGISTER, FORM_STAGED, FORM_FOLDED, FORM_ORTHO = 0, 1, 2, 3
STATUS_WAIT_TIMEOUT = 1
STATUS_GEMM_TIMEOUT = 2
STATUS_BAD_CHUNK = 4
STATUS_PROTOCOL = 8
ORTHO_SCALE_FIXED, ORTHO_SCALE_MATCH_NORM = 0, 1
ORTHO_TF32, ORTHO_FP32, ORTHO_BF16 = 0, 1, 2
ORTHO_SHORT_SIDE = 4  # OR into the precision: iterate in the short side's space

OK, E_ARG, E_STATE, E_STALE, E_BUSY, E_QUORUM, E_KMAX, E_CUDA, E_NOMEM = \
    0, -1, -2, -3, -4, -5, -6, -7, -8


class CamError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"[{code}] {message}")
        self.code = code


class ArgError(CamError, ValueError):
    pass


class StateError(CamError):
    pass


class StaleRoundError(CamError):
    pass


class BusyError(CamError):
    pass


class QuorumError(CamError):
    pass


class KmaxError(CamError):
    pass


class CudaError(CamError):
    pass


_ERRORS = {E_ARG: ArgError, E_STATE: StateError, E_STALE: StaleRoundError,
           E_BUSY: BusyError, E_QUORUM: QuorumError, E_KMAX: KmaxError,
           E_CUDA: CudaError, E_NOMEM: CamError}


class CtxDesc(ctypes.Structure):
    _fields_ = [
        ("n_tensors", ctypes.c_int32),
        ("numel", ctypes.POINTER(ctypes.c_int64)),
        ("fragment_of", ctypes.POINTER(ctypes.c_int32)),
        ("n_fragments", ctypes.c_int32),
        ("quorum", ctypes.c_int32),
        ("master", ctypes.POINTER(ctypes.c_void_p)),
        ("momentum", ctypes.POINTER(ctypes.c_void_p)),
        ("ema", ctypes.POINTER(ctypes.c_void_p)),
        ("device", ctypes.c_int32),
        ("flags", ctypes.c_uint32),
        ("stream", ctypes.c_void_p),
        ("swa", ctypes.POINTER(ctypes.c_void_p)),
        ("rows", ctypes.POINTER(ctypes.c_int64)),
    ]


_lib = None

class CommitRecord(ctypes.Structure):
    """cam_commit_record: what the last commit did."""
    _fields_ = [("round", ctypes.c_int64), ("fragment", ctypes.c_int32), ("K", ctypes.c_int32),
                ("mode", ctypes.c_int32), ("form", ctypes.c_int32), ("elements", ctypes.c_int64),
                ("bytes", ctypes.c_int64), ("launches", ctypes.c_int64), ("ms", ctypes.c_float)]


EXPORTS = ("cam_ctx_create", "cam_ctx_destroy", "cam_merge_begin", "cam_merge_accumulate",
           "cam_merge_accumulate_host", "cam_merge_fold", "cam_merge_publish",
           "cam_swa_update", "cam_swa_reset", "cam_worker_drift_norm", "cam_adopt_keep_drift",
           "cam_merge_orthogonalize", "cam_swa_counts", "cam_swa_set_counts",
           "cam_merge_finalize", "cam_ema_update", "cam_drift_norm", "cam_merge_commit",
           "cam_merge_commit_many", "cam_merge_abort", "cam_merge_round", "cam_fragment_info",
           "cam_ctx_get_last_round",
           "cam_ctx_set_last_round", "cam_ctx_launch_count", "cam_ctx_status",
           "cam_ctx_staged_count", "cam_ctx_last_commit", "cam_stream_capturing",
           "cam_ctx_get_quorum", "cam_ctx_set_quorum",
           "cam_merge_round_noalloc", "cam_last_error", "cam_version")

NOALLOC_MAX_TENSORS = 4096
NOALLOC_MAX_CHUNKS = 131072


def lib() -> ctypes.CDLL:
    """Load libcam.so; raise if it has not been built (there is no fallback)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"libcam.so is missing at {LIB_PATH}: build it with "
            "`python -c 'import __graft_entry__ as g; g.build()'` (needs nvcc)")
    L = ctypes.CDLL(LIB_PATH)
    vp, vpp = ctypes.c_void_p, ctypes.POINTER(ctypes.c_void_p)
    i32, i64 = ctypes.c_int32, ctypes.c_int64
    L.cam_ctx_create.argtypes = [ctypes.POINTER(CtxDesc), vpp]
    L.cam_ctx_destroy.argtypes = [vp]
    L.cam_ctx_destroy.restype = None
    L.cam_merge_begin.argtypes = [vp, i64, i32, vpp]
    L.cam_merge_accumulate.argtypes = [vp, vpp, ctypes.c_int, i64]
    L.cam_merge_accumulate_host.argtypes = [vp, vpp, ctypes.c_int, i64]
    L.cam_merge_fold.argtypes = [vp, vpp, ctypes.c_int, i64, ctypes.c_int, vp]
    L.cam_merge_publish.argtypes = [vp, vpp, vpp]
    L.cam_swa_update.argtypes = [vp]
    L.cam_worker_drift_norm.argtypes = [vp, vp, vp]
    L.cam_merge_orthogonalize.argtypes = [vp, ctypes.c_float, i32, i32, i32]
    L.cam_adopt_keep_drift.argtypes = [i32, ctypes.POINTER(i64), vpp, vpp, vpp, ctypes.c_int, vp]
    L.cam_swa_reset.argtypes = [vp, i32, vp]
    L.cam_swa_counts.argtypes = [vp, ctypes.POINTER(i64)]
    L.cam_swa_set_counts.argtypes = [vp, ctypes.POINTER(i64)]
    L.cam_merge_finalize.argtypes = [vp, ctypes.c_int, ctypes.c_float, ctypes.c_float]
    L.cam_ema_update.argtypes = [vp, ctypes.c_float]
    L.cam_drift_norm.argtypes = [vp, vp, vp]
    L.cam_merge_commit.argtypes = [vp, vp]
    L.cam_merge_commit_many.argtypes = [ctypes.POINTER(ctypes.c_void_p), i32, vp]
    L.cam_merge_abort.argtypes = [vp]
    L.cam_merge_round.argtypes = [vp, i64, i32, i32, ctypes.POINTER(vpp), ctypes.c_int,
                                  ctypes.POINTER(i64), ctypes.c_int, ctypes.c_float,
                                  ctypes.c_float, i32, ctypes.c_float, vp, vp, vp]
    L.cam_fragment_info.argtypes = [vp, i32, ctypes.POINTER(i32), ctypes.POINTER(i64),
                                    ctypes.POINTER(i32)]
    L.cam_ctx_get_last_round.argtypes = [vp, ctypes.POINTER(i64)]
    L.cam_ctx_set_last_round.argtypes = [vp, i64]
    L.cam_ctx_launch_count.argtypes = [vp, ctypes.POINTER(i64)]
    L.cam_ctx_status.argtypes = [vp, ctypes.POINTER(i32)]
    L.cam_ctx_staged_count.argtypes = [vp, ctypes.POINTER(i64)]
    L.cam_ctx_last_commit.argtypes = [vp, ctypes.POINTER(CommitRecord)]
    L.cam_stream_capturing.argtypes = [vp, ctypes.POINTER(i32)]
    L.cam_ctx_get_quorum.argtypes = [vp, ctypes.POINTER(i32)]
    L.cam_ctx_set_quorum.argtypes = [vp, i32]
    L.cam_merge_round_noalloc.argtypes = [i32, ctypes.POINTER(i64), vpp, vpp, vpp, i32, vpp,
                                          ctypes.c_int, ctypes.POINTER(i64), ctypes.c_int,
                                          ctypes.c_float, ctypes.c_float, i32, ctypes.c_float,
                                          vp, vp, vp]
    L.cam_last_error.argtypes = []
    L.cam_last_error.restype = ctypes.c_char_p
    L.cam_version.argtypes = []
    L.cam_version.restype = ctypes.c_char_p
    for name in EXPORTS:
        fn = getattr(L, name)
        if name not in ("cam_ctx_destroy", "cam_last_error", "cam_version"):
            fn.restype = ctypes.c_int
    _lib = L
    return L


def last_error() -> str:
    return lib().cam_last_error().decode()


def version() -> str:
    return lib().cam_version().decode()


def _check(rc: int) -> None:
    if rc != OK:
        raise _ERRORS.get(rc, CamError)(rc, last_error())


def _ptrs(values: Sequence[int] | None):
    if values is None:
        return None
    return (ctypes.c_void_p * max(1, len(values)))(*[int(v) for v in values])


# ---- the C ABI, one function per entry point -----------------------------------

def ctx_create(numel: Sequence[int], master: Sequence[int], *, fragment_of=None,
               n_fragments: int = 1, quorum: int = 1, momentum=None, ema=None,
               device: int = 0, flags: int = 0, stream: int = 0, swa=None, rows=None) -> int:
    n = len(numel)
    numel_a = (ctypes.c_int64 * max(1, n))(*[int(v) for v in numel])
    frag_a = None if fragment_of is None else (ctypes.c_int32 * max(1, n))(*fragment_of)
    rows_a = None if rows is None else (ctypes.c_int64 * max(1, n))(*[int(v) for v in rows])
    keep = [numel_a, frag_a, _ptrs(master), _ptrs(momentum), _ptrs(ema), _ptrs(swa), rows_a]
    d = CtxDesc(n, numel_a,
                None if frag_a is None else ctypes.cast(frag_a, ctypes.POINTER(ctypes.c_int32)),
                n_fragments, quorum,
                ctypes.cast(keep[2], ctypes.POINTER(ctypes.c_void_p)),
                None if keep[3] is None else ctypes.cast(keep[3], ctypes.POINTER(ctypes.c_void_p)),
                None if keep[4] is None else ctypes.cast(keep[4], ctypes.POINTER(ctypes.c_void_p)),
                device, flags, stream or None,
                None if keep[5] is None else ctypes.cast(keep[5], ctypes.POINTER(ctypes.c_void_p)),
                None if rows_a is None else ctypes.cast(rows_a, ctypes.POINTER(ctypes.c_int64)))
    out = ctypes.c_void_p()
    _check(lib().cam_ctx_create(ctypes.byref(d), ctypes.byref(out)))
    return out.value


def ctx_destroy(ctx: int) -> None:
    lib().cam_ctx_destroy(ctx)


def merge_begin(ctx: int, round: int, fragment: int = -1) -> int:
    out = ctypes.c_void_p()
    _check(lib().cam_merge_begin(ctx, round, fragment, ctypes.byref(out)))
    return out.value


def merge_accumulate(rd: int, ckpt: Sequence[int], dtype: int, tokens: int = 0) -> None:
    arr = _ptrs(ckpt)
    _check(lib().cam_merge_accumulate(rd, ctypes.cast(arr, ctypes.POINTER(ctypes.c_void_p)),
                                      dtype, tokens))


def merge_accumulate_host(rd: int, ckpt: Sequence[int], dtype: int, tokens: int = 0) -> None:
    arr = _ptrs(ckpt)
    _check(lib().cam_merge_accumulate_host(
        rd, ctypes.cast(arr, ctypes.POINTER(ctypes.c_void_p)), dtype, tokens))


def merge_finalize(rd: int, mode: int, lr: float = 1.0, mu: float = 0.0) -> None:
    _check(lib().cam_merge_finalize(rd, mode, lr, mu))


def ema_update(rd: int, beta: float) -> None:
    _check(lib().cam_ema_update(rd, beta))


def worker_drift_norm(rd: int, per_worker_tensor: int | None, per_worker: int | None) -> None:
    _check(lib().cam_worker_drift_norm(rd, per_worker_tensor or None, per_worker or None))


def merge_orthogonalize(rd: int, lr: float, scale_mode: int = ORTHO_SCALE_FIXED,
                        precision: int = ORTHO_TF32, iterations: int = 30) -> None:
    _check(lib().cam_merge_orthogonalize(rd, lr, scale_mode, precision, iterations))


def swa_update(rd: int) -> None:
    _check(lib().cam_swa_update(rd))


def swa_reset(ctx: int, fragment: int = -1, stream: int = 0) -> None:
    _check(lib().cam_swa_reset(ctx, fragment, stream or None))


def swa_counts(ctx: int, n_tensors: int) -> list[int]:
    out = (ctypes.c_int64 * max(1, n_tensors))()
    _check(lib().cam_swa_counts(ctx, out))
    return list(out[:n_tensors])


def swa_set_counts(ctx: int, counts: Sequence[int]) -> None:
    arr = (ctypes.c_int64 * max(1, len(counts)))(*[int(c) for c in counts])
    _check(lib().cam_swa_set_counts(ctx, arr))


def drift_norm(rd: int, per_tensor: int | None, per_fragment: int | None) -> None:
    _check(lib().cam_drift_norm(rd, per_tensor or None, per_fragment or None))


def merge_publish(rd: int, theta_out: Sequence[int], ema_out: Sequence[int] | None = None) -> None:
    vpp = ctypes.POINTER(ctypes.c_void_p)
    th = ctypes.cast(_ptrs(theta_out), vpp)
    em = None if ema_out is None else ctypes.cast(_ptrs(ema_out), vpp)
    _check(lib().cam_merge_publish(rd, th, em))


def merge_commit(rd: int, stream: int = 0) -> None:
    _check(lib().cam_merge_commit(rd, stream or None))


def merge_commit_many(rds: Sequence[int], stream: int = 0) -> None:
    arr = (ctypes.c_void_p * len(rds))(*rds)
    _check(lib().cam_merge_commit_many(arr, len(rds), stream or None))


def merge_abort(rd: int) -> None:
    _check(lib().cam_merge_abort(rd))


def fragment_info(ctx: int, fragment: int) -> tuple[list[int], int]:
    nt, ne = ctypes.c_int32(), ctypes.c_int64()
    _check(lib().cam_fragment_info(ctx, fragment, ctypes.byref(nt), ctypes.byref(ne), None))
    ids = (ctypes.c_int32 * max(1, nt.value))()
    _check(lib().cam_fragment_info(ctx, fragment, None, None, ids))
    return list(ids[:nt.value]), ne.value


def ctx_get_last_round(ctx: int) -> int:
    out = ctypes.c_int64()
    _check(lib().cam_ctx_get_last_round(ctx, ctypes.byref(out)))
    return out.value


def ctx_set_last_round(ctx: int, round: int) -> None:
    _check(lib().cam_ctx_set_last_round(ctx, round))


def ctx_launch_count(ctx: int) -> int:
    out = ctypes.c_int64()
    _check(lib().cam_ctx_launch_count(ctx, ctypes.byref(out)))
    return out.value


def ctx_last_commit(ctx: int) -> dict:
    rec = CommitRecord()
    _check(lib().cam_ctx_last_commit(ctx, ctypes.byref(rec)))
    return {name: getattr(rec, name) for name, _ in CommitRecord._fields_}


def ctx_staged_count(ctx: int) -> int:
    out = ctypes.c_int64()
    _check(lib().cam_ctx_staged_count(ctx, ctypes.byref(out)))
    return out.value


def ctx_status(ctx: int) -> int:
    out = ctypes.c_int32()
    _check(lib().cam_ctx_status(ctx, ctypes.byref(out)))
    return out.value


def merge_round_noalloc(numel: Sequence[int], master: Sequence[int], ckpt: Sequence[Sequence[int]],
                        dtype: int, mode: int, *, tokens: Sequence[int] | None = None,
                        lr: float = 1.0, mu: float = 0.0, momentum: Sequence[int] | None = None,
                        ema: Sequence[int] | None = None, beta: float = 0.9,
                        per_tensor: int | None = None, per_round: int | None = None,
                        stream: int = 0) -> None:
    """One whole round through cam_merge_round_noalloc, the entry point that
    allocates nothing (for callers that may not allocate device memory).
    ckpt[k][t] is worker k's device pointer for tensor t, in arrival order.
    The EMA is updated when `ema` is given."""
    n = len(numel)
    K = len(ckpt)
    numel_a = (ctypes.c_int64 * max(1, n))(*[int(v) for v in numel])
    flat = [int(p) for w in ckpt for p in w]
    if len(flat) != K * n:
        raise ValueError("ckpt must hold one pointer per tensor per worker")
    tok = None if tokens is None else (ctypes.c_int64 * max(1, K))(*[int(t) for t in tokens])
    vpp = ctypes.POINTER(ctypes.c_void_p)

    def arr(v):
        return None if v is None else ctypes.cast(_ptrs(v), vpp)

    keep = [arr(master), arr(momentum), arr(ema), arr(flat)]
    _check(lib().cam_merge_round_noalloc(
        n, numel_a, keep[0], keep[1], keep[2], K, keep[3], dtype, tok, mode, lr, mu,
        int(ema is not None), beta, per_tensor or None, per_round or None, stream or None))


def adopt_keep_drift(theta_w, global_, pushed, stream=None) -> None:
    """theta_w[t] += global_[t] - pushed[t] for a worker's tensor list: adopt the
    new global while keeping the progress made since the push (the alternative
    to plain replacement in the DiffuRefill-1B report, section 5.1).
    theta_w and global_ are fp32 CUDA tensors, pushed fp32 or bf16."""
    torch = _torch()
    theta_w, global_, pushed = list(theta_w), list(global_), list(pushed)
    if not (len(theta_w) == len(global_) == len(pushed)):
        raise ValueError("the three tensor lists must have the same length")
    dt = pushed[0].dtype if pushed else torch.float32
    for a, b, c in zip(theta_w, global_, pushed):
        if (a.numel() != b.numel() or a.numel() != c.numel() or a.dtype != torch.float32
                or b.dtype != torch.float32 or c.dtype != dt or a.device.type != "cuda"
                or b.device != a.device or c.device != a.device
                or not (a.is_contiguous() and b.is_contiguous() and c.is_contiguous())):
            raise ValueError("adopt_keep_drift: mismatched tensors")
    n = len(theta_w)
    numel = (ctypes.c_int64 * max(1, n))(*[t.numel() for t in theta_w])
    vpp = ctypes.POINTER(ctypes.c_void_p)
    arrs = [ctypes.cast(_ptrs([t.data_ptr() for t in group]), vpp)
            for group in (theta_w, global_, pushed)]
    _check(lib().cam_adopt_keep_drift(n, numel, arrs[0], arrs[1], arrs[2],
                                      BF16 if dt == torch.bfloat16 else F32,
                                      _stream_handle(stream)))


def average_snapshots(out, snapshots, stream=None) -> None:
    """out[t] = plain mean of snapshots[j][t] over j, for stored globals (the
    averages of the last n snapshots of the DiffuRefill-1B technical report,
    Table 5). One merge pass in plain-mean mode with the snapshots as the
    workers and `out` as the global; at most KMAX snapshots; fp32 or bf16."""
    torch = _torch()
    out = list(out)
    snaps = [list(sn) for sn in snapshots]
    if not 1 <= len(snaps) <= KMAX:
        raise ValueError(f"1..{KMAX} snapshots")
    dt = snaps[0][0].dtype if out else torch.float32
    for sn in snaps:
        if len(sn) != len(out):
            raise ValueError("every snapshot needs one tensor per output tensor")
        for a, b in zip(sn, out):
            if a.numel() != b.numel() or a.dtype != dt or not a.is_contiguous():
                raise ValueError("snapshot tensors must match the outputs")
    for b in out:
        if b.dtype != torch.float32 or not b.is_contiguous() or b.device.type != "cuda":
            raise ValueError("outputs must be contiguous fp32 CUDA tensors")
    merge_round_noalloc([b.numel() for b in out], [b.data_ptr() for b in out],
                        [[a.data_ptr() for a in sn] for sn in snaps],
                        BF16 if dt == torch.bfloat16 else F32, MEAN_REPLACE,
                        stream=_stream_handle(stream))


# ---- torch-facing layer ----------------------------------------------------------

def _torch():
    import torch
    return torch


def stream_capturing(stream: int) -> bool:
    out = ctypes.c_int32()
    _check(lib().cam_stream_capturing(stream or None, ctypes.byref(out)))
    return out.value != 0


def _capturing(stream) -> bool:
    """True while the torch stream `stream` is being captured into a CUDA graph."""
    return stream_capturing(int(stream.cuda_stream))


def _record_streams(tensors, stream, handle: int) -> list:
    """record_stream for each CUDA tensor on `stream`, once per tensor object
    and stream: the caching allocator fences every stream recorded on a block
    when the block is freed, so one record covers every later use on that
    stream while the tensor lives. Returns the CPU tensors, which need their
    own hold."""
    host = []
    for t in tensors:
        if not t.is_cuda:
            host.append(t)
            continue
        seen = getattr(t, "_cam_recorded_streams", None)
        if seen is None:
            seen = set()
            t._cam_recorded_streams = seen
        if handle not in seen:
            t.record_stream(stream)
            seen.add(handle)
    return host


def _stream_handle(stream) -> int:
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


class Merger:
    """The merger's state on one GPU: fp32 master weights (theta), optional
    outer momentum and EMA buffers, the fragment map and the quorum. The
    tensors are borrowed for the Merger's life and updated in place."""

    def __init__(self, master, *, momentum=None, ema=None, fragment_of=None,
                 n_fragments: int = 1, quorum: int = 1, init_ema_from_master=False,
                 zero_momentum=False, stream=None, swa=None, zero_swa=False, rows=None,
                 staging=True, time_commits=False, fused_finish=True, test_stall_staged=False,
                 share_sms=False, test_bad_chunk=False, test_bad_tag=False):
        """rows: optional per-tensor matrix rows (default: the tensors' first
        dimension), used by orthogonalised rounds. staging=False keeps every
        merge pass on the register form (the staged form gives the same
        results). time_commits=True times each commit's device work
        (last_commit()["ms"]). fused_finish=False always launches the
        separate norm pass (small rounds otherwise finish their norms in the
        merge pass; the same bits). share_sms=True (CAM_SHARE_SMS) gives every
        merge pass at most three quarters of the register form's block slots,
        so that rounds in flight on other streams start beside it (the same
        bits). test_stall_staged=True is a test hook
        (CAM_TEST_STALL_STAGED): staged passes withhold their first tile, their
        waits give up after about 1 ms and status() reports the timeout.
        test_bad_chunk=True (CAM_TEST_BAD_CHUNK) and test_bad_tag=True
        (CAM_TEST_BAD_TAG) are test hooks for the passes' own checks: a chunk
        table whose first tensor's last chunk runs 2,048 elements past its end
        (the caller's buffers of that tensor must have that room), and staged
        passes whose end marker carries a wrong fill number."""
        torch = _torch()
        self.master = list(master)
        self.momentum = None if momentum is None else list(momentum)
        self.ema = None if ema is None else list(ema)
        self.swa = None if swa is None else list(swa)
        if not self.master:
            raise ValueError("empty parameter list")
        dev = self.master[0].device
        if dev.type != "cuda":
            raise ValueError("master tensors must be CUDA tensors")
        self.device = dev
        for group in (self.master, self.momentum, self.ema, self.swa):
            if group is None:
                continue
            if len(group) != len(self.master):
                raise ValueError("momentum/ema lists must match the master list")
            for t, ref in zip(group, self.master):
                if (t.device != dev or t.dtype != torch.float32 or not t.is_contiguous()
                        or t.numel() != ref.numel()):
                    raise ValueError("state tensors must be contiguous fp32 on one device")
        self.numel = [t.numel() for t in self.master]
        self.fragment_of = list(fragment_of) if fragment_of is not None else [0] * len(self.master)
        self.n_fragments = n_fragments
        flags = (INIT_EMA_FROM_MASTER if init_ema_from_master else 0) | \
                (INIT_ZERO_MOMENTUM if zero_momentum else 0) | (INIT_ZERO_SWA if zero_swa else 0) | \
                (0 if staging else NO_STAGING) | (TIME_COMMITS if time_commits else 0) | \
                (0 if fused_finish else NO_FUSED_FINISH) | \
                (TEST_STALL_STAGED if test_stall_staged else 0) | (SHARE_SMS if share_sms else 0) | \
                (TEST_BAD_CHUNK if test_bad_chunk else 0) | (TEST_BAD_TAG if test_bad_tag else 0)
        with torch.cuda.device(dev):
            self.ctx = ctx_create(
                self.numel, [t.data_ptr() for t in self.master], fragment_of=self.fragment_of,
                n_fragments=n_fragments, quorum=quorum,
                momentum=None if self.momentum is None else [t.data_ptr() for t in self.momentum],
                ema=None if self.ema is None else [t.data_ptr() for t in self.ema],
                device=dev.index if dev.index is not None else torch.cuda.current_device(),
                flags=flags, stream=_stream_handle(stream),
                swa=None if self.swa is None else [t.data_ptr() for t in self.swa],
                rows=list(rows) if rows is not None else
                [t.shape[0] if t.dim() >= 2 else 0 for t in self.master])
        self._frag_cache = {}
        self._round_args = {}  # merge(): marshalled arguments by (fragment, checkpoints, tokens)
        self._norm_args = {}  # merge(): validated norm outputs by (their ids, fragment)
        self._inflight = []  # (event, host tensors) held until the work reading them ran

    def close(self):
        if getattr(self, "ctx", None):
            # destroying the context frees its open rounds: their handles go too
            for rd in list(getattr(self, "_rounds", ())):
                rd.handle = None
            ctx_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _hold_until_done(self, host_tensors, stream) -> None:
        """Keeps host checkpoints referenced until the work that reads them
        has run (torch cannot record a stream on a CPU tensor)."""
        torch = _torch()
        self._inflight = [(ev, ts) for ev, ts in self._inflight if not ev.query()]
        if host_tensors:
            ev = torch.cuda.Event()
            ev.record(stream)
            self._inflight.append((ev, host_tensors))

    def fragment_tensors(self, fragment: int) -> list[int]:
        if fragment not in self._frag_cache:
            self._frag_cache[fragment] = fragment_info(self.ctx, fragment)[0]
        return self._frag_cache[fragment]

    @property
    def swa_counts(self) -> list[int]:
        """Globals folded into each tensor's running average."""
        return swa_counts(self.ctx, len(self.master))

    @swa_counts.setter
    def swa_counts(self, counts) -> None:
        swa_set_counts(self.ctx, counts)

    def swa_reset(self, fragment: int = -1, stream=None) -> None:
        """Zeroes the running averages of `fragment` (-1: all) and their counts."""
        swa_reset(self.ctx, fragment, _stream_handle(stream))

    @property
    def launch_count(self) -> int:
        return ctx_launch_count(self.ctx)

    def last_commit(self) -> dict:
        """The record of the last commit (round, fragment, K, mode, form,
        elements, bytes, launches, ms); waits for its work when timed."""
        return ctx_last_commit(self.ctx)

    @property
    def staged_count(self) -> int:
        """Merge passes launched in the staged (bulk-copy) form so far."""
        return ctx_staged_count(self.ctx)

    def status(self) -> int:
        """Waits for the device, then returns its status word (0: no merge
        pass gave up waiting on a barrier)."""
        return ctx_status(self.ctx)

    @property
    def quorum(self) -> int:
        """Participants a commit needs; lower it to merge the leftovers of a
        shrunken fleet (down to 1)."""
        out = ctypes.c_int32()
        _check(lib().cam_ctx_get_quorum(self.ctx, ctypes.byref(out)))
        return out.value

    @quorum.setter
    def quorum(self, q: int) -> None:
        _check(lib().cam_ctx_set_quorum(self.ctx, int(q)))

    @property
    def last_round(self) -> int:
        return ctx_get_last_round(self.ctx)

    @last_round.setter
    def last_round(self, r: int) -> None:
        ctx_set_last_round(self.ctx, r)

    def begin(self, round: int, fragment: int = -1) -> "Round":
        rd = Round(self, merge_begin(self.ctx, round, fragment), fragment)
        if not hasattr(self, "_rounds"):
            self._rounds = weakref.WeakSet()
        self._rounds.add(rd)
        return rd

    def merge(self, round: int, ckpts, tokens=None, *, fragment: int = -1,
              mode: int = MEAN_REPLACE, lr: float = 1.0, mu: float = 0.0, ema_beta=None,
              norms=None, stream=None) -> None:
        """One whole round in one host call (cam_merge_round): the same as
        begin(round, fragment), accumulate of each worker of `ckpts` in
        arrival order with its `tokens`, finalize(mode, lr, mu),
        ema_update(ema_beta) when it is given, drift_norm(*norms) when norms
        = (per_tensor, per_fragment) is given, and commit(stream), with the
        same results. ckpts are device-resident Checkpoints made for
        `fragment`, or tensor lists (made into Checkpoints at each call).
        Host-resident workers are not taken here: open the round with begin
        and accumulate them. The marshalled arguments of Checkpoint lists are
        kept for the next call with the same Checkpoints and tokens."""
        torch = _torch()
        ckpts = list(ckpts)
        key = None
        if all(isinstance(c, Checkpoint) for c in ckpts):
            key = (fragment, tuple(map(id, ckpts)), None if tokens is None else tuple(tokens))
        hit = None if key is None else self._round_args.get(key)
        if hit is None:
            cks = [c if isinstance(c, Checkpoint) and c.merger is self and c.fragment == fragment
                   else Checkpoint(self, c, fragment) for c in ckpts]
            if not cks or len(cks) > KMAX:
                raise ValueError(f"a round takes 1 to {KMAX} workers")
            if any(c.host for c in cks):
                raise ValueError("host-resident checkpoints go through Round.accumulate")
            if any(c.dtype_code != cks[0].dtype_code for c in cks):
                raise ValueError("every worker of a round must have the same dtype")
            arr = (ctypes.POINTER(ctypes.c_void_p) * len(cks))(*[c.ptr_array for c in cks])
            tok = None if tokens is None else (ctypes.c_int64 * len(cks))(*map(int, tokens))
            keep = [t for c in cks for t in c.keep]
            # (the entry holds the Checkpoints, so the ids in its key stay
            # theirs; the set names the streams their tensors are recorded on)
            hit = (arr, tok, cks[0].dtype_code, keep, list(ckpts), set())
            if key is not None:
                if len(self._round_args) >= 64:
                    self._round_args.clear()
                self._round_args[key] = hit
        arr, tok, dtype, keep, _, recorded = hit
        pt_p = pf_p = None
        nhit = None
        if norms is not None:
            nkey = (id(norms[0]), id(norms[1]), fragment)
            nhit = self._norm_args.get(nkey)
            if nhit is None:
                pt, pf = norms
                for t, n in ((pt, len(self.fragment_tensors(fragment))), (pf, 1)):
                    if t is not None and (t.device != self.device or t.dtype != torch.float64
                                          or not t.is_contiguous() or t.numel() < n):
                        raise ValueError("norm outputs must be contiguous fp64 device tensors")
                outs = [t for t in (pt, pf) if t is not None]
                nhit = (None if pt is None else pt.data_ptr(), None if pf is None else pf.data_ptr(),
                        outs, set())
                if len(self._norm_args) >= 64:
                    self._norm_args.clear()
                self._norm_args[nkey] = nhit  # (it holds the tensors: their ids stay theirs)
            pt_p, pf_p = nhit[0], nhit[1]
        if stream is None:
            s = torch.cuda.current_stream(self.device)
            sh = int(s.cuda_stream)
            capturing = torch.cuda.is_current_stream_capturing()
        else:
            s = stream
            sh = int(s.cuda_stream)
            capturing = None
        _check(lib().cam_merge_round(
            self.ctx, int(round), int(fragment), len(arr), arr, dtype, tok, int(mode),
            float(lr), float(mu), 0 if ema_beta is None else 1,
            0.0 if ema_beta is None else float(ema_beta), pt_p, pf_p, sh or None))
        if capturing is None:
            capturing = stream_capturing(sh)
        if capturing:
            return  # a captured graph reads its buffers at every replay: they are the caller's
        # record_stream once per tensor and stream covers every later use on it
        if sh not in recorded:
            _record_streams(keep, s, sh)
            recorded.add(sh)
        if nhit is not None and sh not in nhit[3]:
            _record_streams(nhit[2], s, sh)
            nhit[3].add(sh)
        if self._inflight:
            self._hold_until_done([], s)

    def checkpoint(self, ckpt, fragment: int = -1) -> "Checkpoint":
        """Validates a worker's tensors once for rounds on `fragment`."""
        return Checkpoint(self, ckpt, fragment)

    def commit_many(self, rounds, stream=None) -> None:
        """Commits open rounds of this merger as one call (cam_merge_commit_many):
        the same results as committing each in order on `stream`; rounds of
        one register-form variant share one merge pass."""
        torch = _torch()
        rounds = list(rounds)
        s = torch.cuda.current_stream(self.device) if stream is None else stream
        sh = int(s.cuda_stream)
        try:
            merge_commit_many([rd.handle for rd in rounds], sh)
        except CudaError:
            for rd in rounds:
                rd.handle = None  # the library freed the rounds of a shared pass
            raise
        borrowed = []
        for rd in rounds:
            rd.handle = None
            borrowed.extend(rd._borrowed)
            rd._borrowed = []
        if stream_capturing(sh):
            return  # a captured graph reads its buffers at every replay: they are the caller's
        host = _record_streams(borrowed, s, sh)
        if host or self._inflight:
            self._hold_until_done(host, s)


class Checkpoint:
    """One worker's tensors for one fragment of a Merger, validated once.

    The pointer array handed to the C ABI is built here, so accumulating a
    prepared checkpoint is a single library call. CUDA tensors must live on
    the Merger's device; CPU tensors (pinned, or pageable where the GPU reads
    host page tables) are streamed from host memory by the merge pass."""

    def __init__(self, merger: "Merger", ckpt, fragment: int = -1):
        torch = _torch()
        ids = merger.fragment_tensors(fragment)
        ckpt = list(ckpt)
        if len(ckpt) == len(merger.master) and len(ckpt) != len(ids):
            ckpt = [ckpt[g] for g in ids]
        if len(ckpt) != len(ids):
            raise ValueError(f"expected {len(ids)} tensors, got {len(ckpt)}")
        dt = ckpt[0].dtype if ckpt else torch.float32
        if dt not in (torch.float32, torch.bfloat16):
            raise ValueError("checkpoints must be fp32 or bf16")
        host = False
        for t, g in zip(ckpt, ids):
            on_host = t.device.type == "cpu"
            host = host or on_host
            if ((not on_host and t.device != merger.device) or t.dtype != dt
                    or not t.is_contiguous() or t.numel() != merger.numel[g]):
                raise ValueError(f"checkpoint tensor for tensor {g} has wrong device/dtype/shape")
        self.merger, self.fragment, self.host = merger, fragment, host
        self.dtype_code = BF16 if dt == torch.bfloat16 else F32
        self._arr = _ptrs([t.data_ptr() for t in ckpt])
        self.ptr_array = ctypes.cast(self._arr, ctypes.POINTER(ctypes.c_void_p))
        # one tensor per underlying storage is enough to keep memory alive and
        # to record the commit stream on the caching allocator's block
        seen, keep = set(), []
        for t in ckpt:
            key = t.untyped_storage().data_ptr()
            if key not in seen:
                seen.add(key)
                keep.append(t)
        self.keep = keep


class Round:
    def __init__(self, merger: Merger, handle: int, fragment: int):
        self.merger, self.handle, self.fragment = merger, handle, fragment
        self.tensors = merger.fragment_tensors(fragment)
        self._borrowed = []

    def accumulate(self, ckpt, tokens: int = 0) -> None:
        """Adds one worker, in arrival order. ckpt is a Checkpoint made for
        this round's fragment, or its tensors: the fragment's tensors in
        fragment order, or the whole tensor list (the fragment's are taken)."""
        if not isinstance(ckpt, Checkpoint):
            ckpt = Checkpoint(self.merger, ckpt, self.fragment)
        elif ckpt.merger is not self.merger or ckpt.fragment != self.fragment:
            raise ValueError("checkpoint was prepared for another merger or fragment")
        fn = lib().cam_merge_accumulate_host if ckpt.host else lib().cam_merge_accumulate
        _check(fn(self.handle, ckpt.ptr_array, ckpt.dtype_code, int(tokens)))
        self._borrowed.extend(ckpt.keep)

    def fold(self, ckpt, tokens: int = 0, mode: int = MEAN_REPLACE, stream=None) -> None:
        """Folds one arriving worker into the round's running sum at once, on
        `stream` (default: the current stream). The worker's tensors are held
        only until that fold has run; `mode` must match the later finalize."""
        torch = _torch()
        if not isinstance(ckpt, Checkpoint):
            ckpt = Checkpoint(self.merger, ckpt, self.fragment)
        elif ckpt.merger is not self.merger or ckpt.fragment != self.fragment:
            raise ValueError("checkpoint was prepared for another merger or fragment")
        s = torch.cuda.current_stream(self.merger.device) if stream is None else stream
        sh = int(s.cuda_stream)
        _check(lib().cam_merge_fold(self.handle, ckpt.ptr_array, ckpt.dtype_code, int(tokens),
                                    int(mode), sh))
        if stream_capturing(sh):
            return
        self.merger._hold_until_done(_record_streams(ckpt.keep, s, sh), s)

    def finalize(self, mode: int, lr: float = 1.0, mu: float = 0.0) -> None:
        merge_finalize(self.handle, mode, lr, mu)

    def ema_update(self, beta: float) -> None:
        ema_update(self.handle, beta)

    def swa_update(self) -> None:
        swa_update(self.handle)

    def orthogonalize(self, lr: float, scale_mode: int = ORTHO_SCALE_FIXED,
                      precision: int = ORTHO_TF32, iterations: int = 30) -> None:
        """Replace the averaged update of every matrix by its polar factor."""
        merge_orthogonalize(self.handle, lr, scale_mode, precision, iterations)

    def worker_drift_norm(self, per_worker_tensor=None, per_worker=None) -> None:
        """Each worker's drift from the round's starting global: per_worker_tensor
        [K * T_f] (worker-major) and per_worker [K], fp64 CUDA tensors sized for
        the K workers accumulated by commit time."""
        torch = _torch()
        for t in (per_worker_tensor, per_worker):
            if t is not None and (t.device != self.merger.device or t.dtype != torch.float64
                                  or not t.is_contiguous()):
                raise ValueError("worker norm outputs must be contiguous fp64 device tensors")
        worker_drift_norm(self.handle,
                          None if per_worker_tensor is None else per_worker_tensor.data_ptr(),
                          None if per_worker is None else per_worker.data_ptr())
        self._borrowed.extend(t for t in (per_worker_tensor, per_worker) if t is not None)

    def drift_norm(self, per_tensor=None, per_fragment=None) -> None:
        torch = _torch()
        for t, n in ((per_tensor, len(self.tensors)), (per_fragment, 1)):
            if t is not None and (t.device != self.merger.device or t.dtype != torch.float64
                                  or not t.is_contiguous() or t.numel() < n):
                raise ValueError("norm outputs must be contiguous fp64 device tensors")
        drift_norm(self.handle, None if per_tensor is None else per_tensor.data_ptr(),
                   None if per_fragment is None else per_fragment.data_ptr())
        self._borrowed.extend(t for t in (per_tensor, per_fragment) if t is not None)

    def publish(self, theta_out, ema_out=None) -> None:
        """Also write the new theta (and EMA) into these fp32 tensors, fragment
        order, in the same pass: CUDA tensors or (pinned) CPU tensors."""
        torch = _torch()
        for group in (theta_out, ema_out):
            if group is None:
                continue
            if len(group) != len(self.tensors):
                raise ValueError(f"expected {len(self.tensors)} output tensors")
            for t, g in zip(group, self.tensors):
                if (t.dtype != torch.float32 or not t.is_contiguous()
                        or t.numel() != self.merger.numel[g]
                        or (t.device.type != "cpu" and t.device != self.merger.device)):
                    raise ValueError(f"publish buffer for tensor {g} has wrong device/dtype/shape")
        merge_publish(self.handle, [t.data_ptr() for t in theta_out],
                      None if ema_out is None else [t.data_ptr() for t in ema_out])
        self._borrowed.extend(theta_out)
        if ema_out is not None:
            self._borrowed.extend(ema_out)

    def commit(self, stream=None) -> None:
        torch = _torch()
        s = torch.cuda.current_stream(self.merger.device) if stream is None else stream
        sh = int(s.cuda_stream)
        try:
            merge_commit(self.handle, sh)
        except CudaError:
            self.handle = None  # the library freed the round
            raise
        self.handle = None
        borrowed, self._borrowed = self._borrowed, []
        if stream_capturing(sh):
            return  # a captured graph reads its buffers at every replay: they are the caller's
        # freed memory is not reused before the merge ran
        host = _record_streams(borrowed, s, sh)
        if host or self.merger._inflight:
            self.merger._hold_until_done(host, s)

    def abort(self) -> None:
        merge_abort(self.handle)
        self.handle = None

    def __del__(self):
        # a round dropped while open is aborted, so its fragment takes new rounds
        try:
            if getattr(self, "handle", None) is not None and self.merger.ctx:
                merge_abort(self.handle)
                self.handle = None
        except Exception:
            pass
