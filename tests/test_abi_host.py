"""Host-only checks of the C ABI: the library builds and loads, exports every
function include/*.h declares, validates descriptions before any CUDA call, and
fails loudly (never falls back) when no GPU is usable."""
import ctypes
import glob
import os
import re
import subprocess

import pytest
import torch

from checkpoint_averaging_gb300 import binding as B
from checkpoint_averaging_gb300 import build as cam_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    cam_build.build()


def declared_functions():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(cam_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_round_calls():
    names = declared_functions()
    for n in ("cam_merge_begin", "cam_merge_accumulate", "cam_merge_finalize",
              "cam_ema_update", "cam_drift_norm", "cam_merge_commit"):
        assert n in names


def test_library_exports_every_declared_symbol():
    L = ctypes.CDLL(B.LIB_PATH)
    for n in declared_functions():
        assert hasattr(L, n), f"{n} declared in include/ but not exported"
    out = subprocess.run(["nm", "-D", "--defined-only", B.LIB_PATH], capture_output=True,
                         text=True).stdout
    exported = set(re.findall(r" T (\w+)", out))
    assert exported == set(declared_functions()), exported ^ set(declared_functions())
    assert set(B.EXPORTS) == exported


def test_version():
    assert B.version() == "0.1.0"


@pytest.mark.parametrize("kw,msg", [
    (dict(quorum=0), "quorum"),
    (dict(quorum=9), "quorum"),
    (dict(n_fragments=0), "n_fragments"),
    (dict(fragment_of=[3], n_fragments=2), "fragment_of"),
    (dict(device=-1), "device"),
    (dict(flags=1024), "flags"),
    (dict(flags=B.INIT_EMA_FROM_MASTER), "EMA"),
    (dict(flags=B.INIT_ZERO_MOMENTUM), "momentum"),
])
def test_invalid_descriptions_rejected_before_cuda(kw, msg):
    with pytest.raises(B.ArgError) as ei:
        B.ctx_create([16], [0x10000], **kw)
    assert msg in str(ei.value)


def test_null_pointers_and_sizes_rejected():
    with pytest.raises(B.ArgError):
        B.ctx_create([16], [0])             # master pointer NULL
    with pytest.raises(B.ArgError):
        B.ctx_create([-1], [0x10000])       # negative size
    with pytest.raises(B.ArgError):
        B.ctx_create([], [])                # no tensors
    # a zero-size tensor may have a NULL pointer: that is not an argument error
    if not torch.cuda.is_available():
        with pytest.raises(B.CudaError):
            B.ctx_create([0], [0])


def test_null_handles_rejected():
    lib = B.lib()
    assert lib.cam_merge_begin(None, 0, 0, None) == B.E_ARG
    assert lib.cam_merge_accumulate(None, None, 0, 0) == B.E_ARG
    assert lib.cam_merge_fold(None, None, 0, 0, 0, None) == B.E_ARG
    assert lib.cam_merge_finalize(None, 0, 1.0, 0.0) == B.E_ARG
    assert lib.cam_ema_update(None, 0.9) == B.E_ARG
    assert lib.cam_drift_norm(None, None, None) == B.E_ARG
    assert lib.cam_merge_commit(None, None) == B.E_ARG
    assert lib.cam_merge_round(None, 0, 0, 1, None, 0, None, 0, 1.0, 0.0, 0, 0.0, None, None,
                               None) == B.E_ARG
    assert lib.cam_merge_abort(None) == B.E_ARG
    assert lib.cam_ctx_status(None, None) == B.E_ARG
    assert lib.cam_ctx_staged_count(None, None) == B.E_ARG
    assert lib.cam_ctx_last_commit(None, None) == B.E_ARG
    assert lib.cam_stream_capturing(None, None) == B.E_ARG
    assert lib.cam_ctx_get_quorum(None, None) == B.E_ARG
    assert lib.cam_ctx_set_quorum(None, 1) == B.E_ARG
    assert "NULL" in B.last_error()
    lib.cam_ctx_destroy(None)  # no-op


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the GPU-less failure")
def test_no_staging_flag_is_a_valid_description():
    # the description passes validation; only the missing device stops it
    with pytest.raises(B.CudaError):
        B.ctx_create([16], [0x10000], flags=B.NO_STAGING | B.TIME_COMMITS)


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the GPU-less failure")
def test_no_gpu_fails_loudly():
    with pytest.raises(B.CudaError) as ei:
        B.ctx_create([16], [0x10000])
    assert "CUDA" in str(ei.value) or "cuda" in str(ei.value)


def test_noalloc_sizes_beyond_the_scratch_rejected_before_cuda():
    """cam_merge_round_noalloc refuses rounds its fixed scratch cannot hold on
    the host, before any CUDA call: the pointers below are never read, so
    none of them needs to be real device memory."""
    n_t = B.NOALLOC_MAX_TENSORS + 1
    ptrs = [0x10000 + 64 * i for i in range(n_t)]
    with pytest.raises(B.ArgError, match="n_tensors"):
        B.merge_round_noalloc([8] * n_t, ptrs, [ptrs], B.F32, B.MEAN_REPLACE)
    # one tensor cut into more chunks of at most 16,384 elements than the
    # scratch has partials for
    n = B.NOALLOC_MAX_CHUNKS * 16384 + 1
    with pytest.raises(B.ArgError, match="too large"):
        B.merge_round_noalloc([n], [0x10000], [[0x20000]], B.BF16, B.MEAN_REPLACE)
    # the same limit summed over several tensors
    k = 1 << 20
    count = B.NOALLOC_MAX_CHUNKS // 64 + 1
    with pytest.raises(B.ArgError, match="too large"):
        B.merge_round_noalloc([k] * count, [0x10000 + 64 * i for i in range(count)],
                              [[0x20000 + 64 * i for i in range(count)]], B.F32, B.MEAN_REPLACE)


def test_missing_library_is_an_error(monkeypatch, tmp_path):
    monkeypatch.setattr(B, "_lib", None)
    monkeypatch.setattr(B, "LIB_PATH", str(tmp_path / "libcam.so"))
    with pytest.raises(RuntimeError, match="missing"):
        B.lib()
