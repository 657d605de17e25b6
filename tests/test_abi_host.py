"""Host-side checks of the C ABI, which run without a GPU.

The library must build and load, and it must export every function that include/mamba_scan.h
declares. The size queries are checked against hand counts, and argument validation must
reject bad calls with the documented codes before it touches CUDA. The pointers here are fake
integers that every call rejects during validation. These tests never run where a GPU is
visible: a GPU run must never see a fake pointer.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _header_functions():
    with open(os.path.join(ROOT, "include", "mamba_scan.h")) as f:
        src = f.read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mamba_(?:scan|conv)_\w+)\s*\(", src)))


@pytest.fixture(scope="module")
def ms():
    import __graft_entry__
    __graft_entry__.build()
    import selective_state_space_06_gb300 as m
    return m


def test_header_declares_expected_entry_points():
    fns = _header_functions()
    for f in ("mamba_scan_fwd", "mamba_scan_bwd", "mamba_scan_ckpt_bytes",
              "mamba_scan_scratch_bytes", "mamba_scan_status", "mamba_scan_strerror"):
        assert f in fns


def test_library_exports_every_declared_symbol(ms):
    lib = ctypes.CDLL(ms.LIB_PATH)
    for f in _header_functions():
        assert hasattr(lib, f), f"{f} declared in mamba_scan.h but not exported"
    assert set(_header_functions()) <= set(ms.EXPORTED)


def test_buffer_sizes(ms):
    # checkpoint buffer: the state after every 16-step chunk except the last ([b][chunk][d][n]
    # fp32), the forward's per-segment aggregates, and y [b][T][d] for the backward's d_gate
    states = 8 * (1024 // 16 - 1) * 1536 * 16 * 4
    y = 8 * 1024 * 1536 * 4
    ck = ms.mamba_scan_ckpt_bytes(8, 1024, 1536, 16)
    assert states + y <= ck <= 2 * (states + y) and ck % 256 == 0
    assert ms.mamba_scan_ckpt_bytes(1, 16, 32, 16) == 16 * 32 * 4     # one chunk: y only
    assert ms.mamba_scan_ckpt_bytes(1, 17, 32, 16) >= 1 * 1 * 32 * 16 * 4 + 17 * 32 * 4
    assert ms.mamba_scan_ckpt_bytes(0, 16, 32, 16) == 0
    sc = ms.mamba_scan_scratch_bytes(2, 100, 130, 16)
    nblk = -(-130 // 64)
    assert sc >= 4 * (2 * nblk * 2 * 100 * 16 + 2 * 2 * 130 * 16 + 2 * 2 * 130)
    assert sc % 256 == 0
    assert ms.mamba_scan_scratch_bytes(1, 1, 1, 65) == 0
    assert ms.mamba_scan_host_workspace_bytes(1, 64, 32, 16) >= 4 * (8 * 64 * 32 + 4 * 64 * 16)


def test_strerror(ms):
    for code in range(0, 8):
        assert isinstance(ms.mamba_scan_strerror(code), str) and ms.mamba_scan_strerror(code)
    assert "unknown" in ms.mamba_scan_strerror(99)


def _no_gpu():
    try:
        import torch
        return not torch.cuda.is_available()
    except Exception:
        return True


needs_no_gpu = pytest.mark.skipif(not _no_gpu(), reason="fake-pointer validation tests run only without a GPU")

A = 0x10000   # fake, 16-byte aligned "device" addresses (validation rejects before any use)


def _fwd_args(**over):
    b, T, Di, N = over.pop("dims", (2, 40, 64, 16))
    ptr = {k: A * (i + 1) for i, k in enumerate(("delta", "u", "B", "C", "gate", "A_log", "D", "out", "y", "ckpt"))}
    ptr.update(over)
    ck = over.get("ckpt_bytes", 10 ** 9)
    return [ptr["delta"], ptr["u"], ptr["B"], ptr["C"], ptr["gate"], ptr["A_log"], ptr["D"],
            ptr["out"], ptr["y"], ptr["ckpt"], ck, b, T, Di, N, None]


@needs_no_gpu
def test_fwd_validation_codes(ms):
    lib = ms.raw_library()
    assert lib.mamba_scan_fwd(*_fwd_args(delta=None)) == ms.MAMBA_ERR_INVALID_ARG
    assert lib.mamba_scan_fwd(*_fwd_args(out=None)) == ms.MAMBA_ERR_INVALID_ARG
    assert lib.mamba_scan_fwd(*_fwd_args(u=A + 4)) == ms.MAMBA_ERR_MISALIGNED
    assert lib.mamba_scan_fwd(*_fwd_args(ckpt_bytes=16)) == ms.MAMBA_ERR_WORKSPACE
    assert lib.mamba_scan_fwd(*_fwd_args(dims=(0, 40, 64, 16))) == ms.MAMBA_ERR_INVALID_ARG
    assert lib.mamba_scan_fwd(*_fwd_args(dims=(1, 40, 64, 65))) == ms.MAMBA_ERR_UNSUPPORTED
    assert lib.mamba_scan_fwd(*_fwd_args(dims=(70000, 1, 1, 16))) == ms.MAMBA_ERR_INVALID_ARG
    assert lib.mamba_scan_fwd(*_fwd_args(dims=(1, 1 << 20, 1 << 12, 16))) == ms.MAMBA_ERR_INVALID_ARG
    # out overlapping y
    assert lib.mamba_scan_fwd(*_fwd_args(y=A * 8 + 256)) == ms.MAMBA_ERR_INVALID_ARG
    # checkpoint needed (T > 16) but NULL
    assert lib.mamba_scan_fwd(*_fwd_args(ckpt=None)) == ms.MAMBA_ERR_INVALID_ARG


def _bwd_args(**over):
    b, T, Di, N = over.pop("dims", (2, 40, 64, 16))
    big = 1 << 32
    names = ("delta", "u", "B", "C", "gate", "A_log", "D", "dy", "ckpt", "scratch",
             "d_delta", "d_u", "d_B", "d_C", "d_A_log", "d_D", "d_gate")
    ptr = {k: big * (i + 1) for i, k in enumerate(names)}
    ptr.update(over)
    return [ptr["delta"], ptr["u"], ptr["B"], ptr["C"], ptr["gate"], ptr["A_log"], ptr["D"],
            ptr["dy"], ptr["ckpt"], over.get("ckpt_bytes", 10 ** 9), ptr["scratch"],
            over.get("scratch_bytes", 10 ** 9), ptr["d_delta"], ptr["d_u"], ptr["d_B"],
            ptr["d_C"], ptr["d_A_log"], ptr["d_D"], ptr["d_gate"], b, T, Di, N, None]


@needs_no_gpu
def test_bwd_validation_codes(ms):
    lib = ms.raw_library()
    big = 1 << 32
    assert lib.mamba_scan_bwd(*_bwd_args(dy=None)) == ms.MAMBA_ERR_INVALID_ARG
    assert lib.mamba_scan_bwd(*_bwd_args(scratch=None)) == ms.MAMBA_ERR_INVALID_ARG
    assert lib.mamba_scan_bwd(*_bwd_args(d_C=big * 14 + 8)) == ms.MAMBA_ERR_MISALIGNED
    assert lib.mamba_scan_bwd(*_bwd_args(scratch_bytes=1024)) == ms.MAMBA_ERR_WORKSPACE
    assert lib.mamba_scan_bwd(*_bwd_args(ckpt_bytes=0)) == ms.MAMBA_ERR_WORKSPACE
    # two gradients at the same address
    assert lib.mamba_scan_bwd(*_bwd_args(d_u=big * 11)) == ms.MAMBA_ERR_INVALID_ARG
    # scratch overlapping a gradient
    assert lib.mamba_scan_bwd(*_bwd_args(scratch=big * 13 + 64)) == ms.MAMBA_ERR_INVALID_ARG
    assert lib.mamba_scan_bwd(*_bwd_args(dims=(1, 40, 64, 100))) == ms.MAMBA_ERR_UNSUPPORTED


@needs_no_gpu
def test_bwd_test_timeout_takes_only_the_tensor_copy_path(ms):
    """The failure-path test entry point validates like mamba_scan_bwd and refuses sizes that do
    not run the tensor-memory backward with tensor copies, before anything is launched."""
    lib = ms.raw_library()
    f = lib.mamba_scan_bwd_test_timeout
    assert f(*_bwd_args(dims=(1, 40, 64, 8))) == ms.MAMBA_ERR_UNSUPPORTED    # d_state <= 8
    assert f(*_bwd_args(dims=(1, 40, 66, 16))) == ms.MAMBA_ERR_UNSUPPORTED   # d_inner % 4
    assert f(*_bwd_args(dims=(1, 16, 64, 16))) == ms.MAMBA_ERR_UNSUPPORTED   # one chunk
    assert f(*_bwd_args(dims=(1, 40, 64, 100))) == ms.MAMBA_ERR_UNSUPPORTED
    assert f(*_bwd_args(dy=None)) == ms.MAMBA_ERR_INVALID_ARG
    assert f(*_bwd_args(scratch_bytes=1024)) == ms.MAMBA_ERR_WORKSPACE


@needs_no_gpu
def test_fwd_test_timeout_takes_only_the_tensor_copy_path(ms):
    """The forward's failure-path test entry point validates like mamba_scan_fwd and refuses
    sizes that do not run the forward with tensor copies (d_state 33..64, d_inner and d_state
    multiples of 4, more than one chunk), before anything is launched."""
    lib = ms.raw_library()
    f = lib.mamba_scan_fwd_test_timeout
    assert f(*_fwd_args(dims=(1, 40, 64, 16))) == ms.MAMBA_ERR_UNSUPPORTED    # d_state 16
    assert f(*_fwd_args(dims=(1, 40, 64, 32))) == ms.MAMBA_ERR_UNSUPPORTED    # d_state 32
    assert f(*_fwd_args(dims=(1, 40, 66, 64))) == ms.MAMBA_ERR_UNSUPPORTED    # d_inner % 4
    assert f(*_fwd_args(dims=(1, 40, 64, 62))) == ms.MAMBA_ERR_UNSUPPORTED    # d_state % 4
    assert f(*_fwd_args(dims=(1, 16, 64, 64))) == ms.MAMBA_ERR_UNSUPPORTED    # one chunk
    assert f(*_fwd_args(dims=(1, 40, 64, 100))) == ms.MAMBA_ERR_UNSUPPORTED
    assert f(*_fwd_args(dims=(1, 40, 64, 64), delta=None)) == ms.MAMBA_ERR_INVALID_ARG
    assert f(*_fwd_args(dims=(1, 40, 64, 64), ckpt_bytes=64)) == ms.MAMBA_ERR_WORKSPACE


def _fused_args(**over):
    b, T, Di, N = over.pop("dims", (2, 40, 64, 16))
    big = 1 << 32
    names = ("delta", "u", "B", "C", "gate", "A_log", "D", "dy", "out", "ckpt", "scratch",
             "d_delta", "d_u", "d_B", "d_C", "d_A_log", "d_D", "d_gate")
    ptr = {k: big * (i + 1) for i, k in enumerate(names)}
    ptr.update(over)
    return [ptr["delta"], ptr["u"], ptr["B"], ptr["C"], ptr["gate"], ptr["A_log"], ptr["D"],
            ptr["dy"], ptr["out"], ptr["ckpt"], over.get("ckpt_bytes", 10 ** 9), ptr["scratch"],
            over.get("scratch_bytes", 10 ** 9), ptr["d_delta"], ptr["d_u"], ptr["d_B"],
            ptr["d_C"], ptr["d_A_log"], ptr["d_D"], ptr["d_gate"], b, T, Di, N, None]


@needs_no_gpu
def test_fused_validation_codes(ms):
    """mamba_scan_fwd_bwd checks everything, out included, before its first launch."""
    lib = ms.raw_library()
    big = 1 << 32
    f = lib.mamba_scan_fwd_bwd
    assert f(*_fused_args(out=None)) == ms.MAMBA_ERR_INVALID_ARG
    assert f(*_fused_args(out=big * 9 + 8)) == ms.MAMBA_ERR_MISALIGNED
    assert f(*_fused_args(out=big * 12)) == ms.MAMBA_ERR_INVALID_ARG          # out == d_delta
    assert f(*_fused_args(scratch_bytes=1024)) == ms.MAMBA_ERR_WORKSPACE
    assert f(*_fused_args(dims=(1, 40, 64, 65))) == ms.MAMBA_ERR_UNSUPPORTED


@needs_no_gpu
def test_fused_bf16_validation_codes(ms):
    """The bf16 fused call: sizes it does not take are refused before any launch, and the
    overlap checks use 2-byte elements for the bf16 tensors."""
    lib = ms.raw_library()
    big = 1 << 32
    f = lib.mamba_scan_fwd_bwd_bf16
    for dims in ((2, 40, 64, 8), (2, 40, 36, 16), (2, 16, 64, 16), (2, 40, 64, 20)):
        assert f(*_fused_args(dims=dims)) == ms.MAMBA_ERR_UNSUPPORTED, dims
    btd16 = 2 * 40 * 64 * 2                                        # bytes of a bf16 [2, 40, 64]
    # d_u right after out in bf16: no overlap, so validation passes and the launch itself
    # fails here, where there is no device
    assert f(*_fused_args(d_u=big * 9 + btd16)) == ms.MAMBA_ERR_CUDA
    assert f(*_fused_args(d_u=big * 9 + btd16 - 16)) == ms.MAMBA_ERR_INVALID_ARG


@needs_no_gpu
def test_host_entry_validation(ms):
    lib = ms.raw_library()
    args = [A * (i + 1) for i in range(16)] + [A * 40, 16, 1, 64, 32, 16, None]
    assert lib.mamba_scan_fwd_bwd_host(*args) == ms.MAMBA_ERR_WORKSPACE
    args[16] = A * 40 + 8
    args[17] = 1 << 40
    assert lib.mamba_scan_fwd_bwd_host(*args) == ms.MAMBA_ERR_MISALIGNED
    args[3] = None
    assert lib.mamba_scan_fwd_bwd_host(*args) == ms.MAMBA_ERR_INVALID_ARG


def test_binding_rejects_cpu_tensors(ms):
    torch = pytest.importorskip("torch")
    t = torch.zeros(1, 4, 4)
    with pytest.raises(ValueError):
        ms.mamba_scan_fwd(t, t, torch.zeros(1, 4, 16), torch.zeros(1, 4, 16), t,
                          torch.zeros(4, 16), torch.zeros(4), t)


def test_default_build_is_unchecked(ms):
    # the bounds-checked build is a separate library; the default one has no shrink hook and
    # refuses it before touching CUDA
    assert not ms.mamba_scan_bounds_checked()
    lib = ms.raw_library()
    assert lib.mamba_scan_test_bounds_shrink(1) == ms.MAMBA_ERR_UNSUPPORTED
    assert lib.mamba_scan_test_bounds_shrink(-1) == ms.MAMBA_ERR_UNSUPPORTED
    assert "bounds-checked build" in ms.mamba_scan_strerror(ms.MAMBA_ERR_BOUNDS)
