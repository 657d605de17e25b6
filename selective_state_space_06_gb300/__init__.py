"""Python binding of libmambascan.so, the GB300 selective-scan library.

The binding only marshals arguments. Every step of the scan runs in the library's CUDA kernels.
There is no fallback of any kind: if the library has not been built, importing this package
raises ImportError. To build it, run ``python selective_state_space_06_gb300/build.py`` or
``__graft_entry__.build()``.

The functions mirror the C ABI in include/mamba_scan.h and keep its names:
  mamba_scan_ckpt_bytes, mamba_scan_scratch_bytes, mamba_scan_fwd, mamba_scan_bwd,
  mamba_scan_host_workspace_bytes, mamba_scan_fwd_bwd_host, mamba_scan_status,
  mamba_scan_strerror, mamba_scan_last_launch_count, mamba_scan_bounds_checked,
  mamba_scan_test_bounds_shrink (the bounds-checked build: checked_library(), using_library()).
Tensor arguments are torch tensors: float32, contiguous, on a CUDA device. The host entry point
takes CPU tensors instead. ``stream`` defaults to torch's current stream on the tensors' device.
Nonzero return codes raise MambaScanError.
"""
from __future__ import annotations

import contextlib
import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmambascan.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it with `python selective_state_space_06_gb300/build.py` "
        "(nvcc, sm_103a). This package has no CPU or Python fallback.")

_lib = ctypes.CDLL(LIB_PATH)

MAMBA_OK = 0
MAMBA_ERR_INVALID_ARG = 1
MAMBA_ERR_MISALIGNED = 2
MAMBA_ERR_WORKSPACE = 3
MAMBA_ERR_CUDA = 4
MAMBA_ERR_UNSUPPORTED = 5
MAMBA_ERR_NOALLOC_LIMIT = 6
MAMBA_ERR_TIMEOUT = 7
MAMBA_ERR_BOUNDS = 8
MAMBA_SCAN_NOALLOC_SCRATCH_BYTES = 64 << 20

EXPORTED = (
    "mamba_scan_ckpt_bytes", "mamba_scan_scratch_bytes", "mamba_scan_fwd", "mamba_scan_bwd",
    "mamba_scan_host_workspace_bytes", "mamba_scan_fwd_bwd_host", "mamba_scan_status",
    "mamba_scan_strerror", "mamba_scan_last_launch_count", "mamba_scan_bwd_noalloc",
    "mamba_scan_fwd_softplus", "mamba_scan_bwd_softplus", "mamba_scan_fwd_bwd",
    "mamba_scan_fwd_bwd_bf16", "mamba_scan_bwd_test_timeout", "mamba_scan_fwd_test_timeout",
    "mamba_conv_scratch_bytes", "mamba_conv_fwd", "mamba_conv_bwd",
    "mamba_scan_bounds_checked", "mamba_scan_test_bounds_shrink",
)

_vp = ctypes.c_void_p
_i64 = ctypes.c_int64
_sz = ctypes.c_size_t


def _configure(lib: ctypes.CDLL) -> ctypes.CDLL:
    """Sets the argument and result types of every exported function of ``lib``."""
    lib.mamba_scan_ckpt_bytes.argtypes = [_i64] * 4
    lib.mamba_scan_ckpt_bytes.restype = _sz
    lib.mamba_scan_scratch_bytes.argtypes = [_i64] * 4
    lib.mamba_scan_scratch_bytes.restype = _sz
    lib.mamba_scan_host_workspace_bytes.argtypes = [_i64] * 4
    lib.mamba_scan_host_workspace_bytes.restype = _sz
    lib.mamba_scan_fwd.argtypes = [_vp] * 10 + [_sz] + [_i64] * 4 + [_vp]
    lib.mamba_scan_fwd.restype = ctypes.c_int
    lib.mamba_scan_bwd.argtypes = [_vp] * 9 + [_sz, _vp, _sz] + [_vp] * 7 + [_i64] * 4 + [_vp]
    lib.mamba_scan_bwd.restype = ctypes.c_int
    lib.mamba_conv_scratch_bytes.argtypes = [_i64] * 4
    lib.mamba_conv_scratch_bytes.restype = _sz
    lib.mamba_conv_fwd.argtypes = [_vp] * 4 + [_i64] * 4 + [_vp]
    lib.mamba_conv_fwd.restype = ctypes.c_int
    lib.mamba_conv_bwd.argtypes = [_vp] * 5 + [_sz] + [_vp] * 3 + [_i64] * 4 + [_vp]
    lib.mamba_conv_bwd.restype = ctypes.c_int
    lib.mamba_scan_fwd_softplus.argtypes = lib.mamba_scan_fwd.argtypes
    lib.mamba_scan_fwd_softplus.restype = ctypes.c_int
    lib.mamba_scan_bwd_softplus.argtypes = lib.mamba_scan_bwd.argtypes
    lib.mamba_scan_bwd_softplus.restype = ctypes.c_int
    lib.mamba_scan_bwd_test_timeout.argtypes = lib.mamba_scan_bwd.argtypes
    lib.mamba_scan_fwd_test_timeout.argtypes = lib.mamba_scan_fwd.argtypes
    lib.mamba_scan_fwd_test_timeout.restype = ctypes.c_int
    lib.mamba_scan_bwd_test_timeout.restype = ctypes.c_int
    lib.mamba_scan_fwd_bwd.argtypes = [_vp] * 10 + [_sz, _vp, _sz] + [_vp] * 7 + [_i64] * 4 + [_vp]
    lib.mamba_scan_fwd_bwd.restype = ctypes.c_int
    lib.mamba_scan_fwd_bwd_bf16.argtypes = lib.mamba_scan_fwd_bwd.argtypes
    lib.mamba_scan_fwd_bwd_bf16.restype = ctypes.c_int
    lib.mamba_scan_bwd_noalloc.argtypes = [_vp] * 9 + [_sz] + [_vp] * 7 + [_i64] * 4 + [_vp]
    lib.mamba_scan_bwd_noalloc.restype = ctypes.c_int
    lib.mamba_scan_fwd_bwd_host.argtypes = [_vp] * 17 + [_sz] + [_i64] * 4 + [_vp]
    lib.mamba_scan_fwd_bwd_host.restype = ctypes.c_int
    lib.mamba_scan_status.argtypes = [_vp]
    lib.mamba_scan_status.restype = ctypes.c_int
    lib.mamba_scan_strerror.argtypes = [ctypes.c_int]
    lib.mamba_scan_strerror.restype = ctypes.c_char_p
    lib.mamba_scan_last_launch_count.argtypes = []
    lib.mamba_scan_last_launch_count.restype = ctypes.c_int
    lib.mamba_scan_bounds_checked.argtypes = []
    lib.mamba_scan_bounds_checked.restype = ctypes.c_int
    lib.mamba_scan_test_bounds_shrink.argtypes = [_i64]
    lib.mamba_scan_test_bounds_shrink.restype = ctypes.c_int
    return lib


_configure(_lib)


class MambaScanError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: error {code}: {mamba_scan_strerror(code)}")


def raw_library() -> ctypes.CDLL:
    """The ctypes handle of libmambascan.so (for callers that pass raw pointers)."""
    return _lib


def mamba_scan_strerror(code: int) -> str:
    return _lib.mamba_scan_strerror(int(code)).decode()


CHECKED_LIB_PATH = os.path.join(_HERE, "libmambascan_checked.so")


def checked_library() -> ctypes.CDLL:
    """The ctypes handle of the bounds-checked build (libmambascan_checked.so: the same sources
    compiled with -DMAMBA_BOUNDS_CHECK, built by ``build.build(checked=True)``), with the same
    function signatures as the default library."""
    if not os.path.exists(CHECKED_LIB_PATH):
        raise ImportError(f"{CHECKED_LIB_PATH} is missing: build it with build.build(checked=True)")
    return _configure(ctypes.CDLL(CHECKED_LIB_PATH))


@contextlib.contextmanager
def using_library(lib: ctypes.CDLL):
    """Routes every function of this module through ``lib`` (for instance checked_library())
    inside the ``with`` block; the default library again afterwards."""
    global _lib
    old = _lib
    _lib = lib
    try:
        yield lib
    finally:
        _lib = old


def mamba_scan_bounds_checked() -> bool:
    return bool(_lib.mamba_scan_bounds_checked())


def mamba_scan_test_bounds_shrink(elements: int) -> None:
    rc = _lib.mamba_scan_test_bounds_shrink(int(elements))
    if rc != MAMBA_OK:
        raise MambaScanError(rc, "mamba_scan_test_bounds_shrink")


def mamba_scan_ckpt_bytes(batch: int, T: int, d_inner: int, d_state: int) -> int:
    return int(_lib.mamba_scan_ckpt_bytes(batch, T, d_inner, d_state))


def mamba_scan_scratch_bytes(batch: int, T: int, d_inner: int, d_state: int) -> int:
    return int(_lib.mamba_scan_scratch_bytes(batch, T, d_inner, d_state))


def mamba_scan_host_workspace_bytes(batch: int, T: int, d_inner: int, d_state: int) -> int:
    return int(_lib.mamba_scan_host_workspace_bytes(batch, T, d_inner, d_state))


def mamba_scan_last_launch_count() -> int:
    return int(_lib.mamba_scan_last_launch_count())


def _ptr(t, name, device=None, allow_none=False, host=False, dtype=None):
    if t is None:
        if allow_none:
            return None
        raise ValueError(f"{name} is required")
    import torch
    want = torch.float32 if dtype is None else dtype
    if t.dtype != want and name not in ("ckpt", "scratch", "workspace"):
        raise TypeError(f"{name} must be {want}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if host:
        if t.is_cuda:
            raise ValueError(f"{name} must be a host (CPU) tensor")
    else:
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if device is not None and t.device != device:
            raise ValueError(f"{name} is on {t.device}, expected {device}")
    return t.data_ptr()


def _stream_ptr(stream, device):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(device)
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dims(delta, B):
    if delta.dim() != 3 or B.dim() != 3:
        raise ValueError("delta must be [batch, T, d_inner] and B must be [batch, T, d_state]")
    b, T, Di = delta.shape
    return int(b), int(T), int(Di), int(B.shape[2])


def mamba_scan_fwd(delta, u, B, C, gate, A_log, D, out, y=None, ckpt=None, stream=None,
                   _fn="mamba_scan_fwd"):
    """Forward scan on device tensors. ``ckpt`` is a device buffer (any dtype) of at least
    mamba_scan_ckpt_bytes bytes, or None when that size is 0."""
    b, T, Di, N = _dims(delta, B)
    dev = delta.device
    ck_bytes = 0 if ckpt is None else ckpt.numel() * ckpt.element_size()
    rc = getattr(_lib, _fn)(
        _ptr(delta, "delta", dev), _ptr(u, "u", dev), _ptr(B, "B", dev), _ptr(C, "C", dev),
        _ptr(gate, "gate", dev), _ptr(A_log, "A_log", dev), _ptr(D, "D", dev),
        _ptr(out, "out", dev), _ptr(y, "y", dev, allow_none=True),
        _ptr(ckpt, "ckpt", dev, allow_none=True), ck_bytes, b, T, Di, N, _stream_ptr(stream, dev))
    if rc != MAMBA_OK:
        raise MambaScanError(rc, _fn)


def mamba_scan_fwd_softplus(delta_raw, u, B, C, gate, A_log, D, out, y=None, ckpt=None,
                            stream=None):
    """mamba_scan_fwd with delta = softplus(delta_raw) applied inside the kernels."""
    mamba_scan_fwd(delta_raw, u, B, C, gate, A_log, D, out, y, ckpt, stream,
                   _fn="mamba_scan_fwd_softplus")


def mamba_scan_bwd(delta, u, B, C, gate, A_log, D, dy, ckpt, scratch, d_delta, d_u, d_B, d_C,
                   d_A_log, d_D, d_gate, stream=None, _fn="mamba_scan_bwd"):
    """Backward scan on device tensors (all seven gradients are overwritten)."""
    b, T, Di, N = _dims(delta, B)
    dev = delta.device
    ck_bytes = 0 if ckpt is None else ckpt.numel() * ckpt.element_size()
    rc = getattr(_lib, _fn)(
        _ptr(delta, "delta", dev), _ptr(u, "u", dev), _ptr(B, "B", dev), _ptr(C, "C", dev),
        _ptr(gate, "gate", dev), _ptr(A_log, "A_log", dev), _ptr(D, "D", dev),
        _ptr(dy, "dy", dev), _ptr(ckpt, "ckpt", dev, allow_none=True), ck_bytes,
        _ptr(scratch, "scratch", dev), scratch.numel() * scratch.element_size(),
        _ptr(d_delta, "d_delta", dev), _ptr(d_u, "d_u", dev), _ptr(d_B, "d_B", dev),
        _ptr(d_C, "d_C", dev), _ptr(d_A_log, "d_A_log", dev), _ptr(d_D, "d_D", dev),
        _ptr(d_gate, "d_gate", dev), b, T, Di, N, _stream_ptr(stream, dev))
    if rc != MAMBA_OK:
        raise MambaScanError(rc, _fn)


def mamba_scan_bwd_softplus(delta_raw, u, B, C, gate, A_log, D, dy, ckpt, scratch, d_delta_raw,
                            d_u, d_B, d_C, d_A_log, d_D, d_gate, stream=None):
    """mamba_scan_bwd for the softplus variant: d_delta_raw receives the gradient with respect
    to the raw delta."""
    mamba_scan_bwd(delta_raw, u, B, C, gate, A_log, D, dy, ckpt, scratch, d_delta_raw, d_u, d_B,
                   d_C, d_A_log, d_D, d_gate, stream, _fn="mamba_scan_bwd_softplus")


def mamba_scan_fwd_test_timeout(delta, u, B, C, gate, A_log, D, out, y=None, ckpt=None,
                                stream=None):
    """Failure-path test only: mamba_scan_fwd with the copies of each CTA's last chunk left
    unissued and 1 ms copy waits, so that the next mamba_scan_status raises MAMBA_ERR_TIMEOUT."""
    mamba_scan_fwd(delta, u, B, C, gate, A_log, D, out, y, ckpt, stream,
                   _fn="mamba_scan_fwd_test_timeout")


def mamba_scan_bwd_test_timeout(delta, u, B, C, gate, A_log, D, dy, ckpt, scratch, d_delta,
                                d_u, d_B, d_C, d_A_log, d_D, d_gate, stream=None):
    """Failure-path test only: mamba_scan_bwd with the copies of each CTA's last chunk left
    unissued and 1 ms copy waits, so that the next mamba_scan_status raises MAMBA_ERR_TIMEOUT."""
    mamba_scan_bwd(delta, u, B, C, gate, A_log, D, dy, ckpt, scratch, d_delta, d_u, d_B, d_C,
                   d_A_log, d_D, d_gate, stream, _fn="mamba_scan_bwd_test_timeout")


def mamba_scan_fwd_bwd(delta, u, B, C, gate, A_log, D, dy, out, ckpt, scratch, d_delta, d_u,
                       d_B, d_C, d_A_log, d_D, d_gate, stream=None):
    """Forward and backward in one call when dy is known up front: writes out and all seven
    gradients (y is not returned). The same checkpoint and scratch buffers as the separate
    calls."""
    b, T, Di, N = _dims(delta, B)
    dev = delta.device
    ck_bytes = 0 if ckpt is None else ckpt.numel() * ckpt.element_size()
    rc = _lib.mamba_scan_fwd_bwd(
        _ptr(delta, "delta", dev), _ptr(u, "u", dev), _ptr(B, "B", dev), _ptr(C, "C", dev),
        _ptr(gate, "gate", dev), _ptr(A_log, "A_log", dev), _ptr(D, "D", dev),
        _ptr(dy, "dy", dev), _ptr(out, "out", dev), _ptr(ckpt, "ckpt", dev, allow_none=True),
        ck_bytes, _ptr(scratch, "scratch", dev), scratch.numel() * scratch.element_size(),
        _ptr(d_delta, "d_delta", dev), _ptr(d_u, "d_u", dev), _ptr(d_B, "d_B", dev),
        _ptr(d_C, "d_C", dev), _ptr(d_A_log, "d_A_log", dev), _ptr(d_D, "d_D", dev),
        _ptr(d_gate, "d_gate", dev), b, T, Di, N, _stream_ptr(stream, dev))
    if rc != MAMBA_OK:
        raise MambaScanError(rc, "mamba_scan_fwd_bwd")


def mamba_scan_fwd_bwd_bf16(delta, u, B, C, gate, A_log, D, dy, out, ckpt, scratch, d_delta,
                            d_u, d_B, d_C, d_A_log, d_D, d_gate, stream=None):
    """mamba_scan_fwd_bwd with bf16 I/O: delta, u, B, C, gate, dy, out, d_delta, d_u, d_B, d_C
    and d_gate are torch.bfloat16; A_log, D, d_A_log, d_D float32. Needs 9 <= d_state <= 64,
    d_inner and d_state multiples of 8 and T > 16."""
    import torch
    b, T, Di, N = _dims(delta, B)
    dev = delta.device
    h = dict(dtype=torch.bfloat16)
    ck_bytes = 0 if ckpt is None else ckpt.numel() * ckpt.element_size()
    rc = _lib.mamba_scan_fwd_bwd_bf16(
        _ptr(delta, "delta", dev, **h), _ptr(u, "u", dev, **h), _ptr(B, "B", dev, **h),
        _ptr(C, "C", dev, **h), _ptr(gate, "gate", dev, **h), _ptr(A_log, "A_log", dev),
        _ptr(D, "D", dev), _ptr(dy, "dy", dev, **h), _ptr(out, "out", dev, **h),
        _ptr(ckpt, "ckpt", dev, allow_none=True), ck_bytes, _ptr(scratch, "scratch", dev),
        scratch.numel() * scratch.element_size(), _ptr(d_delta, "d_delta", dev, **h),
        _ptr(d_u, "d_u", dev, **h), _ptr(d_B, "d_B", dev, **h), _ptr(d_C, "d_C", dev, **h),
        _ptr(d_A_log, "d_A_log", dev), _ptr(d_D, "d_D", dev), _ptr(d_gate, "d_gate", dev, **h),
        b, T, Di, N, _stream_ptr(stream, dev))
    if rc != MAMBA_OK:
        raise MambaScanError(rc, "mamba_scan_fwd_bwd_bf16")


def mamba_scan_bwd_noalloc(delta, u, B, C, gate, A_log, D, dy, ckpt, d_delta, d_u, d_B, d_C,
                           d_A_log, d_D, d_gate, stream=None):
    """Backward scan without a scratch argument, for callers that may not allocate device
    memory. Scratch comes from the library's static 64 MiB device array, shared by every call
    on the device; calls that overlap on the GPU race on it."""
    b, T, Di, N = _dims(delta, B)
    dev = delta.device
    ck_bytes = 0 if ckpt is None else ckpt.numel() * ckpt.element_size()
    rc = _lib.mamba_scan_bwd_noalloc(
        _ptr(delta, "delta", dev), _ptr(u, "u", dev), _ptr(B, "B", dev), _ptr(C, "C", dev),
        _ptr(gate, "gate", dev), _ptr(A_log, "A_log", dev), _ptr(D, "D", dev),
        _ptr(dy, "dy", dev), _ptr(ckpt, "ckpt", dev, allow_none=True), ck_bytes,
        _ptr(d_delta, "d_delta", dev), _ptr(d_u, "d_u", dev), _ptr(d_B, "d_B", dev),
        _ptr(d_C, "d_C", dev), _ptr(d_A_log, "d_A_log", dev), _ptr(d_D, "d_D", dev),
        _ptr(d_gate, "d_gate", dev), b, T, Di, N, _stream_ptr(stream, dev))
    if rc != MAMBA_OK:
        raise MambaScanError(rc, "mamba_scan_bwd_noalloc")


def mamba_scan_fwd_bwd_host(delta, u, B, C, gate, A_log, D, dy, out, d_delta, d_u, d_B, d_C,
                            d_A_log, d_D, d_gate, workspace, stream=None):
    """End-to-end forward + backward from HOST tensors (ideally pinned) through a device
    workspace of mamba_scan_host_workspace_bytes bytes; returns after the results are on the
    host."""
    b, T, Di, N = _dims(delta, B)
    dev = workspace.device
    h = dict(host=True)
    rc = _lib.mamba_scan_fwd_bwd_host(
        _ptr(delta, "delta", **h), _ptr(u, "u", **h), _ptr(B, "B", **h), _ptr(C, "C", **h),
        _ptr(gate, "gate", **h), _ptr(A_log, "A_log", **h), _ptr(D, "D", **h), _ptr(dy, "dy", **h),
        _ptr(out, "out", **h), _ptr(d_delta, "d_delta", **h), _ptr(d_u, "d_u", **h),
        _ptr(d_B, "d_B", **h), _ptr(d_C, "d_C", **h), _ptr(d_A_log, "d_A_log", **h),
        _ptr(d_D, "d_D", **h), _ptr(d_gate, "d_gate", **h),
        _ptr(workspace, "workspace", dev), workspace.numel() * workspace.element_size(),
        b, T, Di, N, _stream_ptr(stream, dev))
    if rc != MAMBA_OK:
        raise MambaScanError(rc, "mamba_scan_fwd_bwd_host")


def mamba_scan_status(stream=None, device=None) -> None:
    import torch
    dev = device if device is not None else torch.device("cuda", torch.cuda.current_device())
    rc = _lib.mamba_scan_status(_stream_ptr(stream, dev))
    if rc != MAMBA_OK:
        raise MambaScanError(rc, "mamba_scan_status")


# ----------------------------------------------------------------------------------------------
# Convenience layer: allocate outputs and buffers with torch, then call the entry points above.
def alloc_like_outputs(delta, B, A_log, D):
    import torch
    b, T, Di, N = _dims(delta, B)
    dev = delta.device
    ck = mamba_scan_ckpt_bytes(b, T, Di, N)
    sc = mamba_scan_scratch_bytes(b, T, Di, N)
    e = lambda *s: torch.empty(*s, dtype=torch.float32, device=dev)  # noqa: E731
    return {
        "out": e(b, T, Di), "y": e(b, T, Di),
        "ckpt": torch.empty(max(ck, 16), dtype=torch.uint8, device=dev) if ck else None,
        "scratch": torch.empty(max(sc, 16), dtype=torch.uint8, device=dev),
        "d_delta": e(b, T, Di), "d_u": e(b, T, Di), "d_gate": e(b, T, Di),
        "d_B": e(b, T, N), "d_C": e(b, T, N), "d_A_log": e(Di, N), "d_D": e(Di),
    }


# ---- causal depthwise conv1d + SiLU (the step before the scan) -------------------------------
def mamba_conv_scratch_bytes(batch: int, T: int, d_inner: int, d_conv: int) -> int:
    return int(_lib.mamba_conv_scratch_bytes(batch, T, d_inner, d_conv))


def mamba_conv_fwd(x, w, bias, u, stream=None):
    """u = SiLU(causal depthwise conv1d(x, w) + bias); x, u [batch, T, d_inner], w
    [d_inner, d_conv], bias [d_inner] (device tensors)."""
    b, T, Di = x.shape
    K = w.shape[1]
    dev = x.device
    rc = _lib.mamba_conv_fwd(_ptr(x, "x", dev), _ptr(w, "w", dev), _ptr(bias, "bias", dev),
                             _ptr(u, "u", dev), b, T, Di, K, _stream_ptr(stream, dev))
    if rc != MAMBA_OK:
        raise MambaScanError(rc, "mamba_conv_fwd")


def mamba_conv_bwd(x, w, bias, d_u, scratch, d_x, d_w, d_bias, stream=None):
    """Backward of mamba_conv_fwd: d_x, d_w, d_bias (overwritten) from d_u."""
    b, T, Di = x.shape
    K = w.shape[1]
    dev = x.device
    rc = _lib.mamba_conv_bwd(_ptr(x, "x", dev), _ptr(w, "w", dev), _ptr(bias, "bias", dev),
                             _ptr(d_u, "d_u", dev), _ptr(scratch, "scratch", dev),
                             scratch.numel() * scratch.element_size(), _ptr(d_x, "d_x", dev),
                             _ptr(d_w, "d_w", dev), _ptr(d_bias, "d_bias", dev), b, T, Di, K,
                             _stream_ptr(stream, dev))
    if rc != MAMBA_OK:
        raise MambaScanError(rc, "mamba_conv_bwd")


def forward_backward(x: dict, bufs: dict | None = None, with_y: bool = True, stream=None,
                     softplus: bool = False) -> dict:
    """Runs mamba_scan_fwd then mamba_scan_bwd on a dict of device tensors (keys delta, u, B, C,
    gate, A_log, D, dy); returns the dict of outputs (out, y, d_delta, d_u, d_B, d_C, d_A_log,
    d_D, d_gate plus the ckpt/scratch buffers). With softplus=True, x["delta"] holds the raw
    delta, the _softplus entry points run, and bufs["d_delta"] receives d_delta_raw."""
    if bufs is None:
        bufs = alloc_like_outputs(x["delta"], x["B"], x["A_log"], x["D"])
    fwd = mamba_scan_fwd_softplus if softplus else mamba_scan_fwd
    bwd = mamba_scan_bwd_softplus if softplus else mamba_scan_bwd
    fwd(x["delta"], x["u"], x["B"], x["C"], x["gate"], x["A_log"], x["D"], bufs["out"],
        bufs["y"] if with_y else None, bufs["ckpt"], stream=stream)
    bwd(x["delta"], x["u"], x["B"], x["C"], x["gate"], x["A_log"], x["D"], x["dy"],
        bufs["ckpt"], bufs["scratch"], bufs["d_delta"], bufs["d_u"], bufs["d_B"],
        bufs["d_C"], bufs["d_A_log"], bufs["d_D"], bufs["d_gate"], stream=stream)
    return bufs
