"""fp64 sequential oracle of the selective scan: forward and reverse-time BPTT backward.

TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the bench's CPU-baseline leg may
import this package. The CUDA library and its Python binding never do.

The arithmetic lives in ``mamba_oracle.c`` (plain C, float64, one row (b, d) at a time, strictly
sequential in t). This module compiles it with gcc on first use and marshals numpy arrays. The
row-range interface lets a caller split rows across threads. Each thread then gets its own
accumulators, and ``bwd`` sums them in a fixed order. The arithmetic of any one row never changes.
"""
from __future__ import annotations

import concurrent.futures
import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mamba_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libmamba_oracle.so")
_lock = threading.Lock()
_default = None


def build(force: bool = False) -> str:
    """Compile the oracle into oracle/libmamba_oracle.so (gcc, -O2, no fast-math, no FMA
    contraction)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < max(
            os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "mamba_oracle.h"))):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
                               "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _bind(path):
    lib = ctypes.CDLL(path)
    dp = ctypes.POINTER(ctypes.c_double)
    i64 = ctypes.c_int64
    lib.mamba_oracle_fwd_rows.argtypes = [dp] * 7 + [i64] * 6 + [dp, dp]
    lib.mamba_oracle_fwd_rows.restype = ctypes.c_int
    lib.mamba_oracle_bwd_rows.argtypes = [dp] * 8 + [i64] * 6 + [dp] * 7
    lib.mamba_oracle_bwd_rows.restype = ctypes.c_int
    lib.mamba_oracle_softplus.argtypes = [dp, dp, i64]
    lib.mamba_oracle_softplus.restype = None
    lib.mamba_oracle_softplus_bwd.argtypes = [dp, dp, dp, i64]
    lib.mamba_oracle_softplus_bwd.restype = None
    lib.mamba_oracle_conv_fwd.argtypes = [dp] * 3 + [i64] * 4 + [dp, dp]
    lib.mamba_oracle_conv_fwd.restype = ctypes.c_int
    lib.mamba_oracle_conv_bwd.argtypes = [dp] * 4 + [i64] * 4 + [dp] * 3
    lib.mamba_oracle_conv_bwd.restype = ctypes.c_int
    return lib


def _load():
    global _default
    with _lock:
        if _default is None:
            _default = _bind(build())
    return _default


def compile_variant(src_text: str, workdir: str):
    """Compile an edited copy of the oracle's C source (tests plant mistakes this way to show
    that the pins catch them). Returns a handle usable as the ``lib`` argument below."""
    src = os.path.join(workdir, "variant.c")
    with open(src, "w") as f:
        f.write(src_text)
    so = os.path.join(workdir, f"libvariant{abs(hash(src_text))}.so")
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
                           "-I", _HERE, "-o", so, src, "-lm"])
    return _bind(so)


def source() -> str:
    with open(_SRC) as f:
        return f.read()


def _p(a):
    if a is None:
        return None
    assert a.dtype == np.float64 and a.flags.c_contiguous
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def as64(x: dict) -> dict:
    """float64 contiguous copies of an input dict (float32 values are represented exactly)."""
    return {k: np.ascontiguousarray(v, dtype=np.float64) for k, v in x.items()}


def _dims(x):
    b, T, Di = x["delta"].shape
    N = x["B"].shape[-1]
    return b, T, Di, N


_FWD_KEYS = ("delta", "u", "B", "C", "gate", "A_log", "D")


def fwd(x: dict, rows=None, lib=None, out=None, y=None):
    """Forward. Returns (out, y) as float64 [batch, T, d_inner]. ``rows``: optional (begin, end)
    row range (row = b*d_inner + d); other rows are left as NaN, or untouched when the caller
    passes its own float64 ``out`` and ``y`` arrays (threads may fill disjoint rows of them)."""
    x = as64(x)
    b, T, Di, N = _dims(x)
    r0, r1 = rows if rows is not None else (0, b * Di)
    if out is None:
        out = np.full((b, T, Di), np.nan)
    if y is None:
        y = np.full((b, T, Di), np.nan)
    rc = (lib or _load()).mamba_oracle_fwd_rows(*[_p(x[k]) for k in _FWD_KEYS], b, T, Di, N, r0, r1,
                                        _p(out), _p(y))
    if rc != 0:
        raise RuntimeError(f"oracle fwd failed rc={rc}")
    return out, y


def _bwd_range(x, r0, r1, per_row, acc, lib):
    b, T, Di, N = _dims(x)
    rc = (lib or _load()).mamba_oracle_bwd_rows(
        *[_p(x[k]) for k in _FWD_KEYS], _p(x["dy"]), b, T, Di, N, r0, r1,
        _p(per_row["d_delta"]), _p(per_row["d_u"]), _p(per_row["d_gate"]),
        _p(acc["d_B"]), _p(acc["d_C"]), _p(acc["d_A_log"]), _p(acc["d_D"]))
    if rc != 0:
        raise RuntimeError(f"oracle bwd failed rc={rc}")


def bwd(x: dict, threads: int = 1, rows=None, lib=None) -> dict:
    """Forward + backward. Returns float64 gradients d_delta, d_u, d_gate [batch,T,d_inner],
    d_B, d_C [batch,T,d_state], d_A_log [d_inner,d_state], d_D [d_inner].

    ``threads`` > 1 splits the row range into contiguous blocks processed concurrently (ctypes
    releases the GIL), each with private accumulators, summed in block order. ``rows`` restricts
    the computation to a row range; per-row outputs of other rows stay NaN and the accumulated
    outputs then hold only those rows' contributions.
    """
    x = as64(x)
    b, T, Di, N = _dims(x)
    r0, r1 = rows if rows is not None else (0, b * Di)
    per_row = {k: np.full((b, T, Di), np.nan) for k in ("d_delta", "d_u", "d_gate")}

    def new_acc():
        return {"d_B": np.zeros((b, T, N)), "d_C": np.zeros((b, T, N)),
                "d_A_log": np.zeros((Di, N)), "d_D": np.zeros(Di)}

    nthr = max(1, min(threads, r1 - r0))
    bounds = [r0 + (r1 - r0) * i // nthr for i in range(nthr + 1)]
    accs = [new_acc() for _ in range(nthr)]
    if nthr == 1:
        _bwd_range(x, bounds[0], bounds[1], per_row, accs[0], lib)
    else:
        with concurrent.futures.ThreadPoolExecutor(nthr) as ex:
            futs = [ex.submit(_bwd_range, x, bounds[i], bounds[i + 1], per_row, accs[i], lib)
                    for i in range(nthr)]
            for f in futs:
                f.result()
    total = accs[0]
    for a in accs[1:]:
        for k in total:
            total[k] += a[k]
    per_row.update(total)
    return per_row


def bwd_rows_into(x: dict, rows, per_row: dict, acc: dict, lib=None) -> None:
    """The computation of bwd() over the row range ``rows`` into caller-owned float64 arrays:
    per_row holds d_delta, d_u, d_gate [batch,T,d_inner] (rows outside the range untouched);
    acc holds d_B, d_C [batch,T,d_state], d_A_log [d_inner,d_state], d_D [d_inner], which the
    range's contributions are added to. For timing the oracle without allocating its outputs
    in every call."""
    _bwd_range(as64(x), rows[0], rows[1], per_row, acc, lib)


def loss(x: dict, lib=None) -> float:
    """Scalar loss sum(dy * out) whose gradients ``bwd`` returns."""
    out, _ = fwd(x, lib=lib)
    return float(np.sum(np.asarray(x["dy"], dtype=np.float64) * out))


# ---- the softplus before the scan (fused into the CUDA kernels as a variant) ----------------
def softplus(raw, lib=None) -> np.ndarray:
    """delta = softplus(raw), threshold 20 (C: mamba_oracle_softplus)."""
    lib = lib or _load()
    r = np.ascontiguousarray(raw, dtype=np.float64)
    out = np.empty_like(r)
    lib.mamba_oracle_softplus(_p(r), _p(out), r.size)
    return out


def softplus_bwd(raw, d_delta, lib=None) -> np.ndarray:
    """d_raw from d_delta (C: mamba_oracle_softplus_bwd)."""
    lib = lib or _load()
    r = np.ascontiguousarray(raw, dtype=np.float64)
    g = np.ascontiguousarray(d_delta, dtype=np.float64)
    out = np.empty_like(r)
    lib.mamba_oracle_softplus_bwd(_p(r), _p(g), _p(out), r.size)
    return out


def with_softplus(x: dict, lib=None) -> dict:
    """The inputs of the scan when x carries the raw delta under "delta_raw"."""
    y = dict(x)
    y["delta"] = softplus(x["delta_raw"], lib).reshape(np.shape(x["delta_raw"]))
    return y


# ---- causal depthwise conv1d + SiLU (the step before the scan) ------------------------------
def conv_fwd(x, w, bias, lib=None):
    """u = SiLU(causal depthwise conv1d(x) + bias) (C: mamba_oracle_conv_fwd); returns (u, pre)."""
    lib = lib or _load()
    x = np.ascontiguousarray(x, dtype=np.float64)
    w = np.ascontiguousarray(w, dtype=np.float64)
    bias = np.ascontiguousarray(bias, dtype=np.float64)
    b, T, Di = x.shape
    K = w.shape[1]
    u = np.empty_like(x)
    pre = np.empty_like(x)
    rc = lib.mamba_oracle_conv_fwd(_p(x), _p(w), _p(bias), b, T, Di, K, _p(u), _p(pre))
    assert rc == 0, rc
    return u, pre


def conv_bwd(x, w, bias, d_u, lib=None) -> dict:
    """d_x, d_w, d_bias of the conv + SiLU (C: mamba_oracle_conv_bwd)."""
    lib = lib or _load()
    x = np.ascontiguousarray(x, dtype=np.float64)
    w = np.ascontiguousarray(w, dtype=np.float64)
    bias = np.ascontiguousarray(bias, dtype=np.float64)
    d_u = np.ascontiguousarray(d_u, dtype=np.float64)
    b, T, Di = x.shape
    K = w.shape[1]
    d_x = np.empty_like(x)
    d_w = np.empty_like(w)
    d_b = np.empty_like(bias)
    rc = lib.mamba_oracle_conv_bwd(_p(x), _p(w), _p(bias), _p(d_u), b, T, Di, K, _p(d_x),
                                   _p(d_w), _p(d_b))
    assert rc == 0, rc
    return {"d_x": d_x, "d_w": d_w, "d_bias": d_b}
