"""Shared helpers of the GPU tests: run the CUDA path through the C ABI and compare with the
oracle. Tolerance: max|got - ref| <= 1e-4 * max|ref| for every output tensor."""
from __future__ import annotations

import os

import numpy as np

TOL = 1e-4
OUT_KEYS = ("out", "y", "d_delta", "d_u", "d_B", "d_C", "d_A_log", "d_D", "d_gate")
IN_KEYS = ("delta", "u", "B", "C", "gate", "A_log", "D", "dy")


def oracle_threads() -> int:
    return max(1, min(32, os.cpu_count() or 1))


def to_device(x: dict, device="cuda"):
    import torch
    return {k: torch.from_numpy(np.ascontiguousarray(x[k])).to(device) for k in IN_KEYS}


def run_gpu(x: dict, poison: bool = True, stream=None, softplus: bool = False) -> dict:
    """Forward + backward through the C ABI on cuda:0; outputs are NaN-poisoned first so that
    an element the kernels never write shows up as a mismatch. With softplus=True, x["delta"]
    is the raw delta and the _softplus entry points run (d_delta is then d_delta_raw)."""
    import torch
    import selective_state_space_06_gb300 as ms
    xd = to_device(x)
    bufs = ms.alloc_like_outputs(xd["delta"], xd["B"], xd["A_log"], xd["D"])
    if poison:
        for k in OUT_KEYS:
            bufs[k].fill_(float("nan"))
        bufs["scratch"].fill_(0xFF)            # NaN bit patterns in the partial sums
        if bufs["ckpt"] is not None:
            bufs["ckpt"].fill_(0xFF)
    ms.forward_backward(xd, bufs, stream=stream, softplus=softplus)
    torch.cuda.synchronize()
    ms.mamba_scan_status(stream)     # raises on a CUDA error or an expired copy wait
    return {k: bufs[k].cpu().numpy() for k in OUT_KEYS}


def oracle_all(x: dict, threads=None) -> dict:
    import oracle
    ref = oracle.bwd(x, threads=threads or oracle_threads())
    out, y = _oracle_fwd_threaded(x, threads or oracle_threads())
    ref["out"] = out
    ref["y"] = y
    return ref


def _oracle_fwd_threaded(x, threads):
    import concurrent.futures
    import oracle
    b, T, Di = x["delta"].shape
    rows = b * Di
    n = max(1, min(threads, rows))
    bounds = [rows * i // n for i in range(n + 1)]
    x64 = oracle.as64(x)
    out = np.full((b, T, Di), np.nan)
    y = np.full((b, T, Di), np.nan)
    with concurrent.futures.ThreadPoolExecutor(n) as ex:     # disjoint rows of shared arrays
        list(ex.map(lambda i: oracle.fwd(x64, rows=(bounds[i], bounds[i + 1]), out=out, y=y),
                    range(n)))
    return out, y


def rel_errors(got: dict, ref: dict, keys=OUT_KEYS) -> dict:
    errs = {}
    for k in keys:
        g = np.asarray(got[k], dtype=np.float64)
        r = np.asarray(ref[k], dtype=np.float64)
        assert g.shape == r.shape, (k, g.shape, r.shape)
        if not np.all(np.isfinite(g)):
            errs[k] = float("inf")
            continue
        scale = float(np.abs(r).max())
        err = float(np.abs(g - r).max())
        errs[k] = err / scale if scale > 0 else (0.0 if err == 0 else float("inf"))
    return errs


def assert_parity(got: dict, ref: dict, keys=OUT_KEYS, tol=TOL, label=""):
    errs = rel_errors(got, ref, keys)
    bad = {k: v for k, v in errs.items() if not v <= tol}
    assert not bad, f"{label}: max|err|/max|ref| above {tol}: {bad} (all: {errs})"
    return errs
