"""The bounds-checked build (libmambascan_checked.so: the same sources with -DMAMBA_BOUNDS_CHECK).

In that build every global access whose offset a kernel computes is checked against the length
of its buffer (from the call's sizes); an access outside is not made and is recorded for
mamba_scan_status (MAMBA_ERR_BOUNDS). No check traps.

1. Clean runs: on ragged shapes of every kernel family (d_state <= 8 in registers, 16-64 in
   tensor memory, vector and scalar staging, many time segments, the conv1d step) no check
   fires, the outputs equal the default build's bitwise (the checks add predicates, no
   arithmetic), and they match the fp64 oracle within the usual 1e-4 * max|ref|.
2. The check fires without a stray access: with every length taken one element short
   (mamba_scan_test_bounds_shrink(1)) the accesses to each buffer's last element are refused,
   every refused access being inside the real buffer, and mamba_scan_status reports
   MAMBA_ERR_BOUNDS once, then clears. With the real lengths back, the next call passes parity.
"""
import numpy as np
import pytest

import synth
from gpu_helpers import OUT_KEYS, TOL, oracle_all, rel_errors, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def checked():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import selective_state_space_06_gb300 as ms
    from selective_state_space_06_gb300 import build
    build.build(checked=True)
    lib = ms.checked_library()
    assert lib.mamba_scan_bounds_checked() == 1
    assert not ms.mamba_scan_bounds_checked()     # the default library has no checks
    return lib


def _run(x, lib=None):
    import torch
    import selective_state_space_06_gb300 as ms
    xd = to_device(x)
    bufs = ms.alloc_like_outputs(xd["delta"], xd["B"], xd["A_log"], xd["D"])
    for k in OUT_KEYS:
        bufs[k].fill_(float("nan"))
    bufs["scratch"].fill_(0xFF)
    if bufs["ckpt"] is not None:
        bufs["ckpt"].fill_(0xFF)
    if lib is None:
        ms.forward_backward(xd, bufs)
        torch.cuda.synchronize()
        ms.mamba_scan_status()
    else:
        with ms.using_library(lib):
            ms.forward_backward(xd, bufs)
            torch.cuda.synchronize()
            ms.mamba_scan_status()        # raises MambaScanError(MAMBA_ERR_BOUNDS) on a refusal
    return {k: bufs[k].cpu().numpy() for k in OUT_KEYS}


# (batch, T, d_inner, d_state): d_state 3 and 8 (register backward), 13 (scalar staging,
# d_state % 4 != 0), 16 and 64 with one batch row and a long T (many time segments in both
# passes and the backward's segment pre-pass), 32 with d_inner % 4 != 0 (scalar staging)
SHAPES = [(2, 37, 20, 3), (3, 53, 24, 8), (2, 45, 36, 13), (1, 700, 64, 16), (2, 90, 30, 32),
          (1, 700, 64, 64), (2, 33, 132, 16)]


@pytest.mark.parametrize("shape", SHAPES, ids=[f"b{b}_T{T}_d{d}_n{n}" for b, T, d, n in SHAPES])
def test_checked_build_runs_clean_and_bitwise(checked, shape):
    x = synth.random_inputs(*shape, seed=7)
    got = _run(x, checked)
    ref_default = _run(x)
    for k in OUT_KEYS:
        assert np.array_equal(got[k], ref_default[k], equal_nan=True), k
    errs = rel_errors(got, oracle_all(x))
    assert max(errs.values()) <= TOL, errs


def test_conv_checked_runs_clean(checked):
    import torch
    import selective_state_space_06_gb300 as ms
    rng = np.random.default_rng(3)
    b, T, Di, K = 2, 70, 36, 4
    x = torch.from_numpy(rng.standard_normal((b, T, Di)).astype(np.float32)).cuda()
    w = torch.from_numpy(rng.standard_normal((Di, K)).astype(np.float32)).cuda()
    bias = torch.from_numpy(rng.standard_normal(Di).astype(np.float32)).cuda()
    d_u = torch.from_numpy(rng.standard_normal((b, T, Di)).astype(np.float32)).cuda()
    res = []
    for lib in (checked, None):
        with ms.using_library(lib or ms.raw_library()):
            u = torch.full((b, T, Di), float("nan"), device="cuda")
            sc = torch.empty(ms.mamba_conv_scratch_bytes(b, T, Di, K), dtype=torch.uint8,
                             device="cuda")
            dx = torch.full_like(u, float("nan"))
            dw = torch.full((Di, K), float("nan"), device="cuda")
            db = torch.full((Di,), float("nan"), device="cuda")
            ms.mamba_conv_fwd(x, w, bias, u)
            ms.mamba_conv_bwd(x, w, bias, d_u, sc, dx, dw, db)
            ms.mamba_scan_status()
            res.append([t.cpu().numpy() for t in (u, dx, dw, db)])
    for a, b_ in zip(*res):
        assert np.array_equal(a, b_)


def test_check_fires_without_a_stray_access(checked):
    import torch
    import selective_state_space_06_gb300 as ms
    x = synth.random_inputs(1, 300, 64, 64, seed=11)
    with ms.using_library(checked):
        ms.mamba_scan_test_bounds_shrink(1)
        try:
            ms.forward_backward(to_device(x))
            torch.cuda.synchronize()
            with pytest.raises(ms.MambaScanError) as e:
                ms.mamba_scan_status()
            assert e.value.code == ms.MAMBA_ERR_BOUNDS
            ms.mamba_scan_status()       # reported once, then cleared
        finally:
            ms.mamba_scan_test_bounds_shrink(0)
    got = _run(x, checked)               # the real lengths again: clean and correct
    errs = rel_errors(got, oracle_all(x))
    assert max(errs.values()) <= TOL, errs

