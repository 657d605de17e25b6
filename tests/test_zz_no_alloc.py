"""mamba_scan_bwd_noalloc: the backward for callers that may not allocate device memory.

Some callers get only their input and output buffers. A plugin inside a framework that owns
all device memory is one; a latency-critical loop that forbids cudaMalloc is another. For them
the library takes the backward's scratch from a static 64 MiB device array instead of from the
caller.

The GPU test calls the entry point through the C ABI twice in a row, on two different input
sets A and B of the same shape. The first call (A) is checked against mamba_scan_bwd within
the tolerance the parity tests use. The second (B) runs with the array still holding A's
partial sums, and must equal mamba_scan_bwd on B with freshly NaN-filled caller scratch bit for
bit: a read of a scratch word the call did not write would show up there, either as A's stale
value or as NaN. The file is named so that pytest collects it last. It passes when run alone in
a fresh process and when run after the other tests.
"""
import ctypes

import numpy as np
import pytest

import synth
from gpu_helpers import TOL, rel_errors

GRADS = ("d_delta", "d_u", "d_B", "d_C", "d_A_log", "d_D", "d_gate")


def _gpu():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


def _forward_and_reference(ms, xd):
    """Forward, then the regular backward with freshly NaN-filled caller scratch."""
    import torch
    bufs = ms.alloc_like_outputs(xd["delta"], xd["B"], xd["A_log"], xd["D"])
    bufs["scratch"].fill_(0xFF)
    ms.forward_backward(xd, bufs)
    torch.cuda.synchronize()
    return bufs, {k: bufs[k].double().cpu().numpy() for k in GRADS}


def _noalloc(ms, xd, bufs, shape):
    import torch
    b, T, Di, N = shape
    lib = ms.raw_library()
    stream = torch.cuda.current_stream().cuda_stream
    ck = bufs["ckpt"]
    out = {k: torch.full_like(bufs[k], float("nan")) for k in GRADS}
    rc = lib.mamba_scan_bwd_noalloc(
        xd["delta"].data_ptr(), xd["u"].data_ptr(), xd["B"].data_ptr(), xd["C"].data_ptr(),
        xd["gate"].data_ptr(), xd["A_log"].data_ptr(), xd["D"].data_ptr(), xd["dy"].data_ptr(),
        ck.data_ptr() if ck is not None else None, ck.numel() if ck is not None else 0,
        out["d_delta"].data_ptr(), out["d_u"].data_ptr(), out["d_B"].data_ptr(),
        out["d_C"].data_ptr(), out["d_A_log"].data_ptr(), out["d_D"].data_ptr(),
        out["d_gate"].data_ptr(), b, T, Di, N, ctypes.c_void_p(stream))
    assert rc == ms.MAMBA_OK, ms.mamba_scan_strerror(rc)
    torch.cuda.synchronize()
    return {k: out[k].double().cpu().numpy() for k in GRADS}


@pytest.mark.gpu
@pytest.mark.parametrize("shape", [(8, 1024, 1536, 16), (2, 37, 50, 5), (1, 300, 40, 64)],
                         ids=["mamba130m", "ragged", "dstate64"])
def test_noalloc_bwd_two_calls_on_different_inputs(shape):
    if not _gpu():
        pytest.skip("no CUDA device")
    import torch
    import selective_state_space_06_gb300 as ms

    b, T, Di, N = shape
    need = ms.mamba_scan_scratch_bytes(b, T, Di, N)
    assert 0 < need <= ms.MAMBA_SCAN_NOALLOC_SCRATCH_BYTES
    xa = {k: torch.from_numpy(v).to("cuda:0")
          for k, v in synth.random_inputs(b, T, Di, N, seed=11).items()}
    xb = {k: torch.from_numpy(v).to("cuda:0")
          for k, v in synth.random_inputs(b, T, Di, N, seed=12).items()}

    bufs_a, ref_a = _forward_and_reference(ms, xa)
    got_a = _noalloc(ms, xa, bufs_a, shape)                    # call 1: input set A
    errs = rel_errors(got_a, ref_a, GRADS)
    assert all(e <= TOL for e in errs.values()), ("A", errs)

    bufs_b, ref_b = _forward_and_reference(ms, xb)
    got_b = _noalloc(ms, xb, bufs_b, shape)                    # call 2: B, over A's scratch
    for k in GRADS:
        assert np.array_equal(got_b[k], ref_b[k]), f"B: {k} differs from mamba_scan_bwd"


def test_noalloc_rejects_sizes_beyond_the_static_scratch():
    """Host-side check only: the limit is enforced before any device work. Runs without a
    GPU (fake pointers never reach a launch); skipped where a GPU is visible."""
    if _gpu():
        pytest.skip("fake-pointer check runs only without a GPU")
    import __graft_entry__
    __graft_entry__.build()
    import selective_state_space_06_gb300 as ms
    b, T, Di, N = 1, 65536, 2560, 64          # the long-sequence workload
    assert ms.mamba_scan_scratch_bytes(b, T, Di, N) > ms.MAMBA_SCAN_NOALLOC_SCRATCH_BYTES
    lib = ms.raw_library()
    big = 1 << 32
    ptrs = [big * (i + 1) for i in range(9)]
    rc = lib.mamba_scan_bwd_noalloc(*ptrs[:9], 1 << 40, *[big * (20 + i) for i in range(7)],
                                    b, T, Di, N, None)
    assert rc == ms.MAMBA_ERR_NOALLOC_LIMIT
    assert "64 MiB" in ms.mamba_scan_strerror(rc)
