"""mamba_scan_fwd_bwd (forward and backward in one call, dy known up front) against the fp64
oracle.

For d_state 9..16 the forward pass keeps only the chunk-boundary states and the backward forms
y = sum_n C*h + D*u from its recomputed states, so out and d_gate come from a y summed in
another order than the separate forward's; they must meet the parity bar like every other
output. The other six gradients do not depend on y at all: they must equal the separate
calls' bitwise, since both paths run the same recurrence from the same checkpoints. Above
d_state 16 and at d_state <= 8 the call runs the two passes as the separate calls do (with the
backward's pre-pass beside the forward when T spans several segments). The shapes cover both
(d_state 5 to 64; TMA and cp.async staging; one and several time segments; T = 1 and T not a
multiple of the 16-step chunk).
"""
import numpy as np
import pytest

import synth
from gpu_helpers import OUT_KEYS, assert_parity, oracle_all, run_gpu, to_device

pytestmark = pytest.mark.gpu

KEYS = tuple(k for k in OUT_KEYS if k != "y")
Y_FREE = ("d_delta", "d_u", "d_B", "d_C", "d_A_log", "d_D")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import selective_state_space_06_gb300  # noqa: F401


def run_fused(x: dict) -> dict:
    import torch
    import selective_state_space_06_gb300 as ms
    xd = to_device(x)
    bufs = ms.alloc_like_outputs(xd["delta"], xd["B"], xd["A_log"], xd["D"])
    for k in KEYS:
        bufs[k].fill_(float("nan"))
    bufs["scratch"].fill_(0xFF)
    if bufs["ckpt"] is not None:
        bufs["ckpt"].fill_(0xFF)
    ms.mamba_scan_fwd_bwd(xd["delta"], xd["u"], xd["B"], xd["C"], xd["gate"], xd["A_log"],
                          xd["D"], xd["dy"], bufs["out"], bufs["ckpt"], bufs["scratch"],
                          bufs["d_delta"], bufs["d_u"], bufs["d_B"], bufs["d_C"],
                          bufs["d_A_log"], bufs["d_D"], bufs["d_gate"])
    torch.cuda.synchronize()
    ms.mamba_scan_status()
    return {k: bufs[k].cpu().numpy() for k in KEYS}


SHAPES = [(1, 64, 32, 16), (8, 1024, 1536, 16), (1, 300, 64, 64), (2, 31, 20, 32),
          (2, 33, 33, 13), (1, 1, 7, 16), (2, 17, 65, 16), (4, 129, 257, 16), (1, 300, 64, 28),
          (2, 40, 64, 8), (3, 37, 50, 5)]
IDS = ["tiny", "mamba130m", "dstate64_segments", "dstate32_cp_async", "ragged13", "T1",
       "T17_d65", "4x129x257", "dstate28_tma", "dstate8_unfused", "dstate5_unfused"]


@pytest.mark.parametrize("shape", SHAPES, ids=IDS)
def test_fused_matches_oracle(shape):
    if shape == (8, 1024, 1536, 16):
        x = synth.make_inputs(synth.BY_NAME["mamba130m"])
    else:
        x = synth.random_inputs(*shape, seed=sum(shape) + 7, a_log_random=True)
    got = run_fused(x)
    assert_parity(got, oracle_all(x), keys=KEYS, label=f"fused {shape}")


@pytest.mark.parametrize("shape", [(8, 1024, 1536, 16), (1, 300, 64, 64), (2, 31, 20, 32)],
                         ids=["mamba130m", "dstate64_segments", "dstate32_cp_async"])
def test_fused_gradients_equal_separate_calls(shape):
    if shape == (8, 1024, 1536, 16):
        x = synth.make_inputs(synth.BY_NAME["mamba130m"])
    else:
        x = synth.random_inputs(*shape, seed=sum(shape) + 11, a_log_random=True)
    fused = run_fused(x)
    sep = run_gpu(x)
    for k in Y_FREE:
        assert np.array_equal(fused[k], sep[k]), k


def test_fused_call_under_graph_capture():
    """The fused call (whose pre-pass forks to a side stream when T spans several segments)
    captured in a CUDA graph and replayed gives the eager call's outputs bitwise."""
    import torch
    import selective_state_space_06_gb300 as ms
    x = synth.random_inputs(2, 700, 256, 16, seed=5, a_log_random=True)
    xd = to_device(x)
    bufs = ms.alloc_like_outputs(xd["delta"], xd["B"], xd["A_log"], xd["D"])

    def call():
        ms.mamba_scan_fwd_bwd(xd["delta"], xd["u"], xd["B"], xd["C"], xd["gate"], xd["A_log"],
                              xd["D"], xd["dy"], bufs["out"], bufs["ckpt"], bufs["scratch"],
                              bufs["d_delta"], bufs["d_u"], bufs["d_B"], bufs["d_C"],
                              bufs["d_A_log"], bufs["d_D"], bufs["d_gate"])
    call()   # first call: side stream, tensor maps and kernel attributes set up outside capture
    torch.cuda.synchronize()
    eager = {k: bufs[k].clone() for k in KEYS}
    for k in KEYS:
        bufs[k].fill_(float("nan"))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            call()
    g.replay()
    torch.cuda.synchronize()
    ms.mamba_scan_status()
    for k in KEYS:
        assert torch.equal(bufs[k], eager[k]), k
