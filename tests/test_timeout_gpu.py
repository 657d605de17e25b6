"""Failure detection of the bounded copy waits, on the GPU and without a GPU fault.

Every wait of the tensor-memory backward, and of the forward at d_state 64, on its tensor
copies is bounded. When a wait runs
out, the kernel records a fault word, goes on to its end and exits; mamba_scan_status then
reports MAMBA_ERR_TIMEOUT and clears the word. mamba_scan_bwd_test_timeout and
mamba_scan_fwd_test_timeout plant the failure on the host side: the kernel issues no copy for the last chunk each CTA walks, and the waits
give up after 1 ms. Nothing is left in flight (every copy that was issued is waited for before
use), so the context stays usable: the status is read once as TIMEOUT, then as OK, and a normal
call afterwards still matches the oracle.
"""
import pytest

import synth
from gpu_helpers import assert_parity, oracle_all, run_gpu, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@pytest.mark.parametrize("shape", [(2, 96, 128, 16), (1, 80, 64, 64)],
                         ids=["dstate16", "dstate64"])
def test_copy_wait_runs_out_and_is_reported(shape):
    import torch
    import selective_state_space_06_gb300 as ms

    x = synth.random_inputs(*shape, seed=5)
    xd = to_device(x)
    bufs = ms.alloc_like_outputs(xd["delta"], xd["B"], xd["A_log"], xd["D"])
    ms.mamba_scan_status()   # nothing pending before the planted failure
    ms.mamba_scan_fwd(xd["delta"], xd["u"], xd["B"], xd["C"], xd["gate"], xd["A_log"], xd["D"],
                      bufs["out"], None, bufs["ckpt"])
    ms.mamba_scan_bwd_test_timeout(xd["delta"], xd["u"], xd["B"], xd["C"], xd["gate"],
                                   xd["A_log"], xd["D"], xd["dy"], bufs["ckpt"], bufs["scratch"],
                                   bufs["d_delta"], bufs["d_u"], bufs["d_B"], bufs["d_C"],
                                   bufs["d_A_log"], bufs["d_D"], bufs["d_gate"])
    with pytest.raises(ms.MambaScanError) as err:
        ms.mamba_scan_status()
    assert err.value.code == ms.MAMBA_ERR_TIMEOUT
    ms.mamba_scan_status()   # the word was cleared by the read above
    torch.cuda.synchronize()
    # the next regular call is unaffected
    assert_parity(run_gpu(x), oracle_all(x), label=f"after timeout {shape}")


@pytest.mark.parametrize("shape", [(1, 80, 64, 64), (1, 1000, 96, 64), (2, 70, 128, 36)],
                         ids=["one_segment", "segments", "dstate36"])
def test_forward_copy_wait_runs_out_and_is_reported(shape):
    import torch
    import selective_state_space_06_gb300 as ms

    x = synth.random_inputs(*shape, seed=9)
    xd = to_device(x)
    bufs = ms.alloc_like_outputs(xd["delta"], xd["B"], xd["A_log"], xd["D"])
    ms.mamba_scan_status()   # nothing pending before the planted failure
    ms.mamba_scan_fwd_test_timeout(xd["delta"], xd["u"], xd["B"], xd["C"], xd["gate"],
                                   xd["A_log"], xd["D"], bufs["out"], None, bufs["ckpt"])
    with pytest.raises(ms.MambaScanError) as err:
        ms.mamba_scan_status()
    assert err.value.code == ms.MAMBA_ERR_TIMEOUT
    ms.mamba_scan_status()   # the word was cleared by the read above
    torch.cuda.synchronize()
    assert_parity(run_gpu(x), oracle_all(x), label=f"after forward timeout {shape}")
