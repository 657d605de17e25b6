"""The fused softplus variant (mamba_scan_fwd_softplus / mamba_scan_bwd_softplus) against the
fp64 oracle.

delta = softplus(raw) with the threshold 20, and d_raw = d_delta * sigmoid(raw) below it (the
Softplus backward step of mamba-rs src/mamba_ssm/cpu/backward.rs). The expected values come from
the oracle's softplus followed by the oracle scan, and its softplus backward applied to the
oracle's d_delta. The raw values follow the workloads' recipe (0.5*N(0,1) - 2), with some
elements above the threshold and some far below it. The bar is the parity bar of the other
GPU tests, on every element of every output. The shapes run every kernel path: the tensor-memory
backward with TMA (d_state 16, 64) and with cp.async (ragged), and the d_state <= 8 kernels.
"""
import numpy as np
import pytest

import oracle
import synth
from gpu_helpers import OUT_KEYS, assert_parity, oracle_all, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import selective_state_space_06_gb300  # noqa: F401


def _raw_inputs(shape, seed):
    x = synth.random_inputs(*shape, seed=seed, a_log_random=True)
    rng = np.random.default_rng(seed + 1000)
    raw = (0.5 * rng.standard_normal(x["delta"].shape) - 2.0).astype(np.float32)
    flat = raw.reshape(-1)
    k = max(1, flat.size // 97)
    flat[::97][:k] = 21.5                      # the identity branch
    flat[5::89] = -30.0                        # delta ~ 1e-13
    x["delta"] = raw
    return x


def _expected(x):
    xo = dict(x)
    xo["delta_raw"] = x["delta"].astype(np.float64)
    xo = oracle.with_softplus(xo)
    del xo["delta_raw"]
    ref = oracle_all(xo)
    ref["d_delta"] = oracle.softplus_bwd(x["delta"], ref["d_delta"]).reshape(x["delta"].shape)
    return ref


@pytest.mark.parametrize("shape", [(1, 64, 32, 16), (8, 1024, 1536, 16), (1, 300, 64, 64),
                                   (2, 33, 33, 13), (2, 40, 64, 8), (3, 37, 50, 5)],
                         ids=["tiny", "mamba130m", "dstate64_segments", "ragged_cp_async",
                              "dstate8", "dstate5_ragged"])
def test_softplus_variant_matches_oracle(shape):
    x = _raw_inputs(shape, seed=sum(shape))
    got = run_gpu(x, softplus=True)
    assert_parity(got, _expected(x), keys=OUT_KEYS, label=f"softplus {shape}")
