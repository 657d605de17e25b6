"""Causal depthwise conv1d + SiLU (mamba_conv_fwd / mamba_conv_bwd) against the fp64 oracle.

Same bar as the scan: max|got - ref| <= 1e-4 * max|ref| for every output tensor, on every
element, with NaN-poisoned outputs. The shapes cover the vector path (d_inner % 4 == 0) and the
scalar path, kernel sizes 1 to 8, runs that end inside the halo (T not a multiple of the
32-step run), T shorter than the kernel, and the mamba130m size (d_conv 4, the Mamba
default). Two calls in a row must agree bitwise (the weight gradients are fixed-order sums).
"""
import numpy as np
import pytest

import oracle
from gpu_helpers import TOL, rel_errors

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import selective_state_space_06_gb300  # noqa: F401


def _inputs(shape, K, seed):
    rng = np.random.default_rng(seed)
    b, T, Di = shape
    return {"x": rng.standard_normal((b, T, Di)).astype(np.float32),
            "w": (rng.standard_normal((Di, K)) / np.sqrt(K)).astype(np.float32),
            "bias": (0.3 * rng.standard_normal(Di)).astype(np.float32),
            "d_u": rng.standard_normal((b, T, Di)).astype(np.float32)}


def _run(inp):
    import torch
    import selective_state_space_06_gb300 as ms
    dev = "cuda:0"
    t = {k: torch.from_numpy(v).to(dev) for k, v in inp.items()}
    b, T, Di = inp["x"].shape
    K = inp["w"].shape[1]
    u = torch.full((b, T, Di), float("nan"), device=dev)
    ms.mamba_conv_fwd(t["x"], t["w"], t["bias"], u)
    sc = torch.full((ms.mamba_conv_scratch_bytes(b, T, Di, K) // 4,), float("nan"), device=dev)
    out = []
    for _ in range(2):
        g = {"d_x": torch.full((b, T, Di), float("nan"), device=dev),
             "d_w": torch.full((Di, K), float("nan"), device=dev),
             "d_bias": torch.full((Di,), float("nan"), device=dev)}
        ms.mamba_conv_bwd(t["x"], t["w"], t["bias"], t["d_u"], sc, g["d_x"], g["d_w"],
                          g["d_bias"])
        torch.cuda.synchronize()
        out.append({k: v.cpu().numpy() for k, v in g.items()})
    return u.cpu().numpy(), out


@pytest.mark.parametrize("shape,K", [((2, 100, 64), 4), ((3, 37, 50), 4), ((1, 5, 16), 8),
                                    ((2, 64, 32), 1), ((2, 70, 36), 3), ((1, 3, 8), 4),
                                    ((8, 1024, 1536), 4)],
                         ids=["vec_k4", "scalar_k4", "k8_short", "k1", "k3_ragged",
                              "T_below_K", "mamba130m_k4"])
def test_conv_matches_oracle(shape, K):
    inp = _inputs(shape, K, seed=sum(shape) + K)
    u, (g1, g2) = _run(inp)
    ref_u, _ = oracle.conv_fwd(inp["x"], inp["w"], inp["bias"])
    ref = oracle.conv_bwd(inp["x"], inp["w"], inp["bias"], inp["d_u"])
    errs = rel_errors({"u": u, **g1}, {"u": ref_u, **ref}, keys=("u", "d_x", "d_w", "d_bias"))
    assert all(e <= TOL for e in errs.values()), errs
    for k in g1:
        assert np.array_equal(g1[k], g2[k]), k
