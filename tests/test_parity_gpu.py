"""Parity of the CUDA path with the fp64 oracle, through the C ABI on cuda:0.

The bar is max|got - ref| <= 1e-4 * max|ref| per output tensor, where ref is the fp64 oracle
on the same float32 inputs. It is checked element by element on every output, for the five
benchmark workloads at their full sizes (the launch configuration the bench times) and for edge
cases: ragged T, d_inner and d_state, T = 1, delta = 0, saturated gates. Outputs are
NaN-poisoned before every call, so an element the kernels do not write fails too.
"""
import numpy as np
import pytest

import synth
from gpu_helpers import OUT_KEYS, assert_parity, oracle_all, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import selective_state_space_06_gb300  # noqa: F401  (fails loudly if the library is missing)


@pytest.mark.parametrize("name", ["tiny", "mamba130m", "mamba370m", "mamba1p4b"])
def test_workload_full_parity(name):
    x = synth.make_inputs(synth.BY_NAME[name])
    got = run_gpu(x)
    ref = oracle_all(x)
    assert_parity(got, ref, label=name)


def test_longseq_full_parity():
    """batch=1, T=65536, d_inner=2560, d_state=64: every output element against the oracle."""
    x = synth.make_inputs(synth.BY_NAME["longseq"])
    got = run_gpu(x)
    ref = oracle_all(x)
    assert_parity(got, ref, label="longseq")


EDGE_SHAPES = [
    # (batch, T, d_inner, d_state)
    (1, 1, 1, 1),
    (1, 1, 7, 16),
    (2, 15, 3, 4),
    (2, 16, 64, 16),
    (2, 17, 65, 16),
    (3, 37, 50, 5),
    (1, 100, 130, 8),
    (2, 33, 33, 13),
    (1, 48, 40, 17),
    (2, 31, 20, 32),
    (1, 40, 18, 33),
    (1, 64, 33, 63),
    (2, 50, 17, 64),
    (4, 129, 257, 16),
    # vectorised path (d_inner % 4 == 0, d_state % 4 == 0) with d_state below its padding
    (2, 40, 64, 12),
    (1, 50, 32, 20),
    (2, 33, 16, 60),
    (1, 70, 128, 4),
    (2, 45, 96, 8),
    (1, 300, 64, 28),
]


@pytest.mark.parametrize("shape", EDGE_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_edge_shapes(shape):
    x = synth.random_inputs(*shape, seed=sum(shape), a_log_random=True)
    assert_parity(run_gpu(x), oracle_all(x), label=str(shape))


# d_state 32 and 64 with several blocks of channels (32 channels per block at d_state 64, 64
# at d_state 32), vectorised (d_inner and d_state multiples of 4): the d_B / d_C partials of
# the blocks are summed by the reduction in block order.
MULTI_BLOCK_SHAPES = [
    (2, 333, 128, 64),   # 4 blocks, ragged T
    (1, 100, 64, 64),    # 2 blocks
    (1, 200, 256, 48),   # 8 blocks; states 48..63 padding
    (1, 64, 192, 64),    # 6 blocks
    (1, 50, 100, 64),    # 4 blocks, the last one ragged (channels 96..99)
    (2, 90, 256, 32),    # d_state 32: 4 blocks of 64 channels
    (1, 77, 128, 24),    # d_state 24 (padded to 32): 2 blocks
    (3, 1000, 512, 64),  # 16 blocks, several time segments per row
]


@pytest.mark.parametrize("shape", MULTI_BLOCK_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_multi_block_shapes(shape):
    x = synth.random_inputs(*shape, seed=sum(shape) + 1, a_log_random=True)
    assert_parity(run_gpu(x), oracle_all(x), label=str(shape))


def test_multi_block_bitwise_deterministic():
    x = synth.random_inputs(1, 400, 256, 64, seed=5, a_log_random=True)
    a = run_gpu(x)
    b = run_gpu(x)
    for k in OUT_KEYS:
        assert np.array_equal(a[k], b[k], equal_nan=False), k


def test_delta_zero():
    x = synth.random_inputs(2, 40, 70, 16, seed=1)
    x["delta"][:] = 0.0
    got = run_gpu(x)
    ref = oracle_all(x)
    for k in ("d_B", "d_C", "d_A_log"):
        assert np.all(got[k] == 0.0), k
    assert_parity(got, ref, keys=("out", "y", "d_delta", "d_u", "d_D", "d_gate"), label="delta0")


def test_saturated_gates_and_large_delta():
    x = synth.random_inputs(2, 40, 70, 16, seed=2)
    x["gate"] = (x["gate"] * 60).astype(np.float32)          # sigmoid saturates both ways
    x["delta"][:, ::5] = 40.0                                 # exp(delta*A) underflows to 0
    got = run_gpu(x)
    ref = oracle_all(x)
    assert_parity(got, ref, label="saturated")


def test_bitwise_deterministic():
    x = synth.make_inputs(synth.BY_NAME["mamba130m"].resized(batch=2, T=300, name="det"))
    a = run_gpu(x)
    b = run_gpu(x)
    for k in OUT_KEYS:
        assert np.array_equal(a[k], b[k], equal_nan=False), k


def test_euler_identities_full_size_longseq():
    """Exact identities of the method at full size (out is homogeneous of degree 1 in u, B, C
    and D). Checked on the GPU results alone, in float64 sums, at the longseq workload."""
    x = synth.make_inputs(synth.BY_NAME["longseq"])
    g = run_gpu(x)
    f64 = lambda a: np.asarray(a, dtype=np.float64)  # noqa: E731
    s = 1 / (1 + np.exp(-f64(x["gate"])))
    w = f64(x["dy"]) * f64(x["gate"]) * s
    y_minus_du = f64(g["y"]) - f64(x["D"]) * f64(x["u"])
    pairs = {
        "u": (np.sum(f64(g["d_u"]) * f64(x["u"])), np.sum(f64(x["dy"]) * f64(g["out"]))),
        "B": (np.sum(f64(g["d_B"]) * f64(x["B"])), np.sum(w * y_minus_du)),
        "C": (np.sum(f64(g["d_C"]) * f64(x["C"])), np.sum(w * y_minus_du)),
        "D": (np.sum(f64(g["d_D"]) * f64(x["D"])), np.sum(w * f64(x["D"]) * f64(x["u"]))),
    }
    for k, (lhs, rhs) in pairs.items():
        # relative to the sum of magnitudes: fp32 rounding of 1e8 terms
        mag = np.sum(np.abs(w * y_minus_du)) + np.sum(np.abs(f64(x["dy"]) * f64(g["out"])))
        assert abs(lhs - rhs) <= 1e-5 * mag, (k, lhs, rhs, mag)


def test_separate_calls_under_graph_capture():
    """mamba_scan_fwd + mamba_scan_bwd captured in a CUDA graph (their kernels are launched
    with programmatic stream serialization, which capture turns into programmatic edges) and
    replayed give the eager calls' outputs bitwise."""
    import torch
    import selective_state_space_06_gb300 as ms
    x = synth.random_inputs(2, 700, 256, 16, seed=9, a_log_random=True)
    xd = {k: torch.from_numpy(np.ascontiguousarray(v)).to("cuda:0") for k, v in x.items()}
    bufs = ms.alloc_like_outputs(xd["delta"], xd["B"], xd["A_log"], xd["D"])
    keys = ("out", "y", "d_delta", "d_u", "d_B", "d_C", "d_A_log", "d_D", "d_gate")

    def step():
        ms.forward_backward(xd, bufs)
    step()   # first call: tensor maps and kernel attributes set up outside capture
    torch.cuda.synchronize()
    eager = {k: bufs[k].clone() for k in keys}
    for k in keys:
        bufs[k].fill_(float("nan"))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            step()
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    ms.mamba_scan_status()
    for k in keys:
        assert torch.equal(bufs[k], eager[k]), k
