"""mamba_scan_fwd_bwd_bf16 (the fused call with bf16 I/O) against the fp64 oracle and against
the fp32 fused call.

Inputs are the workloads' fp32 inputs rounded to bf16 (nearest even); the oracle takes those
bf16 values exactly. Tolerance, derived: the fp32 path meets |v - ref| <= 1e-4 * max|ref|, and
rounding v to bf16 (8 significant bits, nearest) moves it by at most 2^-8 * |v|, so every bf16
output must satisfy |got - ref| <= 2^-8 * |ref| + 1.01e-4 * max|ref| element by element.
d_A_log and d_D stay fp32 and keep the fp32 bar.

Exactly, since widening bf16 to fp32 is exact and the kernels then run the fp32 arithmetic:
every bf16 output equals the fp32 fused call's output on the same (bf16-valued) inputs,
rounded to nearest even, bit for bit; d_A_log and d_D equal it outright. Above d_state 16 the
fp32 fused call takes y from the forward (summed in another order), while the bf16 call forms
it in the backward at every d_state, so there out and d_gate, the outputs that depend on y,
are left to the oracle bar.
"""
import numpy as np
import pytest

import synth
from gpu_helpers import TOL, oracle_all

pytestmark = pytest.mark.gpu

BF_OUT = ("out", "d_delta", "d_u", "d_B", "d_C", "d_gate")
F32_OUT = ("d_A_log", "d_D")
BF_IN = ("delta", "u", "B", "C", "gate", "dy")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import selective_state_space_06_gb300  # noqa: F401


def _bf16_inputs(x):
    """The inputs rounded to bf16 (torch's conversion, nearest even), as bf16 tensors and as
    the fp32 values they hold."""
    import torch
    bf = {k: torch.from_numpy(np.ascontiguousarray(x[k])).to(torch.bfloat16) for k in BF_IN}
    vals = dict(x)
    for k in BF_IN:
        vals[k] = bf[k].float().numpy()
    return bf, vals


def _outputs(b, T, Di, N, dtype, dev):
    import torch
    o = {k: torch.full((b, T, Di), float("nan"), dtype=dtype, device=dev)
         for k in ("out", "d_delta", "d_u", "d_gate")}
    o["d_B"] = torch.full((b, T, N), float("nan"), dtype=dtype, device=dev)
    o["d_C"] = torch.full((b, T, N), float("nan"), dtype=dtype, device=dev)
    o["d_A_log"] = torch.full((Di, N), float("nan"), device=dev)
    o["d_D"] = torch.full((Di,), float("nan"), device=dev)
    return o


def _workspaces(b, T, Di, N, dev):
    import torch
    import selective_state_space_06_gb300 as ms
    ck = torch.full((ms.mamba_scan_ckpt_bytes(b, T, Di, N) // 4,), float("nan"), device=dev)
    sc = torch.full((ms.mamba_scan_scratch_bytes(b, T, Di, N) // 4,), float("nan"), device=dev)
    return ck, sc


def run_bf16(bf, x):
    import torch
    import selective_state_space_06_gb300 as ms
    dev = "cuda:0"
    b, T, Di = x["delta"].shape
    N = x["B"].shape[2]
    t = {k: v.to(dev) for k, v in bf.items()}
    A_log = torch.from_numpy(x["A_log"]).to(dev)
    D = torch.from_numpy(x["D"]).to(dev)
    o = _outputs(b, T, Di, N, torch.bfloat16, dev)
    ck, sc = _workspaces(b, T, Di, N, dev)
    ms.mamba_scan_fwd_bwd_bf16(t["delta"], t["u"], t["B"], t["C"], t["gate"], A_log, D, t["dy"],
                               o["out"], ck, sc, o["d_delta"], o["d_u"], o["d_B"], o["d_C"],
                               o["d_A_log"], o["d_D"], o["d_gate"])
    torch.cuda.synchronize()
    ms.mamba_scan_status()
    return o


def run_fp32_fused(vals):
    import torch
    import selective_state_space_06_gb300 as ms
    dev = "cuda:0"
    b, T, Di = vals["delta"].shape
    N = vals["B"].shape[2]
    t = {k: torch.from_numpy(np.ascontiguousarray(vals[k])).to(dev)
         for k in BF_IN + ("A_log", "D")}
    o = _outputs(b, T, Di, N, torch.float32, dev)
    ck, sc = _workspaces(b, T, Di, N, dev)
    ms.mamba_scan_fwd_bwd(t["delta"], t["u"], t["B"], t["C"], t["gate"], t["A_log"], t["D"],
                          t["dy"], o["out"], ck, sc, o["d_delta"], o["d_u"], o["d_B"], o["d_C"],
                          o["d_A_log"], o["d_D"], o["d_gate"])
    torch.cuda.synchronize()
    ms.mamba_scan_status()
    return o


def _inputs(shape):
    if shape == (8, 1024, 1536, 16):
        return synth.make_inputs(synth.BY_NAME["mamba130m"])
    return synth.random_inputs(*shape, seed=sum(shape) + 3, a_log_random=True)


SHAPES = [(8, 1024, 1536, 16), (1, 300, 64, 64), (2, 40, 64, 32), (2, 33, 64, 24),
          (4, 129, 256, 16), (1, 17, 8, 16), (1, 100, 72, 40)]
IDS = ["mamba130m", "dstate64_segments", "dstate32", "dstate24_pad32", "4x129x256", "T17_d8",
       "d72_dstate40"]


@pytest.mark.parametrize("shape", SHAPES, ids=IDS)
def test_bf16_matches_oracle(shape):
    bf, vals = _bf16_inputs(_inputs(shape))
    got = {k: v.float().cpu().numpy() for k, v in run_bf16(bf, vals).items()}
    ref = oracle_all(vals)
    for k in BF_OUT:
        r = ref[k].reshape(got[k].shape)
        m = float(np.max(np.abs(r)))
        bound = 2.0 ** -8 * np.abs(r) + 1.01e-4 * m
        err = np.abs(got[k].astype(np.float64) - r)
        assert np.all(err <= bound), (k, float(np.max(err - bound)), m)
    for k in F32_OUT:
        r = ref[k].reshape(got[k].shape)
        m = float(np.max(np.abs(r)))
        assert float(np.max(np.abs(got[k] - r))) <= TOL * m, k


@pytest.mark.parametrize("shape", [(8, 1024, 1536, 16), (1, 300, 64, 64), (2, 33, 64, 24)],
                         ids=["mamba130m", "dstate64_segments", "dstate24_pad32"])
def test_bf16_equals_rounded_fp32_call(shape):
    import torch
    bf, vals = _bf16_inputs(_inputs(shape))
    got = run_bf16(bf, vals)
    f32 = run_fp32_fused(vals)
    same_y = shape[3] <= 16   # both calls form y in the backward
    for k in BF_OUT:
        if not same_y and k in ("out", "d_gate"):
            continue
        want = f32[k].to(torch.bfloat16)
        assert torch.equal(got[k].view(torch.int16), want.view(torch.int16)), k
    for k in F32_OUT:
        assert torch.equal(got[k], f32[k]), k


@pytest.mark.parametrize("shape", [(2, 40, 64, 8), (2, 40, 36, 16), (2, 16, 64, 16),
                                   (2, 40, 64, 20)],
                         ids=["dstate8", "d_inner36", "T16", "dstate20"])
def test_bf16_unsupported_sizes(shape):
    import selective_state_space_06_gb300 as ms
    bf, vals = _bf16_inputs(synth.random_inputs(*shape, seed=1, a_log_random=True))
    with pytest.raises(ms.MambaScanError) as e:
        run_bf16(bf, vals)
    assert e.value.code == ms.MAMBA_ERR_UNSUPPORTED
