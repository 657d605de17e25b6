"""The largest problems the library accepts: batch*T*d_inner just below 2^31 elements.

Two shapes of 2,143,289,344 (b, t, d) elements, 8.6 GB per [batch, T, d_inner] tensor, so every
element offset of the kernels and of their checkpoint, y and partial buffers runs past 2^31
bytes and close to 2^31 elements:
  * batch 2, T 131072, d_inner 8176, d_state 16 (the d_state-16 kernels; the last block of 128
    channels is ragged, 8176 = 63*128 + 112), with the Mamba-370M layer's value recipe;
  * batch 1, T 262144, d_inner 8176, d_state 64 (the tensor-copy forward with its time
    segments, the d_state-64 backward; 34 GB of checkpoints), with the long-sequence layer's.
The inputs are drawn in pieces (synth.iter_input_chunks) so that host memory stays bounded.

Checks, after one forward + backward with NaN-poisoned outputs:
  * no output element is left unwritten (no NaN anywhere);
  * sampled (batch row, channel) rows, the first and last channels and both batch rows among
    them, match the fp64 oracle element by element: out, y, d_delta, d_u, d_gate over all T
    steps, and d_A_log, d_D of the sampled channels (sums over both batch rows);
  * d_B and d_C, sums over all channels, through the method's exact identities (out is linear
    in B alone and in C alone, the other inputs fixed, so Euler's theorem applies to each):
    sum(d_B * B) = sum(d_C * C) = sum(w * (y - D*u)) with w = dy * g * sigmoid(g), in float64.
"""
import numpy as np
import pytest

import oracle
import synth
from gpu_helpers import TOL

pytestmark = pytest.mark.gpu

SHAPES = {"dstate16": ((2, 131072, 8176, 16), "mamba370m"),
          "dstate64": ((1, 262144, 8176, 64), "longseq")}
ROWS_D = (0, 1, 31, 32, 127, 128, 4095, 8063, 8064, 8175)   # channels sampled in every batch row
ROW_KEYS = ("out", "y", "d_delta", "d_u", "d_gate")


@pytest.fixture(scope="module", params=sorted(SHAPES))
def run(request):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import selective_state_space_06_gb300 as ms
    (b, T, Di, N), recipe = SHAPES[request.param]
    assert b * T * Di < 2 ** 31
    torch.cuda.empty_cache()
    free, _ = torch.cuda.mem_get_info()
    need = (4 * 9 * b * T * Di + 4 * 4 * b * T * N + ms.mamba_scan_ckpt_bytes(b, T, Di, N)
            + ms.mamba_scan_scratch_bytes(b, T, Di, N))
    if free < need + 16e9:
        pytest.skip(f"needs {need / 1e9:.0f} GB of device memory and some room, "
                    f"{free / 1e9:.0f} GB free")
    w = synth.BY_NAME[recipe].resized(batch=b, T=T, d_inner=Di, d_state=N, name="max-size")
    dev = torch.device("cuda:0")
    x = {k: torch.empty((b, T, N if k in ("B", "C") else Di), dtype=torch.float32, device=dev)
         for k in synth.CHUNKED_KEYS}
    chunk = 1 << 26
    stage = torch.empty(chunk, dtype=torch.float32).pin_memory()
    for name, start, v in synth.iter_input_chunks(w, seed=0, chunk=chunk):
        stage[:v.size].copy_(torch.from_numpy(v))
        x[name].view(-1)[start:start + v.size].copy_(stage[:v.size])
    small = synth.small_inputs(w, seed=0)
    x["A_log"] = torch.from_numpy(small["A_log"]).to(dev)
    x["D"] = torch.from_numpy(small["D"]).to(dev)
    bufs = ms.alloc_like_outputs(x["delta"], x["B"], x["A_log"], x["D"])
    for k in ("out", "y", "d_delta", "d_u", "d_B", "d_C", "d_A_log", "d_D", "d_gate"):
        bufs[k].fill_(float("nan"))
    bufs["scratch"].fill_(0xFF)
    bufs["ckpt"].fill_(0xFF)
    ms.forward_backward(x, bufs)
    torch.cuda.synchronize()
    ms.mamba_scan_status()
    yield (b, T, Di, N), x, bufs
    del x, bufs
    torch.cuda.empty_cache()


def test_max_size_every_output_written(run):
    import torch
    _, _, bufs = run
    for k in ("out", "y", "d_delta", "d_u", "d_B", "d_C", "d_A_log", "d_D", "d_gate"):
        assert not bool(torch.isnan(bufs[k]).any()), k


def _row_inputs(x, d):
    """Every batch row of channel d, as a (batch, d_inner=1) oracle input."""
    sl = {k: x[k][:, :, d:d + 1].cpu().numpy() for k in ("delta", "u", "gate", "dy")}
    sl["B"] = x["B"].cpu().numpy()
    sl["C"] = x["C"].cpu().numpy()
    sl["A_log"] = x["A_log"][d:d + 1].cpu().numpy()
    sl["D"] = x["D"][d:d + 1].cpu().numpy()
    return sl


def test_max_size_sampled_rows_match_oracle(run):
    _, x, bufs = run
    for d in ROWS_D:
        xi = _row_inputs(x, d)
        ref = oracle.bwd(xi)
        ref["out"], ref["y"] = oracle.fwd(xi)
        for k in ROW_KEYS:
            got = bufs[k][:, :, d:d + 1].cpu().numpy().astype(np.float64)
            r = np.asarray(ref[k], dtype=np.float64).reshape(got.shape)
            scale = float(np.abs(r).max())
            assert float(np.abs(got - r).max()) <= TOL * scale, (d, k)
        for k in ("d_A_log", "d_D"):
            got = bufs[k][d:d + 1].cpu().numpy().astype(np.float64)
            r = np.asarray(ref[k], dtype=np.float64).reshape(got.shape)
            scale = float(np.abs(r).max())
            assert float(np.abs(got - r).max()) <= TOL * scale, (d, k)


def test_max_size_d_B_d_C_identities(run):
    """sum(d_B*B) and sum(d_C*C) both equal sum(w*(y - D*u)), w = dy*g*sigmoid(g): the step's
    output is linear in B and in C for fixed other inputs. Summed in float64 in pieces of T."""
    import torch
    (b, T, Di, N), x, bufs = run
    lhs_B = float((bufs["d_B"].double() * x["B"].double()).sum())
    lhs_C = float((bufs["d_C"].double() * x["C"].double()).sum())
    rhs = 0.0
    mag = 0.0
    Dd = x["D"].double()
    step = 8192
    for t0 in range(0, T, step):
        g = x["gate"][:, t0:t0 + step].double()
        wv = x["dy"][:, t0:t0 + step].double() * g * torch.sigmoid(g)
        ymdu = bufs["y"][:, t0:t0 + step].double() - Dd * x["u"][:, t0:t0 + step].double()
        rhs += float((wv * ymdu).sum())
        mag += float((wv * ymdu).abs().sum())
    for name, lhs in (("B", lhs_B), ("C", lhs_C)):
        assert abs(lhs - rhs) <= 1e-5 * mag, (name, lhs, rhs, mag)
