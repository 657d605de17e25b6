"""mamba_scan_fwd_bwd_host: forward + backward from host buffers, against the fp64 oracle.

The host entry cuts the work into up to four slices, each on its own stream, so that the
copies in both directions overlap the kernels. A batch of four rows or more is cut by batch
rows (d_A_log and d_D are then the slices' sums added in slice order); a smaller batch is cut
into blocks of channels (each slice the whole batch over its channels, moved with 2-D copies;
d_B and d_C are then the slices' sums added in slice order). The outputs must meet the parity
bar of the device entry points on every element (out and the seven gradients; y is not
returned by this call). The shapes cover four batch slices (mamba130m), three with a shorter
last one (batch 5), one slice (rows of T*d_inner not a multiple of 4 floats, where slices
could not start on 16-byte boundaries), and channel slices at batch 1 (d_state 64, with a
narrower last block) and batch 2 (d_state 16).
"""
import numpy as np
import pytest

import synth
from gpu_helpers import IN_KEYS, assert_parity, oracle_all

pytestmark = pytest.mark.gpu

KEYS = ("out", "d_delta", "d_u", "d_B", "d_C", "d_A_log", "d_D", "d_gate")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import selective_state_space_06_gb300  # noqa: F401


def _run_host(x, repeat=2):
    import torch
    import selective_state_space_06_gb300 as ms
    b, T, Di = x["delta"].shape
    N = x["B"].shape[2]
    hin = {k: torch.from_numpy(np.ascontiguousarray(x[k])).pin_memory() for k in IN_KEYS}
    shapes = {"out": (b, T, Di), "d_delta": (b, T, Di), "d_u": (b, T, Di), "d_gate": (b, T, Di),
              "d_B": (b, T, N), "d_C": (b, T, N), "d_A_log": (Di, N), "d_D": (Di,)}
    ws = torch.empty(ms.mamba_scan_host_workspace_bytes(b, T, Di, N), dtype=torch.uint8,
                     device="cuda:0")
    results = []
    for _ in range(repeat):
        hout = {k: torch.full(s, float("nan")).pin_memory() for k, s in shapes.items()}
        ms.mamba_scan_fwd_bwd_host(hin["delta"], hin["u"], hin["B"], hin["C"], hin["gate"],
                                   hin["A_log"], hin["D"], hin["dy"], hout["out"],
                                   hout["d_delta"], hout["d_u"], hout["d_B"], hout["d_C"],
                                   hout["d_A_log"], hout["d_D"], hout["d_gate"], ws)
        ms.mamba_scan_status()
        results.append({k: v.numpy().copy() for k, v in hout.items()})
    return results


@pytest.mark.parametrize("shape", [(8, 1024, 1536, 16), (5, 100, 64, 16), (3, 37, 50, 5),
                                   (1, 300, 260, 64), (2, 200, 512, 16), (1, 150, 600, 64)],
                         ids=["mamba130m_4slices", "batch5_3slices", "ragged_1slice",
                              "batch1_4_channel_slices", "batch2_8_channel_slices",
                              "batch1_8_channel_slices_narrow_last"])
def test_host_entry_matches_oracle(shape):
    if shape[0] == 8:
        x = synth.make_inputs(synth.BY_NAME["mamba130m"])
    else:
        x = synth.random_inputs(*shape, seed=sum(shape), a_log_random=True)
    first, second = _run_host(x)
    ref = oracle_all(x)
    assert_parity(first, ref, keys=KEYS, label=f"host {shape}")
    for k in KEYS:   # bitwise repeatable from call to call
        assert np.array_equal(first[k], second[k]), k


def _host_call(ms, torch, x, stream):
    """One host-entry call on `stream` with its own workspace and pinned outputs."""
    b, T, Di = x["delta"].shape
    N = x["B"].shape[2]
    hin = {k: torch.from_numpy(np.ascontiguousarray(x[k])).pin_memory() for k in IN_KEYS}
    shapes = {"out": (b, T, Di), "d_delta": (b, T, Di), "d_u": (b, T, Di), "d_gate": (b, T, Di),
              "d_B": (b, T, N), "d_C": (b, T, N), "d_A_log": (Di, N), "d_D": (Di,)}
    ws = torch.empty(ms.mamba_scan_host_workspace_bytes(b, T, Di, N), dtype=torch.uint8,
                     device="cuda:0")
    hout = {k: torch.full(s, float("nan")).pin_memory() for k, s in shapes.items()}
    ms.mamba_scan_fwd_bwd_host(hin["delta"], hin["u"], hin["B"], hin["C"], hin["gate"],
                               hin["A_log"], hin["D"], hin["dy"], hout["out"],
                               hout["d_delta"], hout["d_u"], hout["d_B"], hout["d_C"],
                               hout["d_A_log"], hout["d_D"], hout["d_gate"], ws, stream=stream)
    return {k: v.numpy().copy() for k, v in hout.items()}


@pytest.mark.parametrize("shape", [(1, 300, 260, 64), (5, 100, 64, 16)],
                         ids=["channel_slices", "batch_slices"])
def test_host_entry_concurrent_threads(shape):
    """Two host threads call the host entry at the same time, each on its own stream and
    inputs. The calls share the library's streams and events; every result must equal the same
    call made alone, bit for bit."""
    import threading
    import torch
    import selective_state_space_06_gb300 as ms
    xs = [synth.random_inputs(*shape, seed=40 + i, a_log_random=True) for i in range(2)]
    solo = [_host_call(ms, torch, x, torch.cuda.current_stream()) for x in xs]
    got = [[], []]
    errors = []

    def worker(i):
        try:
            torch.cuda.set_device(0)
            s = torch.cuda.Stream()
            for _ in range(3):
                got[i].append(_host_call(ms, torch, xs[i], s))
        except Exception as e:   # reported by the main thread
            errors.append(repr(e))

    th = [threading.Thread(target=worker, args=(i,)) for i in range(2)]
    for t in th:
        t.start()
    for t in th:
        t.join()
    assert errors == []
    for i in range(2):
        assert len(got[i]) == 3
        for r in got[i]:
            for k in KEYS:
                assert np.array_equal(r[k], solo[i][k]), (i, k)
