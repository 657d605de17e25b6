"""The batch-sharded layer's host logic on CPU: world_size 2 over gloo (127.0.0.1).

Each rank takes its slice of the batch from shard_rows, computes that slice's forward and
backward with the fp64 oracle (standing in for the GPU kernels, which need a GPU), and sums
d_A_log and d_D with allreduce_param_grads. The test checks that every rank then holds the
whole-batch oracle's d_A_log and d_D within 1e-12 (relative to the largest entry), and that the
per-row outputs of the slices put together are the whole-batch outputs exactly. The split also
covers a batch that does not divide evenly and a rank with no rows.
"""
import os
import socket
import sys

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def _sharded():
    """The sharded module, loaded by path: its host helpers need neither the built library nor
    a GPU (importing the package itself would load the library)."""
    import importlib.util
    path = os.path.join(ROOT, "selective_state_space_06_gb300", "sharded.py")
    spec = importlib.util.spec_from_file_location("_mamba_sharded", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


shard_rows = _sharded().shard_rows

PER_ROW = ("d_delta", "d_u", "d_gate", "d_B", "d_C")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _slice(x, b0, b1):
    y = dict(x)
    for k in ("delta", "u", "B", "C", "gate", "dy"):
        y[k] = np.ascontiguousarray(x[k][b0:b1])
    return y


def _worker(rank, world, port, shape, out):
    sys.path.insert(0, ROOT)
    import oracle
    import synth
    allreduce_param_grads = _sharded().allreduce_param_grads
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    x = synth.random_inputs(*shape, seed=21, a_log_random=True)
    b0, b1 = shard_rows(shape[0], rank, world)
    Di, N = shape[2], shape[3]
    if b1 > b0:
        g = oracle.bwd(_slice(x, b0, b1))
    else:   # no rows: zero contributions to the sums
        g = {"d_A_log": np.zeros((Di, N)), "d_D": np.zeros(Di)}
    dA = torch.from_numpy(np.ascontiguousarray(g["d_A_log"]))
    dD = torch.from_numpy(np.ascontiguousarray(g["d_D"]))
    allreduce_param_grads(dA, dD)
    out[rank] = {"rows": (b0, b1), "d_A_log": dA.numpy().copy(), "d_D": dD.numpy().copy(),
                 **{k: g[k] for k in PER_ROW if k in g}}
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("shape", [(4, 23, 6, 4), (3, 19, 5, 8), (1, 17, 4, 4)],
                         ids=["even", "uneven", "rank_without_rows"])
def test_two_ranks_match_the_whole_batch(shape):
    import oracle
    import synth
    world, port = 2, _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_worker, args=(world, port, shape, out), nprocs=world, join=True)
        res = {r: dict(out[r]) for r in range(world)}
    whole = oracle.bwd(synth.random_inputs(*shape, seed=21, a_log_random=True))
    for r in range(world):
        for k in ("d_A_log", "d_D"):
            scale = float(np.abs(whole[k]).max())
            err = float(np.abs(res[r][k] - whole[k]).max())
            assert err <= 1e-12 * scale, (r, k, err, scale)
    for k in PER_ROW:
        parts = [res[r][k] for r in range(world) if res[r]["rows"][1] > res[r]["rows"][0]]
        assert np.array_equal(np.concatenate(parts, axis=0), whole[k]), k


def test_shard_rows_covers_the_batch_once():
    for batch in range(0, 13):
        for world in range(1, 6):
            spans = [shard_rows(batch, r, world) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == batch
            for (a0, a1), (b0, b1) in zip(spans, spans[1:]):
                assert a1 == b0 and a1 >= a0
            sizes = [b - a for a, b in spans]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        shard_rows(4, 2, 2)
