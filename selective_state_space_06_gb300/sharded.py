"""Batch-sharded selective scan over several processes, one GPU each.

Every row (b, d) of the scan is independent, so the batch splits across ranks with no exchange
on the data path: rank r runs mamba_scan_fwd and mamba_scan_bwd on its own contiguous slice of
batch rows, and its out, d_delta, d_u, d_gate, d_B and d_C are already that slice of the
whole-batch result. The two parameter gradients are sums over the batch as well as over time
(the d_layer.a_log and d_layer.d_param accumulators of Phase B3 in mamba-rs
src/mamba_ssm/cpu/backward.rs), so each rank holds only its slice's share of d_A_log and d_D.
One all-reduce (sum) of those d_inner * (d_state + 1) floats, packed into one buffer, completes
them on every rank. That is the path's only collective.

The sum over ranks runs in the collective library's order, so d_A_log and d_D agree with a
single-process call up to rounding, not bit for bit.

shard_rows and allreduce_param_grads carry no scan arithmetic and run on any torch.distributed
backend (the tests drive them over gloo on CPU); sharded_fwd_bwd is the CUDA path and needs the
built library.
"""
from __future__ import annotations


def shard_rows(batch: int, rank: int, world_size: int) -> tuple[int, int]:
    """[b0, b1): the contiguous batch rows of `rank`. The first batch % world_size ranks take
    one row more than the others; a rank may get no rows when world_size > batch."""
    if world_size < 1 or not 0 <= rank < world_size or batch < 0:
        raise ValueError(f"bad shard request: batch={batch} rank={rank} world={world_size}")
    base, extra = divmod(batch, world_size)
    b0 = rank * base + min(rank, extra)
    return b0, b0 + base + (1 if rank < extra else 0)


def allreduce_param_grads(d_A_log, d_D, group=None) -> None:
    """Sums d_A_log [d_inner, d_state] and d_D [d_inner] over the ranks of `group`, in place,
    with one all-reduce of a packed buffer."""
    import torch
    import torch.distributed as dist
    n_a = d_A_log.numel()
    buf = torch.cat([d_A_log.reshape(-1), d_D.reshape(-1)])
    dist.all_reduce(buf, op=dist.ReduceOp.SUM, group=group)
    d_A_log.copy_(buf[:n_a].view_as(d_A_log))
    d_D.copy_(buf[n_a:].view_as(d_D))


def sharded_fwd_bwd(x: dict, bufs: dict, group=None, stream=None) -> dict:
    """Forward + backward of this rank's batch slice on its GPU, then the all-reduce of d_A_log
    and d_D.

    x holds this rank's slice of delta, u, B, C, gate, dy ([rows, T, ...] device tensors, the
    rows given by shard_rows) and the full A_log, D; bufs is
    selective_state_space_06_gb300.alloc_like_outputs for that slice. Returns bufs, whose
    d_A_log and d_D then hold the whole batch's sums and the rest this slice's outputs."""
    import selective_state_space_06_gb300 as ms
    ms.forward_backward(x, bufs, stream=stream)
    allreduce_param_grads(bufs["d_A_log"], bufs["d_D"], group=group)
    return bufs
