"""The launch plan's choices for the timed layers, read back through the size queries (host only).

The checkpoint buffer holds, besides the chunk checkpoints and y, one aggregate slot per
forward time segment; the scratch buffer holds the backward's per-block d_B/d_C partials,
per-segment d_A_log/d_D partials and one aggregate slot per backward pre-pass sub-segment.
Each region starts on a 256-byte boundary. So the byte counts fix the segment counts the
planner chose, and a change to the planner shows up here:
  * longseq (1 x 65536 x 2560 x 64): forward in 76 segments (80 blocks of 32 channels: 6080
    CTAs, 8 whole waves of 5 per SM on 152 SMs); backward in 19 segments (1520 CTAs, 5 waves of
    2 per SM), its pre-pass in 8 sub-segments of each (2880 CTAs);
  * mamba370m (8 x 2048 x 2048 x 16): forward in one segment; backward in 7 segments of 16
    blocks (896 CTAs), its pre-pass in 2 sub-segments of each.
"""
import pytest


@pytest.fixture(scope="module")
def ms():
    import __graft_entry__
    __graft_entry__.build()
    import selective_state_space_06_gb300 as m
    return m


def _ru(x, a=64):   # floats, 256-byte regions
    return (x + a - 1) // a * a


def _ckpt_bytes(b, T, Di, N, fwd_nseg):
    bdn, bd = b * Di * N, b * Di
    ck = _ru((T // 16 - 1) * bdn)
    if fwd_nseg > 1:
        ck = _ru(ck + fwd_nseg * bdn)
        ck = _ru(ck + fwd_nseg * bd)
    return 4 * _ru(ck + b * T * Di)


def _scratch_bytes(b, T, Di, N, nblk, nseg, nsub):
    bdn, bd, btn = b * Di * N, b * Di, b * T * N
    off = _ru(nblk * btn)
    off = _ru(off + nblk * btn)
    off = _ru(off + nseg * bdn)
    off = _ru(off + nseg * bd)
    off = _ru(off + nseg * nsub * bdn)
    return 4 * _ru(off + nseg * nsub * bd)


def test_longseq_plan(ms):
    shape = (1, 65536, 2560, 64)
    assert ms.mamba_scan_ckpt_bytes(*shape) == _ckpt_bytes(*shape, fwd_nseg=76)
    assert ms.mamba_scan_scratch_bytes(*shape) == _scratch_bytes(*shape, nblk=80, nseg=19, nsub=8)


def test_mamba370m_plan(ms):
    shape = (8, 2048, 2048, 16)
    assert ms.mamba_scan_ckpt_bytes(*shape) == _ckpt_bytes(*shape, fwd_nseg=1)
    assert ms.mamba_scan_scratch_bytes(*shape) == _scratch_bytes(*shape, nblk=16, nseg=7, nsub=2)
