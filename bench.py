#!/usr/bin/env python3
"""Selective-scan forward + backward throughput on GB300 (one JSON line on stdout).

A step is one mamba_scan_fwd plus one mamba_scan_bwd over one batch of synthetic inputs that
already sit in HBM. That is every step of the hot path: the A = -exp(A_log) prologue, the
chunked forward scan with its checkpoints, the gating backward, the recompute, the reverse
recurrence and the fixed-order reductions.
  metric = (batch * T * d_inner) / (t_fwd + t_bwd), in elements/s.
  e2e    = the same metric through mamba_scan_fwd_bwd_host with pinned HOST buffers: the
           host->device copies of the inputs and the device->host copies of out and all seven
           gradients fall inside the timed region.
The headline workload is the largest single-GPU layer, the long-sequence wide-state scan
(batch 1, T 65536, d_inner 2560, d_state 64). The same run also times the Mamba-370M- and
Mamba-1.4B-width layers (d_state 16) and the Mamba-130M-width layer and reports them under
`per_workload`, each with its forward, backward and step times and its HBM and ALU fractions.
--workload picks another headline. --impl reference times the fp64 CPU oracle on a bounded
sample of the same workload instead.

Besides the step, `variants` reports (unless --no-variants) the softplus-fused calls, the
fused forward + backward call (mamba_scan_fwd_bwd) and its bf16 I/O form, and the causal
conv1d + SiLU step before the scan, each timed on the same workload.

Multi-GPU runs (torchrun) are independent replicas, one per GPU. The scan has no cross-device
exchange, so there is no collective on the data path. value = all ranks' elements / max time.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "selective-scan fwd+bwd (batch*T*d_inner)/sec"
UNIT = "elements/s"
DEFAULT_WORKLOAD = "longseq"
# the other layers timed in the same run (`per_workload`)
PER_WORKLOAD = ("mamba370m", "mamba1p4b", "mamba130m")


def minimal_bytes(w) -> dict:
    """Algorithmic (minimal) HBM bytes: each input read once, each output written once; fp32."""
    btd, btn, dn, d = w.btd, w.btn, w.d_inner * w.d_state, w.d_inner
    return {
        "fwd": 4 * (4 * btd + 2 * btn + dn + d),
        "bwd": 4 * (7 * btd + 4 * btn + 2 * dn + 2 * d),
        "total": 4 * (11 * btd + 6 * btn + 3 * dn + 3 * d),
    }


# Algorithmic compute per (b, t, d, n) of one step (forward + backward): 2 ex2 (the forward's
# decay and the backward's, recomputed or kept) and about 15 fp32 operations (forward 4,
# recompute 3, reverse 8), an FMA counting as one operation.
EX2_PER_ELEMENT_STATE = 2
FP32_OPS_PER_ELEMENT_STATE = 15
# Unit counts of the GB300: 152 SMs, 128 fp32 lanes per SM, and an ex2 rate of 32 per clock per
# SM (measured by a microbenchmark on this GPU); the peaks scale with the sampled SM clock.
SMS, FP32_LANES_PER_SM, EX2_PER_CLK_PER_SM = 152, 128, 32


def alu_roofline(w, step_s: float, sm_mhz: float) -> dict:
    """Achieved fp32 and ex2 rates of the whole step against the unit-count peaks."""
    ns = w.btd * w.d_state
    ghz = sm_mhz / 1e3
    out = {}
    for key, per, lanes in (("fp32", FP32_OPS_PER_ELEMENT_STATE, FP32_LANES_PER_SM),
                            ("ex2", EX2_PER_ELEMENT_STATE, EX2_PER_CLK_PER_SM)):
        achieved = per * ns / step_s / 1e9
        peak = SMS * lanes * ghz
        out[key] = {"achieved": achieved, "peak": peak, "unit": "Gop/s", "frac": achieved / peak,
                    "ops_per_element_state": per}
    out["peak_source"] = f"unit counts x sampled SM clock {sm_mhz:.0f} MHz"
    return out


def read_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "source": "fallback"}


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons; keeps only samples taken inside
    [start, stop] of the timed region."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.samples = []
        self.t0 = self.t1 = None
        self._stop = threading.Event()
        self._thr = None

    def _run(self):
        while not self._stop.is_set():
            try:
                r = subprocess.run(
                    ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                     "--format=csv,noheader,nounits"], capture_output=True, text=True, timeout=5)
                now = time.time()
                if r.returncode == 0 and r.stdout.strip():
                    self.samples.append((now, [c.strip() for c in r.stdout.strip().split(",")]))
            except Exception:
                return
            self._stop.wait(0.05)

    def start(self):
        self._thr = threading.Thread(target=self._run, daemon=True)
        self._thr.start()

    def mark(self, t0, t1):
        self.t0, self.t1 = t0, t1

    def stop(self) -> dict:
        self._stop.set()
        if self._thr:
            self._thr.join(timeout=10)
        inside = [s for t, s in self.samples if self.t0 is not None and self.t0 <= t <= self.t1]
        if not inside and self.samples and self.t0 is not None:   # nearest sample to the region
            mid = 0.5 * (self.t0 + self.t1)
            inside = [min(self.samples, key=lambda ts: abs(ts[0] - mid))[1]]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}

        def num(v):
            try:
                return float(v)
            except ValueError:
                return None
        sm = [num(s[1]) for s in inside if num(s[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in inside for i in range(4) if s[5 + i].strip() == "Active"})
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": num(inside[0][2]), "reasons": reasons, "samples": len(inside)}


def max_over_ranks(pg, value: float, device) -> float:
    """The largest of every rank's value: a replicated job takes as long as its slowest rank.
    pg is torch.distributed (any backend) or None for one rank."""
    if pg is None:
        return value
    import torch
    t = torch.tensor([float(value)], device=device, dtype=torch.float64)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: float, world_size: int, seconds: float) -> float:
    """Whole-job throughput of world_size replicas that each process units_per_rank units."""
    return world_size * units_per_rank / seconds


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# The roofline is that of one mamba_scan_bwd call, the dominant part of the step (its kernels
# together; the call is the unit the minimal-traffic count is defined for).
BWD_CALL_KERNELS = ("mamba_scan_bwd call: segment pre-pass + carry composition + "
                    "scan_bwd_tmem_kernel + scan_reduce_kernel (d_state 16-64)")
# Algorithmic compute of the backward call alone per (b, t, d, n): the recompute (3 fp32
# operations) and the reverse step (8), 1 ex2.
BWD_FP32_OPS_PER_ELEMENT_STATE = 11
BWD_EX2_PER_ELEMENT_STATE = 1

# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum, summed over the call's kernels) of
# one mamba_scan_bwd call, taken from an ncu capture of these kernels (the launch list with
# those two metrics, run on this bench's own command with --steps 3 --warmup 3). Each entry
# carries the digest of the sources of the backward call's kernels and of their launch plan
# (kernel_digest() below); once those sources differ, the entry no longer describes the
# kernels and `traffic` is reported as null. The long-sequence figure was captured at
# T = 8192 (--seq-len 8192) and scaled by 8: every term of it is proportional to T except the
# pre-pass aggregates and the carry composition's reads of them (about 2 % of it).
BWD_TRAFFIC_CAPTURES = {
    # workload: (bytes per call, kernel digest, how the figure was taken)
    "mamba370m": (1625.6e6, "6e01a96729b114b0", "ncu capture at the full size"),
    "mamba1p4b": (1626.1e6, "6e01a96729b114b0", "ncu capture at the full size"),
    "mamba130m": (550.7e6, "6e01a96729b114b0", "ncu capture at the full size"),
    "longseq": (8 * 1962.2e6, "6e01a96729b114b0", "ncu capture at T = 8192, scaled by 8"),
}
# the files that define the backward call's kernels and their launch plan
BWD_KERNEL_SOURCES = ("scan_common.cuh", "scan_plan.h", "scan_plan.cu", "scan_bwd.cu",
                      "scan_bwd_tmem.cu")


def kernel_digest() -> str:
    """sha256 (first 16 hex digits) over the backward call's kernel and plan sources."""
    import hashlib
    d = os.path.join(ROOT, "selective_state_space_06_gb300", "csrc")
    h = hashlib.sha256()
    for name in BWD_KERNEL_SOURCES:
        with open(os.path.join(d, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def bwd_traffic(name: str):
    cap = BWD_TRAFFIC_CAPTURES.get(name)
    if cap is None or cap[1] != kernel_digest():
        return None, None
    return cap[0], cap[2]


def roofline_of(w, fwd_s: float, bwd_s: float, step_s: float, sm_mhz: float, hbm_gbs: float,
                hbm_source: str) -> dict:
    """The backward call's roofline. Both of its bounds are given: HBM (minimal bytes over the
    call's time against the measured copy bandwidth) and fp32 ALU (algorithmic operations over
    the call's time against 152 SMs x 128 lanes x the sampled clock). `bound` names the one
    whose floor is higher for this workload, and the top-level fields are that bound's."""
    mb = minimal_bytes(w)
    ns = w.btd * w.d_state
    ghz = sm_mhz / 1e3
    hbm_ach = mb["bwd"] / bwd_s / 1e9
    alu_ach = BWD_FP32_OPS_PER_ELEMENT_STATE * ns / bwd_s / 1e9
    alu_peak = SMS * FP32_LANES_PER_SM * ghz
    hbm_floor = mb["bwd"] / (hbm_gbs * 1e9)
    alu_floor = BWD_FP32_OPS_PER_ELEMENT_STATE * ns / (alu_peak * 1e9)
    traffic, how = bwd_traffic(w.name)
    hbm = {"achieved": hbm_ach, "peak": hbm_gbs, "unit": "GB/s", "frac": hbm_ach / hbm_gbs,
           "peak_source": f"{hbm_source} (MEASURED_PEAKS.json hbm_gbs)"
           if hbm_source == "measured" else "fallback 6.8 TB/s"}
    alu = {"achieved": alu_ach, "peak": alu_peak, "unit": "Gop/s", "frac": alu_ach / alu_peak,
           "ops_per_element_state": BWD_FP32_OPS_PER_ELEMENT_STATE,
           "peak_source": f"152 SMs x 128 fp32 lanes x sampled SM clock {sm_mhz:.0f} MHz"}
    bound = "alu" if alu_floor > hbm_floor else "hbm"
    top = alu if bound == "alu" else hbm
    return {"kernel": BWD_CALL_KERNELS, "bound": bound, "achieved": top["achieved"],
            "peak": top["peak"], "unit": top["unit"], "frac": top["frac"],
            "peak_source": top["peak_source"], "traffic": traffic, "traffic_capture": how,
            "algorithmic_bytes_per_launch": mb["bwd"],
            "algorithmic_fp32_ops_per_launch": BWD_FP32_OPS_PER_ELEMENT_STATE * ns,
            "hbm": hbm, "alu": alu,
            "hbm_frac_fwd": mb["fwd"] / fwd_s / 1e9 / hbm_gbs,
            "hbm_frac_step": mb["total"] / step_s / 1e9 / hbm_gbs}


def time_conv(ms, w, dev, stream, steps, hbm_gbs, K=4) -> dict:
    """The causal conv1d + SiLU step before the scan (d_conv 4) on this workload's
    [batch, T, d_inner]: CUDA-event times of its forward and backward, and their fractions of
    HBM against the minimal bytes (fwd reads x, writes u; bwd reads x and d_u, writes d_x)."""
    import torch
    b, T, Di = w.batch, w.T, w.d_inner
    g = torch.Generator(device=dev).manual_seed(0)
    # three buffer sets used in turn: one set (x, u, d_u, d_x: 200 MB at mamba130m) would let a
    # launch find the previous one's data in the 126 MB L2; three sets keep each launch on HBM
    nset = 3
    sets = []
    for _ in range(nset):
        x = torch.randn(b, T, Di, device=dev, generator=g)
        sets.append({"x": x, "d_u": torch.randn(b, T, Di, device=dev, generator=g),
                     "u": torch.empty_like(x), "d_x": torch.empty_like(x)})
    wt = torch.randn(Di, K, device=dev, generator=g) * 0.5
    bias = torch.randn(Di, device=dev, generator=g) * 0.3
    d_w, d_b = torch.empty_like(wt), torch.empty_like(bias)
    sc = torch.empty(ms.mamba_conv_scratch_bytes(b, T, Di, K) // 4, device=dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]

    def fwd(i):
        z = sets[i % nset]
        ms.mamba_conv_fwd(z["x"], wt, bias, z["u"], stream=stream)

    def bwd(i):
        z = sets[i % nset]
        ms.mamba_conv_bwd(z["x"], wt, bias, z["d_u"], sc, z["d_x"], d_w, d_b, stream=stream)

    for i in range(3):
        fwd(i)
        bwd(i)
    # back-to-back launches between two events, so that the short kernels are timed with a
    # full queue rather than with the host's launch latency
    torch.cuda.synchronize()
    ev[0].record(stream)
    for i in range(steps):
        fwd(i)
    ev[1].record(stream)
    for i in range(steps):
        bwd(i)
    ev[2].record(stream)
    torch.cuda.synchronize()
    fwd_ms = ev[0].elapsed_time(ev[1]) / steps
    bwd_ms = ev[1].elapsed_time(ev[2]) / steps
    btd = b * T * Di
    fwd_bytes = 4 * (2 * btd + Di * K + Di)
    bwd_bytes = 4 * (3 * btd + 2 * Di * K + 2 * Di)
    return {"d_conv": K, "fwd_ms": fwd_ms, "bwd_ms": bwd_ms, "steps": steps,
            "fwd_hbm_frac": fwd_bytes / (fwd_ms * 1e-3) / 1e9 / hbm_gbs,
            "bwd_hbm_frac": bwd_bytes / (bwd_ms * 1e-3) / 1e9 / hbm_gbs}


def time_steps(ms, x, bufs, stream, steps, warmup, pg=None, sampler=None) -> dict:
    """Times `steps` steps (mamba_scan_fwd + mamba_scan_bwd) after `warmup` untimed ones.

    One pair of events brackets the whole timed region (after a barrier and a synchronize). On a
    regular sample of the steps (every fourth step, or more sparsely beyond 256 steps), events on
    the launching stream also split the forward call from the backward call. An event between
    two calls stops the second call's first kernel from starting early (programmatic dependent
    launch), so the other steps run without them, as a caller's would."""
    import torch

    def step(ev_mid=None):
        ms.mamba_scan_fwd(x["delta"], x["u"], x["B"], x["C"], x["gate"], x["A_log"], x["D"],
                          bufs["out"], None, bufs["ckpt"], stream=stream)
        nf = ms.mamba_scan_last_launch_count()
        if ev_mid is not None:
            ev_mid.record(stream)
        ms.mamba_scan_bwd(x["delta"], x["u"], x["B"], x["C"], x["gate"], x["A_log"], x["D"],
                          x["dy"], bufs["ckpt"], bufs["scratch"], bufs["d_delta"], bufs["d_u"],
                          bufs["d_B"], bufs["d_C"], bufs["d_A_log"], bufs["d_D"], bufs["d_gate"],
                          stream=stream)
        return nf + ms.mamba_scan_last_launch_count()

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    stride = max(4, steps // 64)
    sampled = list(range(0, steps, stride))
    ev = {i: [torch.cuda.Event(enable_timing=True) for _ in range(3)] for i in sampled}
    outer0 = torch.cuda.Event(enable_timing=True)
    outer1 = torch.cuda.Event(enable_timing=True)
    if sampler is not None:
        sampler.start()
        time.sleep(0.3)
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    t_host0 = time.time()
    outer0.record(stream)
    launches = 0
    for i in range(steps):
        e = ev.get(i)
        if e is None:
            launches += step()
        else:
            e[0].record(stream)
            launches += step(e[1])
            e[2].record(stream)
    outer1.record(stream)
    torch.cuda.synchronize()
    if pg:
        pg.barrier()
    t_host1 = time.time()
    clocks = None
    if sampler is not None:
        sampler.mark(t_host0, t_host1)
        clocks = sampler.stop()
    return {"total_ms": outer0.elapsed_time(outer1),
            "fwd_ms": float(np.mean([ev[i][0].elapsed_time(ev[i][1]) for i in sampled])),
            "bwd_ms": float(np.mean([ev[i][1].elapsed_time(ev[i][2]) for i in sampled])),
            "split_steps": len(sampled), "launches": launches, "clocks": clocks}


def time_loop(fn, stream, steps: int, warmup: int = 3) -> float:
    """Mean CUDA-event time in ms of `fn` over `steps` back-to-back calls after `warmup`."""
    import torch
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


def fused_step(ms, x, bufs, stream):
    """The forward and backward in one call (dy known up front)."""
    def f():
        ms.mamba_scan_fwd_bwd(x["delta"], x["u"], x["B"], x["C"], x["gate"], x["A_log"], x["D"],
                              x["dy"], bufs["out"], bufs["ckpt"], bufs["scratch"],
                              bufs["d_delta"], bufs["d_u"], bufs["d_B"], bufs["d_C"],
                              bufs["d_A_log"], bufs["d_D"], bufs["d_gate"], stream=stream)
    return f


def workload_entry(ms, w, dev, stream, steps, warmup, peaks, index) -> dict:
    """The step of another workload, timed on its own (same timing rules as the headline)."""
    import torch
    x = {k: torch.from_numpy(v).to(dev) for k, v in synth.make_inputs(w, seed=0).items()}
    bufs = ms.alloc_like_outputs(x["delta"], x["B"], x["A_log"], x["D"])
    r = time_steps(ms, x, bufs, stream, steps, warmup, sampler=ClockSampler(index))
    fused_ms = time_loop(fused_step(ms, x, bufs, stream), stream, max(3, min(steps, 50)))
    del x, bufs
    torch.cuda.empty_cache()
    step_s = r["total_ms"] * 1e-3 / steps
    sm_mhz = float((r["clocks"] or {}).get("sm_mhz") or 2070.0)
    return {"batch": w.batch, "T": w.T, "d_inner": w.d_inner, "d_state": w.d_state,
            "value": w.btd / step_s, "unit": UNIT, "ms_per_step": 1e3 * step_s,
            "fwd_ms": r["fwd_ms"], "bwd_ms": r["bwd_ms"], "steps": steps,
            "fused_fwd_bwd_ms": fused_ms,
            "roofline": roofline_of(w, r["fwd_ms"] * 1e-3, r["bwd_ms"] * 1e-3, step_s, sm_mhz,
                                    peaks["hbm_gbs"], peaks["source"]),
            "alu_roofline": alu_roofline(w, step_s, sm_mhz), "clocks": r["clocks"]}


def run_gpu(args):
    import torch
    import selective_state_space_06_gb300 as ms

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist
    peaks = read_peaks()
    w = synth.BY_NAME[args.workload]
    if args.seq_len:   # a shorter cut of the workload (same recipe), e.g. for counter captures
        w = w.resized(T=args.seq_len, name=f"{w.name}-T{args.seq_len}")
    x_np = synth.make_inputs(w, seed=0)
    x = {k: torch.from_numpy(v).to(dev) for k, v in x_np.items()}
    bufs = ms.alloc_like_outputs(x["delta"], x["B"], x["A_log"], x["D"])
    stream = torch.cuda.current_stream(dev)

    r = time_steps(ms, x, bufs, stream, args.steps, args.warmup, pg=pg,
                   sampler=ClockSampler(local))
    clocks = r["clocks"]
    total_ms = max_over_ranks(pg, r["total_ms"], dev)
    launches = r["launches"]

    # end-to-end through the host-buffer entry point (pinned host memory)
    e2e = None
    if not args.no_e2e:
        pin = lambda a: torch.from_numpy(a).pin_memory()  # noqa: E731
        hin = {k: pin(v) for k, v in x_np.items()}
        b, T, Di, N = w.shape()
        hout = {k: torch.empty(s, dtype=torch.float32).pin_memory() for k, s in {
            "out": (b, T, Di), "d_delta": (b, T, Di), "d_u": (b, T, Di), "d_gate": (b, T, Di),
            "d_B": (b, T, N), "d_C": (b, T, N), "d_A_log": (Di, N), "d_D": (Di,)}.items()}
        wsb = ms.mamba_scan_host_workspace_bytes(b, T, Di, N)
        wsbuf = torch.empty(wsb, dtype=torch.uint8, device=dev)

        def e2e_step():
            ms.mamba_scan_fwd_bwd_host(hin["delta"], hin["u"], hin["B"], hin["C"], hin["gate"],
                                       hin["A_log"], hin["D"], hin["dy"], hout["out"],
                                       hout["d_delta"], hout["d_u"], hout["d_B"], hout["d_C"],
                                       hout["d_A_log"], hout["d_D"], hout["d_gate"], wsbuf,
                                       stream=stream)
        for _ in range(2):
            e2e_step()
        ke = max(3, min(args.steps, 30))
        if pg:
            pg.barrier()
        t0 = time.perf_counter()
        marks = [t0]
        for _ in range(ke):
            e2e_step()   # returns once the step's results are in host memory
            marks.append(time.perf_counter())
        el = marks[-1] - t0
        el = max_over_ranks(pg, el, dev)
        per_call = sorted(1e3 * (b - a) for a, b in zip(marks, marks[1:]))
        h2d = sum(v.numel() * 4 for k, v in hin.items())
        d2h = sum(v.numel() * 4 for v in hout.values())
        # value and ms_per_step: all steps (the mean); the median and the slowest step show
        # how much of the mean comes from occasional slow calls on the shared host
        e2e = {"value": job_throughput(w.btd * ke, ws, el), "unit": UNIT,
               "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "steps": ke, "ms_per_step": 1e3 * el / ke,
               "median_ms_per_step_rank0": per_call[len(per_call) // 2],
               "max_ms_per_step_rank0": per_call[-1]}
        del wsbuf, hin, hout

    variants = {}
    if not args.no_variants:
        kv = max(3, min(args.steps, 50))
        # the softplus in front of the scan fused into the kernels (raw delta in, d_delta_raw
        # out), on the raw delta that gives this workload's delta
        raw_np = np.log(np.expm1(x_np["delta"].astype(np.float64))).astype(np.float32)
        raw = torch.from_numpy(raw_np).to(dev)
        del raw_np

        def step_sp():
            ms.mamba_scan_fwd_softplus(raw, x["u"], x["B"], x["C"], x["gate"], x["A_log"],
                                       x["D"], bufs["out"], None, bufs["ckpt"], stream=stream)
            ms.mamba_scan_bwd_softplus(raw, x["u"], x["B"], x["C"], x["gate"], x["A_log"],
                                       x["D"], x["dy"], bufs["ckpt"], bufs["scratch"],
                                       bufs["d_delta"], bufs["d_u"], bufs["d_B"], bufs["d_C"],
                                       bufs["d_A_log"], bufs["d_D"], bufs["d_gate"],
                                       stream=stream)
        ms_sp = time_loop(step_sp, stream, kv)
        variants["softplus_fused"] = {"ms_per_step": ms_sp, "value": w.btd / (ms_sp * 1e-3),
                                      "unit": UNIT, "steps": kv}
        del raw
        # forward and backward in one call when dy is known up front
        ms_fu = time_loop(fused_step(ms, x, bufs, stream), stream, kv)
        variants["fused_fwd_bwd"] = {"ms_per_step": ms_fu, "value": w.btd / (ms_fu * 1e-3),
                                     "unit": UNIT, "steps": kv,
                                     "launches": ms.mamba_scan_last_launch_count()}
        # the fused call with bf16 I/O (inputs rounded to bf16; fp32 arithmetic)
        if w.d_state % 8 == 0 and w.d_inner % 8 == 0 and 9 <= w.d_state <= 64 and w.T > 16:
            bf = {k: x[k].to(torch.bfloat16) for k in ("delta", "u", "B", "C", "gate", "dy")}
            ob = {k: torch.empty_like(bf["delta"]) for k in ("out", "d_delta", "d_u", "d_gate")}
            ob["d_B"] = torch.empty_like(bf["B"])
            ob["d_C"] = torch.empty_like(bf["C"])

            def step_bf16():
                ms.mamba_scan_fwd_bwd_bf16(bf["delta"], bf["u"], bf["B"], bf["C"], bf["gate"],
                                           x["A_log"], x["D"], bf["dy"], ob["out"], bufs["ckpt"],
                                           bufs["scratch"], ob["d_delta"], ob["d_u"], ob["d_B"],
                                           ob["d_C"], bufs["d_A_log"], bufs["d_D"],
                                           ob["d_gate"], stream=stream)
            ms_bf = time_loop(step_bf16, stream, kv)
            variants["fused_fwd_bwd_bf16"] = {"ms_per_step": ms_bf,
                                              "value": w.btd / (ms_bf * 1e-3), "unit": UNIT,
                                              "steps": kv, "io": "bf16", "arithmetic": "f32"}
            del bf, ob
        variants["conv1d_silu"] = time_conv(ms, w, dev, stream, kv, peaks["hbm_gbs"])

    del x, bufs
    torch.cuda.empty_cache()
    per_workload = {}
    if not args.no_per_workload:
        for name in PER_WORKLOAD:
            if name != w.name:
                per_workload[name] = workload_entry(ms, synth.BY_NAME[name], dev, stream,
                                                    args.steps, args.warmup, peaks, local)

    step_s = total_ms * 1e-3 / args.steps
    sm_mhz = float((clocks or {}).get("sm_mhz") or 2070.0)
    value = job_throughput(w.btd * args.steps, ws, total_ms * 1e-3)
    mb = minimal_bytes(w)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": w.name, "batch": w.batch, "T": w.T, "d_inner": w.d_inner,
                   "d_state": w.d_state, "seed": 0,
                   "l2": "no flush: inputs larger than the 126 MB L2 "
                         f"({4 * (4 * w.btd + 2 * w.btn) / 1e6:.0f} MB read per step)",
                   "parallelism": f"replicas x{ws}"},
        "fwd_ms": r["fwd_ms"], "bwd_ms": r["bwd_ms"], "fwd_bwd_split_steps": r["split_steps"],
        "hbm_frac_step": (mb["total"] / step_s / 1e9) / peaks["hbm_gbs"],
        "roofline": roofline_of(w, r["fwd_ms"] * 1e-3, r["bwd_ms"] * 1e-3, step_s, sm_mhz,
                                peaks["hbm_gbs"], peaks["source"]),
        "alu_roofline": alu_roofline(w, step_s, sm_mhz),
        "per_workload": per_workload,
        "variants": variants,
        "gpu_launches": launches,
        "clocks": clocks,
        "e2e": e2e,
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, budget_s=args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if pg:
        pg.barrier()
        pg.destroy_process_group()


def _oracle_rows_runner(w):
    """(run(rows) -> seconds) for the oracle over the first `rows` rows of the workload, with
    every output array allocated once outside the timed calls (the forward's out and y, the
    backward's per-row gradients and its accumulators, zeroed before each call)."""
    import oracle
    x = oracle.as64(synth.make_inputs(w, seed=0))
    b, T, Di, N = w.shape()
    out = np.full((b, T, Di), np.nan)
    y = np.full((b, T, Di), np.nan)
    per_row = {k: np.full((b, T, Di), np.nan) for k in ("d_delta", "d_u", "d_gate")}
    acc = {"d_B": np.zeros((b, T, N)), "d_C": np.zeros((b, T, N)),
           "d_A_log": np.zeros((Di, N)), "d_D": np.zeros(Di)}

    def run(rows):
        for a in acc.values():
            a.fill(0.0)
        t0 = time.perf_counter()
        oracle.fwd(x, rows=(0, rows), out=out, y=y)
        oracle.bwd_rows_into(x, (0, rows), per_row, acc)
        return time.perf_counter() - t0
    return run


def _calibrated_rows(w, run, budget_s):
    rows_total = w.batch * w.d_inner
    r = 1
    while True:                        # grow the probe until it takes a measurable time
        el = run(r)
        if el > 0.5 or r >= rows_total:
            break
        r = min(rows_total, r * 4)
    per_row = el / r
    return int(max(1, min(rows_total, budget_s / max(per_row, 1e-12))))


def cpu_info() -> dict:
    """The host's logical CPU count and CPU model (from /proc/cpuinfo, else lscpu)."""
    model = None
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu model")):
                    model = line.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    if model is None:
        try:
            r = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10)
            for line in r.stdout.splitlines():
                if line.strip().lower().startswith("model name"):
                    model = line.split(":", 1)[1].strip()
                    break
        except Exception:
            pass
    return {"nproc": os.cpu_count(), "cpu_model": model or "unknown"}


def cpu_baseline(w, budget_s: float = 12.0) -> dict:
    """The oracle as it stands (single-threaded fp64 C, forward + backward per row) on a bounded
    sample of rows of the workload; scaled to elements/s."""
    run = _oracle_rows_runner(w)
    rows = _calibrated_rows(w, run, budget_s)
    el = run(rows)
    return {"value": rows * w.T / el, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{rows} of {w.batch * w.d_inner} rows (b,d) x T={w.T}, fwd+bwd, fp64, "
                      f"1 thread; {el:.1f} s", **cpu_info()}


def run_reference(args):
    """Reference arm: the fp64 CPU oracle timed on the host cores, on a bounded sample of the
    same workload per step; rank 0 only."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    w = synth.BY_NAME[args.workload]
    run = _oracle_rows_runner(w)
    total_budget = 120.0
    rows = _calibrated_rows(w, run, total_budget / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        run(rows)
    el = sum(run(rows) for _ in range(args.steps))
    value = rows * w.T * args.steps / el
    sample = (f"{rows} of {w.batch * w.d_inner} rows (b,d) x T={w.T} per step, fwd+bwd, fp64, "
              "1 thread")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": w.name, "batch": w.batch, "T": w.T, "d_inner": w.d_inner,
                   "d_state": w.d_state, "seed": 0},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": sample, **cpu_info()},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(synth.BY_NAME))
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-variants", action="store_true",
                    help="skip timing the variants (softplus, fused, bf16, conv1d)")
    ap.add_argument("--no-per-workload", action="store_true",
                    help="time the headline workload only")
    ap.add_argument("--seq-len", type=int, default=0,
                    help="run the workload at this T instead of its own (same value recipe)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
