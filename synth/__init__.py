"""Seeded synthetic inputs for the selective scan (shared by the tests, the bench and the oracle).

This module holds only the input recipe: shapes, value distributions and seeds. It contains none of
the scan's arithmetic. Every tensor is drawn from its own PCG64 stream keyed by
(seed, workload id, tensor id), in float64, and then cast to float32. Both the CUDA path and the
oracle receive these exact float32 values.

The workloads are the five selective-scan layers used to benchmark the path:
  tiny          batch=1, T=64,    d_inner=32,   d_state=16
  mamba130m     batch=8, T=1024,  d_inner=1536, d_state=16
  mamba370m     batch=8, T=2048,  d_inner=2048, d_state=16
  mamba1p4b     batch=4, T=2048,  d_inner=4096, d_state=16
  longseq       batch=1, T=65536, d_inner=2560, d_state=64

The value distributions are:
  delta = softplus(scale * N(0,1) + shift), with softplus(x) = x for x > 20, else log1p(exp(x));
  u, gate, dy ~ N(0,1);  B, C ~ bc_scale * N(0,1);
  A_log[d, n] = log(n + 1) (the S4D-real initialisation, n zero-based);
  D = 1 (tiny) or U(0.5, 1.5).
The softplus threshold of 20 follows the softplus-backward step of mamba-rs
`src/mamba_ssm/cpu/backward.rs` (Phase B3, "Softplus backward").
"""
from __future__ import annotations

import dataclasses

import numpy as np

# tensor ids: fixed forever, they key the random streams
TENSOR_IDS = {"delta": 0, "u": 1, "B": 2, "C": 3, "gate": 4, "dy": 5, "D": 6}


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    wid: int            # workload id, part of the stream key
    batch: int
    T: int
    d_inner: int
    d_state: int
    delta_scale: float  # delta = softplus(delta_scale * N(0,1) + delta_shift)
    delta_shift: float
    bc_scale: float     # B, C ~ bc_scale * N(0,1)
    d_const: bool       # D == 1 (else U(0.5, 1.5))

    @property
    def btd(self) -> int:
        return self.batch * self.T * self.d_inner

    @property
    def btn(self) -> int:
        return self.batch * self.T * self.d_state

    def shape(self):
        return (self.batch, self.T, self.d_inner, self.d_state)

    def resized(self, batch=None, T=None, d_inner=None, d_state=None, name=None) -> "Workload":
        """Same value distributions, other sizes (used for edge cases and bounded samples)."""
        return dataclasses.replace(
            self,
            name=name or self.name + "-resized",
            batch=batch or self.batch, T=T or self.T,
            d_inner=d_inner or self.d_inner, d_state=d_state or self.d_state)


WORKLOADS = [
    Workload("tiny", 0, 1, 64, 32, 16, 1.0, -1.0, 1.0, True),
    Workload("mamba130m", 1, 8, 1024, 1536, 16, 0.5, -2.0, 0.25, False),
    Workload("mamba370m", 2, 8, 2048, 2048, 16, 0.5, -2.0, 0.25, False),
    Workload("mamba1p4b", 3, 4, 2048, 4096, 16, 0.5, -2.0, 0.25, False),
    Workload("longseq", 4, 1, 65536, 2560, 64, 0.5, -3.0, 0.25, False),
]
BY_NAME = {w.name: w for w in WORKLOADS}


def _rng(seed: int, wid: int, tensor: str) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, wid, TENSOR_IDS[tensor]])))


def _normal(seed, wid, tensor, shape):
    return _rng(seed, wid, tensor).standard_normal(size=shape, dtype=np.float64)


def softplus64(x: np.ndarray) -> np.ndarray:
    """softplus in float64 with the pass-through above 20 (input distribution only)."""
    out = np.empty_like(x)
    big = x > 20.0
    out[big] = x[big]
    out[~big] = np.log1p(np.exp(x[~big]))
    return out


def make_inputs(w: Workload, seed: int = 0, with_dy: bool = True) -> dict:
    """All inputs of one forward + backward call, as contiguous float32 numpy arrays.

    Shapes: delta, u, gate, dy [batch, T, d_inner]; B, C [batch, T, d_state];
    A_log [d_inner, d_state]; D [d_inner].
    """
    b, T, Di, N = w.shape()
    x = {}
    x["delta"] = softplus64(w.delta_scale * _normal(seed, w.wid, "delta", (b, T, Di)) + w.delta_shift).astype(np.float32)
    x["u"] = _normal(seed, w.wid, "u", (b, T, Di)).astype(np.float32)
    x["B"] = (w.bc_scale * _normal(seed, w.wid, "B", (b, T, N))).astype(np.float32)
    x["C"] = (w.bc_scale * _normal(seed, w.wid, "C", (b, T, N))).astype(np.float32)
    x["gate"] = _normal(seed, w.wid, "gate", (b, T, Di)).astype(np.float32)
    x["A_log"] = np.ascontiguousarray(
        np.broadcast_to(np.log(np.arange(1, N + 1, dtype=np.float64)), (Di, N))).astype(np.float32)
    if w.d_const:
        x["D"] = np.ones(Di, dtype=np.float32)
    else:
        x["D"] = _rng(seed, w.wid, "D").uniform(0.5, 1.5, size=Di).astype(np.float32)
    if with_dy:
        x["dy"] = _normal(seed, w.wid, "dy", (b, T, Di)).astype(np.float32)
    return x


# the [batch, T, *] inputs in the order iter_input_chunks yields them
CHUNKED_KEYS = ("delta", "u", "gate", "dy", "B", "C")


def iter_input_chunks(w: Workload, seed: int = 0, chunk: int = 1 << 26):
    """The [batch, T, *] inputs of make_inputs(w, seed) in pieces, for sizes whose float64 draws
    would not fit in host memory at once. Yields (name, start, values): float32 values of the
    flattened (C-order) tensor from element `start` on. Each tensor's stream is drawn in the
    same order as in make_inputs, so the pieces join into exactly make_inputs' values."""
    b, T, Di, N = w.shape()
    for name in CHUNKED_KEYS:
        n = b * T * (N if name in ("B", "C") else Di)
        g = _rng(seed, w.wid, name)
        for start in range(0, n, chunk):
            v = g.standard_normal(size=min(chunk, n - start), dtype=np.float64)
            if name == "delta":
                v = softplus64(w.delta_scale * v + w.delta_shift)
            elif name in ("B", "C"):
                v = w.bc_scale * v
            yield name, start, v.astype(np.float32)


def small_inputs(w: Workload, seed: int = 0) -> dict:
    """A_log [d_inner, d_state] and D [d_inner] of make_inputs(w, seed)."""
    b, T, Di, N = w.shape()
    A_log = np.ascontiguousarray(
        np.broadcast_to(np.log(np.arange(1, N + 1, dtype=np.float64)), (Di, N))).astype(np.float32)
    if w.d_const:
        D = np.ones(Di, dtype=np.float32)
    else:
        D = _rng(seed, w.wid, "D").uniform(0.5, 1.5, size=Di).astype(np.float32)
    return {"A_log": A_log, "D": D}


def random_inputs(batch, T, d_inner, d_state, seed=0, a_log_random=False) -> dict:
    """Generic asymmetric inputs for small cases (edge cases, pins).

    Same recipe as the mamba130m workload; with a_log_random, A_log ~ U(-1, 1.5) so that no
    structure of the S4D-real initialisation can hide an indexing mistake.
    """
    w = Workload("random", 100 + seed, batch, T, d_inner, d_state, 0.5, -1.0, 0.5, False)
    x = make_inputs(w, seed)
    if a_log_random:
        x["A_log"] = _rng(seed, w.wid, "D").uniform(-1.0, 1.5, size=(d_inner, d_state)).astype(np.float32)
    return x
