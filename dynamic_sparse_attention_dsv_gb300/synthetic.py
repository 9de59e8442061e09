"""Seeded synthetic inputs shaped like video-latent attention (no method arithmetic).

This module only builds inputs: shapes, the five workload configurations and
the seeded random tensors. It computes nothing the DSV method computes, so both
the CUDA path and the CPU oracle may consume its output.

Input recipe (the DSV pages evaluate on video datasets that are not available
here; these seeded tensors stand in for video-latent Q/K/V):

* Tokens lie on a T x Y x X latent grid, flattened as s = (t*Y + y)*X + x.
* P is a per-token 3D sinusoidal embedding of width d: d/4 channels for the
  time axis and 3d/8 each for the two spatial axes; each axis uses the
  textbook 1D sinusoid [sin(p*w_m), cos(p*w_m)], w_m = 10000^(-2m/n).
* Per head h, in this draw order from numpy ``default_rng(20250000 + cfg)``:
  G_h (d x d, N(0,1)/sqrt(d)), Wq_h and Wk_h (d x r, N(0, 1/d)), the head's
  Q scale (constant or uniform, per config), then noise N_Q, N_K, N_V
  (S x d, N(0,1)).  Q = qscale_h*(P G_h + 0.5 N_Q), K = P G_h + 0.5 N_K,
  V = P G_h + 0.5 N_V.  After all heads, dO ~ N(0,1) of shape [H, S, d].
* Every tensor is rounded fp64 -> fp32 -> bf16 (round to nearest even) on the
  host; the CUDA path and the oracle read the identical bf16 bits.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    """One workload: B=1, H heads, a T x Y x X latent grid, head dim d, rank r,
    query-group cube gt x gy x gx and k selected keys per group."""

    name: str
    cfg: int
    H: int
    T: int
    Y: int
    X: int
    d: int
    r: int
    gt: int
    gy: int
    gx: int
    k: int                      # keys per group (0: set per head by coverage)
    qscale: tuple               # ("const", c) or ("uniform", lo, hi)
    backward: bool

    @property
    def S(self) -> int:
        return self.T * self.Y * self.X

    @property
    def G(self) -> int:
        return self.gt * self.gy * self.gx

    @property
    def n_groups(self) -> int:
        return self.S // self.G


def k_of_fraction(p: float, S: int) -> int:
    """Keys per group for a fraction p of S, rounded half up (1638 = 10% of 16384)."""
    return int(math.floor(p * S + 0.5))


WORKLOADS = {
    0: Workload("oracle-scale forward: H=1, 4x16x16 (S=1024), d=64, r=16, cube 4x4x4, k=128",
                0, 1, 4, 16, 16, 64, 16, 4, 4, 4, 128, ("const", 4.0), False),
    1: Workload("forward+backward: H=8, 8x32x64 (S=16384), d=64, r=32, cube 4x4x4, k=1638",
                1, 8, 8, 32, 64, 64, 32, 4, 4, 4, 1638, ("const", 4.0), True),
    2: Workload("video-DiT layer forward+backward: H=24, 16x64x64 (S=65536), d=128, r=32, cube 2x8x8, k=6554",
                2, 24, 16, 64, 64, 128, 32, 2, 8, 8, 6554, ("uniform", 2.0, 8.0), True),
    3: Workload("low-rank top-k sweep: H=24, 32x64x64 (S=131072), d=128, r in {16,32,64}, cube 2x8x8",
                3, 24, 32, 64, 64, 128, 32, 2, 8, 8, 13107, ("uniform", 2.0, 8.0), False),
    4: Workload("dispatcher-driven layer: H=16, 64x64x64 (S=262144), d=128, r=32, cube 2x8x8, per-head k",
                4, 16, 64, 64, 64, 128, 32, 2, 8, 8, 0, ("uniform", 1.0, 8.0), True),
}

#: the k sweep of the low-rank top-k workload, as fractions of S
TOPK_SWEEP_FRACTIONS = (0.01, 0.05, 0.10, 0.20)
TOPK_SWEEP_RANKS = (16, 32, 64)


def workload(cfg: int, **overrides) -> Workload:
    return dataclasses.replace(WORKLOADS[cfg], **overrides) if overrides else WORKLOADS[cfg]


def sinusoid_3d(T: int, Y: int, X: int, d: int) -> np.ndarray:
    """[S, d] float64 3D sinusoidal embedding (time d/4, height 3d/8, width 3d/8)."""
    dt = d // 4
    dy = (d - dt) // 2
    dx = d - dt - dy

    def axis(n_pos: int, n: int) -> np.ndarray:
        pos = np.arange(n_pos, dtype=np.float64)[:, None]
        m = np.arange(n // 2, dtype=np.float64)[None, :]
        w = 10000.0 ** (-2.0 * m / n)
        return np.concatenate([np.sin(pos * w), np.cos(pos * w)], axis=1)

    et, ey, ex = axis(T, dt), axis(Y, dy), axis(X, dx)
    t = np.repeat(np.arange(T), Y * X)
    y = np.tile(np.repeat(np.arange(Y), X), T)
    x = np.tile(np.arange(X), T * Y)
    return np.concatenate([et[t], ey[y], ex[x]], axis=1)


def to_bf16(a: np.ndarray) -> torch.Tensor:
    """fp64 -> fp32 -> bf16 (round to nearest even), as a CPU tensor."""
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


def make_inputs(w: Workload, seed: Optional[int] = None, with_grad_out: Optional[bool] = None,
                heads: Optional[int] = None) -> dict:
    """Builds the seeded inputs of workload ``w`` as CPU bf16 tensors.

    Returns a dict with Q, K, V ([H,S,d]), Wq, Wk ([H,d,r]), dO ([H,S,d] or
    None) and qscale (float64 [H]). ``heads`` truncates H (the draw order for
    the first heads is unchanged).
    """
    H = w.H if heads is None else heads
    S, d, r = w.S, w.d, w.r
    rng = np.random.default_rng(20250000 + w.cfg if seed is None else seed)
    P = sinusoid_3d(w.T, w.Y, w.X, d)
    Q = torch.empty((H, S, d), dtype=torch.bfloat16)
    K = torch.empty_like(Q)
    V = torch.empty_like(Q)
    Wq = torch.empty((H, d, r), dtype=torch.bfloat16)
    Wk = torch.empty_like(Wq)
    qs = np.empty(H)
    for h in range(H):
        Gh = rng.standard_normal((d, d)) / math.sqrt(d)
        Wq[h] = to_bf16(rng.standard_normal((d, r)) / math.sqrt(d))
        Wk[h] = to_bf16(rng.standard_normal((d, r)) / math.sqrt(d))
        if w.qscale[0] == "const":
            qs[h] = w.qscale[1]
        else:
            qs[h] = rng.uniform(w.qscale[1], w.qscale[2])
        base = P @ Gh
        Q[h] = to_bf16(qs[h] * (base + 0.5 * rng.standard_normal((S, d))))
        K[h] = to_bf16(base + 0.5 * rng.standard_normal((S, d)))
        V[h] = to_bf16(base + 0.5 * rng.standard_normal((S, d)))
    want = w.backward if with_grad_out is None else with_grad_out
    dO = None
    if want:
        dO = torch.empty((H, S, d), dtype=torch.bfloat16)
        for h in range(H):
            dO[h] = to_bf16(rng.standard_normal((S, d)))
    return dict(Q=Q, K=K, V=V, Wq=Wq, Wk=Wk, dO=dO, qscale=qs)
