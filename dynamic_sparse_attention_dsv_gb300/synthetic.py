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
* Per head h, in this draw order from numpy ``default_rng(20250000 + index)``
  (index: the workload's position in ``WORKLOADS``):
  G_h (d x d, N(0,1)/sqrt(d)), Wq_h and Wk_h (d x r, N(0, 1/d)), the head's
  Q scale (constant or uniform, per workload), then noise N_Q, N_K, N_V
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
    index: int                  # position in WORKLOADS; offsets the default seed
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


def workload(n: int, **overrides) -> Workload:
    return dataclasses.replace(WORKLOADS[n], **overrides) if overrides else WORKLOADS[n]


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
    rng = np.random.default_rng(20250000 + w.index if seed is None else seed)
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


def make_clustered_inputs(T: int, Y: int, X: int, d: int, r: int, H: int, mode: str = "spread",
                          seed: int = 7) -> dict:
    """Adversarial predictor inputs for the top-k boundary: one key far above
    and one far below the others, and every other key in a narrow cluster.

    W_lr^Q = W_lr^K = [I_r; 0], so the predictor's q_lr, k_lr are the first r
    channels of Q and K. Every query of head h is e_0 + c_h e_1 with c_h a
    power of two, and key j carries a_j in channel 0 and b_j in channel 1:
    a = 1 except a_0 = 100 and a_1 = -100; b is a seeded bf16 multiple of
    2^-12 in [-1, 1] ("spread": many distinct values, some repeated) or one of
    {-1, -1/2, 0, 1/2, 1} ("ties": large groups of exactly equal keys).
    Channels past 1 hold small seeded noise. Every a_j + c_h b_j is exact in
    fp32 (at most 21 significant bits), so any correct fp32 computation of
    the predictor scores gives them exactly.

    Two peaked shapes for the coverage search set b = 0: "two_level" puts
    every 32nd key at a = 32 and the rest at a = 0, besides a_1 = -64 (so the
    lower level sits inside the score range, not at its edge); "dominant"
    puts key 0 at a = 256 and every other key at a = 0.
    Returns Q, K, V, Wq, Wk as CPU bf16 tensors ([H,S,d] and [H,d,r]) and
    the per-head c (float64 [H]).
    """
    S = T * Y * X
    rng = np.random.default_rng(seed)
    eye = np.zeros((d, r))
    eye[np.arange(r), np.arange(r)] = 1.0
    Wq = to_bf16(np.broadcast_to(eye, (H, d, r)))
    Wk = Wq.clone()
    c = np.array([2.0 ** -(3 + 2 * (h % 3)) * (-1) ** h for h in range(H)])
    Q = np.zeros((H, S, d))
    Q[:, :, 0] = 1.0
    Q[:, :, 1] = c[:, None]
    K = 0.01 * rng.standard_normal((H, S, d))
    K[:, :, 0] = 1.0
    K[:, 0, 0], K[:, 1, 0] = 100.0, -100.0
    if mode == "spread":
        K[:, :, 1] = np.round(rng.uniform(-1.0, 1.0, (H, S)) * 4096.0) / 4096.0
    elif mode == "ties":
        K[:, :, 1] = rng.choice(np.array([-1.0, -0.5, 0.0, 0.5, 1.0]), (H, S))
    elif mode == "two_level":
        K[:, :, 0] = 0.0
        K[:, ::32, 0] = 32.0
        K[:, 1, 0] = -64.0
        K[:, :, 1] = 0.0
    elif mode == "dominant":
        K[:, :, 0] = 0.0
        K[:, 0, 0] = 256.0
        K[:, :, 1] = 0.0
    else:
        raise ValueError(mode)
    V = rng.standard_normal((H, S, d))
    return dict(Q=to_bf16(Q), K=to_bf16(K), V=to_bf16(V), Wq=Wq, Wk=Wk, c=c)


def make_inputs_device(w: Workload, device, heads: Optional[int] = None, seed: Optional[int] = None,
                       with_grad_out: Optional[bool] = None, r: Optional[int] = None) -> dict:
    """The recipe of ``make_inputs`` drawn on ``device`` with torch's seeded
    generator: the same distributions and structure, not the same bits. For
    timing runs at sizes where drawing on the host takes minutes (the 128K
    sweep, the 256K layer); parity tests use ``make_inputs``. ``r``
    overrides the workload's predictor rank."""
    H = w.H if heads is None else heads
    S, d = w.S, w.d
    r = w.r if r is None else r
    gen = torch.Generator(device=device)
    gen.manual_seed(20250000 + w.index if seed is None else seed)
    host = np.random.default_rng(20250000 + w.index if seed is None else seed)
    P = torch.from_numpy(sinusoid_3d(w.T, w.Y, w.X, d)).to(device=device, dtype=torch.float32)
    kw = dict(device=device, dtype=torch.float32, generator=gen)
    Q = torch.empty((H, S, d), dtype=torch.bfloat16, device=device)
    K = torch.empty_like(Q)
    V = torch.empty_like(Q)
    Wq = torch.empty((H, d, r), dtype=torch.bfloat16, device=device)
    Wk = torch.empty_like(Wq)
    qs = np.empty(H)
    for h in range(H):
        Gh = torch.randn((d, d), **kw) / math.sqrt(d)
        Wq[h] = (torch.randn((d, r), **kw) / math.sqrt(d)).to(torch.bfloat16)
        Wk[h] = (torch.randn((d, r), **kw) / math.sqrt(d)).to(torch.bfloat16)
        qs[h] = w.qscale[1] if w.qscale[0] == "const" else host.uniform(w.qscale[1], w.qscale[2])
        base = P @ Gh
        Q[h] = (qs[h] * (base + 0.5 * torch.randn((S, d), **kw))).to(torch.bfloat16)
        K[h] = (base + 0.5 * torch.randn((S, d), **kw)).to(torch.bfloat16)
        V[h] = (base + 0.5 * torch.randn((S, d), **kw)).to(torch.bfloat16)
    want = w.backward if with_grad_out is None else with_grad_out
    dO = torch.randn((H, S, d), **kw).to(torch.bfloat16) if want else None
    return dict(Q=Q, K=K, V=V, Wq=Wq, Wk=Wk, dO=dO, qscale=qs)
