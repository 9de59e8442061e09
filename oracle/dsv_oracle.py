"""CPU oracle for the DSV hot path -- TEST INFRASTRUCTURE, not product code.

Only the test suite, ``__graft_entry__.smoke()`` and ``bench.py`` (its
``cpu_baseline`` leg and its ``--impl reference`` arm) may import this module.
The CUDA path never calls it, and it shares no code with the CUDA path.

Plain numpy, float64 throughout. Inputs are the bf16 tensors the GPU receives,
upcast exactly to fp64. Every step follows the DSV method as the pages
describe it ("DSV: Exploiting Dynamic Sparsity to Accelerate Large-Scale Video
DiT Training", gist.science summaries of arXiv 2502.07590):

* low-rank predictor (technical summary, section 2.1 "two-stage training"):
  per-head matrices W_lr^Q, W_lr^K (d x r) whose product approximates QK^T;
* critical KV (section 2.1): the keys that carry 90% of the attention mass;
* fused low-rank MatMul + Top-K (section 2.2 "efficient kernels"): the S x S
  score matrix is never needed, only each query group's top-k key set;
* query grouping (section 2.2): spatio-temporally adjacent queries share one
  key index set;
* sparse attention (section 2.1): full softmax attention over the selected
  keys only; the dense case is the same computation over all keys.

Readings taken where the pages are silent:
* group score of key j = mean over the group's queries of q_lr . k_lr (a
  design choice: the pages do not fix the aggregation);
* top-k ties go to the lower key index; each index row is returned ascending;
* coverage: per head, C(k) = mean over groups of the mass of the group's k
  largest predicted softmax probabilities, softmax of (1/sqrt(d)) * score;
  k_cov = smallest k with C(k) >= mass (0.9);
* dispatcher: k_h = clamp(k_cov, round(0.01 S), round(0.25 S)) with
  round-half-up, dense (k = S) when k_cov > 0.5 S;
* attention scale 1/sqrt(d); LSE is the natural log of the row's sum of
  exp(scale * q.k) over the selected keys;
* the backward pass treats the index sets as constants (no gradient flows
  into the selection or into W_lr).

Parity status: every function below is pinned by ``tests/test_oracle.py``
against closed forms, brute force or library routines; none is unpinned.
"""
from __future__ import annotations

import itertools
import math
from typing import Optional, Sequence

import numpy as np


# ------------------------------------------------------------------ helpers
def as_f64(x) -> np.ndarray:
    """bf16/fp32 torch tensor or numpy array -> float64 numpy (exact upcast)."""
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").float().numpy()
    return np.asarray(x, dtype=np.float64)


def round_half_up(x: float) -> int:
    return int(math.floor(x + 0.5))


# --------------------------------------------------------- query grouping
def group_members(T: int, Y: int, X: int, gt: int, gy: int, gx: int) -> np.ndarray:
    """Token positions of each query group (section 2.2, query grouping).

    Tokens sit on a T x Y x X grid at s = (t*Y + y)*X + x. A group is one
    gt x gy x gx cube; groups are numbered row-major over the (T/gt, Y/gy,
    X/gx) grid of cubes, members listed in (t, y, x) lexicographic order.
    Returns int64 [n_groups, gt*gy*gx].
    """
    if T % gt or Y % gy or X % gx:
        raise ValueError("the group cube must divide the latent grid")
    out = []
    for ct in range(T // gt):
        for cy in range(Y // gy):
            for cx in range(X // gx):
                mem = []
                for t in range(ct * gt, ct * gt + gt):
                    for y in range(cy * gy, cy * gy + gy):
                        for x in range(cx * gx, cx * gx + gx):
                            mem.append((t * Y + y) * X + x)
                out.append(mem)
    return np.asarray(out, dtype=np.int64)


# ----------------------------------------------------- low-rank predictor
def lowrank_project(X, W) -> np.ndarray:
    """q_lr = Q W_lr^Q (or k_lr = K W_lr^K) in fp64 (section 2.1: per-head
    low-rank matrices approximating QK^T). X: [S, d], W: [d, r] -> [S, r]."""
    return as_f64(X) @ as_f64(W)


def group_scores(q_lr: np.ndarray, k_lr: np.ndarray, members: np.ndarray,
                 groups: Optional[Sequence[int]] = None) -> np.ndarray:
    """Group score s_gj = mean over queries i of group g of q_lr[i] . k_lr[j].

    This is the literal mean of the per-query predicted logits (the
    aggregation is a design choice; the pages only say the group shares one
    key set). Returns [len(groups), S] float64.
    """
    gs = range(members.shape[0]) if groups is None else groups
    out = np.empty((len(gs), k_lr.shape[0]))
    for n, g in enumerate(gs):
        per_query = q_lr[members[g]] @ k_lr.T          # [G, S] predicted q.k
        out[n] = per_query.mean(axis=0)
    return out


def topk_ascending(scores_row: np.ndarray, k: int) -> np.ndarray:
    """The k keys with the largest group score, ties to the lower key index,
    returned in ascending key order (section 2.2: fused MatMul + Top-K)."""
    S = scores_row.shape[0]
    if not 1 <= k <= S:
        raise ValueError("k out of range")
    order = np.lexsort((np.arange(S), -scores_row))   # score desc, then index asc
    return np.sort(order[:k]).astype(np.int64)


def lowrank_topk(Q, K, Wq, Wk, members: np.ndarray, k: int,
                 groups: Optional[Sequence[int]] = None):
    """One head: projection, group scores and top-k. Returns (idx [n, k]
    int64 ascending, scores [n, S])."""
    s = group_scores(lowrank_project(Q, Wq), lowrank_project(K, Wk), members, groups)
    idx = np.stack([topk_ascending(row, k) for row in s])
    return idx, s


# ---------------------------------------------------------------- coverage
def coverage_curve(scores: np.ndarray, scale: float) -> np.ndarray:
    """C(k) for k = 1..S: mean over groups of the total predicted softmax mass
    of each group's k most probable keys (section 2.1: critical KV are those
    holding 90% of the attention mass; the predictor's logits are scale*s)."""
    logits = scale * scores
    logits = logits - logits.max(axis=1, keepdims=True)
    p = np.exp(logits)
    p /= p.sum(axis=1, keepdims=True)
    p_desc = -np.sort(-p, axis=1)
    return np.cumsum(p_desc, axis=1).mean(axis=0)


def coverage_k(scores: np.ndarray, scale: float, mass: float = 0.9) -> int:
    """Smallest k with C(k) >= mass (1-based)."""
    C = coverage_curve(scores, scale)
    hit = np.nonzero(C >= mass)[0]
    return int(hit[0]) + 1 if hit.size else scores.shape[1]


# -------------------------------------------------------------- dispatcher
def plan_heads(k_cov: Sequence[int], S: int, lo_frac: float = 0.01, hi_frac: float = 0.25,
               dense_frac: float = 0.5):
    """OP dispatcher (section 2.1: sparse or dense per block, here per head).

    Dense (k = S) when k_cov > dense_frac*S, else k = clamp(k_cov, lo, hi)
    with lo, hi = round-half-up(lo_frac*S), round-half-up(hi_frac*S).
    Returns (k_h list, dense list of bool).
    """
    lo, hi = round_half_up(lo_frac * S), round_half_up(hi_frac * S)
    ks, dense = [], []
    for kc in k_cov:
        if kc > dense_frac * S:
            ks.append(S)
            dense.append(True)
        else:
            ks.append(min(max(int(kc), lo), hi))
            dense.append(False)
    return ks, dense


def plan_gpus(cost: Sequence[int], n_gpus: int, equal_counts: bool = True):
    """Head-wise context-parallel re-balancing (section 2.3: each head's
    assignment to a GPU follows its sparsity so that the compute balances).

    Longest processing time first: heads in order of decreasing cost (ties:
    lower head first), each to the GPU with the least load so far (ties: lower
    GPU); with ``equal_counts`` only GPUs holding fewer than ceil(n / n_gpus)
    heads take one. Returns (gpu_of list, load list).
    """
    n = len(cost)
    cap = -(-n // n_gpus) if equal_counts else n
    order = sorted(range(n), key=lambda p: (-int(cost[p]), p))
    load, count, gpu_of = [0] * n_gpus, [0] * n_gpus, [0] * n
    for p in order:
        g = min((q for q in range(n_gpus) if count[q] < cap), key=lambda q: (load[q], q))
        gpu_of[p] = g
        load[g] += int(cost[p])
        count[g] += 1
    return gpu_of, load


def best_makespan(cost: Sequence[int], n_gpus: int, equal_counts: bool = True) -> int:
    """Smallest possible largest per-GPU load, by trying every assignment
    (tiny inputs only)."""
    n = len(cost)
    cap = -(-n // n_gpus) if equal_counts else n
    best = None
    for assign in itertools.product(range(n_gpus), repeat=n):
        if max(assign.count(g) for g in range(n_gpus)) > cap:
            continue
        loads = [0] * n_gpus
        for p, g in enumerate(assign):
            loads[g] += int(cost[p])
        m = max(loads)
        best = m if best is None else min(best, m)
    return best


# ------------------------------------------------------ sparse attention
def _group_forward(Qg, Ksel, Vsel, scale):
    logits = scale * (Qg @ Ksel.T)
    m = logits.max(axis=1, keepdims=True)
    e = np.exp(logits - m)
    ssum = e.sum(axis=1, keepdims=True)
    P = e / ssum
    lse = (m + np.log(ssum))[:, 0]
    return P, P @ Vsel, lse


def sparse_attn_fwd(Q, K, V, idx: Optional[np.ndarray], members: np.ndarray, scale: float,
                    groups: Optional[Sequence[int]] = None):
    """One head of query-grouped sparse attention (section 2.1: attention on
    the critical KV only; section 2.2: a group shares its key set).

    For each query i of group g: O_i = sum_{j in I_g} softmax_j(scale q_i.k_j) v_j,
    LSE_i = ln sum_{j in I_g} exp(scale q_i.k_j). ``idx=None`` is the dense
    case (I_g = all keys). Returns (O [S, d], LSE [S]); rows of groups not in
    ``groups`` are left NaN.
    """
    Q, K, V = as_f64(Q), as_f64(K), as_f64(V)
    S, d = Q.shape
    O = np.full((S, V.shape[1]), np.nan)
    LSE = np.full(S, np.nan)
    gs = range(members.shape[0]) if groups is None else groups
    for g in gs:
        I = np.arange(K.shape[0]) if idx is None else idx[g]
        mem = members[g]
        _, Og, lse = _group_forward(Q[mem], K[I], V[I], scale)
        O[mem] = Og
        LSE[mem] = lse
    return O, LSE


def true_mass(Q, K, idx: np.ndarray, members: np.ndarray, scale: float) -> np.ndarray:
    """Share of each query's true attention mass that its group's selected keys
    carry (section 2.1: the critical KV pairs are those carrying over 90% of
    the attention score, here measured on the real scores q_i.k_j rather than
    the predictor's). For query i of group g: the softmax over all S keys of
    scale q_i.k_j, summed over j in I_g. Returns [S]."""
    Q, K = as_f64(Q), as_f64(K)
    S = Q.shape[0]
    out = np.full(S, np.nan)
    for g in range(members.shape[0]):
        mem = members[g]
        logits = scale * (Q[mem] @ K.T)
        e = np.exp(logits - logits.max(axis=1, keepdims=True))
        P = e / e.sum(axis=1, keepdims=True)
        out[mem] = P[:, idx[g]].sum(axis=1)
    return out


def predicted_mass(Q, K, Wq, Wk, idx: np.ndarray, members: np.ndarray, scale: float) -> np.ndarray:
    """Share of each query's own predicted softmax mass that its group's
    selected keys carry (section 2.1: critical KV carry over 90% of the
    attention score; the per-query reading of the coverage criterion, on the
    low-rank predictor's logits). For query i of group g, with the
    predictor's logits scale * q_lr,i . k_lr,j over all S keys (q_lr = Q
    W_lr^Q, k_lr = K W_lr^K): the softmax of those logits summed over j in
    I_g. Returns [S]."""
    q_lr, k_lr = lowrank_project(Q, Wq), lowrank_project(K, Wk)
    S = q_lr.shape[0]
    out = np.full(S, np.nan)
    for g in range(members.shape[0]):
        mem = members[g]
        logits = scale * (q_lr[mem] @ k_lr.T)
        e = np.exp(logits - logits.max(axis=1, keepdims=True))
        P = e / e.sum(axis=1, keepdims=True)
        out[mem] = P[:, idx[g]].sum(axis=1)
    return out


def sparse_attn_bwd(Q, K, V, dO, idx: Optional[np.ndarray], members: np.ndarray, scale: float):
    """Gradients of sum(dO * O) for one head of sparse attention, with the
    index sets held constant. Per group g and selected key j:
    P = softmax(scale Q_g K_I^T), dP = dO_g V_I^T, Delta_i = sum_c dO_ic O_ic,
    dS = P (dP - Delta), dQ_g = scale dS K_I, dK_j += scale sum_i dS_ij q_i,
    dV_j += sum_i P_ij dO_i (each key summed over every group that selected it).
    Returns (dQ, dK, dV), each [S, d] float64.
    """
    Q, K, V, dO = as_f64(Q), as_f64(K), as_f64(V), as_f64(dO)
    dQ = np.zeros_like(Q)
    dK = np.zeros_like(K)
    dV = np.zeros_like(V)
    for g in range(members.shape[0]):
        I = np.arange(K.shape[0]) if idx is None else idx[g]
        mem = members[g]
        P, Og, _ = _group_forward(Q[mem], K[I], V[I], scale)
        dOg = dO[mem]
        delta = (dOg * Og).sum(axis=1, keepdims=True)
        dP = dOg @ V[I].T
        dS = P * (dP - delta)
        dQ[mem] = scale * (dS @ K[I])
        np.add.at(dK, I, scale * (dS.T @ Q[mem]))
        np.add.at(dV, I, P.T @ dOg)
    return dQ, dK, dV


def sparse_attn_group_dq(Q, K, V, dO, idx_row: Optional[np.ndarray], mem: np.ndarray, scale: float):
    """dQ and O for one group only (they depend on that group alone); used to
    check sampled groups of full-size workloads."""
    Q, K, V, dO = as_f64(Q), as_f64(K), as_f64(V), as_f64(dO)
    I = np.arange(K.shape[0]) if idx_row is None else idx_row
    P, Og, lse = _group_forward(Q[mem], K[I], V[I], scale)
    dOg = dO[mem]
    delta = (dOg * Og).sum(axis=1, keepdims=True)
    dS = P * (dOg @ V[I].T - delta)
    return Og, lse, scale * (dS @ K[I])


# ------------------------------------------------- full-size check helpers
def group_scores_via_mean(q_lr: np.ndarray, k_lr: np.ndarray, members: np.ndarray,
                          groups: Optional[Sequence[int]] = None) -> np.ndarray:
    """Same group scores as `group_scores`, formed as (mean of q_lr over the
    group) . k_lr, which equals the mean of q_lr . k_lr by linearity. Used
    where the literal form is too slow (all groups of a 64K-262K token head)."""
    gs = range(members.shape[0]) if groups is None else groups
    qbar = np.stack([q_lr[members[g]].mean(axis=0) for g in gs])
    return qbar @ k_lr.T


def sparse_attn_key_grads(Q, K, V, dO, idx: np.ndarray, members: np.ndarray, scale: float, key: int):
    """dK and dV of one key only: sum over the groups whose index set holds the
    key of that group's contribution (each group's softmax over its own
    selected keys). Returns (dK_key [d], dV_key [d], number of groups)."""
    Q, K, V, dO = as_f64(Q), as_f64(K), as_f64(V), as_f64(dO)
    dk = np.zeros(K.shape[1])
    dv = np.zeros(V.shape[1])
    hits = 0
    for g in range(members.shape[0]):
        row = idx[g]
        pos = np.searchsorted(row, key)
        if pos >= row.shape[0] or row[pos] != key:
            continue
        hits += 1
        mem = members[g]
        P, Og, _ = _group_forward(Q[mem], K[row], V[row], scale)
        dOg = dO[mem]
        delta = (dOg * Og).sum(axis=1)
        pj = P[:, pos]
        dpj = dOg @ V[key]
        dsj = pj * (dpj - delta)
        dv += pj @ dOg
        dk += scale * (dsj @ Q[mem])
    return dk, dv, hits
