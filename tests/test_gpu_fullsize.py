"""Parity at the workloads' full sizes, in the launch configuration the bench
uses, on outputs the oracle can compute one by one (sampled index rows,
sampled query groups' O/LSE/dQ, sampled keys' dK/dV) plus identities that
hold at any size (sum_j dV_j = sum_i dO_i, sum_j dK_j = 0) and the pooled
coverage of whole heads."""
import math

import numpy as np
import pytest
import torch

import dynamic_sparse_attention_dsv_gb300 as dsv
from dynamic_sparse_attention_dsv_gb300 import synthetic as syn
from oracle import dsv_oracle as ora

from .parity import (GRAD_REL_L2, LSE_MAX_ABS, O_MAX_ABS, O_MEAN_ABS, check_idx_row, check_kcov, o_errors,
                     rel_l2)

pytestmark = pytest.mark.gpu


def _dev(inp):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


def _rows(idx, off, k, n_groups):
    return idx[off: off + n_groups * k].view(n_groups, k).cpu().numpy()


def _check_topk_rows(w, inp, idx, ks, offs, heads, groups):
    mem = ora.group_members(w.T, w.Y, w.X, w.gt, w.gy, w.gx)
    for h in heads:
        ridx, s = ora.lowrank_topk(inp["Q"][h], inp["K"][h], inp["Wq"][h], inp["Wk"][h], mem, ks[h], groups)
        rows = _rows(idx, offs[h], ks[h], w.n_groups)
        for n, g in enumerate(groups):
            why = check_idx_row(rows[g], s[n], ks[h], ridx[n])
            assert not why, f"head {h} group {g}: {why}"


def _pooled_curve(w, inp, h, chunk=128):
    """The oracle's coverage curve of a whole head, accumulated over chunks of
    groups (its curve is a mean over groups, so chunk means combine exactly)."""
    mem = ora.group_members(w.T, w.Y, w.X, w.gt, w.gy, w.gx)
    q = ora.lowrank_project(inp["Q"][h], inp["Wq"][h])
    k = ora.lowrank_project(inp["K"][h], inp["Wk"][h])
    total = np.zeros(w.S)
    for g0 in range(0, w.n_groups, chunk):
        gs = list(range(g0, min(w.n_groups, g0 + chunk)))
        total += len(gs) * ora.coverage_curve(ora.group_scores_via_mean(q, k, mem, gs), 1.0 / math.sqrt(w.d))
    return total / w.n_groups


def _check_kcov(w, inp, k_cov, heads):
    for h in heads:
        why = check_kcov(_pooled_curve(w, inp, h), int(k_cov[h]))
        assert not why, f"head {h}: {why}"


def _check_attention(w, inp, idx_rows, O, L, dQ, h, groups):
    """O, LSE, dQ of sampled groups against the oracle on the GPU's (accepted) index sets."""
    mem = ora.group_members(w.T, w.Y, w.X, w.gt, w.gy, w.gx)
    scale = 1.0 / math.sqrt(w.d)
    Oh, Lh, dQh = O[h].float().cpu().numpy(), L[h].cpu().numpy(), dQ[h].float().cpu().numpy()
    errs_o = []
    for g in groups:
        row = None if idx_rows is None else idx_rows[g].astype(np.int64)
        Og, lse, dq = ora.sparse_attn_group_dq(inp["Q"][h], inp["K"][h], inp["V"][h], inp["dO"][h], row, mem[g], scale)
        errs_o.append(np.abs(Oh[mem[g]] - Og))
        assert np.abs(Lh[mem[g]] - lse).max() <= LSE_MAX_ABS, (h, g)
        assert rel_l2(dQh[mem[g]], dq) <= GRAD_REL_L2, (h, g)
    e = np.concatenate(errs_o)
    assert e.max() <= O_MAX_ABS and e.mean() <= O_MEAN_ABS, (h, e.max(), e.mean())


def _check_grad_identities(dK, dV, dO, heads):
    for h in heads:
        dk, dv, do = dK[h].float(), dV[h].float(), dO[h].float()
        sv, so = dv.sum(0), do.sum(0)
        assert torch.all((sv - so).abs() <= 1e-2 * dv.abs().sum(0) + 1e-2), h
        assert torch.all(dk.sum(0).abs() <= 1e-2 * dk.abs().sum(0) + 1e-2), h


def _check_keys(w, inp, idx_rows, dK, dV, h, n_keys=2, max_hits=80):
    """dK, dV of a few keys, summed by the oracle over every group that chose them."""
    mem = ora.group_members(w.T, w.Y, w.X, w.gt, w.gy, w.gx)
    counts = np.bincount(idx_rows.ravel(), minlength=w.S)
    cand = np.nonzero((counts > 0) & (counts <= max_hits))[0]
    assert cand.size > 0
    picks = cand[np.linspace(0, cand.size - 1, n_keys).astype(int)]
    for key in picks:
        dk, dv, hits = ora.sparse_attn_key_grads(inp["Q"][h], inp["K"][h], inp["V"][h], inp["dO"][h],
                                                 idx_rows.astype(np.int64), mem, 1.0 / math.sqrt(w.d), int(key))
        assert hits == counts[key]
        assert rel_l2(dK[h, key].float().cpu().numpy(), dk) <= GRAD_REL_L2, (h, key)
        assert rel_l2(dV[h, key].float().cpu().numpy(), dv) <= GRAD_REL_L2, (h, key)


# --------------------------------------------- S=16K forward+backward
def test_fullsize_16k_forward_backward():
    """H=8, 8x32x64 (S=16384), d=64, r=32, cube 4x4x4, k=1638: every output of
    one head against the full oracle, sampled rows of the others."""
    w = syn.workload(1)
    inp = syn.make_inputs(w)
    d = _dev(inp)
    grid, group = (w.T, w.Y, w.X), (w.gt, w.gy, w.gx)
    st = dsv.new_status()
    k_cov, _ = dsv.coverage(d["Q"], d["K"], d["Wq"], d["Wk"], grid, group, status=st)
    idx, ks, offs = dsv.lowrank_topk(d["Q"], d["K"], d["Wq"], d["Wk"], grid, group, w.k, status=st)
    O, L = dsv.sparse_attn_fwd(d["Q"], d["K"], d["V"], idx, ks, offs, grid, group, status=st)
    dQ, dK, dV = dsv.sparse_attn_bwd(d["Q"], d["K"], d["V"], O, L, d["dO"], idx, ks, offs, grid, group, status=st)
    dsv.check_status(st, "16k")
    _check_topk_rows(w, inp, idx, ks, offs, [0, 3, 7], [0, 100, w.n_groups - 1])
    _check_kcov(w, inp, k_cov.cpu().numpy(), [0, 5])
    mem = ora.group_members(w.T, w.Y, w.X, w.gt, w.gy, w.gx)
    h = 2
    rows = _rows(idx, offs[h], ks[h], w.n_groups).astype(np.int64)
    scale = 1.0 / math.sqrt(w.d)
    Oref, Lref = ora.sparse_attn_fwd(inp["Q"][h], inp["K"][h], inp["V"][h], rows, mem, scale)
    mx, mean = o_errors(O[h].float().cpu().numpy(), Oref)
    assert mx <= O_MAX_ABS and mean <= O_MEAN_ABS
    assert np.abs(L[h].cpu().numpy() - Lref).max() <= LSE_MAX_ABS
    grads = ora.sparse_attn_bwd(inp["Q"][h], inp["K"][h], inp["V"][h], inp["dO"][h], rows, mem, scale)
    for name, got, ref in zip(("dQ", "dK", "dV"), (dQ, dK, dV), grads):
        assert rel_l2(got[h].float().cpu().numpy(), ref) <= GRAD_REL_L2, name
    _check_grad_identities(dK, dV, d["dO"], range(w.H))


# --------------------------------------------- S=64K video-DiT layer
def test_fullsize_64k_bench_step():
    """The bench step itself (H=24, 16x64x64, d=128, r=32, cube 2x8x8, k=6554):
    coverage, top-k, forward and backward with the bench's buffers."""
    import bench
    w = syn.workload(2)
    inp = syn.make_inputs(w)
    step = bench.Step(w, inp, torch.device("cuda", 0))
    step.run()
    torch.cuda.synchronize()
    assert dsv.read_status(step.status) == 0
    _check_topk_rows(w, inp, step.idx, step.ks, step.offs, [0, 11, 23], [0, 257, w.n_groups - 1])
    _check_kcov(w, inp, step.k_cov.cpu().numpy(), [4, 17])
    for h in (1, 22):
        rows = _rows(step.idx, step.offs[h], step.ks[h], w.n_groups)
        _check_attention(w, inp, rows, step.O, step.LSE, step.dQ, h, [0, 200, w.n_groups - 1])
        _check_keys(w, inp, rows, step.dK, step.dV, h)
    _check_grad_identities(step.dK, step.dV, step.dO, range(w.H))


# --------------------------------------------- S=128K top-k sweep
@pytest.mark.parametrize("r", syn.TOPK_SWEEP_RANKS)
def test_fullsize_128k_topk_sweep(r):
    """32x64x64 (S=131072), d=128, cube 2x8x8, k in {1, 5, 10, 20}% of S, for
    each rank. Each head is its own launch chunk at this size, so four heads
    exercise the same launch configuration as twenty-four."""
    w = syn.workload(3, r=r)
    inp = syn.make_inputs(w, heads=4, with_grad_out=False)
    d = _dev(inp)
    grid, group = (w.T, w.Y, w.X), (w.gt, w.gy, w.gx)
    st = dsv.new_status()
    for frac in syn.TOPK_SWEEP_FRACTIONS:
        k = syn.k_of_fraction(frac, w.S)
        idx, ks, offs = dsv.lowrank_topk(d["Q"], d["K"], d["Wq"], d["Wk"], grid, group, k, status=st)
        dsv.check_status(st, f"128k r={r} k={k}")
        _check_topk_rows(w, inp, idx, ks, offs, [0, 3], [1, w.n_groups // 2])
    k_cov, _ = dsv.coverage(d["Q"], d["K"], d["Wq"], d["Wk"], grid, group, status=st)
    dsv.check_status(st, f"128k coverage r={r}")
    _check_kcov(w, inp, k_cov.cpu().numpy(), [1])


# --------------------------------------------- S=256K dispatcher-driven layer
def test_fullsize_256k_dispatcher_layer():
    """H=16, 64x64x64 (S=262144), d=128, r=32, cube 2x8x8: coverage -> per-head
    plan (clamp to [1%, 25%] S, dense above 50%) -> top-k for sparse heads ->
    forward and backward over all heads."""
    w = syn.workload(4)
    inp = syn.make_inputs(w)
    d = _dev(inp)
    grid, group = (w.T, w.Y, w.X), (w.gt, w.gy, w.gx)
    st = dsv.new_status()
    k_cov, _ = dsv.coverage(d["Q"], d["K"], d["Wq"], d["Wk"], grid, group, status=st)
    kc = k_cov.cpu().tolist()
    k_h, dense, offs, total = dsv.plan_heads(kc, w.S, w.n_groups)
    assert (k_h, dense) == tuple(map(list, ora.plan_heads(kc, w.S)))
    idx = torch.empty(max(total, 1), dtype=torch.int32, device="cuda")
    if total:
        dsv.lowrank_topk(d["Q"], d["K"], d["Wq"], d["Wk"], grid, group, k_h, idx_offset=offs, idx=idx, status=st)
    O, L = dsv.sparse_attn_fwd(d["Q"], d["K"], d["V"], idx, k_h, offs, grid, group, status=st)
    dQ, dK, dV = dsv.sparse_attn_bwd(d["Q"], d["K"], d["V"], O, L, d["dO"], idx, k_h, offs, grid, group, status=st)
    dsv.check_status(st, "256k")
    _check_kcov(w, inp, kc, [int(np.argmin(kc))])
    sparse_heads = [h for h in range(w.H) if not dense[h]]
    dense_heads = [h for h in range(w.H) if dense[h]]
    # every head: 16 sampled groups of each sparse head (index rows, O, LSE, dQ)
    # and one key's dK/dV; 2 sampled groups of each dense head (O, LSE, dQ)
    for n, h in enumerate(sparse_heads):
        groups = sorted({int(g) for g in (np.linspace(0, w.n_groups - 1, 16) + 37 * n) % w.n_groups})
        _check_topk_rows(w, inp, idx, k_h, offs, [h], groups)
        rows = _rows(idx, offs[h], k_h[h], w.n_groups)
        _check_attention(w, inp, rows, O, L, dQ, h, groups)
        _check_keys(w, inp, rows, dK, dV, h, n_keys=1, max_hits=8)
    for n, h in enumerate(dense_heads):
        _check_attention(w, inp, None, O, L, dQ, h, [(7 + 211 * n) % w.n_groups, (w.n_groups - 1 - 97 * n) % w.n_groups])
    _check_grad_identities(dK, dV, d["dO"], range(w.H))
