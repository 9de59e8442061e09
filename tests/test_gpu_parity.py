"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on the
same seeded bf16 inputs, element by element, at sizes the oracle finishes in
seconds that still span several key tiles and a ragged last tile."""
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

CASES = {
    # the oracle-scale workload exactly: H=1, 4x16x16, d=64, r=16, cube 4x4x4, k=128
    "oracle_scale": syn.workload(0, backward=True),
    # d=128, G=128, two full key tiles and a 44-key tail
    "ragged_d128": syn.Workload("ragged", 101, 2, 4, 16, 32, 128, 32, 2, 8, 8, 300, ("uniform", 2.0, 8.0), True),
    # d=64, G=64, r=64 (two 128-byte atoms per predictor row)
    "d64_r64": syn.Workload("d64r64", 102, 2, 4, 8, 16, 64, 64, 4, 4, 4, 200, ("const", 4.0), True),
    # three heads, r=16, one tile plus one key
    "r16_h3": syn.Workload("r16", 103, 3, 8, 16, 16, 64, 16, 4, 4, 4, 129, ("uniform", 1.0, 8.0), True),
}


def _cuda(inp):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


def _grid(w):
    return (w.T, w.Y, w.X)


def _group(w):
    return (w.gt, w.gy, w.gx)


@pytest.fixture(scope="module", params=list(CASES))
def case(request):
    w = CASES[request.param]
    inp = syn.make_inputs(w)
    mem = ora.group_members(w.T, w.Y, w.X, w.gt, w.gy, w.gx)
    scale = 1.0 / math.sqrt(w.d)
    ref = []
    for h in range(w.H):
        idx, s = ora.lowrank_topk(inp["Q"][h], inp["K"][h], inp["Wq"][h], inp["Wk"][h], mem, w.k)
        ref.append(dict(idx=idx, scores=s))
    return dict(name=request.param, w=w, inp=inp, dev=_cuda(inp), mem=mem, scale=scale, ref=ref)


def _rows(idx_flat, offs, ks, n_groups, h):
    return idx_flat[offs[h]: offs[h] + n_groups * ks[h]].view(n_groups, ks[h]).cpu().numpy()


def test_lowrank_topk_matches_oracle(case):
    w, d = case["w"], case["dev"]
    st = dsv.new_status()
    idx, ks, offs = dsv.lowrank_topk(d["Q"], d["K"], d["Wq"], d["Wk"], _grid(w), _group(w), w.k, status=st)
    dsv.check_status(st, "lowrank_topk")
    for h in range(w.H):
        rows = _rows(idx, offs, ks, w.n_groups, h)
        for g in range(w.n_groups):
            why = check_idx_row(rows[g], case["ref"][h]["scores"][g], w.k, case["ref"][h]["idx"][g])
            assert not why, f"head {h} group {g}: {why}"


def test_coverage_matches_oracle(case):
    w, d = case["w"], case["dev"]
    st = dsv.new_status()
    k_cov, curve = dsv.coverage(d["Q"], d["K"], d["Wq"], d["Wk"], _grid(w), _group(w), mass=0.9, curve_points=8,
                                status=st)
    dsv.check_status(st, "coverage")
    k_cov = k_cov.cpu().numpy()
    for h in range(w.H):
        C = ora.coverage_curve(case["ref"][h]["scores"], case["scale"])
        why = check_kcov(C, int(k_cov[h]))
        assert not why, f"head {h}: {why}"
        pts = [int(math.ceil((i + 1) * w.S / 8)) for i in range(8)]
        np.testing.assert_allclose(curve[h].cpu().numpy(), C[np.array(pts) - 1], atol=2e-4)


def test_coverage_topk_equals_the_two_calls(case):
    """One combined call writes exactly what dsv_coverage and dsv_lowrank_topk
    write separately (shared projections and row ranges change no bit)."""
    w, d = case["w"], case["dev"]
    st = dsv.new_status()
    k1, c1 = dsv.coverage(d["Q"], d["K"], d["Wq"], d["Wk"], _grid(w), _group(w), mass=0.9, curve_points=8, status=st)
    i1, _, _ = dsv.lowrank_topk(d["Q"], d["K"], d["Wq"], d["Wk"], _grid(w), _group(w), w.k, status=st)
    k2, c2, i2, ks, offs = dsv.coverage_topk(d["Q"], d["K"], d["Wq"], d["Wk"], _grid(w), _group(w), w.k, mass=0.9,
                                             curve_points=8, status=st)
    dsv.check_status(st, "coverage_topk")
    assert torch.equal(k1, k2) and torch.equal(c1, c2) and torch.equal(i1, i2)


def _oracle_attention(case, h, idx):
    inp = case["inp"]
    O, L = ora.sparse_attn_fwd(inp["Q"][h], inp["K"][h], inp["V"][h], idx, case["mem"], case["scale"])
    return O, L


def _idx_tensor(case):
    w = case["w"]
    flat = np.concatenate([case["ref"][h]["idx"].ravel() for h in range(w.H)]).astype(np.int32)
    ks, offs, _ = dsv.topk_layout(w.H, w.n_groups, w.k)
    return torch.from_numpy(flat).cuda(), ks, offs


def test_sparse_fwd_matches_oracle(case):
    w, d = case["w"], case["dev"]
    idx, ks, offs = _idx_tensor(case)
    st = dsv.new_status()
    O, L = dsv.sparse_attn_fwd(d["Q"], d["K"], d["V"], idx, ks, offs, _grid(w), _group(w), status=st)
    dsv.check_status(st, "sparse_attn_fwd")
    for h in range(w.H):
        Oref, Lref = _oracle_attention(case, h, case["ref"][h]["idx"])
        mx, mean = o_errors(O[h].float().cpu().numpy(), Oref)
        assert mx <= O_MAX_ABS and mean <= O_MEAN_ABS, (h, mx, mean)
        assert np.abs(L[h].cpu().numpy() - Lref).max() <= LSE_MAX_ABS


def test_sparse_bwd_matches_oracle(case):
    w, d = case["w"], case["dev"]
    idx, ks, offs = _idx_tensor(case)
    O, L = dsv.sparse_attn_fwd(d["Q"], d["K"], d["V"], idx, ks, offs, _grid(w), _group(w))
    st = dsv.new_status()
    dQ, dK, dV = dsv.sparse_attn_bwd(d["Q"], d["K"], d["V"], O, L, d["dO"], idx, ks, offs, _grid(w), _group(w),
                                     status=st)
    dsv.check_status(st, "sparse_attn_bwd")
    inp = case["inp"]
    for h in range(w.H):
        rq, rk, rv = ora.sparse_attn_bwd(inp["Q"][h], inp["K"][h], inp["V"][h], inp["dO"][h], case["ref"][h]["idx"],
                                         case["mem"], case["scale"])
        for name, got, ref in (("dQ", dQ, rq), ("dK", dK, rk), ("dV", dV, rv)):
            e = rel_l2(got[h].float().cpu().numpy(), ref)
            assert e <= GRAD_REL_L2, (h, name, e)


def test_small_backward_workspace_changes_no_bit(case):
    """A backward workspace below the reported size makes the call keep fewer
    (group, key) pairs in flight per launch. Where a head's partial rows
    outweigh the fp32 running sums (ragged_d128, d64_r64, r16_h3), the
    minimum size leaves one query group per launch, so every head's groups
    are split over launches with running sums. The summation order, and so
    every bit of dQ, dK and dV, stays the same."""
    w, d = case["w"], case["dev"]
    idx, ks, offs = _idx_tensor(case)
    O, L = dsv.sparse_attn_fwd(d["Q"], d["K"], d["V"], idx, ks, offs, _grid(w), _group(w))
    ref = dsv.sparse_attn_bwd(d["Q"], d["K"], d["V"], O, L, d["dO"], idx, ks, offs, _grid(w), _group(w))
    need = dsv.sparse_attn_bwd_workspace_size(d["Q"], _grid(w), _group(w), ks, offs)
    least = dsv.sparse_attn_bwd_min_workspace_size(d["Q"], _grid(w), _group(w), ks, offs)
    assert 0 < least <= need
    for nbytes in (least, (least + need) // 2):
        ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        st = dsv.new_status()
        got = dsv.sparse_attn_bwd(d["Q"], d["K"], d["V"], O, L, d["dO"], idx, ks, offs, _grid(w), _group(w),
                                  workspace=ws, status=st)
        dsv.check_status(st, "small workspace")
        for a, b in zip(got, ref):
            assert torch.equal(a, b)


def test_true_attention_mass_matches_oracle(case):
    """Share of each query's true softmax mass carried by its group's selected
    keys, from the forward's sparse and dense LSE, against the oracle's direct
    sum of the fp64 softmax over all keys."""
    w, d = case["w"], case["dev"]
    idx, ks, offs = _idx_tensor(case)
    _, Ls = dsv.sparse_attn_fwd(d["Q"], d["K"], d["V"], idx, ks, offs, _grid(w), _group(w))
    _, La = dsv.sparse_attn_fwd(d["Q"], d["K"], d["V"], None, None, None, _grid(w), _group(w))
    mass, per_q = dsv.attn_mass(Ls, La, per_query=True)
    for h in range(w.H):
        ref = ora.true_mass(case["inp"]["Q"][h], case["inp"]["K"][h], case["ref"][h]["idx"], case["mem"],
                            case["scale"])
        got = per_q[h].cpu().numpy()
        assert np.abs(got - ref).max() <= 3e-2, h
        assert abs(float(mass[h]) - ref.mean()) <= 1e-2, h


def test_dense_fwd_bwd_matches_oracle(case):
    w, d = case["w"], case["dev"]
    st = dsv.new_status()
    O, L = dsv.sparse_attn_fwd(d["Q"], d["K"], d["V"], None, None, None, _grid(w), _group(w), status=st)
    dQ, dK, dV = dsv.sparse_attn_bwd(d["Q"], d["K"], d["V"], O, L, d["dO"], None, None, None, _grid(w), _group(w),
                                     status=st)
    dsv.check_status(st, "dense")
    inp = case["inp"]
    h = w.H - 1
    Oref, Lref = ora.sparse_attn_fwd(inp["Q"][h], inp["K"][h], inp["V"][h], None, case["mem"], case["scale"])
    mx, mean = o_errors(O[h].float().cpu().numpy(), Oref)
    assert mx <= O_MAX_ABS and mean <= O_MEAN_ABS
    assert np.abs(L[h].cpu().numpy() - Lref).max() <= LSE_MAX_ABS
    rq, rk, rv = ora.sparse_attn_bwd(inp["Q"][h], inp["K"][h], inp["V"][h], inp["dO"][h], None, case["mem"],
                                     case["scale"])
    for name, got, ref in (("dQ", dQ, rq), ("dK", dK, rk), ("dV", dV, rv)):
        assert rel_l2(got[h].float().cpu().numpy(), ref) <= GRAD_REL_L2, name


def test_determinism_bitwise(case):
    w, d = case["w"], case["dev"]

    def run():
        idx, ks, offs = dsv.lowrank_topk(d["Q"], d["K"], d["Wq"], d["Wk"], _grid(w), _group(w), w.k)
        O, L = dsv.sparse_attn_fwd(d["Q"], d["K"], d["V"], idx, ks, offs, _grid(w), _group(w))
        g = dsv.sparse_attn_bwd(d["Q"], d["K"], d["V"], O, L, d["dO"], idx, ks, offs, _grid(w), _group(w))
        torch.cuda.synchronize()
        return [t.clone() for t in (idx, O, L) + tuple(g)]

    a, b = run(), run()
    for x, y in zip(a, b):
        assert torch.equal(x, y)


# ------------------------------------------------------------- edge cases
def test_k_equals_S_selects_every_key_and_matches_dense():
    w = syn.Workload("kS", 104, 1, 2, 8, 16, 64, 16, 2, 4, 8, 256, ("const", 2.0), True)
    inp = _cuda(syn.make_inputs(w))
    idx, ks, offs = dsv.lowrank_topk(inp["Q"], inp["K"], inp["Wq"], inp["Wk"], _grid(w), _group(w), w.S)
    rows = _rows(idx, offs, ks, w.n_groups, 0)
    assert np.array_equal(rows, np.tile(np.arange(w.S), (w.n_groups, 1)))
    O1, L1 = dsv.sparse_attn_fwd(inp["Q"], inp["K"], inp["V"], idx, ks, offs, _grid(w), _group(w))
    O2, L2 = dsv.sparse_attn_fwd(inp["Q"], inp["K"], inp["V"], None, None, None, _grid(w), _group(w))
    assert torch.equal(O1, O2) and torch.equal(L1, L2)


def test_equal_scores_take_the_lowest_keys():
    """W_lr^Q = 0 makes every group score 0: all ties, so each row is 0..k-1."""
    w = syn.Workload("ties", 105, 2, 2, 16, 16, 128, 32, 2, 8, 8, 77, ("const", 1.0), False)
    inp = _cuda(syn.make_inputs(w))
    Wq = torch.zeros_like(inp["Wq"])
    st = dsv.new_status()
    idx, ks, offs = dsv.lowrank_topk(inp["Q"], inp["K"], Wq, inp["Wk"], _grid(w), _group(w), w.k, status=st)
    dsv.check_status(st, "ties")
    for h in range(w.H):
        assert np.array_equal(_rows(idx, offs, ks, w.n_groups, h), np.tile(np.arange(w.k), (w.n_groups, 1)))
    k_cov, _ = dsv.coverage(inp["Q"], inp["K"], Wq, inp["Wk"], _grid(w), _group(w), mass=0.9)
    # uniform predicted distribution: C(k) = k/S
    assert k_cov.cpu().tolist() == [math.ceil(0.9 * w.S)] * w.H


def test_mixed_plan_sparse_and_dense_heads():
    w = syn.Workload("mixed", 106, 3, 4, 16, 32, 128, 32, 2, 8, 8, 0, ("uniform", 1.0, 8.0), True)
    inp = syn.make_inputs(w)
    d = _cuda(inp)
    mem = ora.group_members(w.T, w.Y, w.X, w.gt, w.gy, w.gx)
    plan_k = [150, w.S, 400]
    dense = [False, True, False]
    ks, offs, total = dsv.topk_layout(w.H, w.n_groups, plan_k, skip=dense)
    idx = torch.empty(total, dtype=torch.int32, device="cuda")
    st = dsv.new_status()
    dsv.lowrank_topk(d["Q"], d["K"], d["Wq"], d["Wk"], _grid(w), _group(w), ks, idx_offset=offs, idx=idx, status=st)
    # the combined call takes its two-call path on a plan with a dense head: same bits
    kc, _, idx2, _, _ = dsv.coverage_topk(d["Q"], d["K"], d["Wq"], d["Wk"], _grid(w), _group(w), ks, idx_offset=offs,
                                          status=st)
    kc1, _ = dsv.coverage(d["Q"], d["K"], d["Wq"], d["Wk"], _grid(w), _group(w), status=st)
    assert torch.equal(idx2, idx) and torch.equal(kc, kc1)
    O, L = dsv.sparse_attn_fwd(d["Q"], d["K"], d["V"], idx, ks, offs, _grid(w), _group(w), status=st)
    dQ, dK, dV = dsv.sparse_attn_bwd(d["Q"], d["K"], d["V"], O, L, d["dO"], idx, ks, offs, _grid(w), _group(w),
                                     status=st)
    dsv.check_status(st, "mixed plan")
    scale = 1.0 / math.sqrt(w.d)
    for h in range(w.H):
        if dense[h]:
            ridx = None
        else:
            ridx, s = ora.lowrank_topk(inp["Q"][h], inp["K"][h], inp["Wq"][h], inp["Wk"][h], mem, ks[h])
            rows = _rows(idx, offs, ks, w.n_groups, h)
            for g in range(w.n_groups):
                assert not check_idx_row(rows[g], s[g], ks[h], ridx[g])
            ridx = rows.astype(np.int64)   # attention parity on the GPU's own (accepted) sets
        Oref, _ = ora.sparse_attn_fwd(inp["Q"][h], inp["K"][h], inp["V"][h], ridx, mem, scale)
        mx, mean = o_errors(O[h].float().cpu().numpy(), Oref)
        assert mx <= O_MAX_ABS and mean <= O_MEAN_ABS, h
        grads = ora.sparse_attn_bwd(inp["Q"][h], inp["K"][h], inp["V"][h], inp["dO"][h], ridx, mem, scale)
        for got, ref in zip((dQ, dK, dV), grads):
            assert rel_l2(got[h].float().cpu().numpy(), ref) <= GRAD_REL_L2, h
