"""The device-side failure path. Every pipeline wait inside the kernels is
bounded; when one runs out, the call raises DSV_ERR_TIMEOUT in its status
word and each block unwinds (it waits for the copies and MMAs it already
issued, frees its tensor memory and exits), leaving the context usable. A
wait limit of 0 makes every wait that has not already completed give up at
once, so one call with that limit runs the failure path on purpose; the
next call, with the normal limit, must match the oracle (nothing was left
allocated or in flight)."""
import math

import numpy as np
import pytest
import torch

import dynamic_sparse_attention_dsv_gb300 as dsv
from dynamic_sparse_attention_dsv_gb300 import synthetic as syn
from oracle import dsv_oracle as ora

from .parity import (GRAD_REL_L2, LSE_MAX_ABS, O_MAX_ABS, O_MEAN_ABS, check_idx_row, o_errors, rel_l2)

pytestmark = pytest.mark.gpu

TIMEOUT = 5          # DSV_ERR_TIMEOUT
NORMAL = 2_000_000_000


@pytest.fixture(scope="module")
def case():
    w = syn.workload(0, backward=True)
    inp = syn.make_inputs(w)
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    mem = ora.group_members(w.T, w.Y, w.X, w.gt, w.gy, w.gx)
    idx, s = ora.lowrank_topk(inp["Q"][0], inp["K"][0], inp["Wq"][0], inp["Wk"][0], mem, w.k)
    return dict(w=w, inp=inp, dev=dev, mem=mem, idx=idx, scores=s, scale=1.0 / math.sqrt(w.d))


@pytest.fixture
def limit():
    prev = dsv.set_wait_limit_ns(NORMAL)
    yield
    dsv.set_wait_limit_ns(prev)


def _run_timed_out(fn):
    dsv.set_wait_limit_ns(0)
    try:
        st = dsv.new_status()
        fn(st)
        code = dsv.read_status(st)
    finally:
        dsv.set_wait_limit_ns(NORMAL)
    return code


def _grid(w):
    return (w.T, w.Y, w.X), (w.gt, w.gy, w.gx)


def _idx_dev(case):
    w = case["w"]
    ks, offs, _ = dsv.topk_layout(1, w.n_groups, w.k)
    return torch.from_numpy(case["idx"].astype(np.int32).ravel()).cuda(), ks, offs


def test_limit_setter_round_trip(limit):
    assert dsv.set_wait_limit_ns(123) == NORMAL
    assert dsv.set_wait_limit_ns(NORMAL) == 123


def test_forward_times_out_then_recovers(case, limit):
    w, d = case["w"], case["dev"]
    grid, group = _grid(w)
    idx, ks, offs = _idx_dev(case)
    code = _run_timed_out(lambda st: dsv.sparse_attn_fwd(d["Q"], d["K"], d["V"], idx, ks, offs, grid, group, status=st))
    assert code == TIMEOUT
    st = dsv.new_status()
    O, L = dsv.sparse_attn_fwd(d["Q"], d["K"], d["V"], idx, ks, offs, grid, group, status=st)
    dsv.check_status(st, "forward after a timed-out call")
    Oref, Lref = ora.sparse_attn_fwd(case["inp"]["Q"][0], case["inp"]["K"][0], case["inp"]["V"][0], case["idx"],
                                     case["mem"], case["scale"])
    mx, mean = o_errors(O[0].float().cpu().numpy(), Oref)
    assert mx <= O_MAX_ABS and mean <= O_MEAN_ABS
    assert np.abs(L[0].cpu().numpy() - Lref).max() <= LSE_MAX_ABS


def test_dense_forward_times_out_then_recovers(case, limit):
    """The dense path's TMA tile loads unwind the same way."""
    w, d = case["w"], case["dev"]
    grid, group = _grid(w)
    code = _run_timed_out(lambda st: dsv.sparse_attn_fwd(d["Q"], d["K"], d["V"], None, None, None, grid, group,
                                                         status=st))
    assert code == TIMEOUT
    st = dsv.new_status()
    O, L = dsv.sparse_attn_fwd(d["Q"], d["K"], d["V"], None, None, None, grid, group, status=st)
    dsv.check_status(st, "dense forward after a timed-out call")
    Oref, Lref = ora.sparse_attn_fwd(case["inp"]["Q"][0], case["inp"]["K"][0], case["inp"]["V"][0], None,
                                     case["mem"], case["scale"])
    mx, mean = o_errors(O[0].float().cpu().numpy(), Oref)
    assert mx <= O_MAX_ABS and mean <= O_MEAN_ABS


def test_topk_and_coverage_time_out_then_recover(case, limit):
    w, d = case["w"], case["dev"]
    grid, group = _grid(w)
    code = _run_timed_out(lambda st: dsv.lowrank_topk(d["Q"], d["K"], d["Wq"], d["Wk"], grid, group, w.k, status=st))
    assert code == TIMEOUT
    code = _run_timed_out(lambda st: dsv.coverage(d["Q"], d["K"], d["Wq"], d["Wk"], grid, group, status=st))
    assert code == TIMEOUT
    st = dsv.new_status()
    idx, ks, offs = dsv.lowrank_topk(d["Q"], d["K"], d["Wq"], d["Wk"], grid, group, w.k, status=st)
    dsv.check_status(st, "top-k after timed-out calls")
    rows = idx.view(w.n_groups, w.k).cpu().numpy()
    for g in range(w.n_groups):
        why = check_idx_row(rows[g], case["scores"][g], w.k, case["idx"][g])
        assert not why, f"group {g}: {why}"


@pytest.mark.parametrize("dense", [False, True])
def test_backward_times_out_then_recovers(case, limit, dense):
    """Sparse: group-major kernel with its dK/dV partials; dense: group-major
    dQ and the key-major dK/dV kernel."""
    w, d, inp = case["w"], case["dev"], case["inp"]
    grid, group = _grid(w)
    idx, ks, offs = _idx_dev(case) if not dense else (None, None, None)
    st = dsv.new_status()
    O, L = dsv.sparse_attn_fwd(d["Q"], d["K"], d["V"], idx, ks, offs, grid, group, status=st)
    dsv.check_status(st, "forward")
    code = _run_timed_out(lambda s: dsv.sparse_attn_bwd(d["Q"], d["K"], d["V"], O, L, d["dO"], idx, ks, offs, grid,
                                                        group, status=s))
    assert code == TIMEOUT
    st = dsv.new_status()
    dQ, dK, dV = dsv.sparse_attn_bwd(d["Q"], d["K"], d["V"], O, L, d["dO"], idx, ks, offs, grid, group, status=st)
    dsv.check_status(st, "backward after a timed-out call")
    ref = ora.sparse_attn_bwd(inp["Q"][0], inp["K"][0], inp["V"][0], inp["dO"][0], None if dense else case["idx"],
                              case["mem"], case["scale"])
    for name, got, r in zip(("dQ", "dK", "dV"), (dQ, dK, dV), ref):
        assert rel_l2(got[0].float().cpu().numpy(), r) <= GRAD_REL_L2, name
