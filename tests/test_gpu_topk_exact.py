"""Top-k exactness where a linear score histogram puts thousands of keys into
the boundary bin: one key far above and one far below a dense cluster of
near-equal keys, with and without large groups of exactly equal scores
(technical summary section 2.2: the fused low-rank MatMul + Top-K must return
each group's exact top-k key set).

The predictor scores of these inputs are exact in fp32 (see
``synthetic.make_clustered_inputs``), so every GPU index row must equal the
oracle's row exactly, ties to the lower key included."""
import math

import numpy as np
import pytest
import torch

import dynamic_sparse_attention_dsv_gb300 as dsv
from dynamic_sparse_attention_dsv_gb300 import synthetic as syn
from oracle import dsv_oracle as ora

from .parity import check_kcov

pytestmark = pytest.mark.gpu

GROUP = (2, 8, 8)

# (grid, d, r, heads, mode, k values)
CASES = {
    "spread_r32": ((16, 32, 32), 128, 32, 2, "spread", (5000, 16381, 1)),
    "spread_r64": ((16, 32, 32), 128, 64, 2, "spread", (5000, 12000)),
    "ties_r64_d64": ((16, 32, 32), 64, 64, 1, "ties", (9000, 2)),
    "ties_64k_r32": ((16, 64, 64), 128, 32, 1, "ties", (20000, 6554)),
    "ties_64k_r64": ((16, 64, 64), 128, 64, 1, "ties", (40000,)),
}


def _oracle_row(inp, h, grid, k):
    mem = ora.group_members(*grid, *GROUP)
    q = ora.lowrank_project(inp["Q"][h], inp["Wq"][h])
    kk = ora.lowrank_project(inp["K"][h], inp["Wk"][h])
    s = ora.group_scores(q, kk, mem, [0])[0]   # every group's queries are equal: one row serves all
    return ora.topk_ascending(s, k), s


def _check_all_rows(idx, ks, offs, n_groups, h, ref):
    rows = idx[offs[h]: offs[h] + n_groups * ks[h]].view(n_groups, ks[h]).cpu().numpy()
    bad = np.nonzero(~np.all(rows == ref[None, :], axis=1))[0]
    assert bad.size == 0, f"head {h}: {bad.size} rows differ from the oracle (first group {bad[:1]})"


@pytest.mark.parametrize("name", list(CASES))
def test_topk_exact_on_clustered_scores(name):
    grid, d, r, H, mode, kvals = CASES[name]
    inp = syn.make_clustered_inputs(*grid, d, r, H, mode)
    dev = {n: inp[n].cuda() for n in ("Q", "K", "Wq", "Wk")}
    S = grid[0] * grid[1] * grid[2]
    n_groups = S // (GROUP[0] * GROUP[1] * GROUP[2])
    for k in kvals:
        st = dsv.new_status()
        idx, ks, offs = dsv.lowrank_topk(dev["Q"], dev["K"], dev["Wq"], dev["Wk"], grid, GROUP, k, status=st)
        dsv.check_status(st, f"{name} k={k}")
        for h in range(H):
            ref, _ = _oracle_row(inp, h, grid, k)
            _check_all_rows(idx, ks, offs, n_groups, h, ref)


@pytest.mark.parametrize("name", list(CASES))
def test_coverage_topk_exact_on_clustered_scores(name):
    """The combined call writes the same exact rows on the same inputs. Its
    bracket for the k-th score comes from the coverage pass's half-bin counts
    (no histogram pass), so these inputs also drive the REFINE rounds, the
    tied rows and the resolve from that bracket."""
    grid, d, r, H, mode, kvals = CASES[name]
    inp = syn.make_clustered_inputs(*grid, d, r, H, mode)
    dev = {n: inp[n].cuda() for n in ("Q", "K", "Wq", "Wk")}
    S = grid[0] * grid[1] * grid[2]
    n_groups = S // (GROUP[0] * GROUP[1] * GROUP[2])
    for k in tuple(kvals) + (7000,):
        st = dsv.new_status()
        _, _, idx, ks, offs = dsv.coverage_topk(dev["Q"], dev["K"], dev["Wq"], dev["Wk"], grid, GROUP, k, status=st)
        dsv.check_status(st, f"coverage_topk {name} k={k}")
        for h in range(H):
            ref, _ = _oracle_row(inp, h, grid, k)
            _check_all_rows(idx, ks, offs, n_groups, h, ref)


@pytest.mark.parametrize("k", [65536, 2621])
def test_topk_exact_on_clustered_scores_256k(k):
    """One head at the dispatcher layer's size (64x64x64, S=262144, d=128,
    r=32, cube 2x8x8): 262,142 keys in the cluster, every one of the 2048
    index rows exact."""
    grid = (64, 64, 64)
    inp = syn.make_clustered_inputs(*grid, 128, 32, 1, "spread", seed=11)
    dev = {n: inp[n].cuda() for n in ("Q", "K", "Wq", "Wk")}
    st = dsv.new_status()
    idx, ks, offs = dsv.lowrank_topk(dev["Q"], dev["K"], dev["Wq"], dev["Wk"], grid, GROUP, k, status=st)
    dsv.check_status(st, f"256k k={k}")
    ref, _ = _oracle_row(inp, 0, grid, k)
    _check_all_rows(idx, ks, offs, 2048, 0, ref)
