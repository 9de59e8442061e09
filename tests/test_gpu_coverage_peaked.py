"""Coverage (the smallest k whose pooled predicted softmax mass reaches 90%)
on peaked predictor scores, where a bin-interpolated estimate goes wrong
(technical summary section 2.1: the critical KV carry over 90% of the
attention score): a two-level score row with the 90% point inside the
lower level, a single dominant key, and a narrow cluster with one key far
above and one far below it. Every group of these inputs has the same score
row, so the oracle's curve of one row is the pooled curve."""
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
GRID = (8, 32, 32)   # S = 8192


def _oracle_curve(inp, h, grid, d):
    mem = ora.group_members(*grid, *GROUP)
    q = ora.lowrank_project(inp["Q"][h], inp["Wq"][h])
    k = ora.lowrank_project(inp["K"][h], inp["Wk"][h])
    s = ora.group_scores(q, k, mem, [0])
    return ora.coverage_curve(s, 1.0 / math.sqrt(d))


@pytest.mark.parametrize("mode", ["two_level", "dominant", "spread", "ties"])
@pytest.mark.parametrize("r", [32, 64])
def test_coverage_exact_on_peaked_scores(mode, r):
    d, H = 128, 2
    inp = syn.make_clustered_inputs(*GRID, d, r, H, mode)
    dev = {n: inp[n].cuda() for n in ("Q", "K", "Wq", "Wk")}
    S = GRID[0] * GRID[1] * GRID[2]
    st = dsv.new_status()
    k_cov, curve = dsv.coverage(dev["Q"], dev["K"], dev["Wq"], dev["Wk"], GRID, GROUP, mass=0.9, curve_points=16,
                                status=st)
    dsv.check_status(st, f"coverage {mode} r={r}")
    k_cov = k_cov.cpu().numpy()
    pts = np.array([int(math.ceil((i + 1) * S / 16)) for i in range(16)])
    for h in range(H):
        C = _oracle_curve(inp, h, GRID, d)
        why = check_kcov(C, int(k_cov[h]))
        assert not why, f"{mode} r={r} head {h}: {why} (oracle k_cov {int(np.argmax(C >= 0.9)) + 1})"
        np.testing.assert_allclose(curve[h].cpu().numpy(), C[pts - 1], atol=2e-4)
    if mode == "dominant":
        assert list(k_cov) == [1] * H


def test_coverage_topk_on_peaked_scores():
    """The combined call gives the same k_cov and curve on a peaked row."""
    d, r, H = 128, 32, 2
    inp = syn.make_clustered_inputs(*GRID, d, r, H, "two_level")
    dev = {n: inp[n].cuda() for n in ("Q", "K", "Wq", "Wk")}
    st = dsv.new_status()
    k1, c1 = dsv.coverage(dev["Q"], dev["K"], dev["Wq"], dev["Wk"], GRID, GROUP, curve_points=8, status=st)
    k2, c2, _, _, _ = dsv.coverage_topk(dev["Q"], dev["K"], dev["Wq"], dev["Wk"], GRID, GROUP, 300, curve_points=8,
                                        status=st)
    dsv.check_status(st, "coverage_topk peaked")
    assert torch.equal(k1, k2) and torch.equal(c1, c2)
