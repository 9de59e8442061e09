"""Per-query predicted mass (the share of each query's own predicted softmax
mass that its group's selected keys carry; technical summary section 2.1)
against the oracle, on the oracle's exact index sets: every query's share
within 1e-4 (the predictor scores carry ~2^-21 relative error, which moves
a logit of size <= 50 by <= 2.5e-5), and the per-head mean within 1e-5."""
import math

import numpy as np
import pytest
import torch

import dynamic_sparse_attention_dsv_gb300 as dsv
from dynamic_sparse_attention_dsv_gb300 import synthetic as syn
from oracle import dsv_oracle as ora

pytestmark = pytest.mark.gpu

PQ_ABS, MEAN_ABS = 1e-4, 1e-5

CASES = {
    "oracle_scale": syn.workload(0),
    "ragged_d128_g128": syn.Workload("ragged", 101, 2, 4, 16, 32, 128, 32, 2, 8, 8, 300, ("uniform", 2.0, 8.0), False),
    "d64_r64": syn.Workload("d64r64", 102, 2, 4, 8, 16, 64, 64, 4, 4, 4, 200, ("const", 4.0), False),
    "r16_h3": syn.Workload("r16", 103, 3, 8, 16, 16, 64, 16, 4, 4, 4, 129, ("uniform", 1.0, 8.0), False),
}


def _run(w, inp, dense_heads=()):
    mem = ora.group_members(w.T, w.Y, w.X, w.gt, w.gy, w.gx)
    scale = 1.0 / math.sqrt(w.d)
    refs, flat = [], []
    for h in range(w.H):
        idx, _ = ora.lowrank_topk(inp["Q"][h], inp["K"][h], inp["Wq"][h], inp["Wk"][h], mem, w.k)
        if h in dense_heads:
            idx = np.tile(np.arange(w.S), (w.n_groups, 1))
        else:
            flat.append(idx.astype(np.int32).ravel())
        refs.append(ora.predicted_mass(inp["Q"][h], inp["K"][h], inp["Wq"][h], inp["Wk"][h], idx, mem, scale))
    ks, offs, _ = dsv.topk_layout(w.H, w.n_groups, w.k, skip=[h in dense_heads for h in range(w.H)])
    d = {n: inp[n].cuda() for n in ("Q", "K", "Wq", "Wk")}
    idx_dev = torch.from_numpy(np.concatenate(flat)).cuda() if flat else torch.zeros(1, dtype=torch.int32).cuda()
    st = dsv.new_status()
    mass, pq = dsv.predicted_mass(d["Q"], d["K"], d["Wq"], d["Wk"], (w.T, w.Y, w.X), (w.gt, w.gy, w.gx), idx_dev, ks,
                                  offs, per_query=True, status=st)
    dsv.check_status(st, "predicted_mass")
    return refs, mass.cpu().numpy(), pq.cpu().numpy()


@pytest.mark.parametrize("name", list(CASES))
def test_predicted_mass_matches_oracle(name):
    w = CASES[name]
    inp = syn.make_inputs(w)
    refs, mass, pq = _run(w, inp)
    for h in range(w.H):
        assert np.abs(pq[h] - refs[h]).max() <= PQ_ABS, (h, np.abs(pq[h] - refs[h]).max())
        assert abs(float(mass[h]) - refs[h].mean()) <= MEAN_ABS, (h, float(mass[h]), refs[h].mean())


def test_predicted_mass_dense_head_is_one():
    """A head without index sets (offset -1) selects every key: m_i = 1."""
    w = CASES["r16_h3"]
    inp = syn.make_inputs(w)
    refs, mass, pq = _run(w, inp, dense_heads=(1,))
    assert np.all(pq[1] == 1.0) and float(mass[1]) == 1.0
    for h in (0, 2):
        assert np.abs(pq[h] - refs[h]).max() <= PQ_ABS


def test_predicted_mass_16k_head():
    """One head of the 16K workload (8x32x64, d=64, r=32, cube 4x4x4,
    k=1638): 256 groups x 16384 keys, every query against the oracle."""
    w = syn.workload(1, H=1)
    inp = syn.make_inputs(w, with_grad_out=False)
    refs, mass, pq = _run(w, inp)
    assert np.abs(pq[0] - refs[0]).max() <= PQ_ABS
    assert abs(float(mass[0]) - refs[0].mean()) <= MEAN_ABS
