"""dsv_lowrank_topk_noalloc: the top-k for callers that cannot allocate device
memory (its scratch is a fixed array inside libdsv). Checked through the C ABI
against dsv_lowrank_topk on two calls in a row. This file is collected last."""
import ctypes

import numpy as np
import pytest
import torch

import dynamic_sparse_attention_dsv_gb300 as dsv
from dynamic_sparse_attention_dsv_gb300 import api, native
from dynamic_sparse_attention_dsv_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu


def _call_noalloc(lib, d, w, ks, offs, idx, status):
    shape = api.make_shape(d["Q"], (w.T, w.Y, w.X))
    group = api.make_group((w.gt, w.gy, w.gx))
    return lib.dsv_lowrank_topk_noalloc(api._ptr(d["Q"]), api._ptr(d["K"]), api._ptr(d["Wq"]), api._ptr(d["Wk"]),
                                        shape, int(w.r), group, api._i32(ks), api._i64(offs), api._ptr(idx),
                                        api._ptr(status), api._stream())


def test_noalloc_matches_workspace_topk_twice():
    lib = native.load()
    runs = [syn.workload(0), syn.Workload("second", 107, 2, 4, 16, 32, 128, 32, 2, 8, 8, 300, ("uniform", 2.0, 8.0),
                                          False)]
    for w in runs:   # two calls in a row, the second on a different shape and k
        d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in syn.make_inputs(w).items()}
        st = dsv.new_status()
        ref, ks, offs = dsv.lowrank_topk(d["Q"], d["K"], d["Wq"], d["Wk"], (w.T, w.Y, w.X), (w.gt, w.gy, w.gx), w.k,
                                         status=st)
        got = torch.full_like(ref, -1)
        assert _call_noalloc(lib, d, w, ks, offs, got, st) == 0
        dsv.check_status(st, "noalloc")
        # index work is compared bit for bit
        assert torch.equal(got, ref)


def test_noalloc_rejects_shapes_beyond_its_scratch():
    lib = native.load()
    w = syn.workload(3)       # S = 131072: its top-k scratch is far above 64 MiB
    q = torch.empty((1, w.S, w.d), dtype=torch.bfloat16, device="cuda")
    wq = torch.empty((1, w.d, w.r), dtype=torch.bfloat16, device="cuda")
    need = api.lowrank_topk_workspace_size(q, (w.T, w.Y, w.X), (w.gt, w.gy, w.gx), w.r)
    assert need > (64 << 20)
    idx = torch.empty(1, dtype=torch.int32, device="cuda")
    st = dsv.new_status()
    d = dict(Q=q, K=q, Wq=wq, Wk=wq)
    code = _call_noalloc(lib, d, w.__class__(**{**w.__dict__, "H": 1}), [w.k], [0], idx, st)
    assert code == 3   # DSV_ERR_WORKSPACE, nothing launched
    assert dsv.read_status(st) == 0
