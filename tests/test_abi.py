"""CPU-only checks of the C ABI: the library loads, exports every symbol the
header declares, validates arguments before launching anything, and its host
logic (dispatcher, workspace sizing) matches the oracle and the O(S*k) claim."""
import ctypes
import os
import re

import numpy as np
import pytest

from dynamic_sparse_attention_dsv_gb300 import api, native
from oracle import dsv_oracle as ora

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    with open(os.path.join(ROOT, "include", "libdsv.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"\b(dsv_[a-z_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    return native.load()


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert "dsv_lowrank_topk" in names and "dsv_sparse_attn_bwd" in names
    for n in names:
        assert hasattr(lib, n), n
    # the binding declares exactly the header's entry points
    assert sorted(n for n, _, _ in native.SIGNATURES) == names


def test_status_strings(lib):
    for code, name in native.DSV_STATUS.items():
        assert lib.dsv_status_string(code).decode().startswith(name)


@pytest.mark.parametrize("S,kcovs", [(262144, [1, 2621, 50000, 65536, 70000, 131072, 131073, 262144]),
                                     (16384, [1, 163, 164, 2000, 4096, 4097, 8192, 8193]),
                                     (1024, [1, 10, 11, 256, 257, 512, 513])])
def test_plan_heads_matches_oracle(S, kcovs):
    n_groups = S // 128
    k_h, dense, offs, total = api.plan_heads(kcovs, S, n_groups)
    ok, od = ora.plan_heads(kcovs, S)
    assert k_h == ok and dense == od
    run = 0
    for k, dn, off in zip(k_h, dense, offs):
        if dn:
            assert off == -1
        else:
            assert off == run
            run += n_groups * k
    assert total == run


def test_plan_heads_rejects_bad_input(lib):
    kc = (ctypes.c_int32 * 1)(0)
    out_k = (ctypes.c_int32 * 1)()
    out_d = (ctypes.c_uint8 * 1)()
    out_o = (ctypes.c_int64 * 1)()
    tot = ctypes.c_int64()
    assert lib.dsv_plan_heads(kc, 1, 1024, 8, 0.01, 0.25, 0.5, out_k, out_d, out_o, ctypes.byref(tot)) == 1


def _shape(B, H, T, Y, X, d):
    return native.dsv_shape(B, H, T, Y, X, d)


def test_workspace_is_order_S_k_not_S_squared(lib):
    """At a fixed k, scratch bytes per token stay bounded as S grows 8x (an
    S x S term would grow 8x); the backward's grows with k as O(S k)."""
    g = native.dsv_group(2, 8, 8)
    sizes = []
    for T in (8, 16, 32, 64):
        s = _shape(1, 1, T, 64, 64, 128)
        k = (ctypes.c_int32 * 1)(2048)
        off = (ctypes.c_int64 * 1)(0)
        sizes.append(lib.dsv_lowrank_topk_workspace_size(s, 32, g) + lib.dsv_coverage_workspace_size(s, 32, g) +
                     lib.dsv_sparse_attn_bwd_workspace_size(s, g, k, off))
    S = np.array([8, 16, 32, 64]) * 4096
    ratio = np.array(sizes) / S
    assert ratio.max() / ratio.min() < 1.6, ratio
    # backward scratch: O(n_groups * k) partial rows
    s = _shape(1, 1, 16, 64, 64, 128)
    small = lib.dsv_sparse_attn_bwd_workspace_size(s, g, (ctypes.c_int32 * 1)(1000), (ctypes.c_int64 * 1)(0))
    big = lib.dsv_sparse_attn_bwd_workspace_size(s, g, (ctypes.c_int32 * 1)(4000), (ctypes.c_int64 * 1)(0))
    n_groups = 16 * 64 * 64 // 128
    assert big - small >= n_groups * 3000 * 128 * 4 * 0.99
    # the minimum (one query group per launch) is far below the full plan and is accepted
    least = lib.dsv_sparse_attn_bwd_min_workspace_size(s, g, (ctypes.c_int32 * 1)(4000), (ctypes.c_int64 * 1)(0))
    assert 0 < least < big // 8
    fake = ctypes.c_void_p(256)
    args = lambda nbytes: (fake, fake, fake, fake, fake, fake, fake, (ctypes.c_int32 * 1)(4000),
                           (ctypes.c_int64 * 1)(0), s, g, ctypes.c_float(0.1), fake, fake, fake, fake, nbytes, None,
                           None)
    assert lib.dsv_sparse_attn_bwd(*args(least)) != 3       # past the workspace check (no GPU here: launch fails)
    assert lib.dsv_sparse_attn_bwd(*args(least // 2)) == 3
    # dense-only problems need almost nothing
    assert lib.dsv_sparse_attn_bwd_workspace_size(s, g, None, None) < 64 << 20


def test_argument_validation_before_launch(lib):
    g = native.dsv_group(2, 8, 8)
    s = _shape(1, 1, 16, 64, 64, 128)
    fake = ctypes.c_void_p(256)
    ks = (ctypes.c_int32 * 1)(10)
    offs = (ctypes.c_int64 * 1)(0)
    # group does not divide the grid
    assert lib.dsv_lowrank_topk(fake, fake, fake, fake, s, 32, native.dsv_group(3, 8, 8), ks, offs, fake, fake, 1 << 30,
                                None, None) == 1
    # unsupported rank / head dim / group size
    assert lib.dsv_lowrank_topk(fake, fake, fake, fake, s, 48, g, ks, offs, fake, fake, 1 << 30, None, None) == 2
    assert lib.dsv_sparse_attn_fwd(fake, fake, fake, None, None, None, _shape(1, 1, 16, 64, 64, 96), g,
                                   ctypes.c_float(0.1), fake, fake, None, 0, None, None) == 2
    assert lib.dsv_sparse_attn_fwd(fake, fake, fake, None, None, None, s, native.dsv_group(1, 4, 8),
                                   ctypes.c_float(0.1), fake, fake, None, 0, None, None) == 2
    # null / misaligned pointers
    assert lib.dsv_sparse_attn_fwd(None, fake, fake, None, None, None, s, g, ctypes.c_float(0.1), fake, fake, None, 0,
                                   None, None) == 1
    assert lib.dsv_sparse_attn_fwd(ctypes.c_void_p(258), fake, fake, None, None, None, s, g, ctypes.c_float(0.1), fake,
                                   fake, None, 0, None, None) == 1
    # k out of range
    bad = (ctypes.c_int32 * 1)(s.T * s.Y * s.X + 1)
    assert lib.dsv_lowrank_topk(fake, fake, fake, fake, s, 32, g, bad, offs, fake, fake, 1 << 40, None, None) == 1
    # missing or short workspace
    assert lib.dsv_lowrank_topk(fake, fake, fake, fake, s, 32, g, ks, offs, fake, None, 0, None, None) == 3
    assert lib.dsv_sparse_attn_bwd(fake, fake, fake, fake, fake, fake, None, None, None, s, g, ctypes.c_float(0.1),
                                   fake, fake, fake, fake, 16, None, None) == 3
    # S not a multiple of 128
    assert lib.dsv_coverage(fake, fake, fake, fake, _shape(1, 1, 1, 8, 8, 64), 16, native.dsv_group(1, 8, 8),
                            ctypes.c_float(0.1), ctypes.c_float(0.9), fake, None, 0, fake, 1 << 30, None, None) == 2


def test_coverage_topk_workspace_and_validation(lib):
    """The combined call holds both calls' buffers with the projections and
    row ranges once, and rejects bad arguments before anything launches."""
    g = native.dsv_group(2, 8, 8)
    s = _shape(1, 2, 16, 64, 64, 128)
    both = lib.dsv_coverage_topk_workspace_size(s, 32, g)
    topk = lib.dsv_lowrank_topk_workspace_size(s, 32, g)
    cov = lib.dsv_coverage_workspace_size(s, 32, g)
    assert max(topk, cov) < both < topk + cov
    fake = ctypes.c_void_p(256)
    ks = (ctypes.c_int32 * 2)(10, 10)
    offs = (ctypes.c_int64 * 2)(0, 10 * 512)
    args = lambda k, mass, ws_bytes: (fake, fake, fake, fake, s, 32, g, ctypes.c_float(0.1), ctypes.c_float(mass),
                                      fake, None, 0, k, offs, fake, fake, ws_bytes, None, None)
    assert lib.dsv_coverage_topk(*args((ctypes.c_int32 * 2)(10, s.T * s.Y * s.X + 1), 0.9, 1 << 40)) == 1
    assert lib.dsv_coverage_topk(*args(ks, 1.5, 1 << 40)) == 1
    assert lib.dsv_coverage_topk(*args(ks, 0.9, both - 1)) == 3
    assert lib.dsv_coverage_topk(fake, fake, fake, fake, s, 48, g, ctypes.c_float(0.1), ctypes.c_float(0.9), fake,
                                 None, 0, ks, offs, fake, fake, 1 << 40, None, None) == 2


def test_attn_mass_validation(lib):
    fake = ctypes.c_void_p(256)
    assert lib.dsv_attn_mass(None, fake, 1024, 2, fake, None, None) == 1
    assert lib.dsv_attn_mass(fake, fake, 0, 2, fake, None, None) == 1
    assert lib.dsv_attn_mass(fake, fake, 1024, 257, fake, None, None) == 1
    assert lib.dsv_attn_mass(ctypes.c_void_p(258), fake, 1024, 2, fake, None, None) == 1


def test_plan_gpus_matches_oracle(lib):
    rng = np.random.default_rng(5)
    for _ in range(50):
        n, N = int(rng.integers(1, 40)), int(rng.integers(1, 9))
        cost = [int(c) for c in rng.integers(0, 1 << 20, n)]
        for eq in (False, True):
            assert api.plan_gpus(cost, N, eq) == ora.plan_gpus(cost, N, eq)
    # ties: equal costs keep head order, lower GPUs first
    assert api.plan_gpus([7, 7, 7], 2, False) == ora.plan_gpus([7, 7, 7], 2, False)
    gpu_of = (ctypes.c_int32 * 2)()
    assert lib.dsv_plan_gpus((ctypes.c_int64 * 2)(1, -1), 2, 2, 1, gpu_of, None) == 1
    assert lib.dsv_plan_gpus((ctypes.c_int64 * 2)(1, 1), 2, 0, 1, gpu_of, None) == 1
    assert lib.dsv_plan_gpus(None, 2, 2, 1, gpu_of, None) == 1


def test_topk_layout_packs_rows():
    ks, offs, total = api.topk_layout(3, 16, [5, 7, 9], skip=[False, True, False])
    assert offs == [0, -1, 80] and total == 80 + 16 * 9


def test_wait_limit_setter_is_host_only(lib):
    """dsv_set_wait_limit_ns only swaps a host value (no CUDA call): it works
    without a GPU and returns the previous limit (2 s by default)."""
    prev = lib.dsv_set_wait_limit_ns(7)
    try:
        assert prev == 2_000_000_000
        assert lib.dsv_set_wait_limit_ns(11) == 7
    finally:
        lib.dsv_set_wait_limit_ns(prev)
