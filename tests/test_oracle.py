"""Pins for the CPU oracle, checked against things other than the oracle itself:
a hand-derived worked example, closed forms, brute force over the full S x S
matrix, and library routines (numpy sorting, torch SDPA and autograd)."""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import dsv_oracle as ora

pytestmark = pytest.mark.filterwarnings("ignore::DeprecationWarning")


def _golden(golden_dir):
    with open(os.path.join(golden_dir, "tiny_hand_example.json")) as f:
        return json.load(f)


# ------------------------------------------------------------ query groups
def test_group_members_hand_cube():
    mem = ora.group_members(4, 4, 4, 2, 2, 2)
    assert mem.shape == (8, 8)
    # first cube: t in {0,1}, y in {0,1}, x in {0,1} on a 4x4x4 grid
    assert mem[0].tolist() == [0, 1, 4, 5, 16, 17, 20, 21]
    # second cube is the next one along x
    assert mem[1].tolist() == [2, 3, 6, 7, 18, 19, 22, 23]
    # the cubes partition the grid
    assert sorted(mem.ravel().tolist()) == list(range(64))


def test_group_members_rejects_non_dividing_cube():
    with pytest.raises(ValueError):
        ora.group_members(4, 4, 6, 2, 2, 4)


# -------------------------------------------------- hand-derived example
def test_golden_scores_topk_coverage(golden_dir):
    g = _golden(golden_dir)
    grid = g["grid"]
    mem = ora.group_members(grid["T"], grid["Y"], grid["X"], grid["gt"], grid["gy"], grid["gx"])
    assert mem.tolist() == g["groups"]
    Q, K = np.array(g["Q"], float), np.array(g["K"], float)
    Wq, Wk = np.array(g["Wq"], float), np.array(g["Wk"], float)
    s = ora.group_scores(ora.lowrank_project(Q, Wq), ora.lowrank_project(K, Wk), mem)
    np.testing.assert_allclose(s, g["group_scores"]["value"], atol=1e-12)
    for kk in (1, 2, 3):
        idx, _ = ora.lowrank_topk(Q, K, Wq, Wk, mem, kk)
        assert idx.tolist() == g["topk"][f"k{kk}"]
    scale = 1.0 / math.sqrt(g["d"])
    np.testing.assert_allclose(ora.coverage_curve(s, scale), g["coverage"]["C"], atol=2e-6)
    for mass, kc in g["coverage"]["k_cov"].items():
        assert ora.coverage_k(s, scale, float(mass)) == kc


def test_golden_attention(golden_dir):
    g = _golden(golden_dir)
    grid = g["grid"]
    mem = ora.group_members(grid["T"], grid["Y"], grid["X"], grid["gt"], grid["gy"], grid["gx"])
    a = g["attention_k2"]
    O, L = ora.sparse_attn_fwd(np.array(g["Q"], float), np.array(g["K"], float), np.array(g["V"], float),
                               np.array(a["idx"]), mem, 1.0 / math.sqrt(g["d"]))
    np.testing.assert_allclose(O, a["O"], atol=2e-6)
    np.testing.assert_allclose(L, a["LSE"], atol=2e-6)


# ------------------------------------------------------- predictor + top-k
def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def test_mean_of_dots_equals_dot_of_mean():
    mem = ora.group_members(2, 4, 4, 1, 2, 2)
    q, k = _rand((32, 8), 1), _rand((32, 8), 2)
    s = ora.group_scores(q, k, mem)
    alt = np.stack([q[m].mean(axis=0) for m in mem]) @ k.T
    np.testing.assert_allclose(s, alt, rtol=0, atol=1e-12)
    np.testing.assert_allclose(ora.group_scores_via_mean(q, k, mem), s, rtol=0, atol=1e-12)
    np.testing.assert_allclose(ora.group_scores_via_mean(q, k, mem, [3, 1]), s[[3, 1]], rtol=0, atol=1e-12)


def test_identity_predictor_gives_true_group_topk():
    """r = d, W = I: the predicted group score must equal the group mean of the
    true QK^T, taken from the full S x S matrix (brute force)."""
    T, Y, X, d = 2, 4, 8, 8
    mem = ora.group_members(T, Y, X, 1, 2, 4)
    S = T * Y * X
    Q, K = _rand((S, d), 3), _rand((S, d), 4)
    full = Q @ K.T                                            # [S, S]
    brute = np.stack([full[m].mean(axis=0) for m in mem])
    eye = np.eye(d)
    for k in (1, 5, 17, S):
        idx, s = ora.lowrank_topk(Q, K, eye, eye, mem, k)
        np.testing.assert_allclose(s, brute, atol=1e-12)
        want = np.sort(np.argsort(-brute, axis=1, kind="stable")[:, :k], axis=1)
        assert np.array_equal(idx, want)


def test_truncated_identity_predictor():
    """W = first r columns of I: scores use only the first r channels."""
    T, Y, X, d, r = 1, 8, 8, 16, 4
    mem = ora.group_members(T, Y, X, 1, 4, 4)
    S = T * Y * X
    Q, K = _rand((S, d), 5), _rand((S, d), 6)
    W = np.eye(d)[:, :r]
    full = Q[:, :r] @ K[:, :r].T
    brute = np.stack([full[m].mean(axis=0) for m in mem])
    idx, s = ora.lowrank_topk(Q, K, W, W, mem, 9)
    np.testing.assert_allclose(s, brute, atol=1e-12)
    assert np.array_equal(idx, np.sort(np.argsort(-brute, axis=1, kind="stable")[:, :9], axis=1))


def test_topk_ties_go_to_lower_index():
    s = np.array([1.0, 3.0, 3.0, 2.0, 3.0, 0.0])
    assert ora.topk_ascending(s, 1).tolist() == [1]
    assert ora.topk_ascending(s, 2).tolist() == [1, 2]
    assert ora.topk_ascending(s, 4).tolist() == [1, 2, 3, 4]
    rng = np.random.default_rng(7)
    for _ in range(20):
        row = rng.integers(0, 5, size=64).astype(float)        # heavy ties
        k = int(rng.integers(1, 65))
        want = np.sort(np.argsort(-row, kind="stable")[:k])     # stable: lower index first
        assert ora.topk_ascending(row, k).tolist() == want.tolist()


def test_topk_rejects_bad_k():
    with pytest.raises(ValueError):
        ora.topk_ascending(np.zeros(4), 0)
    with pytest.raises(ValueError):
        ora.topk_ascending(np.zeros(4), 5)


# ----------------------------------------------------------------- coverage
def test_coverage_monotone_and_reaches_one():
    s = 3.0 * _rand((16, 300), 8)
    C = ora.coverage_curve(s, 0.125)
    assert np.all(np.diff(C) >= -1e-15)
    assert abs(C[-1] - 1.0) < 1e-12
    assert ora.coverage_k(s, 0.125, 1.0 - 1e-15) <= 300


def test_coverage_uniform_scores_closed_form():
    S = 1024                                  # C(k) = k/S, 0.9 S = 921.6
    s = np.zeros((3, S))
    np.testing.assert_allclose(ora.coverage_curve(s, 1.0), np.arange(1, S + 1) / S, atol=1e-12)
    assert ora.coverage_k(s, 1.0, 0.9) == 922


def test_coverage_dominant_key():
    s = np.zeros((2, 50))
    s[0, 7] = 1000.0
    s[1, 3] = 1000.0
    assert ora.coverage_k(s, 0.125, 0.9) == 1


def test_coverage_two_level_closed_form():
    """m keys at score a, the rest at 0; with scale 1/sqrt(64) the high keys
    carry weight w = exp(a/8) = 37.3 each: C(k) = k w/Z for k <= m, then adds
    1/Z per low key, Z = m w + S - m. With S=100, m=10: the high keys hold
    373/463 of the mass, 0.9*463 = 416.7 needs 43.7 more low keys -> k = 54."""
    S, m, wgt = 100, 10, 37.3
    a = 8.0 * math.log(wgt)
    s = np.zeros((1, S))
    s[0, 20:30] = a
    Z = m * wgt + S - m
    C = ora.coverage_curve(s, 1.0 / math.sqrt(64))
    k = np.arange(1, S + 1)
    want = np.where(k <= m, k * wgt / Z, (m * wgt + (k - m)) / Z)
    np.testing.assert_allclose(C, want, atol=1e-12)
    assert ora.coverage_k(s, 1.0 / math.sqrt(64), 0.9) == 54


# --------------------------------------------------------------- dispatcher
@pytest.mark.parametrize("kcov,k,dense", [
    (1, 2621, False), (2621, 2621, False), (50000, 50000, False), (65536, 65536, False),
    (70000, 65536, False), (131072, 65536, False), (131073, 262144, True), (262144, 262144, True)])
def test_plan_heads_table_s262144(kcov, k, dense):
    ks, ds = ora.plan_heads([kcov], 262144)
    assert ks == [k] and ds == [dense]


def test_plan_heads_rounding_half_up():
    # 1% of 16384 = 163.84 -> 164; 25% = 4096
    ks, _ = ora.plan_heads([1, 5000], 16384)
    assert ks == [164, 4096]
    assert ora.round_half_up(1638.4) == 1638 and ora.round_half_up(6553.6) == 6554
    assert ora.round_half_up(2.5) == 3


# -------------------------------------------------------- attention forward
def _tiny_problem(seed, T=2, Y=4, X=4, cube=(1, 2, 2), d=8, k=5):
    rng = np.random.default_rng(seed)
    mem = ora.group_members(T, Y, X, *cube)
    S = T * Y * X
    Q, K, V, dO = (rng.standard_normal((S, d)) for _ in range(4))
    idx = np.stack([np.sort(rng.choice(S, size=k, replace=False)) for _ in range(mem.shape[0])])
    return mem, Q, K, V, dO, idx


def _mask(mem, idx, S):
    m = np.zeros((S, S), dtype=bool)
    for g, members in enumerate(mem):
        for i in members:
            m[i, idx[g]] = True
    return m


def _sdpa(Q, K, V, mask, scale):
    t = lambda a: torch.tensor(a, dtype=torch.float64)
    am = None if mask is None else torch.tensor(mask)
    return torch.nn.functional.scaled_dot_product_attention(t(Q)[None], t(K)[None], t(V)[None],
                                                            attn_mask=am, scale=scale)[0].numpy()


def test_dense_attention_equals_sdpa():
    mem, Q, K, V, _, _ = _tiny_problem(11)
    scale = 1 / math.sqrt(Q.shape[1])
    O, L = ora.sparse_attn_fwd(Q, K, V, None, mem, scale)
    np.testing.assert_allclose(O, _sdpa(Q, K, V, None, scale), atol=1e-12)
    full = scale * Q @ K.T
    np.testing.assert_allclose(L, np.log(np.exp(full).sum(axis=1)), atol=1e-12)
    # k = S through an explicit index set is the same computation
    all_idx = np.tile(np.arange(Q.shape[0]), (mem.shape[0], 1))
    O2, L2 = ora.sparse_attn_fwd(Q, K, V, all_idx, mem, scale)
    np.testing.assert_allclose(O2, O, atol=1e-14)
    np.testing.assert_allclose(L2, L, atol=1e-14)


def test_sparse_attention_equals_masked_sdpa():
    mem, Q, K, V, _, idx = _tiny_problem(12)
    scale = 0.37
    O, L = ora.sparse_attn_fwd(Q, K, V, idx, mem, scale)
    mask = _mask(mem, idx, Q.shape[0])
    np.testing.assert_allclose(O, _sdpa(Q, K, V, mask, scale), atol=1e-12)
    logits = np.where(mask, scale * Q @ K.T, -np.inf)
    np.testing.assert_allclose(L, torch.logsumexp(torch.tensor(logits), dim=1).numpy(), atol=1e-12)


def test_zero_query_closed_form():
    mem, Q, K, V, _, idx = _tiny_problem(13)
    O, L = ora.sparse_attn_fwd(np.zeros_like(Q), K, V, idx, mem, 0.5)
    for g, members in enumerate(mem):
        np.testing.assert_allclose(O[members], np.tile(V[idx[g]].mean(axis=0), (len(members), 1)), atol=1e-14)
        np.testing.assert_allclose(L[members], math.log(idx.shape[1]), atol=1e-14)


# ------------------------------------------------------- attention backward
def test_backward_central_finite_differences():
    mem, Q, K, V, dO, idx = _tiny_problem(14, T=1, Y=2, X=4, cube=(1, 1, 2), d=4, k=3)
    scale = 0.6

    def loss(Qx, Kx, Vx):
        O, _ = ora.sparse_attn_fwd(Qx, Kx, Vx, idx, mem, scale)
        return float((dO * O).sum())

    dQ, dK, dV = ora.sparse_attn_bwd(Q, K, V, dO, idx, mem, scale)
    h = 1e-6
    for name, base, grad in (("Q", Q, dQ), ("K", K, dK), ("V", V, dV)):
        num = np.zeros_like(base)
        for pos in np.ndindex(base.shape):
            plus, minus = base.copy(), base.copy()
            plus[pos] += h
            minus[pos] -= h
            args_p = [Q, K, V]
            args_m = [Q, K, V]
            which = "QKV".index(name)
            args_p[which], args_m[which] = plus, minus
            num[pos] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        np.testing.assert_allclose(grad, num, rtol=1e-6, atol=1e-8, err_msg=name)


def test_backward_equals_torch_autograd():
    mem, Q, K, V, dO, idx = _tiny_problem(15)
    scale = 0.29
    mask = torch.tensor(_mask(mem, idx, Q.shape[0]))
    tq, tk, tv = (torch.tensor(a, dtype=torch.float64, requires_grad=True) for a in (Q, K, V))
    out = torch.nn.functional.scaled_dot_product_attention(tq[None], tk[None], tv[None], attn_mask=mask,
                                                           scale=scale)[0]
    (out * torch.tensor(dO)).sum().backward()
    dQ, dK, dV = ora.sparse_attn_bwd(Q, K, V, dO, idx, mem, scale)
    np.testing.assert_allclose(dQ, tq.grad.numpy(), atol=1e-11)
    np.testing.assert_allclose(dK, tk.grad.numpy(), atol=1e-11)
    np.testing.assert_allclose(dV, tv.grad.numpy(), atol=1e-11)
    # the per-group helper agrees with the full backward
    for g in (0, 3):
        Og, lse, dq = ora.sparse_attn_group_dq(Q, K, V, dO, idx[g], mem[g], scale)
        np.testing.assert_allclose(dq, dQ[mem[g]], atol=1e-12)


def test_key_grads_equal_full_backward_rows():
    mem, Q, K, V, dO, idx = _tiny_problem(17, k=9)
    scale = 0.41
    _, dK, dV = ora.sparse_attn_bwd(Q, K, V, dO, idx, mem, scale)
    for key in range(Q.shape[0]):
        dk, dv, hits = ora.sparse_attn_key_grads(Q, K, V, dO, idx, mem, scale, key)
        assert hits == int(sum(key in row for row in idx))
        np.testing.assert_allclose(dk, dK[key], atol=1e-12)
        np.testing.assert_allclose(dv, dV[key], atol=1e-12)


def test_backward_column_sums_identities():
    """sum_j dV_j = sum_i dO_i (softmax rows sum to 1) and sum_j dK_j = 0
    (sum_j P_ij dP_ij = Delta_i); both hold for any index sets."""
    mem, Q, K, V, dO, idx = _tiny_problem(18, k=7)
    _, dK, dV = ora.sparse_attn_bwd(Q, K, V, dO, idx, mem, 0.5)
    np.testing.assert_allclose(dV.sum(axis=0), dO.sum(axis=0), atol=1e-12)
    np.testing.assert_allclose(dK.sum(axis=0), 0.0, atol=1e-12)


def test_backward_dense_equals_all_keys():
    mem, Q, K, V, dO, _ = _tiny_problem(16)
    all_idx = np.tile(np.arange(Q.shape[0]), (mem.shape[0], 1))
    a = ora.sparse_attn_bwd(Q, K, V, dO, None, mem, 0.3)
    b = ora.sparse_attn_bwd(Q, K, V, dO, all_idx, mem, 0.3)
    for x, y in zip(a, b):
        np.testing.assert_allclose(x, y, atol=1e-13)


# ------------------------------------------------------- true attention mass
def test_true_mass_all_keys_is_one_and_uniform_scores_give_k_over_S():
    """Selecting every key captures all of each query's mass; with Q = 0 every
    key has the same probability 1/S, so k selected keys carry exactly k/S."""
    rng = np.random.default_rng(7)
    T, Y, X, d = 2, 4, 8, 16
    S = T * Y * X
    mem = ora.group_members(T, Y, X, 2, 2, 2)
    K = rng.standard_normal((S, d))
    Q = rng.standard_normal((S, d))
    everything = np.tile(np.arange(S), (mem.shape[0], 1))
    np.testing.assert_allclose(ora.true_mass(Q, K, everything, mem, 0.25), 1.0, rtol=0, atol=1e-12)
    k = 11
    some = np.stack([np.sort(rng.choice(S, k, replace=False)) for _ in range(mem.shape[0])])
    np.testing.assert_allclose(ora.true_mass(np.zeros_like(Q), K, some, mem, 0.25), k / S, rtol=0, atol=1e-12)


def test_true_mass_single_dominant_key():
    """A key whose logit exceeds every other by L carries 1 / (1 + (S-1) e^-L)
    of the mass when the others are equal."""
    T, Y, X, d = 1, 2, 4, 8
    S = T * Y * X
    mem = ora.group_members(T, Y, X, 1, 2, 2)
    K = np.zeros((S, d))
    K[3, 0] = 5.0
    Q = np.zeros((S, d))
    Q[:, 0] = 1.0
    idx = np.tile(np.array([3]), (mem.shape[0], 1))
    want = 1.0 / (1.0 + (S - 1) * np.exp(-5.0))
    np.testing.assert_allclose(ora.true_mass(Q, K, idx, mem, 1.0), want, rtol=1e-12)


def test_predicted_mass_equals_true_mass_with_identity_predictor():
    """With r = d and W_lr^Q = W_lr^K = I the predictor's logits are the true
    ones, so the per-query predicted mass is the true mass (a separate
    function that works on Q K^T directly)."""
    rng = np.random.default_rng(5)
    T, Y, X, d = 2, 4, 4, 8
    S = T * Y * X
    mem = ora.group_members(T, Y, X, 1, 2, 2)
    Q, K = rng.standard_normal((S, d)), rng.standard_normal((S, d))
    idx = np.stack([np.sort(rng.choice(S, 5, replace=False)) for _ in range(mem.shape[0])])
    eye = np.eye(d)
    np.testing.assert_allclose(ora.predicted_mass(Q, K, eye, eye, idx, mem, 0.3), ora.true_mass(Q, K, idx, mem, 0.3),
                               rtol=0, atol=1e-13)


def test_predicted_mass_closed_forms():
    """All keys selected gives 1; W_lr^Q = 0 makes every logit 0, so each key
    carries 1/S and k selected keys carry k/S; one key whose predicted logit
    is L above all others (which are equal) carries 1/(1 + (S-1) e^-L)."""
    rng = np.random.default_rng(6)
    T, Y, X, d, r = 1, 4, 8, 8, 4
    S = T * Y * X
    mem = ora.group_members(T, Y, X, 1, 2, 2)
    Q, K = rng.standard_normal((S, d)), rng.standard_normal((S, d))
    Wq, Wk = rng.standard_normal((d, r)), rng.standard_normal((d, r))
    everything = np.tile(np.arange(S), (mem.shape[0], 1))
    np.testing.assert_allclose(ora.predicted_mass(Q, K, Wq, Wk, everything, mem, 0.5), 1.0, rtol=0, atol=1e-12)
    k = 7
    some = np.stack([np.sort(rng.choice(S, k, replace=False)) for _ in range(mem.shape[0])])
    np.testing.assert_allclose(ora.predicted_mass(Q, K, np.zeros((d, r)), Wk, some, mem, 0.5), k / S, rtol=0,
                               atol=1e-12)
    # q_lr = e_0 for every query, k_lr,j = 0 except k_lr,3 = L e_0 (scale 1)
    L = 4.0
    Q1 = np.zeros((S, d)); Q1[:, 0] = 1.0
    K1 = np.zeros((S, d)); K1[3, 0] = L
    W = np.zeros((d, r)); W[0, 0] = 1.0
    idx = np.tile(np.array([3]), (mem.shape[0], 1))
    np.testing.assert_allclose(ora.predicted_mass(Q1, K1, W, W, idx, mem, 1.0), 1.0 / (1.0 + (S - 1) * np.exp(-L)),
                               rtol=1e-12)


# ------------------------------------------------- head-wise CP re-balancing
def test_plan_gpus_hand_example():
    """Costs 9, 8, 7, 5, 3, 1 on 3 GPUs: 9 -> 0, 8 -> 1, 7 -> 2, 5 -> 2 (7 is
    least), 3 -> 1 (8 < 9 < 12), 1 -> 0 (9 < 11 < 12); loads 10, 11, 12."""
    gpu_of, load = ora.plan_gpus([5, 9, 3, 7, 1, 8], 3)
    assert gpu_of == [2, 0, 1, 2, 0, 1] and load == [10, 11, 12]


def test_best_makespan_hand_examples():
    """Optima worked out by hand. [3, 3, 2, 2, 2] on 2 GPUs: the total is 12,
    so 6 is a lower bound, reached by {3, 3} | {2, 2, 2} (longest processing
    time first only reaches 7). [5, 4, 3, 3, 3]: {5, 4} | {3, 3, 3} = 9 = 18/2.
    [10, 1, 1, 1]: alone, 10 is the largest cost and {10} | {1, 1, 1} reaches
    it; with at most two heads per GPU the best is {10, 1} | {1, 1} = 11."""
    assert ora.best_makespan([3, 3, 2, 2, 2], 2, False) == 6
    assert ora.best_makespan([3, 3, 2, 2, 2], 2, True) == 6
    assert max(ora.plan_gpus([3, 3, 2, 2, 2], 2, False)[1]) == 7
    assert ora.best_makespan([5, 4, 3, 3, 3], 2, True) == 9
    assert ora.best_makespan([10, 1, 1, 1], 2, False) == 10
    assert ora.best_makespan([10, 1, 1, 1], 2, True) == 11
    assert ora.best_makespan([7], 3, True) == 7


def test_plan_gpus_within_graham_bound_of_brute_force():
    """Longest-processing-time first is within (4/3 - 1/(3N)) of the best
    makespan (Graham 1969); with equal head counts the result is still a valid
    split and never better than the constrained optimum."""
    rng = np.random.default_rng(11)
    for _ in range(60):
        n, N = int(rng.integers(1, 8)), int(rng.integers(1, 4))
        cost = [int(c) for c in rng.integers(0, 50, n)]
        for eq in (False, True):
            gpu_of, load = ora.plan_gpus(cost, N, eq)
            assert len(gpu_of) == n and all(0 <= g < N for g in gpu_of)
            assert [sum(c for c, g in zip(cost, gpu_of) if g == q) for q in range(N)] == load
            if eq:
                assert max(gpu_of.count(q) for q in range(N)) <= -(-n // N)
            best = ora.best_makespan(cost, N, eq)
            assert max(load) >= best
            if not eq:
                assert max(load) <= (4 / 3 - 1 / (3 * N)) * best + 1e-9


def test_plan_gpus_special_cases():
    # equal costs spread evenly; fewer heads than GPUs: one head each
    gpu_of, load = ora.plan_gpus([4] * 8, 4)
    assert load == [8, 8, 8, 8] and sorted(gpu_of) == [0, 0, 1, 1, 2, 2, 3, 3]
    gpu_of, load = ora.plan_gpus([3, 1], 4)
    assert gpu_of == [0, 1] and load == [3, 1, 0, 0]
