"""Torch-facing wrappers of the libdsv C ABI (argument marshalling only).

Tensors: Q, K, V, O, dO, dQ, dK, dV are CUDA bf16 [B, H, S, d] (or [H, S, d]
for B = 1), contiguous; W_lr^Q, W_lr^K are bf16 [H, d, r]. ``grid`` is the
latent grid (T, Y, X) with S = T*Y*X, ``group`` the query-group cube
(gt, gy, gx). Outputs and workspaces are allocated here with torch; every
arithmetic step runs in libdsv's CUDA kernels on the current stream.
"""
from __future__ import annotations

import ctypes
import math
from typing import Optional, Sequence, Union

import torch

from . import native as N


def _ptr(t: Optional[torch.Tensor]):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _dims(x: torch.Tensor):
    if x.dim() == 3:
        return 1, x.shape[0], x.shape[1], x.shape[2]
    if x.dim() == 4:
        return tuple(x.shape)
    raise ValueError("expected [B, H, S, d] or [H, S, d]")


def _check_bf16(*ts):
    for t in ts:
        if t is None:
            continue
        if not t.is_cuda or t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError("expected contiguous CUDA bf16 tensors")


def make_shape(x: torch.Tensor, grid: Sequence[int]) -> N.dsv_shape:
    B, H, S, d = _dims(x)
    T, Y, X = grid
    if T * Y * X != S:
        raise ValueError(f"grid {tuple(grid)} does not match S={S}")
    return N.dsv_shape(B, H, T, Y, X, d)


def make_group(group: Sequence[int]) -> N.dsv_group:
    return N.dsv_group(*[int(v) for v in group])


def _i32(vals):
    return (ctypes.c_int32 * len(vals))(*[int(v) for v in vals])


def _i64(vals):
    return (ctypes.c_int64 * len(vals))(*[int(v) for v in vals])


def set_wait_limit_ns(ns: int) -> int:
    """dsv_set_wait_limit_ns: the limit (ns) of every pipeline wait inside the
    kernels launched from now on, for this process; returns the previous one."""
    return int(N.load().dsv_set_wait_limit_ns(int(ns)))


def new_status(device=None) -> torch.Tensor:
    """A zeroed device status word (int32) for one or more calls."""
    return torch.zeros(1, dtype=torch.int32, device=device or "cuda")


def read_status(status: torch.Tensor) -> int:
    lib = N.load()
    out = ctypes.c_int32(0)
    N.check(lib.dsv_read_status(_ptr(status), ctypes.byref(out), _stream()), "dsv_read_status")
    return int(out.value)


def check_status(status: torch.Tensor, where: str = "libdsv") -> None:
    code = read_status(status)
    if code != 0:
        raise N.DsvError(code, where + " (device)")


def _workspace(nbytes: int, device, workspace: Optional[torch.Tensor], any_size: bool = False) -> torch.Tensor:
    """The caller's workspace (uint8) or a new one of nbytes. With any_size the
    library itself decides whether a smaller workspace is enough."""
    if workspace is not None:
        if workspace.dtype != torch.uint8 or workspace.device != torch.device(device):
            raise ValueError("workspace must be a uint8 tensor on the call's device")
        if not any_size and workspace.numel() < nbytes:
            raise ValueError("workspace too small")
        return workspace
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


def topk_layout(P: int, n_groups: int, k: Union[int, Sequence[int]], skip: Optional[Sequence[bool]] = None):
    """Packed index layout: per-problem k, offsets (-1 = skipped) and total."""
    ks = [int(k)] * P if isinstance(k, int) else [int(v) for v in k]
    offs, total = [], 0
    for p in range(P):
        if skip is not None and skip[p]:
            offs.append(-1)
        else:
            offs.append(total)
            total += n_groups * ks[p]
    return ks, offs, total


# ------------------------------------------------------------------- calls
def lowrank_topk_workspace_size(x, grid, group, r) -> int:
    return int(N.load().dsv_lowrank_topk_workspace_size(make_shape(x, grid), int(r), make_group(group)))


def lowrank_topk(Q, K, Wq, Wk, grid, group, k, idx_offset: Optional[Sequence[int]] = None,
                 idx: Optional[torch.Tensor] = None, workspace=None, status=None):
    """dsv_lowrank_topk. Returns (idx int32 flat tensor, k list, offset list)."""
    _check_bf16(Q, K, Wq, Wk)
    lib = N.load()
    shape, grp = make_shape(Q, grid), make_group(group)
    P = shape.B * shape.H
    n_groups = (shape.T * shape.Y * shape.X) // (grp.gt * grp.gy * grp.gx)
    ks, offs, total = topk_layout(P, n_groups, k)
    if idx_offset is not None:
        offs = [int(v) for v in idx_offset]
        total = max([o + n_groups * kk for o, kk in zip(offs, ks) if o >= 0] + [0])
    if idx is None:
        idx = torch.empty(max(total, 1), dtype=torch.int32, device=Q.device)
    r = Wq.shape[-1]
    ws = _workspace(int(lib.dsv_lowrank_topk_workspace_size(shape, r, grp)), Q.device, workspace)
    st = status if status is not None else new_status(Q.device)
    code = lib.dsv_lowrank_topk(_ptr(Q), _ptr(K), _ptr(Wq), _ptr(Wk), shape, r, grp, _i32(ks), _i64(offs), _ptr(idx),
                                _ptr(ws), ws.numel(), _ptr(st), _stream())
    N.check(code, "dsv_lowrank_topk")
    return idx, ks, offs


def coverage(Q, K, Wq, Wk, grid, group, scale: Optional[float] = None, mass: float = 0.9, curve_points: int = 0,
             workspace=None, status=None):
    """dsv_coverage. Returns (k_cov int32 device tensor [P], curve or None)."""
    _check_bf16(Q, K, Wq, Wk)
    lib = N.load()
    shape, grp = make_shape(Q, grid), make_group(group)
    P = shape.B * shape.H
    scale = 1.0 / math.sqrt(shape.d) if scale is None else float(scale)
    k_cov = torch.empty(P, dtype=torch.int32, device=Q.device)
    curve = torch.empty((P, curve_points), dtype=torch.float32, device=Q.device) if curve_points else None
    r = Wq.shape[-1]
    ws = _workspace(int(lib.dsv_coverage_workspace_size(shape, r, grp)), Q.device, workspace)
    st = status if status is not None else new_status(Q.device)
    code = lib.dsv_coverage(_ptr(Q), _ptr(K), _ptr(Wq), _ptr(Wk), shape, r, grp, ctypes.c_float(scale),
                            ctypes.c_float(mass), _ptr(k_cov), _ptr(curve), int(curve_points), _ptr(ws), ws.numel(),
                            _ptr(st), _stream())
    N.check(code, "dsv_coverage")
    return k_cov, curve


def coverage_workspace_size(x, grid, group, r) -> int:
    return int(N.load().dsv_coverage_workspace_size(make_shape(x, grid), int(r), make_group(group)))


def coverage_topk_workspace_size(x, grid, group, r) -> int:
    return int(N.load().dsv_coverage_topk_workspace_size(make_shape(x, grid), int(r), make_group(group)))


def coverage_topk(Q, K, Wq, Wk, grid, group, k, scale: Optional[float] = None, mass: float = 0.9,
                  curve_points: int = 0, idx_offset: Optional[Sequence[int]] = None,
                  idx: Optional[torch.Tensor] = None, workspace=None, status=None):
    """dsv_coverage_topk. Returns (k_cov int32 device tensor [P], curve or None,
    idx int32 flat tensor, k list, offset list)."""
    _check_bf16(Q, K, Wq, Wk)
    lib = N.load()
    shape, grp = make_shape(Q, grid), make_group(group)
    P = shape.B * shape.H
    n_groups = (shape.T * shape.Y * shape.X) // (grp.gt * grp.gy * grp.gx)
    scale = 1.0 / math.sqrt(shape.d) if scale is None else float(scale)
    ks, offs, total = topk_layout(P, n_groups, k)
    if idx_offset is not None:
        offs = [int(v) for v in idx_offset]
        total = max([o + n_groups * kk for o, kk in zip(offs, ks) if o >= 0] + [0])
    if idx is None:
        idx = torch.empty(max(total, 1), dtype=torch.int32, device=Q.device)
    k_cov = torch.empty(P, dtype=torch.int32, device=Q.device)
    curve = torch.empty((P, curve_points), dtype=torch.float32, device=Q.device) if curve_points else None
    r = Wq.shape[-1]
    ws = _workspace(int(lib.dsv_coverage_topk_workspace_size(shape, r, grp)), Q.device, workspace)
    st = status if status is not None else new_status(Q.device)
    code = lib.dsv_coverage_topk(_ptr(Q), _ptr(K), _ptr(Wq), _ptr(Wk), shape, r, grp, ctypes.c_float(scale),
                                 ctypes.c_float(mass), _ptr(k_cov), _ptr(curve), int(curve_points), _i32(ks),
                                 _i64(offs), _ptr(idx), _ptr(ws), ws.numel(), _ptr(st), _stream())
    N.check(code, "dsv_coverage_topk")
    return k_cov, curve, idx, ks, offs


def plan_heads(k_cov: Sequence[int], S: int, n_groups: int, lo_frac: float = 0.01, hi_frac: float = 0.25,
               dense_frac: float = 0.5):
    """dsv_plan_heads (host only). Returns (k_h list, dense list, offsets list, total)."""
    lib = N.load()
    n = len(k_cov)
    kc = _i32(k_cov)
    k_h = (ctypes.c_int32 * n)()
    dense = (ctypes.c_uint8 * n)()
    offs = (ctypes.c_int64 * n)()
    total = ctypes.c_int64(0)
    code = lib.dsv_plan_heads(kc, n, int(S), int(n_groups), lo_frac, hi_frac, dense_frac, k_h, dense, offs,
                              ctypes.byref(total))
    N.check(code, "dsv_plan_heads")
    return list(k_h), [bool(v) for v in dense], list(offs), int(total.value)


def plan_gpus(cost: Sequence[int], n_gpus: int, equal_counts: bool = True):
    """dsv_plan_gpus (host only): heads to GPUs by cost, longest first.
    Returns (gpu_of list, load per GPU list)."""
    n = len(cost)
    gpu_of = (ctypes.c_int32 * n)()
    load = (ctypes.c_int64 * n_gpus)()
    code = N.load().dsv_plan_gpus(_i64(cost), n, int(n_gpus), 1 if equal_counts else 0, gpu_of, load)
    N.check(code, "dsv_plan_gpus")
    return list(gpu_of), list(load)


def sparse_attn_fwd(Q, K, V, idx, k_per_head, idx_offset, grid, group, scale: Optional[float] = None, O=None,
                    LSE=None, status=None):
    """dsv_sparse_attn_fwd. idx=None runs every problem dense. Returns (O, LSE)."""
    _check_bf16(Q, K, V, O)
    lib = N.load()
    shape, grp = make_shape(Q, grid), make_group(group)
    scale = 1.0 / math.sqrt(shape.d) if scale is None else float(scale)
    O = torch.empty_like(Q) if O is None else O
    if LSE is None:
        LSE = torch.empty(Q.shape[:-1], dtype=torch.float32, device=Q.device)
    st = status if status is not None else new_status(Q.device)
    kp = _i32(k_per_head) if idx is not None else None
    op = _i64(idx_offset) if idx is not None else None
    code = lib.dsv_sparse_attn_fwd(_ptr(Q), _ptr(K), _ptr(V), _ptr(idx), kp, op, shape, grp, ctypes.c_float(scale),
                                   _ptr(O), _ptr(LSE), None, 0, _ptr(st), _stream())
    N.check(code, "dsv_sparse_attn_fwd")
    return O, LSE


def sparse_attn_bwd_workspace_size(x, grid, group, k_per_head=None, idx_offset=None) -> int:
    kp = _i32(k_per_head) if k_per_head is not None else None
    op = _i64(idx_offset) if k_per_head is not None else None
    return int(N.load().dsv_sparse_attn_bwd_workspace_size(make_shape(x, grid), make_group(group), kp, op))


def attn_mass(LSE_sel, LSE_all, per_query: bool = False):
    """dsv_attn_mass: the share of each query's true attention mass that its
    selected keys carry, from the forward's LSE on the index sets and dense.
    Returns (mean per problem, shape LSE.shape[:-1]; per-query shares or None)."""
    if LSE_sel.dtype != torch.float32 or LSE_all.dtype != torch.float32 or LSE_sel.shape != LSE_all.shape:
        raise TypeError("LSE_sel and LSE_all must be float32 tensors of one shape")
    if not (LSE_sel.is_contiguous() and LSE_all.is_contiguous()):
        raise ValueError("LSE tensors must be contiguous")
    S = LSE_sel.shape[-1]
    P = LSE_sel.numel() // S
    mass = torch.empty(LSE_sel.shape[:-1], dtype=torch.float32, device=LSE_sel.device)
    pq = torch.empty_like(LSE_sel) if per_query else None
    code = N.load().dsv_attn_mass(_ptr(LSE_sel), _ptr(LSE_all), int(S), int(P), _ptr(mass), _ptr(pq), _stream())
    N.check(code, "dsv_attn_mass")
    return mass, pq


def predicted_mass(Q, K, Wq, Wk, grid, group, idx=None, k_per_head=None, idx_offset=None,
                   scale: Optional[float] = None, per_query: bool = False, workspace=None, status=None):
    """dsv_predicted_mass: the share of each query's own predicted softmax
    mass that its group's selected keys carry. idx=None: every key.
    Returns (mean per problem float32 [P], per-query shares [P, S] or None)."""
    _check_bf16(Q, K, Wq, Wk)
    lib = N.load()
    shape, grp = make_shape(Q, grid), make_group(group)
    P, S = shape.B * shape.H, shape.T * shape.Y * shape.X
    scale = 1.0 / math.sqrt(shape.d) if scale is None else float(scale)
    r = Wq.shape[-1]
    mass = torch.empty(P, dtype=torch.float32, device=Q.device)
    pq = torch.empty((P, S), dtype=torch.float32, device=Q.device) if per_query else None
    ws = _workspace(int(lib.dsv_predicted_mass_workspace_size(shape, r, grp)), Q.device, workspace)
    st = status if status is not None else new_status(Q.device)
    kp = _i32(k_per_head) if idx is not None else None
    op = _i64(idx_offset) if idx is not None else None
    code = lib.dsv_predicted_mass(_ptr(Q), _ptr(K), _ptr(Wq), _ptr(Wk), shape, r, grp, _ptr(idx), kp, op,
                                  ctypes.c_float(scale), _ptr(mass), _ptr(pq), _ptr(ws), ws.numel(), _ptr(st),
                                  _stream())
    N.check(code, "dsv_predicted_mass")
    return mass, pq


def sparse_attn_bwd_min_workspace_size(x, grid, group, k_per_head=None, idx_offset=None) -> int:
    kp = _i32(k_per_head) if k_per_head is not None else None
    op = _i64(idx_offset) if idx_offset is not None else None
    return int(N.load().dsv_sparse_attn_bwd_min_workspace_size(make_shape(x, grid), make_group(group), kp, op))


def sparse_attn_bwd(Q, K, V, O, LSE, dO, idx, k_per_head, idx_offset, grid, group, scale: Optional[float] = None,
                    dQ=None, dK=None, dV=None, workspace=None, status=None):
    """dsv_sparse_attn_bwd. Returns (dQ, dK, dV). A workspace smaller than
    dsv_sparse_attn_bwd_workspace_size() is accepted down to the library's
    minimum (more, smaller launches; the same result bits)."""
    _check_bf16(Q, K, V, O, dO)
    lib = N.load()
    shape, grp = make_shape(Q, grid), make_group(group)
    scale = 1.0 / math.sqrt(shape.d) if scale is None else float(scale)
    dQ = torch.empty_like(Q) if dQ is None else dQ
    dK = torch.empty_like(K) if dK is None else dK
    dV = torch.empty_like(V) if dV is None else dV
    kp = _i32(k_per_head) if idx is not None else None
    op = _i64(idx_offset) if idx is not None else None
    ws = _workspace(int(lib.dsv_sparse_attn_bwd_workspace_size(shape, grp, kp, op)), Q.device, workspace,
                    any_size=True)
    st = status if status is not None else new_status(Q.device)
    code = lib.dsv_sparse_attn_bwd(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(LSE), _ptr(dO), _ptr(idx), kp, op, shape,
                                   grp, ctypes.c_float(scale), _ptr(dQ), _ptr(dK), _ptr(dV), _ptr(ws), ws.numel(),
                                   _ptr(st), _stream())
    N.check(code, "dsv_sparse_attn_bwd")
    return dQ, dK, dV
