"""libdsv: the DSV hot path (low-rank critical-KV selection + query-grouped
sparse attention) as sm_103a CUDA kernels behind a C ABI (include/libdsv.h).

The Python functions below only marshal arguments into libdsv.so; every step
of the computation runs in its CUDA kernels.
"""
from .api import (attn_mass, check_status, coverage, coverage_topk, coverage_topk_workspace_size,
                  coverage_workspace_size, lowrank_topk,
                  lowrank_topk_workspace_size, new_status, plan_gpus, plan_heads, predicted_mass, read_status, set_wait_limit_ns, sparse_attn_bwd,
                  sparse_attn_bwd_min_workspace_size, sparse_attn_bwd_workspace_size, sparse_attn_fwd, topk_layout)
from .native import DsvError

__all__ = ["attn_mass", "check_status", "coverage", "coverage_topk", "coverage_topk_workspace_size",
           "coverage_workspace_size", "lowrank_topk",
           "lowrank_topk_workspace_size", "new_status", "plan_gpus", "plan_heads", "predicted_mass", "read_status", "set_wait_limit_ns", "sparse_attn_bwd",
           "sparse_attn_bwd_min_workspace_size", "sparse_attn_bwd_workspace_size", "sparse_attn_fwd", "topk_layout",
           "DsvError"]
