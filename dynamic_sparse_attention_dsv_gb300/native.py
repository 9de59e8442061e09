"""ctypes binding of libdsv (include/libdsv.h): same names, argument marshalling only.

Every computation runs in the CUDA kernels of libdsv.so. Tensors are passed as
raw device pointers, the stream as the current torch CUDA stream. There is no
fallback: if libdsv.so is missing, importing the loader raises.
"""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libdsv.so")

DSV_STATUS = {0: "DSV_OK", 1: "DSV_ERR_INVALID_ARG", 2: "DSV_ERR_UNSUPPORTED", 3: "DSV_ERR_WORKSPACE",
              4: "DSV_ERR_CUDA", 5: "DSV_ERR_TIMEOUT", 6: "DSV_ERR_OVERFLOW", 7: "DSV_ERR_CANDIDATES"}


class DsvError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {DSV_STATUS.get(code, code)}")


class dsv_shape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int64), ("H", ctypes.c_int64), ("T", ctypes.c_int64), ("Y", ctypes.c_int64),
                ("X", ctypes.c_int64), ("d", ctypes.c_int64)]


class dsv_group(ctypes.Structure):
    _fields_ = [("gt", ctypes.c_int32), ("gy", ctypes.c_int32), ("gx", ctypes.c_int32)]


_P = ctypes.c_void_p
_I32P = ctypes.POINTER(ctypes.c_int32)
_I64P = ctypes.POINTER(ctypes.c_int64)
_F32P = ctypes.POINTER(ctypes.c_float)
_U8P = ctypes.POINTER(ctypes.c_uint8)

#: (name, restype, argtypes) of every entry point declared in include/libdsv.h
SIGNATURES = [
    ("dsv_status_string", ctypes.c_char_p, [ctypes.c_int]),
    ("dsv_read_status", ctypes.c_int, [_P, _I32P, _P]),
    ("dsv_set_wait_limit_ns", ctypes.c_uint64, [ctypes.c_uint64]),
    ("dsv_lowrank_topk_workspace_size", ctypes.c_size_t, [dsv_shape, ctypes.c_int32, dsv_group]),
    ("dsv_lowrank_topk", ctypes.c_int, [_P, _P, _P, _P, dsv_shape, ctypes.c_int32, dsv_group, _I32P, _I64P, _P, _P,
                                        ctypes.c_size_t, _P, _P]),
    ("dsv_lowrank_topk_noalloc", ctypes.c_int, [_P, _P, _P, _P, dsv_shape, ctypes.c_int32, dsv_group, _I32P, _I64P,
                                                _P, _P, _P]),
    ("dsv_coverage_workspace_size", ctypes.c_size_t, [dsv_shape, ctypes.c_int32, dsv_group]),
    ("dsv_predicted_mass_workspace_size", ctypes.c_size_t, [dsv_shape, ctypes.c_int32, dsv_group]),
    ("dsv_predicted_mass", ctypes.c_int, [_P, _P, _P, _P, dsv_shape, ctypes.c_int32, dsv_group, _P, _I32P, _I64P,
                                          ctypes.c_float, _P, _P, _P, ctypes.c_size_t, _P, _P]),
    ("dsv_coverage", ctypes.c_int, [_P, _P, _P, _P, dsv_shape, ctypes.c_int32, dsv_group, ctypes.c_float,
                                    ctypes.c_float, _P, _P, ctypes.c_int32, _P, ctypes.c_size_t, _P, _P]),
    ("dsv_coverage_topk_workspace_size", ctypes.c_size_t, [dsv_shape, ctypes.c_int32, dsv_group]),
    ("dsv_coverage_topk", ctypes.c_int, [_P, _P, _P, _P, dsv_shape, ctypes.c_int32, dsv_group, ctypes.c_float,
                                         ctypes.c_float, _P, _P, ctypes.c_int32, _I32P, _I64P, _P, _P,
                                         ctypes.c_size_t, _P, _P]),
    ("dsv_plan_heads", ctypes.c_int, [_I32P, ctypes.c_int32, ctypes.c_int64, ctypes.c_int64, ctypes.c_double,
                                      ctypes.c_double, ctypes.c_double, _I32P, _U8P, _I64P, _I64P]),
    ("dsv_plan_gpus", ctypes.c_int, [_I64P, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, _I32P, _I64P]),
    ("dsv_sparse_attn_fwd_workspace_size", ctypes.c_size_t, [dsv_shape, dsv_group]),
    ("dsv_sparse_attn_fwd", ctypes.c_int, [_P, _P, _P, _P, _I32P, _I64P, dsv_shape, dsv_group, ctypes.c_float, _P,
                                           _P, _P, ctypes.c_size_t, _P, _P]),
    ("dsv_attn_mass", ctypes.c_int, [_P, _P, ctypes.c_int64, ctypes.c_int32, _P, _P, _P]),
    ("dsv_sparse_attn_bwd_workspace_size", ctypes.c_size_t, [dsv_shape, dsv_group, _I32P, _I64P]),
    ("dsv_sparse_attn_bwd_min_workspace_size", ctypes.c_size_t, [dsv_shape, dsv_group, _I32P, _I64P]),
    ("dsv_sparse_attn_bwd", ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _I32P, _I64P, dsv_shape, dsv_group,
                                           ctypes.c_float, _P, _P, _P, _P, ctypes.c_size_t, _P, _P]),
]

_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Loads libdsv.so (once) and declares every signature. Raises if missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libdsv.so not built ({path}); run `python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(path)
    for name, res, args in SIGNATURES:
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def check(code: int, where: str) -> None:
    if code != 0:
        raise DsvError(code, where)
