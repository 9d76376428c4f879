"""ctypes view of libsparse_mla.so (the C ABI declared in include/sparse_mla.h)."""
from __future__ import annotations

import ctypes as C
import os

from . import build as _build

_LIB = None


class SmlaDims(C.Structure):
    _fields_ = [("batch", C.c_int32), ("num_heads", C.c_int32), ("topk", C.c_int32),
                ("page_size", C.c_int32), ("max_pages_per_seq", C.c_int32), ("d_latent", C.c_int32),
                ("d_rope", C.c_int32), ("nsplit", C.c_int32), ("num_pages", C.c_int64),
                ("heads_per_cta", C.c_int32), ("queries_per_request", C.c_int32), ("merge", C.c_int32)]


class SmlaAppendDims(C.Structure):
    _fields_ = [("tokens", C.c_int32), ("num_requests", C.c_int32), ("page_size", C.c_int32),
                ("max_pages_per_seq", C.c_int32), ("d_latent", C.c_int32), ("d_rope", C.c_int32),
                ("num_pages", C.c_int64)]


class SmlaTopkDims(C.Structure):
    _fields_ = [("batch", C.c_int32), ("num_cols", C.c_int32), ("row_stride", C.c_int64), ("k", C.c_int32),
                ("cluster_ctas", C.c_int32)]


class SmlaPlan(C.Structure):
    _fields_ = [("nsplit", C.c_int32), ("tokens_per_split", C.c_int32), ("head_groups", C.c_int32),
                ("ctas", C.c_int32), ("ctas_per_sm", C.c_int32), ("sm_count", C.c_int32),
                ("waves", C.c_double), ("est_us", C.c_double), ("workspace_bytes", C.c_size_t),
                ("heads_per_cta", C.c_int32), ("fused", C.c_int32)]


_P = C.c_void_p
_SIGS = {
    "sparse_mla_plan_for": (C.c_int, [C.POINTER(SmlaDims), C.c_int32, C.POINTER(SmlaPlan)]),
    "sparse_mla_plan": (C.c_int, [C.POINTER(SmlaDims), C.c_int32, C.POINTER(SmlaPlan)]),
    "sparse_mla_workspace_size": (C.c_size_t, [C.POINTER(SmlaDims), C.c_int32]),
    "sparse_mla_kv_append": (C.c_int, [C.POINTER(SmlaAppendDims), _P, _P, _P, _P, _P, _P, _P, _P]),
    "sparse_mla_topk_select": (C.c_int, [C.POINTER(SmlaTopkDims), _P, _P, _P, _P, _P]),
    "sparse_mla_topk_plan_for": (C.c_int, [C.POINTER(SmlaTopkDims), C.c_int32, C.POINTER(C.c_int32),
                                         C.POINTER(C.c_int32)]),
    "sparse_mla_decode": (C.c_int, [C.POINTER(SmlaDims), _P, _P, _P, _P, _P, C.c_float, _P, _P, _P,
                                    C.c_size_t, _P]),
    "sparse_mla_split": (C.c_int, [C.POINTER(SmlaDims), C.c_int32, _P, _P, _P, _P, _P, C.c_float, _P, _P,
                                   _P, _P]),
    "sparse_mla_combine": (C.c_int, [C.c_int32, C.c_int32, C.c_int32, _P, _P, _P, _P, _P]),
    "sparse_mla_gather_rows": (C.c_int, [C.POINTER(SmlaDims), _P, _P, _P, _P, _P]),
    "sparse_mla_clear_errors": (C.c_int, [_P, _P]),
    "sparse_mla_read_errors": (C.c_int, [_P, C.POINTER(C.c_uint32), _P]),
    "sparse_mla_status_string": (C.c_char_p, [C.c_int]),
    "sparse_mla_decode_noalloc": (C.c_int, [C.POINTER(SmlaDims), _P, _P, _P, _P, _P, C.c_float, _P, _P, _P]),
    "sparse_mla_noalloc_read_errors": (C.c_int, [C.POINTER(C.c_uint32), _P]),
    "sparse_mla_decode_rows": (C.c_int, [C.POINTER(SmlaDims), _P, _P, _P, _P, _P, C.c_float, _P, _P, _P,
                                         C.c_size_t, _P, _P]),
    "sparse_mla_debug_set_wait_limit": (C.c_int, [C.c_uint64]),
}

STATUS = {0: "SMLA_OK", 1: "SMLA_ERR_INVALID_ARG", 2: "SMLA_ERR_UNSUPPORTED", 3: "SMLA_ERR_WORKSPACE",
          4: "SMLA_ERR_CUDA"}
DEVERR_PAGE_RANGE, DEVERR_TIMEOUT, DEVERR_RANGE = 0x1, 0x2, 0x4


def lib_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """Load the native library, building it in-tree first when it is missing or stale.

    Raises if it cannot be built: there is no fallback path.
    """
    global _LIB
    if _LIB is not None:
        return _LIB
    if build_if_missing and not _build.up_to_date():
        _build.build()
    if not os.path.exists(lib_path()):
        raise FileNotFoundError(f"{lib_path()} is missing; run sparse_mla_decode_paged_gb300.build.build()")
    lib = C.CDLL(lib_path())
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _LIB = lib
    return lib


class SmlaError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} returned {STATUS.get(status, status)}")
        self.status = status


def check(fn: str, status: int) -> None:
    if status != 0:
        raise SmlaError(fn, status)
