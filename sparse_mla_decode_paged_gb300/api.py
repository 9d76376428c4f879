"""Thin PyTorch binding of the C ABI: argument marshalling only.

Every step of the decode runs in the CUDA library; torch provides device
memory and the current stream.  Names follow include/sparse_mla.h.
"""
from __future__ import annotations

import ctypes as C
from typing import Optional, Tuple

import torch

from . import _native
from ._native import SmlaAppendDims, SmlaDims, SmlaPlan, SmlaTopkDims, check

PAGE_SIZE, D_LATENT, D_ROPE, D_QK = 64, 512, 64, 576


def _lib():
    return _native.load()


def _ptr(t: Optional[torch.Tensor]):
    """Device address for a void* argument (the library's argument types convert a plain int)."""
    return t.data_ptr() if t is not None else None


def _stream(stream=None):
    return (stream if stream is not None else torch.cuda.current_stream()).cuda_stream


def _need(t: torch.Tensor, name: str, dtype, ndim: int):
    # the common case in one expression; the checks below only name what is wrong
    if type(t) is torch.Tensor and t.is_cuda and t.dtype is dtype and t.dim() == ndim and t.is_contiguous():
        return
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous {ndim}-d tensor")


MERGE_AUTO, MERGE_KERNEL, MERGE_FUSED = 0, 1, 2


def make_dims(B: int, H: int, topk: int, max_pages_per_seq: int, num_pages: int, nsplit: int = 0,
              heads_per_cta: int = 0, queries_per_request: int = 1, merge: int = MERGE_AUTO) -> SmlaDims:
    return SmlaDims(B, H, topk, PAGE_SIZE, max_pages_per_seq, D_LATENT, D_ROPE, nsplit, num_pages, heads_per_cta,
                    queries_per_request, merge)


def dims_of(q, kv_cache, block_table, topk_idx, nsplit: int = 0, heads_per_cta: int = 0,
            merge: int = MERGE_AUTO) -> SmlaDims:
    """Shapes of a call; several queries per request when q has a multiple of block_table's rows."""
    return make_dims(q.shape[0], q.shape[1], topk_idx.shape[1], block_table.shape[1], kv_cache.shape[0], nsplit,
                     heads_per_cta, q.shape[0] // block_table.shape[0], merge)


# Decode dims by call shape and device, with the split count the library's scheduler chose filled in: a
# call with the same shapes as an earlier one reuses them (the library reads dims, never writes them).
_DECODE_DIMS = {}


def _decode_dims(q, kv_cache, block_table, topk_idx, nsplit: int, heads_per_cta: int, merge: int) -> SmlaDims:
    key = (q.shape, kv_cache.shape[0], block_table.shape, topk_idx.shape[1], nsplit, heads_per_cta, merge,
           q.device.index)
    d = _DECODE_DIMS.get(key)
    if d is None:
        d = dims_of(q, kv_cache, block_table, topk_idx, nsplit, heads_per_cta, merge)
        if nsplit == 0:
            d.nsplit = plan(d, q.device.index).nsplit
        if len(_DECODE_DIMS) > 256:
            _DECODE_DIMS.clear()
        _DECODE_DIMS[key] = d
    return d


def plan_for(dims: SmlaDims, sm_count: int) -> SmlaPlan:
    p = SmlaPlan()
    check("sparse_mla_plan_for", _lib().sparse_mla_plan_for(C.byref(dims), sm_count, C.byref(p)))
    return p


def plan(dims: SmlaDims, device: Optional[int] = None) -> SmlaPlan:
    p = SmlaPlan()
    dev = torch.cuda.current_device() if device is None else device
    check("sparse_mla_plan", _lib().sparse_mla_plan(C.byref(dims), dev, C.byref(p)))
    return p


def workspace_size(dims: SmlaDims, nsplit: int) -> int:
    return int(_lib().sparse_mla_workspace_size(C.byref(dims), nsplit))


def alloc_workspace(dims: SmlaDims, nsplit: int, device=None) -> torch.Tensor:
    """Caller-owned workspace (zeroed, so the device error word starts clear)."""
    n = workspace_size(dims, nsplit)
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")


def _check_inputs(q, kv_cache, block_table, topk_idx, seq_lens):
    _need(q, "q", torch.bfloat16, 3)
    _need(kv_cache, "kv_cache", torch.uint8, 3)
    _need(block_table, "block_table", torch.int32, 2)
    _need(topk_idx, "topk_idx", torch.int32, 2)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    if q.shape[2] != D_QK or kv_cache.shape[1] != PAGE_SIZE or kv_cache.shape[2] != 656:
        raise ValueError("q must be [B,H,576] and kv_cache [pages,64,656]")
    B = q.shape[0]
    R = block_table.shape[0]
    if R < 1 or B % R != 0 or topk_idx.shape[0] != B or seq_lens.shape[0] != B:
        raise ValueError("q, topk_idx and seq_lens need one row per query, block_table one row per request "
                         "(a divisor of the query count)")


def sparse_mla_decode(q: torch.Tensor, kv_cache: torch.Tensor, block_table: torch.Tensor, topk_idx: torch.Tensor,
                      seq_lens: torch.Tensor, sm_scale: float, out: Optional[torch.Tensor] = None,
                      lse: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                      nsplit: int = 0, stream=None, heads_per_cta: int = 0,
                      merge: int = MERGE_AUTO) -> Tuple[torch.Tensor, torch.Tensor]:
    """out bf16 [B,H,512], lse fp32 [B,H].  nsplit = 0, heads_per_cta = 0 and merge = MERGE_AUTO let the
    library's scheduler choose."""
    _check_inputs(q, kv_cache, block_table, topk_idx, seq_lens)
    dims = _decode_dims(q, kv_cache, block_table, topk_idx, nsplit, heads_per_cta, merge)
    if out is None:
        out = torch.empty((q.shape[0], q.shape[1], D_LATENT), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((q.shape[0], q.shape[1]), dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = alloc_workspace(dims, dims.nsplit, q.device)
    st = _lib().sparse_mla_decode(
        dims, q.data_ptr(), kv_cache.data_ptr(), block_table.data_ptr(), topk_idx.data_ptr(), seq_lens.data_ptr(),
        sm_scale, out.data_ptr(), lse.data_ptr(), workspace.data_ptr(), workspace.numel(), _stream(stream))
    if st != 0:
        check("sparse_mla_decode", st)
    return out, lse


def sparse_mla_decode_rows(q: torch.Tensor, kv_cache: torch.Tensor, block_table: torch.Tensor,
                           topk_idx: torch.Tensor, seq_lens: torch.Tensor, sm_scale: float,
                           workspace: Optional[torch.Tensor] = None, nsplit: int = 0, stream=None,
                           heads_per_cta: int = 0, rows: Optional[torch.Tensor] = None, merge: int = MERGE_AUTO):
    """sparse_mla_decode that also returns the rows the decode's split kernel loaded:
    (out bf16 [B,H,512], lse fp32 [B,H], rows int64 [B,topk], -1 for skipped entries)."""
    _check_inputs(q, kv_cache, block_table, topk_idx, seq_lens)
    B, H = q.shape[0], q.shape[1]
    dims = dims_of(q, kv_cache, block_table, topk_idx, nsplit, heads_per_cta, merge)
    if nsplit == 0:
        nsplit = plan(dims, q.device.index).nsplit
        dims.nsplit = nsplit
    out = torch.empty((B, H, D_LATENT), dtype=torch.bfloat16, device=q.device)
    lse = torch.empty((B, H), dtype=torch.float32, device=q.device)
    if rows is None:
        rows = torch.empty(topk_idx.shape, dtype=torch.int64, device=q.device)
    _need(rows, "rows", torch.int64, 2)
    if workspace is None:
        workspace = alloc_workspace(dims, nsplit, q.device)
    check("sparse_mla_decode_rows", _lib().sparse_mla_decode_rows(
        C.byref(dims), _ptr(q), _ptr(kv_cache), _ptr(block_table), _ptr(topk_idx), _ptr(seq_lens),
        C.c_float(sm_scale), _ptr(out), _ptr(lse), _ptr(workspace), C.c_size_t(workspace.numel()),
        _ptr(rows), _stream(stream)))
    return out, lse, rows


def debug_set_wait_limit(ns: int) -> None:
    """Time limit of the split kernel's pipeline waits for later launches (0 = the default, 1 s)."""
    check("sparse_mla_debug_set_wait_limit", _lib().sparse_mla_debug_set_wait_limit(int(ns)))


def sparse_mla_split(q, kv_cache, block_table, topk_idx, seq_lens, sm_scale: float, nsplit: int,
                     err_word: Optional[torch.Tensor] = None, stream=None, heads_per_cta: int = 0):
    """Partials: o_part fp32 [B,nsplit,H,512], lse_part fp32 [B,nsplit,H]."""
    _check_inputs(q, kv_cache, block_table, topk_idx, seq_lens)
    B, H = q.shape[0], q.shape[1]
    dims = dims_of(q, kv_cache, block_table, topk_idx, nsplit, heads_per_cta)
    o_part = torch.empty((B, nsplit, H, D_LATENT), dtype=torch.float32, device=q.device)
    lse_part = torch.empty((B, nsplit, H), dtype=torch.float32, device=q.device)
    check("sparse_mla_split", _lib().sparse_mla_split(
        C.byref(dims), nsplit, _ptr(q), _ptr(kv_cache), _ptr(block_table), _ptr(topk_idx), _ptr(seq_lens),
        C.c_float(sm_scale), _ptr(o_part), _ptr(lse_part), _ptr(err_word), _stream(stream)))
    return o_part, lse_part


def sparse_mla_kv_append(latent: torch.Tensor, rope: torch.Tensor, block_table: torch.Tensor,
                         positions: torch.Tensor, kv_cache: torch.Tensor, requests: Optional[torch.Tensor] = None,
                         err_word: Optional[torch.Tensor] = None, stream=None) -> None:
    """Quantise new tokens (latent bf16 [T,512], rope bf16 [T,64]) into the paged FP8 cache at
    (requests[i] or i, positions[i]) through block_table; kv_cache is written in place."""
    _need(latent, "latent", torch.bfloat16, 2)
    _need(rope, "rope", torch.bfloat16, 2)
    _need(block_table, "block_table", torch.int32, 2)
    _need(positions, "positions", torch.int32, 1)
    _need(kv_cache, "kv_cache", torch.uint8, 3)
    T = latent.shape[0]
    if latent.shape[1] != D_LATENT or rope.shape != (T, D_ROPE) or positions.shape[0] != T:
        raise ValueError("latent must be [T,512], rope [T,64], positions [T]")
    if kv_cache.shape[1] != PAGE_SIZE or kv_cache.shape[2] != 656:
        raise ValueError("kv_cache must be [pages,64,656]")
    if requests is not None:
        _need(requests, "requests", torch.int32, 1)
        if requests.shape[0] != T:
            raise ValueError("requests must be [T]")
    dims = SmlaAppendDims(T, block_table.shape[0], PAGE_SIZE, block_table.shape[1], D_LATENT, D_ROPE,
                          kv_cache.shape[0])
    check("sparse_mla_kv_append", _lib().sparse_mla_kv_append(
        C.byref(dims), _ptr(latent), _ptr(rope), _ptr(block_table), _ptr(requests), _ptr(positions),
        _ptr(kv_cache), _ptr(err_word), _stream(stream)))


def sparse_mla_topk_select(scores: torch.Tensor, seq_lens: torch.Tensor, k: int, cluster_ctas: int = 0,
                           err_word: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """int32 [B,k]: per query the k positions below seq_lens[b] of largest score (IEEE totalOrder,
    ties to the lower position), in increasing order, -1 padded when seq_lens[b] <= k.
    scores float32 [B, num_cols] with unit stride along positions."""
    _need(seq_lens, "seq_lens", torch.int32, 1)
    if scores.dtype != torch.float32 or scores.dim() != 2 or not scores.is_cuda:
        raise ValueError("scores must be a float32 [B, num_cols] CUDA tensor")
    if scores.stride(1) != 1 or (scores.shape[0] > 1 and scores.stride(0) < scores.shape[1]):
        raise ValueError("scores rows must be contiguous")
    B, n = scores.shape
    if seq_lens.shape[0] != B:
        raise ValueError("seq_lens must be [B]")
    out = torch.empty((B, k), dtype=torch.int32, device=scores.device)
    dims = SmlaTopkDims(B, n, scores.stride(0) if B > 1 else n, k, cluster_ctas)
    check("sparse_mla_topk_select", _lib().sparse_mla_topk_select(
        C.byref(dims), _ptr(scores), _ptr(seq_lens), _ptr(out), _ptr(err_word), _stream(stream)))
    return out


def sparse_mla_combine(o_part: torch.Tensor, lse_part: torch.Tensor, stream=None):
    _need(o_part, "o_part", torch.float32, 4)
    _need(lse_part, "lse_part", torch.float32, 3)
    B, S, H, D = o_part.shape
    out = torch.empty((B, H, D), dtype=torch.bfloat16, device=o_part.device)
    lse = torch.empty((B, H), dtype=torch.float32, device=o_part.device)
    check("sparse_mla_combine", _lib().sparse_mla_combine(B, H, S, _ptr(o_part), _ptr(lse_part), _ptr(out),
                                                          _ptr(lse), _stream(stream)))
    return out, lse


def sparse_mla_gather_rows(block_table, topk_idx, seq_lens, num_pages: int, stream=None) -> torch.Tensor:
    _need(block_table, "block_table", torch.int32, 2)
    _need(topk_idx, "topk_idx", torch.int32, 2)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    B, K = topk_idx.shape
    if block_table.shape[0] < 1 or B % block_table.shape[0] != 0:
        raise ValueError("block_table needs one row per request (a divisor of the query count)")
    dims = make_dims(B, 64, K, block_table.shape[1], num_pages, queries_per_request=B // block_table.shape[0])
    rows = torch.empty((B, K), dtype=torch.int64, device=topk_idx.device)
    check("sparse_mla_gather_rows", _lib().sparse_mla_gather_rows(
        C.byref(dims), _ptr(block_table), _ptr(topk_idx), _ptr(seq_lens), _ptr(rows), _stream(stream)))
    return rows


def clear_errors(workspace: torch.Tensor, stream=None) -> None:
    check("sparse_mla_clear_errors", _lib().sparse_mla_clear_errors(_ptr(workspace), _stream(stream)))


def read_errors(workspace: torch.Tensor, stream=None) -> int:
    v = C.c_uint32(0)
    check("sparse_mla_read_errors", _lib().sparse_mla_read_errors(_ptr(workspace), C.byref(v), _stream(stream)))
    return int(v.value)
