"""The decode entry point that allocates nothing (static device scratch) against the regular
entry point with a caller workspace, through the C ABI.

It serves callers that cannot allocate device memory (engine-hosted plugins without a workspace,
code running under stream capture, host paths that must not synchronise).  This file is collected
last so that a run stopping at the first failure has already run every other test."""
import ctypes as C

import pytest
import torch

from sparse_mla_decode_paged_gb300 import _native, api
from sparse_mla_decode_paged_gb300 import workloads as wl
from parity_util import LSE_ATOL, OUT_RTOL, compare, oracle_on

pytestmark = pytest.mark.gpu


def _noalloc(lib, w, nsplit, out, lse):
    dims = api.dims_of(w.q, w.kv_cache, w.block_table, w.topk_idx, nsplit)
    return lib.sparse_mla_decode_noalloc(C.byref(dims), api._ptr(w.q), api._ptr(w.kv_cache),
                                         api._ptr(w.block_table), api._ptr(w.topk_idx), api._ptr(w.seq_lens),
                                         C.c_float(w.sm_scale), api._ptr(out), api._ptr(lse), api._stream())


def _close(out_a, lse_a, out_b, lse_b):
    a, b = out_a.float(), out_b.float()
    denom = b.abs().amax(-1).clamp_min(1e-30)
    assert float(((a - b).abs().amax(-1) / denom).max()) <= OUT_RTOL
    fin = torch.isfinite(lse_b)
    assert torch.equal(fin, torch.isfinite(lse_a))
    assert float((lse_a[fin] - lse_b[fin]).abs().max()) <= LSE_ATOL if fin.any() else True


@pytest.mark.parametrize("cfg,nsplit", [("tiny", 0), ("b32_ctx32k", 4), ("b32_ctx32k", 0)])
def test_noalloc_matches_workspace_entry_point_twice(cfg, nsplit):
    lib = _native.load()
    w = wl.make_workload(wl.CONFIGS[cfg], device="cuda")
    ref_out, ref_lse = api.sparse_mla_decode(w.q, w.kv_cache, w.block_table, w.topk_idx, w.seq_lens,
                                             w.sm_scale, nsplit=nsplit)
    for _ in range(2):                      # the scratch keeps the previous call's contents
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        assert _noalloc(lib, w, nsplit, out, lse) == 0
        torch.cuda.synchronize()
        _close(out, lse, ref_out, ref_lse)


def test_noalloc_rejects_shapes_beyond_the_scratch():
    lib = _native.load()
    w = wl.make_custom(B=64, H=128, topk=64, ctx_lens=[64] * 64, seed=3, device="cuda")
    dims = api.dims_of(w.q, w.kv_cache, w.block_table, w.topk_idx, 16)
    assert lib.sparse_mla_workspace_size(C.byref(dims), 16) > (32 << 20)
    out = torch.zeros((64, 128, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((64, 128), dtype=torch.float32, device="cuda")
    assert _noalloc(lib, w, 16, out, lse) == 3          # SMLA_ERR_WORKSPACE, nothing launched
    torch.cuda.synchronize()
    assert torch.all(out == 0)


def _flags(lib):
    v = C.c_uint32(0xFFFFFFFF)
    assert lib.sparse_mla_noalloc_read_errors(C.byref(v), api._stream()) == 0
    return int(v.value)


@pytest.mark.parametrize("nsplit", [1, 3])
def test_noalloc_matches_the_oracle_and_reports_bad_pages(nsplit):
    """Checked against the float64 oracle directly; a block-table entry outside the cache sets the
    page-range flag, which the error getter reads back, and the next clean call clears it."""
    lib = _native.load()
    w = wl.make_custom(B=3, H=64, topk=300, ctx_lens=[2000, 700, 90], seed=81 + nsplit, device="cuda")
    w.block_table[1, 2] = w.num_pages + 11
    out = torch.empty((w.B, w.H, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((w.B, w.H), dtype=torch.float32, device="cuda")
    assert _noalloc(lib, w, nsplit, out, lse) == 0
    torch.cuda.synchronize()
    compare(out, lse, *oracle_on(w))
    assert _flags(lib) & _native.DEVERR_PAGE_RANGE
    clean = wl.make_custom(B=3, H=64, topk=300, ctx_lens=[2000, 700, 90], seed=81 + nsplit, device="cuda")
    assert _noalloc(lib, clean, nsplit, out, lse) == 0
    torch.cuda.synchronize()
    compare(out, lse, *oracle_on(clean))
    assert _flags(lib) == 0
