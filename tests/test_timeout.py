"""The split kernel's failure path on the GPU: every internal pipeline wait is bounded, and a wait that
runs out sets SMLA_DEVERR_TIMEOUT in the device error word, leaves the call's outputs unwritten and
the context usable.  The test shortens the limit to 1 ns so that the waits of a normal call run out
(nothing faults, traps or hangs: the roles finish their loops without work, then drain their MMAs
and copies before the CTA leaves), reads the flag back, restores the limit and checks that the next
call on the same workspace matches the oracle with no flag set."""
import pytest
import torch

from sparse_mla_decode_paged_gb300 import _native, api
from sparse_mla_decode_paged_gb300 import workloads as wl
from parity_util import compare, oracle_on

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("nsplit,merge", [(1, api.MERGE_AUTO), (2, api.MERGE_KERNEL), (2, api.MERGE_FUSED)])
def test_wait_that_runs_out_is_reported_and_recoverable(nsplit, merge):
    w = wl.make_workload(wl.CONFIGS["tiny"], device="cuda")
    dims = api.dims_of(w.q, w.kv_cache, w.block_table, w.topk_idx, nsplit, 0, merge)
    ws = api.alloc_workspace(dims, nsplit)
    out = torch.full((w.B, w.H, 512), 3.0, dtype=torch.bfloat16, device="cuda")
    lse = torch.full((w.B, w.H), 3.0, dtype=torch.float32, device="cuda")
    try:
        api.debug_set_wait_limit(1)
        api.sparse_mla_decode(w.q, w.kv_cache, w.block_table, w.topk_idx, w.seq_lens, w.sm_scale, out=out,
                              lse=lse, workspace=ws, nsplit=nsplit, merge=merge)
        torch.cuda.synchronize()                         # the call returns; no fault
    finally:
        api.debug_set_wait_limit(0)
    assert api.read_errors(ws) & _native.DEVERR_TIMEOUT
    if nsplit == 1:                                      # the split kernel writes the outputs itself
        assert torch.all(out == 3.0) and torch.all(lse == 3.0)
    api.clear_errors(ws)
    out2, lse2 = api.sparse_mla_decode(w.q, w.kv_cache, w.block_table, w.topk_idx, w.seq_lens, w.sm_scale,
                                       workspace=ws, nsplit=nsplit, merge=merge)
    torch.cuda.synchronize()
    assert api.read_errors(ws) == 0
    compare(out2, lse2, *oracle_on(w))
