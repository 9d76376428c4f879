"""Comparison of the CUDA path with the float64 oracle.

Tolerances (from the stated target): out within max relative error 5e-3,
read per (query, head) row as max_d |gpu - ref| / max_d |ref|; lse within
1e-3 absolute; rows with no valid entry must give out == 0 and lse == -inf
exactly; gathered row indices bit-exact.
"""
import numpy as np
import torch

import oracle
from sparse_mla_decode_paged_gb300 import workloads as wl

OUT_RTOL = 5e-3
LSE_ATOL = 1e-3


def oracle_on(w: wl.Workload, batch_index=None):
    """Run the oracle on (a subset of) a workload; only the touched pages are copied to the host."""
    idx = list(range(w.B)) if batch_index is None else list(batch_index)
    q, kv, bt, tk, sl = wl.host_subset(w, idx)
    out, lse = oracle.sparse_mla_decode(q.view(torch.int16).numpy().view(np.uint16), kv.numpy(), bt.numpy(),
                                        tk.numpy(), sl.numpy(), w.sm_scale)
    return out, lse


def compare(out_gpu: torch.Tensor, lse_gpu: torch.Tensor, out_ref: np.ndarray, lse_ref: np.ndarray):
    """Return (worst normwise out error, worst lse error); raise AssertionError on failure."""
    g = out_gpu.float().cpu().double().numpy()
    lg = lse_gpu.float().cpu().double().numpy()
    assert g.shape == out_ref.shape and lg.shape == lse_ref.shape
    empty = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lg), empty), "empty rows differ"
    if empty.any():
        assert np.all(g[empty] == 0.0), "empty rows must give out == 0"
    full = ~empty
    if not full.any():
        return 0.0, 0.0
    assert np.all(np.isfinite(g[full])) and np.all(np.isfinite(lg[full])), "non-finite output"
    denom = np.abs(out_ref[full]).max(axis=-1)
    err = np.abs(g[full] - out_ref[full]).max(axis=-1) / np.where(denom > 0, denom, 1.0)
    lerr = np.abs(lg[full] - lse_ref[full])
    worst, lworst = float(err.max()), float(lerr.max())
    assert worst <= OUT_RTOL, f"out normwise relative error {worst:.3e} > {OUT_RTOL}"
    assert lworst <= LSE_ATOL, f"lse abs error {lworst:.3e} > {LSE_ATOL}"
    return worst, lworst


def oracle_rows(w: wl.Workload) -> np.ndarray:
    return oracle.gathered_rows(w.block_table.cpu().numpy(), w.topk_idx.cpu().numpy(), w.seq_lens.cpu().numpy(),
                                w.num_pages)
