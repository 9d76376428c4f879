"""CUDA path vs the float64 oracle, element by element, through the C ABI."""
import math

import numpy as np
import pytest
import torch

import oracle
from sparse_mla_decode_paged_gb300 import api
from sparse_mla_decode_paged_gb300 import workloads as wl
from parity_util import compare, oracle_on, oracle_rows

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _run(w, nsplit=0):
    out, lse = api.sparse_mla_decode(w.q, w.kv_cache, w.block_table, w.topk_idx, w.seq_lens, w.sm_scale,
                                     nsplit=nsplit)
    torch.cuda.synchronize()
    return out, lse


def _custom(B, H, topk, ctx, seed, **kw):
    return wl.make_custom(B=B, H=H, topk=topk, ctx_lens=ctx, seed=seed, device=DEV, **kw)


def test_tiny_config():
    w = wl.make_workload(wl.CONFIGS["tiny"], device=DEV)
    out, lse = _run(w)
    compare(out, lse, *oracle_on(w))


@pytest.mark.parametrize("H", [16, 32, 64, 128])
def test_ragged_small_all_head_counts(H):
    # several tiles per partition, a ragged tail, padding (ctx < topk), a one-token context
    w = _custom(B=5, H=H, topk=300, ctx=[1000, 250, 64, 1, 5000], seed=20 + H, outlier_channels=5)
    out, lse = _run(w)
    compare(out, lse, *oracle_on(w))


@pytest.mark.parametrize("nsplit", [1, 2, 3, 4, 7, 8, 13, 16])
def test_every_split_count(nsplit):
    w = _custom(B=3, H=64, topk=512, ctx=[4096, 700, 300], seed=31)
    out, lse = _run(w, nsplit=nsplit)
    compare(out, lse, *oracle_on(w))


@pytest.mark.parametrize("nh", [16, 32, 64])
@pytest.mark.parametrize("H,nsplit", [(16, 1), (32, 3), (64, 1), (64, 4), (128, 2)])
def test_every_head_group_size(H, nsplit, nh):
    # the split kernel's 16-, 32- and 64-head variants on every head count (fewer heads than a group:
    # padded rows), one partition of several tiles and several partitions
    w = _custom(B=3, H=H, topk=400, ctx=[5000, 400, 77], seed=50 + nh + H + nsplit, outlier_channels=2)
    out, lse = api.sparse_mla_decode(w.q, w.kv_cache, w.block_table, w.topk_idx, w.seq_lens, w.sm_scale,
                                     nsplit=nsplit, heads_per_cta=nh)
    torch.cuda.synchronize()
    compare(out, lse, *oracle_on(w))


@pytest.mark.parametrize("nh", [16, 32, 64])
@pytest.mark.parametrize("topk", [256, 258])
def test_one_tile_partitions_and_the_next_size(nh, topk):
    # two partitions of 128 entries (every partition one tile: the launch takes the one-tile
    # instantiation, whose QK gather warp 0 issues) and of 129 entries (the general instantiation)
    w = _custom(B=3, H=64, topk=topk, ctx=[3000, 257, 129], seed=70 + nh + topk, outlier_channels=2)
    out, lse = api.sparse_mla_decode(w.q, w.kv_cache, w.block_table, w.topk_idx, w.seq_lens, w.sm_scale,
                                     nsplit=2, heads_per_cta=nh)
    torch.cuda.synchronize()
    compare(out, lse, *oracle_on(w))


@pytest.mark.parametrize("H,nsplit", [(16, 4), (32, 8), (64, 5), (128, 3), (64, 2)])
def test_split_merge_heads_and_partitions(H, nsplit):
    # head counts of one or two groups, partitions made only of padding (ctx 40 < topk), several
    # tiles per partition, partition counts that do not divide the top-k list
    w = _custom(B=4, H=H, topk=448, ctx=[3000, 40, 448, 1200], seed=40 + nsplit, outlier_channels=3)
    out, lse = _run(w, nsplit=nsplit)
    compare(out, lse, *oracle_on(w))


@pytest.mark.parametrize("merge", [api.MERGE_KERNEL, api.MERGE_FUSED])
@pytest.mark.parametrize("H,nsplit,nh", [(64, 2, 64), (64, 4, 64), (64, 8, 64), (64, 4, 32), (32, 8, 16),
                                         (16, 2, 16), (128, 4, 64)])
def test_merge_kernel_and_in_kernel_merge(H, nsplit, nh, merge):
    # the same partitions merged by the merge kernel or inside the split kernel (a cluster of the
    # partitions): several tiles per partition, partitions made only of padding (ctx 40), a one-token
    # context, duplicated entries
    w = _custom(B=4, H=H, topk=480, ctx=[6000, 40, 1, 900], seed=60 + H + nsplit + nh, outlier_channels=2)
    w.topk_idx[3, :4] = torch.tensor([3, 3, 3, 899], dtype=torch.int32, device=DEV)
    out, lse = api.sparse_mla_decode(w.q, w.kv_cache, w.block_table, w.topk_idx, w.seq_lens, w.sm_scale,
                                     nsplit=nsplit, heads_per_cta=nh, merge=merge)
    torch.cuda.synchronize()
    compare(out, lse, *oracle_on(w))
    assert torch.all(torch.isneginf(lse[2]) == False)      # noqa: E712  (one valid token: finite lse)


def test_in_kernel_merge_rows_and_flags():
    w = _custom(B=3, H=64, topk=512, ctx=[3000, 700, 5], seed=77)
    w.block_table[0, 5] = w.num_pages + 1
    dims = api.dims_of(w.q, w.kv_cache, w.block_table, w.topk_idx, 4, 64, api.MERGE_FUSED)
    ws = api.alloc_workspace(dims, 4)
    out, lse, rows = api.sparse_mla_decode_rows(w.q, w.kv_cache, w.block_table, w.topk_idx, w.seq_lens,
                                                w.sm_scale, workspace=ws, nsplit=4, heads_per_cta=64,
                                                merge=api.MERGE_FUSED)
    torch.cuda.synchronize()
    assert api.read_errors(ws) == 0x1
    assert np.array_equal(rows.cpu().numpy(), oracle_rows(w))
    compare(out, lse, *oracle_on(w))


@pytest.mark.parametrize("s_q,nsplit", [(2, 0), (3, 2), (4, 1)])
def test_several_queries_per_request(s_q, nsplit):
    # the MTP / verify shape: s_q queries per request, each with its own top-k and causal length
    # (query j of a request sees positions < ctx - (s_q - 1 - j)); one block-table row per request
    R = 3
    base = wl.make_custom(B=R, H=64, topk=200, ctx_lens=[900, 150, 1500], seed=70 + s_q, device=DEV)
    g = torch.Generator(device="cpu").manual_seed(71 + s_q)
    seq, rows = [], []
    for r in range(R):
        for j in range(s_q):
            L = int(base.seq_lens[r]) - (s_q - 1 - j)
            seq.append(L)
            pick = torch.randperm(L, generator=g)[:200]
            rows.append(torch.cat([pick, torch.full((200 - pick.numel(),), -1)]).to(torch.int32))
    seq_lens = torch.tensor(seq, dtype=torch.int32, device=DEV)
    topk = torch.stack(rows).to(DEV)
    q = torch.randn((R * s_q, 64, 576), generator=g).to(torch.bfloat16).to(DEV)
    out, lse = api.sparse_mla_decode(q, base.kv_cache, base.block_table, topk, seq_lens, base.sm_scale,
                                     nsplit=nsplit)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle.sparse_mla_decode(q.cpu().view(torch.int16).numpy().view(np.uint16),
                                            base.kv_cache.cpu().numpy(), base.block_table.cpu().numpy(),
                                            topk.cpu().numpy(), seq_lens.cpu().numpy(), base.sm_scale)
    compare(out, lse, ref_o, ref_l)
    rows_gpu = api.sparse_mla_gather_rows(base.block_table, topk, seq_lens, base.kv_cache.shape[0])
    torch.cuda.synchronize()
    assert np.array_equal(rows_gpu.cpu().numpy(), oracle.gathered_rows(base.block_table.cpu().numpy(),
                                                                       topk.cpu().numpy(), seq_lens.cpu().numpy(),
                                                                       base.kv_cache.shape[0]))


def test_split_and_combine_entry_points():
    w = _custom(B=2, H=64, topk=200, ctx=[900, 150], seed=32)
    o_part, lse_part = api.sparse_mla_split(w.q, w.kv_cache, w.block_table, w.topk_idx, w.seq_lens, w.sm_scale, 3)
    torch.cuda.synchronize()
    q, kv, bt, tk, sl = wl.host_subset(w, range(w.B))
    o_ref, l_ref = oracle.split_partials(q.view(torch.int16).numpy().view(np.uint16), kv.numpy(), bt.numpy(),
                                         tk.numpy(), sl.numpy(), w.sm_scale, 3)
    for s in range(3):
        compare(o_part[:, s].clone(), lse_part[:, s].clone(), o_ref[:, s], l_ref[:, s])
    out, lse = api.sparse_mla_combine(o_part, lse_part)
    torch.cuda.synchronize()
    compare(out, lse, *oracle.combine(o_ref, l_ref))


def test_edge_cases_padding_empty_duplicates():
    w = _custom(B=6, H=64, topk=64, ctx=[300, 300, 300, 300, 0, 70], seed=33)
    w.topk_idx[0] = -1                                   # all padding
    w.topk_idx[1, :] = -1
    w.topk_idx[1, 17] = 123                              # one valid token
    w.topk_idx[2, :8] = torch.tensor([5, 5, 5, 9, 9, 299, 300, 10_000], dtype=torch.int32, device=DEV)  # dups, bounds
    w.topk_idx[3] = w.topk_idx[3].flip(0)
    out, lse = _run(w)
    ref_out, ref_lse = oracle_on(w)
    compare(out, lse, ref_out, ref_lse)
    assert torch.all(out[0] == 0) and torch.all(torch.isneginf(lse[0]))
    assert torch.all(torch.isneginf(lse[4]))


@pytest.mark.parametrize("topk,ctx", [(1, [5, 1]), (1024, [1500, 900]), (2048, [3000, 2048]), (17, [17, 400])])
def test_topk_extremes(topk, ctx):
    w = _custom(B=2, H=64, topk=topk, ctx=ctx, seed=34 + topk)
    out, lse = _run(w)
    compare(out, lse, *oracle_on(w))


def test_bad_pages_are_skipped_and_flagged():
    w = _custom(B=2, H=64, topk=64, ctx=[500, 500], seed=35)
    ref_w = _custom(B=2, H=64, topk=64, ctx=[500, 500], seed=35)
    w.block_table[0, 2] = w.num_pages + 7               # physical page outside the cache
    w.block_table[1, 0] = -3
    dims = api.dims_of(w.q, w.kv_cache, w.block_table, w.topk_idx, 2)
    ws = api.alloc_workspace(dims, 2)
    out, lse = api.sparse_mla_decode(w.q, w.kv_cache, w.block_table, w.topk_idx, w.seq_lens, w.sm_scale,
                                     workspace=ws, nsplit=2)
    flags = api.read_errors(ws)
    assert flags & 0x1
    compare(out, lse, *oracle_on(w))                     # the oracle skips the same entries
    api.clear_errors(ws)
    out2, lse2 = api.sparse_mla_decode(ref_w.q, ref_w.kv_cache, ref_w.block_table, ref_w.topk_idx,
                                       ref_w.seq_lens, ref_w.sm_scale, workspace=ws, nsplit=2)
    assert api.read_errors(ws) == 0


def test_gather_rows_bit_exact_small():
    w = _custom(B=4, H=64, topk=100, ctx=[5000, 90, 1, 640], seed=36)
    w.topk_idx[0, 3] = 5000
    w.topk_idx[0, 4] = -1
    rows = api.sparse_mla_gather_rows(w.block_table, w.topk_idx, w.seq_lens, w.num_pages)
    torch.cuda.synchronize()
    assert np.array_equal(rows.cpu().numpy(), oracle_rows(w))


def _sample(B, n, seed):
    rng = np.random.default_rng(seed)
    return sorted(rng.choice(B, size=min(n, B), replace=False).tolist())


def _decode_rows(w, nsplit=0, heads_per_cta=0, merge=api.MERGE_AUTO):
    """Decode that also returns the rows its split kernel loaded; the row buffer starts as a sentinel
    no entry can produce, so an entry the kernel never resolved shows up."""
    rows = torch.full(tuple(w.topk_idx.shape), -7, dtype=torch.int64, device=DEV)
    out, lse, rows = api.sparse_mla_decode_rows(w.q, w.kv_cache, w.block_table, w.topk_idx, w.seq_lens,
                                                w.sm_scale, nsplit=nsplit, heads_per_cta=heads_per_cta, rows=rows,
                                                merge=merge)
    torch.cuda.synchronize()
    return out, lse, rows


@pytest.mark.parametrize("nh", [16, 32, 64])
@pytest.mark.parametrize("nsplit", [1, 3, 4])
def test_decode_gathers_exactly_the_oracle_rows(nh, nsplit):
    # the rows the decode kernel itself loaded, bit-exact: several tiles per partition, ragged tails,
    # padding, entries at or past the length, duplicates, pages outside the table and the cache
    w = _custom(B=5, H=64, topk=448, ctx=[5000, 300, 64, 1, 2000], seed=90 + nh + nsplit)
    w.topk_idx[0, :6] = torch.tensor([7, 7, 4999, 5000, -1, 130], dtype=torch.int32, device=DEV)
    w.block_table[4, 3] = w.num_pages + 2               # a physical page outside the cache
    out, lse, rows = _decode_rows(w, nsplit=nsplit, heads_per_cta=nh)
    assert np.array_equal(rows.cpu().numpy(), oracle_rows(w))
    compare(out, lse, *oracle_on(w))


@pytest.mark.parametrize("name", ["tiny", "bs1_ctx8k", "b32_ctx32k", "b80_ctx128k", "b96_ragged_h64",
                                  "b96_ragged_h16"])
def test_full_size_configs_sampled(name):
    """The full configurations with the scheduler's launch choice (the one the benchmark times):
    every row the decode kernel gathered is bit-exact for all queries; out and lse are checked against
    the oracle on sampled queries (the oracle copies only the pages those queries touch)."""
    w = wl.make_workload(wl.CONFIGS[name], device=DEV)
    try:
        out, lse = _run(w)
        out_r, lse_r, rows = _decode_rows(w)
        assert np.array_equal(rows.cpu().numpy(), oracle_rows(w))
        assert torch.equal(out_r, out) and torch.equal(lse_r, lse)    # recording rows changes nothing else
        rows = api.sparse_mla_gather_rows(w.block_table, w.topk_idx, w.seq_lens, w.num_pages)
        torch.cuda.synchronize()
        assert np.array_equal(rows.cpu().numpy(), oracle_rows(w))
        idx = _sample(w.B, 6, seed=len(name))
        if name.startswith("b96"):
            lens = w.seq_lens.cpu().numpy()
            idx = sorted(set(idx) | {int(np.argmin(lens)), int(np.argmax(lens))})   # shortest and longest context
        ref_out, ref_lse = oracle_on(w, idx)
        compare(out[idx], lse[idx], ref_out, ref_lse)
        assert torch.isfinite(lse[w.seq_lens > 0]).all()
    finally:
        del w
        torch.cuda.empty_cache()


@pytest.mark.parametrize("case", range(10))
def test_random_shapes(case):
    # seeded random shapes through the decode with its rows: batch, heads, top-k, ragged lengths (some
    # shorter than top-k, some of one token), partition count, head-group size and merge path
    rng = np.random.default_rng(3000 + case)
    H = int(rng.choice([16, 32, 64, 128]))
    B = int(rng.integers(1, 7))
    topk = int(rng.choice([1, 33, 128, 200, 512, 1000, 2048]))
    ctx = [int(rng.choice([1, int(rng.integers(2, topk + 2)), int(rng.integers(topk, 9000))])) for _ in range(B)]
    nh = int(rng.choice([0, 16, 32, 64]))
    nh = nh if nh <= H else 0
    nsplit = int(rng.choice([0, 1, 2, 3, 4, 8, 16]))
    merge = int(rng.choice([api.MERGE_AUTO, api.MERGE_KERNEL, api.MERGE_FUSED]))
    w = _custom(B=B, H=H, topk=topk, ctx=ctx, seed=3100 + case, outlier_channels=int(rng.integers(0, 3)))
    try:
        out, lse, rows = _decode_rows(w, nsplit=nsplit, heads_per_cta=nh, merge=merge)
    except Exception as e:
        # a merge inside the kernel that no launch shape of these dims allows is refused on the host
        assert merge == api.MERGE_FUSED and "UNSUPPORTED" in str(e), e
        return
    assert np.array_equal(rows.cpu().numpy(), oracle_rows(w)), f"case {case}"
    compare(out, lse, *oracle_on(w))
