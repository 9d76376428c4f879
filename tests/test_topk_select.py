"""Top-k selection kernel against the oracle: bit-exact kept positions.

The rule (IEEE totalOrder, ties to the lower position, positions ascending, -1 padding) is a reading of
"Inside the Decode Performance Investigation", The Setup (index_topk = 512 per query)."""
import numpy as np
import pytest
import torch

from oracle import topk_select_oracle as T
from sparse_mla_decode_paged_gb300 import _native, api
from sparse_mla_decode_paged_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _check(scores, lens, k, cluster_ctas=0):
    got = api.sparse_mla_topk_select(scores, lens, k, cluster_ctas=cluster_ctas)
    torch.cuda.synchronize()
    ref = T.topk_select(scores.cpu().numpy(), lens.cpu().numpy(), k)
    g = got.cpu().numpy()
    bad = np.flatnonzero(np.any(g != ref, axis=1))
    assert bad.size == 0, f"rows {bad[:8].tolist()} differ"
    return got


@pytest.mark.parametrize("csize", [1, 2, 3, 5, 8])
@pytest.mark.parametrize("pattern", wl.SCORE_PATTERNS)
def test_every_cluster_size_and_pattern(csize, pattern):
    B, n = 6, 9000
    s = wl.make_indexer_scores(B, n, seed=10 + csize, device=DEV, pattern=pattern)
    lens = torch.tensor([9000, 8999, 4097, 513, 512, 1], dtype=torch.int32, device=DEV)
    _check(s, lens, 512, cluster_ctas=csize)


@pytest.mark.parametrize("k", [1, 17, 512, 1000, 2048])
def test_k_values(k):
    s = wl.make_indexer_scores(5, 6000, seed=k, device=DEV, pattern="ties")
    lens = torch.tensor([6000, 2049, 2047, k + 1, k], dtype=torch.int32, device=DEV)
    _check(s, lens, k)


def test_all_equal_and_two_level_rows():
    n = 5000
    s = torch.zeros((4, n), dtype=torch.float32, device=DEV)
    s[1, ::7] = 1.0                          # 715 ones: the top 512 are ones, lowest positions first
    s[2, 4000:] = -1.0
    s[3] = -0.0
    s[3, 100:200] = 0.0                      # +0 above -0
    lens = torch.full((4,), n, dtype=torch.int32, device=DEV)
    for c in (1, 4):
        _check(s, lens, 512, cluster_ctas=c)


def test_lengths_short_zero_and_out_of_range():
    s = wl.make_indexer_scores(6, 3000, seed=3, device=DEV)
    lens = torch.tensor([0, 1, 511, 512, 513, 3000], dtype=torch.int32, device=DEV)
    _check(s, lens, 512)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    bad = torch.tensor([-4, 5000, 700, 3000, 0, 12], dtype=torch.int32, device=DEV)
    got = api.sparse_mla_topk_select(s, bad, 512, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) & 0x8
    ref = T.topk_select(s.cpu().numpy(), bad.cpu().numpy(), 512)   # the oracle clamps the same way
    assert np.array_equal(got.cpu().numpy(), ref)


def test_unaligned_rows_take_scalar_loads():
    # a row stride that is not a multiple of 4 elements and a base one element past a 16-byte boundary
    base = wl.make_indexer_scores(5, 7003, seed=4, device=DEV)
    s = base[:, 1:7002]
    lens = torch.tensor([7001, 7000, 6999, 4096, 2000], dtype=torch.int32, device=DEV)
    for c in (1, 3):
        _check(s, lens, 512, cluster_ctas=c)


def test_padded_row_stride():
    big = wl.make_indexer_scores(3, 8192, seed=5, device=DEV)
    s = big[:, :5000]                        # rows 8192 apart, 5000 scored
    lens = torch.tensor([5000, 4999, 600], dtype=torch.int32, device=DEV)
    _check(s, lens, 512)


@pytest.mark.parametrize("B,n,k", [(32, 32768, 512), (80, 131072, 512), (1, 8192, 512), (4, 393216, 2048),
                                   (3, 524288, 512), (2, 786432, 1024), (1, 1048576, 2048)])
def test_decode_sizes(B, n, k):
    s = wl.make_indexer_scores(B, n, seed=B, device=DEV, pattern="relu")
    g = torch.Generator(device="cpu").manual_seed(B)
    lens = torch.randint(n // 2, n + 1, (B,), generator=g, dtype=torch.int32)
    lens[0] = n
    _check(s, lens.to(DEV), k)


def test_selected_lists_feed_the_decode():
    # scores -> top-k lists -> decode, compared with the decode of the oracle's lists
    w = wl.make_custom(B=3, H=64, topk=512, ctx_lens=[3000, 700, 200], seed=6, device=DEV)
    s = wl.make_indexer_scores(3, 3000, seed=6, device=DEV)
    topk = api.sparse_mla_topk_select(s, w.seq_lens, 512)
    ref_topk = torch.from_numpy(T.topk_select(s.cpu().numpy(), w.seq_lens.cpu().numpy(), 512)).to(DEV)
    assert torch.equal(topk, ref_topk)
    out, lse = api.sparse_mla_decode(w.q, w.kv_cache, w.block_table, topk, w.seq_lens, w.sm_scale)
    out2, lse2 = api.sparse_mla_decode(w.q, w.kv_cache, w.block_table, ref_topk, w.seq_lens, w.sm_scale)
    torch.cuda.synchronize()
    assert torch.equal(out, out2) and torch.equal(lse, lse2)


@pytest.mark.parametrize("csize", [1, 4])
def test_one_top_digit_bin_overflows_the_lists(csize):
    # every score in [1, 1.25): one top-digit bin (same exponent and top mantissa bits), distinct keys,
    # so more candidates than a warp lists and the later steps read the segment again
    g = torch.Generator(device=DEV).manual_seed(8)
    s = 1.0 + 0.2499 * torch.rand((3, 40000), generator=g, device=DEV)
    s[2, ::3] = 1.125                         # plus heavy ties inside that bin
    lens = torch.tensor([40000, 39999, 40000], dtype=torch.int32, device=DEV)
    _check(s, lens, 512, cluster_ctas=csize)


@pytest.mark.parametrize("scale", [1e-9, 1e-6, 1e7, 3e38])
def test_scores_at_extreme_magnitudes(scale):
    # tiny, huge and near-overflow scores: every exponent lands in its own top-digit bins
    s = wl.make_indexer_scores(4, 6000, seed=9, device=DEV) * scale
    lens = torch.tensor([6000, 5000, 3000, 600], dtype=torch.int32, device=DEV)
    for c in (1, 2):
        _check(s, lens, 512, cluster_ctas=c)


def _row(parts, n):
    # parts: [(count, value)], the rest filled with `fill`; positions shuffled with a fixed seed
    vals = []
    for c, v in parts[:-1]:
        vals += [v] * c
    vals += [parts[-1][1]] * (n - len(vals))
    g = np.random.default_rng(len(vals) + len(parts))
    return np.array(vals, dtype=np.float32)[g.permutation(n)]


@pytest.mark.parametrize("csize", [1, 3])
def test_bins_taken_whole(csize):
    # rows where the k-th entry closes a top-digit bin or a refinement digit exactly, so the select stops
    # early and keeps "everything from a bin boundary up": positive, negative, infinite and signed-zero
    # boundaries, and a digit boundary inside one top-digit bin
    n, k = 6000, 512
    rows = [
        _row([(k, 10.0), (0, 1.0)], n),
        _row([(k, -1.0), (0, -10.0)], n),
        _row([(k, np.inf), (0, 1.0)], n),
        _row([(k, 0.0), (0, -0.0)], n),
        _row([(412, 3.0), (100, 1.2), (1000, 1.1), (0, 0.5)], n),
        _row([(412, 3.0), (101, 1.2), (1000, 1.1), (0, 0.5)], n),
        _row([(k - 1, 7.0), (0, -np.inf)], n),
    ]
    s = torch.from_numpy(np.stack(rows)).to(DEV)
    lens = torch.full((len(rows),), n, dtype=torch.int32, device=DEV)
    _check(s, lens, k, cluster_ctas=csize)


@pytest.mark.parametrize("csize", [0, 4, 16])
def test_ragged_rows_share_clusters(csize):
    # log-uniform lengths: most rows need one CTA and share a cluster with other rows, a few need several
    B, n = 48, 200000
    g = torch.Generator(device="cpu").manual_seed(12)
    u = torch.rand(B, generator=g, dtype=torch.float64)
    lens = (64 * (n / 64) ** u).floor().to(torch.int32)
    lens[0] = n
    lens[1] = 0
    s = wl.make_indexer_scores(B, n, seed=12, device=DEV)
    _check(s, lens.to(DEV), 512, cluster_ctas=csize)


@pytest.mark.parametrize("B", [2048, 2100])
def test_many_rows(B):
    # 2048 rows packed into clusters of 2 (each CTA reads every length and finds its row among four
    # 512-row rounds); past 2048 rows every row takes a cluster of its own
    n, k = 4096, 64
    g = torch.Generator(device="cpu").manual_seed(13)
    lens = torch.randint(0, n + 1, (B,), generator=g, dtype=torch.int32)
    lens[-1] = n
    s = wl.make_indexer_scores(B, n, seed=13, device=DEV)
    _check(s, lens.to(DEV), k, cluster_ctas=2)


@pytest.mark.parametrize("case", range(12))
def test_random_shapes(case):
    # seeded random shapes: batch, row width, stride (aligned or not), k, cluster size, score pattern and
    # lengths (including 0, k, k + 1 and out-of-range values, which the oracle clamps the same way)
    rng = np.random.default_rng(1000 + case)
    B = int(rng.integers(1, 40))
    n = int(rng.integers(1, 60000))
    k = int(rng.choice([1, 7, 64, 512, 2048]))
    csize = int(rng.choice([0, 1, 2, 3, 4, 8, 16]))
    pattern = wl.SCORE_PATTERNS[case % len(wl.SCORE_PATTERNS)]
    pad = int(rng.choice([0, 1, 3, 64]))
    base = wl.make_indexer_scores(B, n + pad + 1, seed=2000 + case, device=DEV, pattern=pattern)
    s = base[:, 1:n + 1] if pad % 2 else base[:, :n]
    lens = rng.integers(0, n + 1, size=B)
    for i, v in enumerate([0, k, k + 1, n, n + 5, -3]):
        if i < B:
            lens[i] = v
    lens = torch.from_numpy(lens.astype(np.int32)).to(DEV)
    try:
        got = api.sparse_mla_topk_select(s, lens, k, cluster_ctas=csize)
    except _native.SmlaError as e:
        # a fixed cluster size whose chunk would exceed the per-CTA limit is refused on the host
        assert csize > 0 and e.status == 2, e
        return
    torch.cuda.synchronize()
    ref = T.topk_select(s.cpu().numpy(), lens.cpu().numpy(), k)
    bad = np.flatnonzero(np.any(got.cpu().numpy() != ref, axis=1))
    assert bad.size == 0, f"case {case} (B={B}, n={n}, k={k}, csize={csize}, {pattern}): rows {bad[:8].tolist()}"
