"""Pins for the float64 oracle: each test ties it to something other than itself
(the OCP FP8 table, library decoders, textbook dense softmax, closed forms,
invariants, high-precision brute force, hand-derived fixtures)."""
import json
import math
import os
import struct

import numpy as np
import pytest
import torch

import oracle
from sparse_mla_decode_paged_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ----------------------------------------------------------------------------- decoders

def test_e4m3_ocp_table_values():
    g = _golden("e4m3_ocp_values.json")
    for code, val in g["values"].items():
        got = oracle.e4m3_to_f64(np.array([int(code, 16)]))[0]
        assert got == val and math.copysign(1, got) == math.copysign(1, val), code
    for code in g["nan"]:
        assert np.isnan(oracle.e4m3_to_f64(np.array([int(code, 16)]))[0])


def test_e4m3_exhaustive_vs_torch_float8():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float32).double().numpy()
    got = oracle.e4m3_to_f64(codes.numpy())
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok], got[ok])
    assert np.array_equal(np.signbit(ref[ok]), np.signbit(got[ok]))


def test_bf16_decode_vs_torch():
    bits = torch.randint(0, 1 << 16, (20000,), generator=torch.Generator().manual_seed(3), dtype=torch.int32)
    t = bits.to(torch.int16).view(torch.bfloat16).float().double().numpy()
    got = oracle.bf16_bits_to_f64(bits.numpy().astype(np.uint16))
    ok = ~np.isnan(t)
    assert np.array_equal(np.isnan(t), np.isnan(got))
    assert np.array_equal(t[ok], got[ok])
    assert oracle.bf16_bits_to_f64(np.array([0x3F80, 0xC000, 0x0000]))[:3].tolist() == [1.0, -2.0, 0.0]


def test_record_layout_fields():
    lat_codes = bytes([0x38] * 128 + [0x40] * 128 + [0xB8] * 128 + [0x00] * 128)   # 1, 2, -1, 0
    scales = struct.pack("<4f", 0.5, 0.25, 4.0, 3.0)
    rope = struct.pack("<64H", *([0x3F80] * 32 + [0xC000] * 32))                   # 1.0, -2.0
    rec = np.frombuffer(lat_codes + scales + rope, dtype=np.uint8)
    assert rec.size == oracle.RECORD_BYTES
    k = oracle.dequantize_record(rec)
    assert np.all(k[:128] == 0.5) and np.all(k[128:256] == 0.5)
    assert np.all(k[256:384] == -4.0) and np.all(k[384:512] == 0.0)
    assert np.all(k[512:544] == 1.0) and np.all(k[544:576] == -2.0)


# ----------------------------------------------------------------------------- a1 gather

def test_gathered_rows_golden():
    g = _golden("gather_rows_small.json")
    rows = oracle.gathered_rows(g["block_table"], g["topk_idx"], g["seq_lens"], g["num_pages"], g["page_size"])
    assert rows.tolist() == g["rows"]


# ----------------------------------------------------------------------------- helpers

def _small(seed=0, B=2, H=4, topk=40, ctx=(100, 37), pool=None, outliers=0):
    w = wl.make_custom(B=B, H=H, topk=topk, ctx_lens=ctx, seed=seed, pool_pages=pool,
                       outlier_channels=outliers)
    return w


def _np(w):
    return (w.q.view(torch.int16).numpy().view(np.uint16), w.kv_cache.numpy(), w.block_table.numpy(),
            w.topk_idx.numpy(), w.seq_lens.numpy(), w.sm_scale)


def _torch_dequant_rows(kv_cache: torch.Tensor, rows: np.ndarray) -> np.ndarray:
    """Independent dequantisation through torch's float8/bf16 views (library decoders)."""
    flat = kv_cache.reshape(-1, wl.RECORD_BYTES)[torch.as_tensor(rows, dtype=torch.long)]
    lat = flat[:, :512].contiguous().view(torch.float8_e4m3fn).to(torch.float64)
    sc = flat[:, 512:528].contiguous().view(torch.float32).to(torch.float64)
    rope = flat[:, 528:].contiguous().view(torch.bfloat16).to(torch.float64)
    lat = lat * sc.repeat_interleave(128, dim=1)
    return torch.cat([lat, rope], 1).numpy()


# ----------------------------------------------------------------------------- a3..a5

def test_full_coverage_equals_dense_softmax_attention():
    """top-k = every position of the context => textbook dense softmax attention."""
    from scipy.special import logsumexp, softmax
    ctx = 150
    w = wl.make_custom(B=1, H=8, topk=ctx, ctx_lens=[ctx], seed=11, outlier_channels=3)
    perm = torch.randperm(ctx, generator=torch.Generator().manual_seed(2)).to(torch.int32)
    w.topk_idx[0] = perm
    out, lse = oracle.sparse_mla_decode(*_np(w))
    t = np.arange(ctx)
    rows = w.block_table[0].numpy()[t // 64].astype(np.int64) * 64 + t % 64
    K = _torch_dequant_rows(w.kv_cache, rows)
    q = w.q[0].double().numpy()
    S = w.sm_scale * q @ K.T
    ref = softmax(S, axis=1) @ K[:, :512]
    assert np.allclose(out[0], ref, rtol=1e-12, atol=1e-13)
    assert np.allclose(lse[0], logsumexp(S, axis=1), rtol=0, atol=1e-12)


def test_q_zero_gives_mean_of_v():
    w = _small(seed=5)
    w.q.zero_()
    out, lse = oracle.sparse_mla_decode(*_np(w))
    rows = oracle.gathered_rows(w.block_table, w.topk_idx, w.seq_lens, w.num_pages)
    for b in range(w.B):
        r = rows[b][rows[b] >= 0]
        V = _torch_dequant_rows(w.kv_cache, r)[:, :512]
        for h in range(w.H):
            assert np.allclose(out[b, h], V.mean(0), rtol=1e-12, atol=1e-14)
            assert abs(lse[b, h] - math.log(len(r))) < 1e-12


def test_single_valid_token_gives_its_value_and_score():
    w = _small(seed=6, B=1, H=5, topk=16, ctx=(300,))
    w.topk_idx[0] = -1
    w.topk_idx[0, 9] = 257
    out, lse = oracle.sparse_mla_decode(*_np(w))
    row = int(w.block_table[0, 257 // 64]) * 64 + 257 % 64
    k = _torch_dequant_rows(w.kv_cache, np.array([row]))[0]
    q = w.q[0].double().numpy()
    for h in range(w.H):
        assert np.array_equal(out[0, h], k[:512])
        assert abs(lse[0, h] - w.sm_scale * float(np.dot(q[h], k))) < 1e-12


def test_all_padding_and_empty_context():
    w = _small(seed=7)
    w.topk_idx[0] = -1
    w.seq_lens[1] = 0
    out, lse = oracle.sparse_mla_decode(*_np(w))
    assert np.all(out == 0) and np.all(np.isneginf(lse))


def test_entries_at_or_beyond_seq_len_are_ignored():
    w = _small(seed=8, B=1, topk=30, ctx=(200,))
    ref = oracle.sparse_mla_decode(*_np(w))
    w2 = _small(seed=8, B=1, topk=30, ctx=(200,))
    w2.topk_idx[0, 3] = 200          # == seq_len
    w2.topk_idx[0, 4] = 10_000       # far beyond
    base = _np(w)
    t = base[3].copy()
    t[0, 3] = -1
    t[0, 4] = -1
    expect = oracle.sparse_mla_decode(base[0], base[1], base[2], t, base[4], base[5])
    got = oracle.sparse_mla_decode(*_np(w2))
    assert np.array_equal(got[0], expect[0]) and np.array_equal(got[1], expect[1])
    assert not np.array_equal(ref[1], got[1])


def test_permutation_and_padding_invariance():
    w = _small(seed=9, B=2, topk=48, ctx=(400, 48))
    base = _np(w)
    out, lse = oracle.sparse_mla_decode(*base)
    rng = np.random.default_rng(0)
    t = base[3].copy()
    for b in range(t.shape[0]):
        t[b] = t[b][rng.permutation(t.shape[1])]
    o2, l2 = oracle.sparse_mla_decode(base[0], base[1], base[2], t, base[4], base[5])
    assert np.allclose(o2, out, rtol=1e-13, atol=1e-15) and np.allclose(l2, lse, rtol=0, atol=1e-13)
    t3 = np.concatenate([np.full((2, 7), -1, np.int32), base[3][:, :20], np.full((2, 5), -1, np.int32),
                         base[3][:, 20:]], axis=1)
    o3, l3 = oracle.sparse_mla_decode(base[0], base[1], base[2], t3, base[4], base[5])
    assert np.allclose(o3, out, rtol=1e-13, atol=1e-15) and np.allclose(l3, lse, rtol=0, atol=1e-13)


def test_duplicate_entry_counts_twice():
    """Two tokens a, b with a listed twice: weights 2e^{s_a} : e^{s_b} (closed form)."""
    w = _small(seed=10, B=1, H=3, topk=3, ctx=(128,))
    w.topk_idx[0] = torch.tensor([5, 77, 5], dtype=torch.int32)
    out, lse = oracle.sparse_mla_decode(*_np(w))
    bt = w.block_table[0].numpy()
    rows = np.array([bt[0] * 64 + 5, bt[1] * 64 + 13])
    K = _torch_dequant_rows(w.kv_cache, rows)
    q = w.q[0].double().numpy()
    for h in range(3):
        sa, sb = (w.sm_scale * float(np.dot(q[h], K[i])) for i in range(2))
        z = 2 * math.exp(sa) + math.exp(sb)
        ref = (2 * math.exp(sa) * K[0, :512] + math.exp(sb) * K[1, :512]) / z
        assert np.allclose(out[0, h], ref, rtol=1e-12, atol=1e-14)
        assert abs(lse[0, h] - math.log(z)) < 1e-12


def test_score_shift_leaves_out_and_shifts_lse():
    """Adding c to every score (through one rope dimension held constant) leaves out unchanged
    and adds c to lse; a large c also checks the max subtraction."""
    w = _small(seed=12, B=1, H=4, topk=40, ctx=(200,))
    base = _np(w)
    out, lse = oracle.sparse_mla_decode(*base)
    q = w.q.clone()
    kv = w.kv_cache.clone()
    q[..., 512] = 0.0
    kv.view(-1, 656)[:, 528:530] = torch.tensor([0.0], dtype=torch.bfloat16).view(torch.uint8)
    o0, l0 = oracle.sparse_mla_decode(q.view(torch.int16).numpy().view(np.uint16), kv.numpy(), *base[2:])
    q[..., 512] = 64.0
    kv.view(-1, 656)[:, 528:530] = torch.tensor([96.0], dtype=torch.bfloat16).view(torch.uint8)
    o1, l1 = oracle.sparse_mla_decode(q.view(torch.int16).numpy().view(np.uint16), kv.numpy(), *base[2:])
    c = w.sm_scale * 64.0 * 96.0          # = 256
    assert np.allclose(o1, o0, rtol=1e-11, atol=1e-13)
    assert np.allclose(l1 - l0, c, rtol=0, atol=1e-10)


def test_brute_force_high_precision():
    """Tiny case recomputed with scalar loops in 50-digit arithmetic (mpmath)."""
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = 50
    w = _small(seed=13, B=2, H=2, topk=5, ctx=(70, 130))
    w.topk_idx[1, 2] = -1
    out, lse = oracle.sparse_mla_decode(*_np(w))
    flat = w.kv_cache.reshape(-1, 656).numpy()
    for b in range(2):
        for h in range(2):
            ks, ss = [], []
            for t in w.topk_idx[b].tolist():
                if t < 0 or t >= int(w.seq_lens[b]):
                    continue
                rec = flat[int(w.block_table[b, t // 64]) * 64 + t % 64]
                sc = struct.unpack("<4f", rec[512:528].tobytes())
                k = []
                for d in range(512):
                    c = int(rec[d])
                    s, e, m = (-1 if c >> 7 else 1), (c >> 3) & 15, c & 7
                    val = mp.mpf(m) / 8 * mp.mpf(2) ** -6 if e == 0 else (1 + mp.mpf(m) / 8) * mp.mpf(2) ** (e - 7)
                    k.append(s * val * mp.mpf(sc[d // 128]))
                for j in range(64):
                    bits = int(rec[528 + 2 * j]) | (int(rec[529 + 2 * j]) << 8)
                    k.append(mp.mpf(struct.unpack("<f", struct.pack("<I", bits << 16))[0]))
                qv = [mp.mpf(x) for x in w.q[b, h].float().tolist()]
                ss.append(mp.mpf(w.sm_scale) * mp.fsum(qv[d] * k[d] for d in range(576)))
                ks.append(k)
            z = mp.fsum(mp.e ** s for s in ss)
            assert abs(float(mp.log(z)) - lse[b, h]) < 1e-12
            for d in range(0, 512, 37):
                ref = mp.fsum(mp.e ** ss[i] * ks[i][d] for i in range(len(ss))) / z
                assert abs(float(ref) - out[b, h, d]) < 1e-12 * max(1.0, abs(float(ref)))


# ----------------------------------------------------------------------------- a6, a7

@pytest.mark.parametrize("nsplit", [1, 2, 3, 5, 8])
def test_split_partials_merge_to_full(nsplit):
    w = _small(seed=14, B=3, H=4, topk=40, ctx=(300, 25, 64))
    base = _np(w)
    out, lse = oracle.sparse_mla_decode(*base)
    o_s, l_s = oracle.split_partials(*base, nsplit=nsplit)
    o, l = oracle.combine(o_s, l_s)
    assert np.allclose(o, out, rtol=1e-12, atol=1e-14)
    fin = np.isfinite(lse)
    assert np.array_equal(fin, np.isfinite(l))
    assert np.allclose(l[fin], lse[fin], rtol=0, atol=1e-12)


def test_combine_closed_form_two_partials():
    o = np.zeros((1, 2, 1, 512))
    o[0, 0, 0] = 1.0
    o[0, 1, 0] = 3.0
    l = np.array([[[math.log(1.0)], [math.log(3.0)]]])
    out, lse = oracle.combine(o, l)
    assert np.allclose(out[0, 0], 2.5) and abs(lse[0, 0] - math.log(4.0)) < 1e-15
    l2 = np.array([[[0.5], [-np.inf]]])
    out2, lse2 = oracle.combine(o, l2)
    assert np.allclose(out2[0, 0], 1.0) and abs(lse2[0, 0] - 0.5) < 1e-15


def test_split_positions_cover_topk():
    for K in (1, 7, 64, 512, 513):
        for s in range(1, 17):
            ps = oracle.split_positions(K, s)
            assert sum(len(p) for p in ps) == K and [i for p in ps for i in p] == list(range(K))


# ----------------------------------------------------------------------------- pages' numbers

def test_pages_split_numbers():
    g = _golden("pages_split_numbers.json")
    for b, n in g["grid_by_batch"].items():
        assert oracle.pages_grid(int(b)) == n
        assert oracle.pages_nsplit(int(b)) == g["nsplit_by_batch"][b]
    for b, wv in g["waves_by_batch"].items():
        assert round(oracle.waves(oracle.pages_grid(int(b)), g["sms"]), 2) == wv
    waste = 1 - oracle.wave_efficiency(oracle.pages_grid(64), g["sms"])     # 120 idle of 376 slots
    assert round(waste, 2) == g["b64_second_wave_waste"]
    assert 1 * 64 == g["bs1_grid_b_h"] and 1 * 64 * 8 == g["split_k_prescription_blocks"]


def test_queries_per_request_share_the_request_row():
    # several queries of one request (block table row b // s_q) equal the same queries with the row
    # repeated per query
    g = np.random.default_rng(21)
    R, s_q, K, pages = 3, 2, 12, 10
    bt = g.permutation(pages)[: R * 3].reshape(R, 3).astype(np.int32)
    seq = np.array([150, 151, 60, 61, 190, 191], dtype=np.int32)
    tk = np.stack([g.integers(-1, seq[b] + 5, K) for b in range(R * s_q)]).astype(np.int32)
    rows = oracle.gathered_rows(bt, tk, seq, pages)
    assert np.array_equal(rows, oracle.gathered_rows(np.repeat(bt, s_q, axis=0), tk, seq, pages))
    cache = g.integers(0, 256, size=(pages, 64, 656), dtype=np.uint8)
    cache[..., 512:528] = np.frombuffer(np.full(pages * 64 * 4, 0.01, "<f4").tobytes(), np.uint8).reshape(pages, 64, 16)
    cache[..., :512] &= 0x77                                              # finite codes
    cache[..., 528:] = 0
    q = (g.standard_normal((R * s_q, 2, 576))).astype(np.float64)
    o1, l1 = oracle.sparse_mla_decode(q, cache, bt, tk, seq, 0.05)
    o2, l2 = oracle.sparse_mla_decode(q, cache, np.repeat(bt, s_q, axis=0), tk, seq, 0.05)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
