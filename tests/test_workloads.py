"""The seeded input recipes produce the structure the workloads state."""
import math

import numpy as np
import torch

from sparse_mla_decode_paged_gb300 import workloads as wl


def test_recent_random_pattern():
    spec = wl.custom_spec("t", B=3, H=4, topk=64, ctx=1000, pattern="recent_random", seed=3)
    w = wl.make_workload(spec)
    for b in range(3):
        t = w.topk_idx[b].tolist()
        assert len(set(t)) == 64
        assert set(range(1000 - 32, 1000)) <= set(t)
        assert all(0 <= x < 1000 for x in t)
        assert t != sorted(t)


def test_uniform_pad_and_ragged_lengths():
    spec = wl.custom_spec("t", B=40, H=4, topk=512, ctx=None, pattern="uniform_pad", seed=4,
                          ragged_lo=64, ragged_hi=4096)
    w = wl.make_workload(spec)
    lens = w.seq_lens.tolist()
    assert min(lens) >= 64 and max(lens) < 4096
    for b, c in enumerate(lens):
        t = w.topk_idx[b]
        valid = t[t >= 0]
        assert len(set(valid.tolist())) == valid.numel()
        if c >= 512:
            assert valid.numel() == 512 and int(valid.max()) < c
        else:
            assert sorted(valid.tolist()) == list(range(c)) and int((t < 0).sum()) == 512 - c


def test_block_table_pages_distinct_and_in_pool():
    spec = wl.custom_spec("t", B=4, H=4, topk=16, ctx=300, pattern="uniform", seed=5, pool_pages=100)
    w = wl.make_workload(spec)
    used = w.block_table[w.block_table >= 0].tolist()
    assert len(used) == 4 * 5 and len(set(used)) == len(used) and max(used) < 100
    assert w.num_pages == 100


def test_large_range_sampler_is_distinct_and_uniformish():
    g = torch.Generator().manual_seed(0)
    r = wl._uniform_without_replacement(0, 1 << 20, 512, g, "cpu")
    assert r.numel() == 512 and len(set(r.tolist())) == 512
    assert 0 <= int(r.min()) and int(r.max()) < (1 << 20)
    assert abs(float(r.double().mean()) / (1 << 20) - 0.5) < 0.05


def test_quantiser_round_trip_and_record_layout():
    g = torch.Generator().manual_seed(1)
    lat = torch.randn((3, 64, 512), generator=g)
    codes, scales = wl.quantize_latent_fp8(lat)
    deq = codes.view(torch.float8_e4m3fn).float().reshape(3, 64, 4, 128) * scales.unsqueeze(-1)
    rel = (deq.reshape(3, 64, 512) - lat).abs() / lat.abs().reshape(3, 64, 4, 128).amax(-1).repeat_interleave(128, -1)
    assert float(rel.max()) <= 2.0 ** -4 + 1e-6            # half an E4M3 ulp at the block max
    amax_code = codes.view(torch.float8_e4m3fn).float().abs().reshape(3, 64, 4, 128).amax(-1)
    assert torch.all(amax_code == 448.0)
    rope = torch.randn((3, 64, 64), generator=g).to(torch.bfloat16)
    rec = wl.pack_records(codes, scales, rope)
    assert rec.shape == (3, 64, 656)
    assert torch.equal(rec[..., :512], codes)
    assert torch.equal(rec[..., 512:528].contiguous().view(torch.float32), scales)
    assert torch.equal(rec[..., 528:].contiguous().view(torch.bfloat16), rope)


def test_named_configs_match_their_recipes():
    c = wl.CONFIGS
    assert (c["tiny"].B, c["tiny"].topk, c["tiny"].ctx) == (1, 64, 256)
    assert (c["bs1_ctx8k"].B, c["bs1_ctx8k"].ctx, c["bs1_ctx8k"].pattern) == (1, 8192, "recent_random")
    assert (c["b32_ctx32k"].B, c["b32_ctx32k"].ctx, c["b32_ctx32k"].outlier_channels) == (32, 32768, 5)
    assert (c["b80_ctx128k"].B, c["b80_ctx128k"].ctx) == (80, 131072)
    assert c["b96_ragged_h64"].pool_pages * 64 * 656 > 32e9 and c["b96_ragged_h16"].H == 16
    w = wl.make_workload(c["tiny"])
    assert w.q.shape == (1, 64, 576) and w.kv_cache.shape == (4, 64, 656)
    assert abs(w.sm_scale - 1 / math.sqrt(576)) < 1e-15


def test_host_subset_remaps_pages():
    spec = wl.custom_spec("t", B=3, H=2, topk=20, ctx=500, pattern="uniform", seed=6, pool_pages=64)
    w = wl.make_workload(spec)
    q, kv, bt, tk, sl = wl.host_subset(w, [2, 0])
    for j, b in enumerate([2, 0]):
        for t in tk[j].tolist():
            p_new = int(bt[j, t // 64])
            p_old = int(w.block_table[b, t // 64])
            assert torch.equal(kv[p_new, t % 64], w.kv_cache[p_old, t % 64])
