"""Pins of the KV-append oracle (CPU): the E4M3 encoder and the per-block quantiser against
library routines and closed forms, and the record layout against the decode oracle."""
import numpy as np
import pytest
import torch

import oracle
from oracle import kv_append_oracle as ka
from sparse_mla_decode_paged_gb300 import workloads as wl


def _torch_e4m3(x):
    x = np.clip(np.asarray(x, dtype=np.float32), -448, 448)
    return torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_every_finite_code_encodes_to_itself():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)   # no NaNs
    vals = oracle.e4m3_to_f64(codes)
    assert np.array_equal(ka.e4m3_encode(vals), codes)


def test_ties_and_neighbours_match_the_library_cast():
    mags = ka._MAGS
    mids = (mags[:-1] + mags[1:]) / 2                        # exact midpoints (ties)
    m32 = mids.astype(np.float32)
    assert np.array_equal(m32.astype(np.float64), mids)       # representable in float32
    near = np.concatenate([m32, np.nextafter(m32, np.float32(0)), np.nextafter(m32, np.float32(1e9))])
    x = np.concatenate([near, -near])
    assert np.array_equal(ka.e4m3_encode(x), _torch_e4m3(x))
    # a tie goes to the even code: 2^-10 lies between 0 and the smallest subnormal 2^-9
    assert ka.e4m3_encode(np.float32(2.0 ** -10)) == 0
    assert ka.e4m3_encode(np.float32(3 * 2.0 ** -10)) == 2   # between codes 1 and 2: even code 2


def test_random_values_match_the_library_cast():
    g = np.random.default_rng(7)
    x = (g.standard_normal(200_000) * np.exp(g.uniform(-12, 6, 200_000))).astype(np.float32)
    assert np.array_equal(ka.e4m3_encode(x), _torch_e4m3(x))


def test_saturation_and_signed_zero():
    assert np.array_equal(ka.e4m3_encode(np.array([448, 463.9, 464, 1e30], dtype=np.float32)),
                          np.full(4, 0x7E, np.uint8))
    assert np.array_equal(ka.e4m3_encode(np.array([-448, -1e30], dtype=np.float32)), np.full(2, 0xFE, np.uint8))
    assert ka.e4m3_encode(np.float32(-0.0)) == 0x80
    assert ka.e4m3_encode(np.float32(-1e-9)) == 0x80
    assert ka.e4m3_encode(np.float32(0.0)) == 0


def test_quantiser_equals_the_generator_quantiser():
    # the input generator's torch quantiser follows the same definition (fp32 scale, fp32 quotient)
    g = torch.Generator().manual_seed(3)
    lat = torch.randn(64, 512, generator=g) * torch.exp(torch.randn(64, 512, generator=g))
    lat[5, 128:256] = 0                                     # an all-zero block: scale 1, codes 0
    lat[9, 7] = 1e4                                          # an outlier
    codes_t, scales_t = wl.quantize_latent_fp8(lat)
    codes_o, scales_o = ka.quantize_latent(lat.numpy())
    assert np.array_equal(codes_o, codes_t.numpy())
    assert np.array_equal(scales_o.view(np.uint32), scales_t.numpy().view(np.uint32))
    assert scales_o[5, 1] == 1.0 and not codes_o[5, 128:256].any()


def test_block_max_gets_the_largest_code_and_the_error_bound_holds():
    g = np.random.default_rng(11)
    lat = g.standard_normal((16, 512)).astype(np.float32)
    codes, scales = ka.quantize_latent(lat)
    blk = lat.reshape(16, 4, 128)
    cb = codes.reshape(16, 4, 128)
    amax_idx = np.abs(blk).argmax(-1)
    top = np.take_along_axis(cb, amax_idx[..., None], -1)[..., 0]
    assert np.all((top & 0x7F) == 0x7E)
    deq = oracle.e4m3_to_f64(codes).reshape(16, 4, 128) * scales[..., None]
    # E4M3 keeps 3 fraction bits: |x - deq| <= 2^-4 |x| for normal codes, <= 2^-10 * scale below them
    err = np.abs(deq - blk)
    bound = np.maximum(2.0 ** -4 * np.abs(blk), 2.0 ** -10 * scales[..., None]) * (1 + 1e-6)
    assert np.all(err <= bound)


def test_records_read_back_through_the_decode_oracle():
    g = np.random.default_rng(5)
    T, pages = 6, 8
    cache = g.integers(0, 256, size=(pages, 64, 656), dtype=np.uint8)
    bt = np.array([[3, 1], [0, 6]], dtype=np.int32)
    lat = g.standard_normal((T, 512)).astype(np.float32)
    lat_bits = (lat.view(np.uint32) >> 16).astype(np.uint16)          # bf16 by truncation (any bf16 input)
    rope_bits = g.integers(0, 1 << 15, size=(T, 64), dtype=np.uint16)
    req = np.array([0, 0, 1, 1, 0, 1], dtype=np.int32)
    pos = np.array([5, 70, 0, 127, 128, -1], dtype=np.int32)           # the last two are out of range
    new = ka.kv_append(cache, lat_bits, rope_bits, bt, pos, req)
    lat_in = ka.bf16_bits_to_f32(lat_bits)
    for i, (r, t) in enumerate(zip(req[:4], pos[:4])):
        page, slot = bt[r, t // 64], t % 64
        codes, scales, rope = oracle.decode_record(new[page, slot])
        c_ref, s_ref = ka.quantize_latent(lat_in[i])
        assert np.array_equal(oracle.e4m3_to_f64(c_ref), codes)
        assert np.array_equal(s_ref.astype(np.float64), scales)
        assert np.array_equal(np.ascontiguousarray(new[page, slot, 528:]).view("<u2"), rope_bits[i])
        finite = np.isfinite(rope)
        assert np.array_equal(oracle.bf16_bits_to_f64(rope_bits[i])[finite], rope[finite])
    touched = {(bt[r, t // 64], t % 64) for r, t in zip(req[:4], pos[:4])}
    for p in range(pages):
        for s in range(64):
            if (p, s) not in touched:
                assert np.array_equal(new[p, s], cache[p, s])
