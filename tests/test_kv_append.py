"""FP8 KV append kernel vs the oracle, through the C ABI: written records bit-exact, every other
byte of the cache untouched, out-of-range tokens skipped and flagged, and a decode that reads the
appended tokens matching the decode oracle."""
import numpy as np
import pytest
import torch

import oracle
from oracle import kv_append_oracle as ka
from sparse_mla_decode_paged_gb300 import api
from sparse_mla_decode_paged_gb300 import workloads as wl
from parity_util import compare, oracle_on

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _inputs(T, seed, extreme=True):
    """bf16 latent and rope; `extreme` adds log-normal magnitudes, a zero block and a 3e4 outlier (for
    the byte-exact checks), else N(0,1) with one channel x8 (the decode workloads' recipe)."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    lat = torch.randn(T, 512, generator=g)
    if extreme:
        lat = lat * torch.exp(torch.randn(T, 512, generator=g))
        if T > 3:
            lat[3, 256:384] = 0                                      # an all-zero block
            lat[1, 17] = 3.0e4                                       # an outlier
    else:
        lat[:, 41] *= 8
    rope = torch.randn(T, 64, generator=g)
    return lat.to(torch.bfloat16), rope.to(torch.bfloat16)


def _bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _cache_and_table(pages, R, P, seed):
    g = torch.Generator(device="cpu").manual_seed(seed)
    cache = torch.randint(0, 256, (pages, 64, 656), generator=g, dtype=torch.uint8)
    bt = torch.randperm(pages, generator=g)[: R * P].reshape(R, P).to(torch.int32)
    return cache, bt


@pytest.mark.parametrize("with_requests", [True, False])
def test_append_bit_exact(with_requests):
    R, P, pages = 8, 12, 120
    cache, bt = _cache_and_table(pages, R, P, seed=1)
    g = torch.Generator(device="cpu").manual_seed(2)
    if with_requests:
        T = 300
        flat = torch.randperm(R * P * 64, generator=g)[:T]                 # distinct (request, position)
        req, pos = (flat // (P * 64)).to(torch.int32), (flat % (P * 64)).to(torch.int32)
    else:
        T = R
        req, pos = None, torch.randint(0, P * 64, (T,), generator=g, dtype=torch.int32)
    lat, rope = _inputs(T, seed=3)
    ref = ka.kv_append(cache.numpy(), _bits(lat), _bits(rope), bt.numpy(), pos.numpy(),
                       None if req is None else req.numpy())
    dcache = cache.to(DEV)
    api.sparse_mla_kv_append(lat.to(DEV), rope.to(DEV), bt.to(DEV), pos.to(DEV), dcache,
                             requests=None if req is None else req.to(DEV))
    torch.cuda.synchronize()
    got = dcache.cpu().numpy()
    assert np.array_equal(got, ref)
    assert not np.array_equal(got, cache.numpy())                      # something was written


def test_out_of_range_tokens_skipped_and_flagged():
    R, P, pages = 3, 2, 8
    cache, bt = _cache_and_table(pages, R, P, seed=4)
    bt[2, 1] = 99                                                      # a page outside the cache
    req = torch.tensor([0, 1, 2, 5, 0, 2], dtype=torch.int32)          # request 5 does not exist
    pos = torch.tensor([3, 127, 100, 0, -1, 64], dtype=torch.int32)    # -1; page 99 for request 2
    lat, rope = _inputs(6, seed=5)
    ref = ka.kv_append(cache.numpy(), _bits(lat), _bits(rope), bt.numpy(), pos.numpy(), req.numpy())
    dcache = cache.to(DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    api.sparse_mla_kv_append(lat.to(DEV), rope.to(DEV), bt.to(DEV), pos.to(DEV), dcache, requests=req.to(DEV),
                             err_word=err)
    torch.cuda.synchronize()
    assert np.array_equal(dcache.cpu().numpy(), ref)
    assert int(err.item()) & 0x1                                       # SMLA_DEVERR_PAGE_RANGE
    ok_err = torch.zeros(1, dtype=torch.int32, device=DEV)
    api.sparse_mla_kv_append(lat[:2].to(DEV), rope[:2].to(DEV), bt.to(DEV), pos[:2].to(DEV), dcache,
                             requests=req[:2].to(DEV), err_word=ok_err)     # both in range
    torch.cuda.synchronize()
    assert int(ok_err.item()) == 0


def test_decode_reads_the_appended_tokens():
    # append one new token per request at position seq_len (inside the last page), make it part of
    # the top-k, and decode: the result matches the decode oracle on the oracle-appended cache
    w = wl.make_custom(B=4, H=64, topk=96, ctx_lens=[700, 63, 130, 1000], seed=61, device=DEV)
    lat, rope = _inputs(w.B, seed=62, extreme=False)
    pos = w.seq_lens.clone()
    ref_cache = ka.kv_append(w.kv_cache.cpu().numpy(), _bits(lat), _bits(rope), w.block_table.cpu().numpy(),
                             pos.cpu().numpy())
    api.sparse_mla_kv_append(lat.to(DEV), rope.to(DEV), w.block_table, pos, w.kv_cache)
    torch.cuda.synchronize()
    assert np.array_equal(w.kv_cache.cpu().numpy(), ref_cache)
    w.seq_lens += 1
    w.topk_idx[:, 0] = pos                                             # the new token is selected
    out, lse = api.sparse_mla_decode(w.q, w.kv_cache, w.block_table, w.topk_idx, w.seq_lens, w.sm_scale)
    torch.cuda.synchronize()
    compare(out, lse, *oracle_on(w))
