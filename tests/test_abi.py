"""The C-ABI library loads, exports every declared entry point, and rejects bad
arguments on the host (no GPU needed: nothing here launches a kernel)."""
import ctypes as C
import glob
import math
import os
import re

import pytest

import oracle
from sparse_mla_decode_paged_gb300 import _native
from sparse_mla_decode_paged_gb300.api import make_dims

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_symbols():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        txt = open(h).read()
        txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
        names |= set(re.findall(r"\b(sparse_mla_\w+)\s*\(", txt))
    return sorted(names)


def test_every_declared_symbol_is_exported(lib):
    names = _declared_symbols()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for code, name in _native.STATUS.items():
        assert lib.sparse_mla_status_string(code)
    assert lib.sparse_mla_status_string(99) == b"unknown status"


FAKE = C.c_void_p(1 << 20)   # aligned non-null stand-in; never dereferenced by these calls


def _decode(lib, dims, ws=FAKE, ws_bytes=1 << 30, q=FAKE):
    return lib.sparse_mla_decode(C.byref(dims), q, FAKE, FAKE, FAKE, FAKE, C.c_float(0.04), FAKE, FAKE,
                                 ws, C.c_size_t(ws_bytes), None)


def test_host_side_rejections(lib):
    d = make_dims(4, 64, 512, 16, 100, nsplit=4)
    assert _decode(lib, d, q=C.c_void_p(0)) == 1                      # null q
    assert _decode(lib, d, q=C.c_void_p((1 << 20) + 8)) == 1          # misaligned q
    bad = make_dims(4, 64, 512, 16, 100, nsplit=4); bad.page_size = 32
    assert _decode(lib, bad) == 2
    bad = make_dims(4, 48, 512, 16, 100, nsplit=4)
    assert _decode(lib, bad) == 2                                     # unsupported head count
    bad = make_dims(4, 64, 4096, 16, 100, nsplit=4)
    assert _decode(lib, bad) == 2                                     # top-k too long
    bad = make_dims(0, 64, 512, 16, 100, nsplit=4)
    assert _decode(lib, bad) == 1
    bad = make_dims(65536, 64, 512, 16, 100, nsplit=4)
    assert _decode(lib, bad) == 2                                     # more queries than the grid holds
    need = lib.sparse_mla_workspace_size(C.byref(d), 4)
    assert need == 256 + 4 * 4 * 64 * 4 + 4 * 4 * 64 * 512 * 4
    assert _decode(lib, d, ws_bytes=need - 1) == 3                    # workspace too small
    assert _decode(lib, d, ws=C.c_void_p(0)) == 3
    assert lib.sparse_mla_combine(4, 64, 0, FAKE, FAKE, FAKE, FAKE, None) == 1
    assert lib.sparse_mla_combine(4, 64, 65, FAKE, FAKE, FAKE, FAKE, None) == 1
    assert lib.sparse_mla_split(C.byref(d), 0, FAKE, FAKE, FAKE, FAKE, FAKE, C.c_float(1.0), FAKE, FAKE,
                                None, None) == 1
    assert lib.sparse_mla_gather_rows(None, FAKE, FAKE, FAKE, FAKE, None) == 1
    assert lib.sparse_mla_read_errors(None, None, None) == 1
    assert lib.sparse_mla_workspace_size(None, 2) == 0


def test_noalloc_dims_statuses_match_the_workspace_entry_point(lib):
    """The workspace-free decode checks dims the way sparse_mla_decode does, before any CUDA call."""
    for dims, want in ((make_dims(4, 48, 512, 16, 100, nsplit=4), 2),      # unsupported head count
                       (make_dims(4, 48, 512, 16, 100, nsplit=0), 2),
                       (make_dims(4, 64, 4096, 16, 100, nsplit=2), 2),     # top-k too long
                       (make_dims(0, 64, 512, 16, 100, nsplit=0), 1)):     # no queries
        assert _decode(lib, dims) == want
        assert lib.sparse_mla_decode_noalloc(C.byref(dims), FAKE, FAKE, FAKE, FAKE, FAKE, C.c_float(0.04),
                                             FAKE, FAKE, None) == want
    assert lib.sparse_mla_decode_noalloc(None, FAKE, FAKE, FAKE, FAKE, FAKE, C.c_float(0.04), FAKE, FAKE,
                                         None) == 1
    assert lib.sparse_mla_noalloc_read_errors(None, None) == 1


def test_merge_selector(lib):
    d = make_dims(32, 64, 512, 16, 100, nsplit=4, merge=3)
    assert _decode(lib, d) == 1                                        # no such merge mode
    p = _native.SmlaPlan()
    d = make_dims(32, 64, 512, 16, 100, nsplit=3, heads_per_cta=64, merge=2)
    assert lib.sparse_mla_plan_for(C.byref(d), 152, C.byref(p)) == 2   # 3 partitions do not divide 64 heads
    for merge, fused in ((1, 0), (2, 1)):
        d = make_dims(32, 64, 512, 16, 100, nsplit=4, heads_per_cta=64, merge=merge)
        assert lib.sparse_mla_plan_for(C.byref(d), 152, C.byref(p)) == 0 and p.fused == fused
    d = make_dims(32, 64, 512, 16, 100, merge=2)                       # automatic split count, in-kernel merge
    assert lib.sparse_mla_plan_for(C.byref(d), 152, C.byref(p)) == 0
    assert p.nsplit == 1 or (p.fused == 1 and p.heads_per_cta % p.nsplit == 0 and p.nsplit <= 8)


def test_debug_entry_points_host_checks(lib):
    d = make_dims(4, 64, 512, 16, 100, nsplit=4)
    assert lib.sparse_mla_decode_rows(C.byref(d), FAKE, FAKE, FAKE, FAKE, FAKE, C.c_float(0.04), FAKE, FAKE,
                                      FAKE, C.c_size_t(1 << 30), None, None) == 1            # no row buffer
    assert lib.sparse_mla_decode_rows(C.byref(d), FAKE, FAKE, FAKE, FAKE, FAKE, C.c_float(0.04), FAKE, FAKE,
                                      FAKE, C.c_size_t(1 << 30), C.c_void_p((1 << 20) + 4), None) == 1
    bad = make_dims(4, 48, 512, 16, 100, nsplit=4)
    assert lib.sparse_mla_decode_rows(C.byref(bad), FAKE, FAKE, FAKE, FAKE, FAKE, C.c_float(0.04), FAKE, FAKE,
                                      FAKE, C.c_size_t(1 << 30), FAKE, None) == 2
    assert lib.sparse_mla_debug_set_wait_limit(5) == 0
    assert lib.sparse_mla_debug_set_wait_limit(0) == 0     # back to the default


def _plan(lib, B, H, K, sms, nsplit=0):
    p = _native.SmlaPlan()
    st = lib.sparse_mla_plan_for(C.byref(make_dims(B, H, K, 8192, 1 << 20, nsplit)), sms, C.byref(p))
    assert st == 0
    return p


def test_plan_fields_consistent(lib):
    for B in (1, 7, 32, 64, 80, 96):
        for H in (16, 64, 128):
            p = _plan(lib, B, H, 512, 152)
            assert 1 <= p.nsplit <= 16
            assert p.tokens_per_split == math.ceil(512 / p.nsplit)
            assert math.ceil(512 / p.tokens_per_split) == p.nsplit          # no empty partition
            assert p.heads_per_cta in (16, 32, 64) and p.heads_per_cta <= H
            assert p.head_groups == math.ceil(H / p.heads_per_cta)
            assert p.ctas == B * p.head_groups * p.nsplit
            assert abs(p.waves - p.ctas / (152 * p.ctas_per_sm)) < 1e-12
            ws = 256 if p.nsplit == 1 else 256 + math.ceil(B * p.nsplit * H * 4 / 256) * 256 + B * p.nsplit * H * 2048
            assert p.workspace_bytes == ws


def test_plan_is_argmin_of_its_cost_model(lib):
    """The automatic choice is the cheapest fixed choice (brute force over 1..16)."""
    for B in range(1, 97, 5):
        for sms in (148, 152, 188):
            auto = _plan(lib, B, 64, 512, sms)
            costs = {}
            for n in range(1, 17):
                if math.ceil(512 / math.ceil(512 / n)) != n:
                    continue
                costs[n] = _plan(lib, B, 64, 512, sms, nsplit=n).est_us
            best = min(costs.values())
            assert auto.est_us == pytest.approx(best)
            assert auto.nsplit == min(n for n, c in costs.items() if c <= best + 1e-9)


def test_plan_fixed_split_kept(lib):
    p = _plan(lib, 4, 64, 10, 152, nsplit=16)
    assert p.nsplit == 16 and p.tokens_per_split == 1


def test_plan_fixed_heads_per_cta_kept(lib):
    for nh in (16, 32, 64):
        for H in (16, 64, 128):
            p = _native.SmlaPlan()
            d = make_dims(8, H, 512, 8192, 1 << 20, 0, nh)
            assert lib.sparse_mla_plan_for(C.byref(d), 152, C.byref(p)) == 0
            assert p.heads_per_cta == nh and p.head_groups == math.ceil(H / nh)
    p = _native.SmlaPlan()
    assert lib.sparse_mla_plan_for(C.byref(make_dims(8, 64, 512, 8192, 1 << 20, 0, 48)), 152, C.byref(p)) == 1


def test_wave_count_matches_pages_arithmetic(lib):
    """With the pages' grid (B * 2 head groups * nsplit) the waves are the pages' numbers."""
    for B in (32, 96):
        ctas = oracle.pages_grid(B)
        assert round(ctas / 188, 2) == {32: 1.36, 96: 2.04}[B]
    p = _plan(lib, 64, 128, 512, 188, nsplit=2)     # 2 head groups per query, as in the pages' B=64 case
    assert p.ctas == 256 and round(p.waves, 2) == round(256 / 188, 2)
    assert round(1 - oracle.wave_efficiency(p.ctas, 188), 2) == 0.32


def test_kv_append_argument_checks_without_cuda(lib):
    d = _native.SmlaAppendDims(4, 2, 64, 8, 512, 64, 100)
    p = C.c_void_p(1 << 20)
    call = lambda dims, *ptrs: lib.sparse_mla_kv_append(C.byref(dims), *ptrs)
    ok_ptrs = [p, p, p, None, p, p, None, None]
    assert call(d, None, p, p, None, p, p, None, None) == 1                 # null latent
    assert call(d, C.c_void_p((1 << 20) + 8), p, p, None, p, p, None, None) == 1   # misaligned latent
    assert call(d, p, p, p, C.c_void_p((1 << 20) + 2), p, p, None, None) == 1      # misaligned requests
    bad = _native.SmlaAppendDims(4, 2, 32, 8, 512, 64, 100)                  # page size 32
    assert call(bad, *ok_ptrs) == 2
    bad = _native.SmlaAppendDims(-1, 2, 64, 8, 512, 64, 100)                 # negative token count
    assert call(bad, *ok_ptrs) == 1
    bad = _native.SmlaAppendDims(4, 0, 64, 8, 512, 64, 100)                  # no requests
    assert call(bad, *ok_ptrs) == 1


def test_topk_select_argument_checks_without_cuda(lib):
    p = C.c_void_p(1 << 20)
    call = lambda d, *ptrs: lib.sparse_mla_topk_select(C.byref(d), *ptrs)
    D = _native.SmlaTopkDims
    ok = [p, p, p, None, None]
    assert call(D(4, 1000, 1000, 512, 0), None, p, p, None, None) == 1      # null scores
    assert call(D(4, 1000, 1000, 512, 0), C.c_void_p((1 << 20) + 2), p, p, None, None) == 1   # misaligned
    assert call(D(4, 1000, 999, 512, 0), *ok) == 1                          # stride below the row
    assert call(D(4, 1000, 1000, 0, 0), *ok) == 1                           # k = 0
    assert call(D(4, 0, 1000, 8, 0), *ok) == 1                              # no positions
    assert call(D(4, 1000, 1000, 8, 17), *ok) == 1                          # cluster of 17 CTAs
    assert call(D(4, 1000, 1000, 4096, 0), *ok) == 2                        # k beyond 2048
    assert call(D(4, 16 * 65536 + 1, 16 * 65536 + 1, 512, 0), *ok) == 2     # row too long
    assert call(D(0, 1000, 1000, 512, 0), None, None, None, None, None) == 0   # empty batch: nothing to do


def _topk_plan(lib, B, n, k=512, forced=0, sms=152):
    d = _native.SmlaTopkDims(B, n, n, k, forced)
    c, ch = C.c_int32(0), C.c_int32(0)
    st = lib.sparse_mla_topk_plan_for(C.byref(d), sms, C.byref(c), C.byref(ch))
    return st, c.value, ch.value


@pytest.mark.parametrize("B,n", [(1, 256), (1, 8192), (32, 32768), (80, 131072), (96, 464028), (128, 65536),
                                 (4, 786432), (2, 1048576), (7, 1000)])
def test_topk_plan_shapes_cover_the_row(lib, B, n):
    st, c, ch = _topk_plan(lib, B, n)
    assert st == 0
    assert 1 <= c <= 16 and ch % 2048 == 0 and 2048 <= ch <= 65536
    assert c * ch >= n                       # every position has a CTA
    assert c == 1 or (c - 1) * ch < n         # no CTA of an automatic choice is empty
    assert (c > 8) == (n > 8 * 65536)         # clusters past the portable size only for long rows


def test_topk_plan_keeps_one_cta_per_sm_when_it_can(lib):
    st, c, ch = _topk_plan(lib, 32, 32768)
    assert st == 0 and (c, ch) == (4, 8192)   # 128 CTAs on 152 SMs (8-CTA clusters would double up)
    for B, n in [(1, 8192), (16, 65536), (150, 4096)]:
        st, c, ch = _topk_plan(lib, B, n)
        assert st == 0 and B * c <= 152


def test_topk_plan_fixed_and_rejected(lib):
    assert _topk_plan(lib, 8, 20000, forced=3)[:2] == (0, 3)
    assert _topk_plan(lib, 8, 20000, forced=16)[:2] == (0, 16)   # kept as given, even with empty CTAs
    assert _topk_plan(lib, 8, 100000, forced=1)[0] == 2          # one CTA cannot hold 100000 positions
    assert _topk_plan(lib, 8, 1048577)[0] == 2                   # longer than 16 chunks
    assert _topk_plan(lib, 8, 1000, k=4096)[0] == 2
    assert _topk_plan(lib, 8, 1000, forced=17)[0] == 1
    assert _topk_plan(lib, 8, 1000, sms=0)[0] == 1
