"""Pins of the top-k selection oracle against what the ranking rule and IEEE 754 fix.

The rule (the k largest scores among positions below the length, IEEE
totalOrder, ties by lower position, kept positions in increasing order) is a
reading of "Inside the Decode Performance Investigation", The Setup
(index_topk = 512); these tests pin the oracle to it by independent routes.
"""
import itertools
import math

import numpy as np
import pytest

from oracle import topk_select_oracle as T

F32 = np.float32


def _bits(x):
    return np.frombuffer(np.array(x, dtype=F32).tobytes(), dtype=np.uint32)


def test_distinct_finite_scores_match_argsort():
    # distinct values: the kept set is the one a descending float sort gives
    g = np.random.default_rng(1)
    s = g.standard_normal((4, 3000)).astype(F32)
    lens = np.array([3000, 2500, 900, 1201])
    out = T.topk_select(s, lens, 512)
    for b in range(4):
        ref = np.sort(np.argsort(-s[b, :lens[b]].astype(np.float64), kind="stable")[:512])
        assert np.array_equal(out[b], ref)


def test_brute_force_subsets_with_ties():
    # tiny rows drawn from three values: enumerate every k-subset and keep the one whose members all
    # outrank every non-member (greater float value, or equal value and lower position)
    g = np.random.default_rng(2)
    for trial in range(60):
        n, k = int(g.integers(4, 9)), int(g.integers(1, 4))
        v = g.choice(np.array([-1.5, 0.25, 2.0], dtype=F32), size=n)
        good = []
        for sub in itertools.combinations(range(n), k):
            rest = [j for j in range(n) if j not in sub]
            if all(v[i] > v[j] or (v[i] == v[j] and i < j) for i in sub for j in rest):
                good.append(list(sub))
        assert len(good) == 1
        assert T.topk_select(v[None], np.array([n]), k)[0].tolist() == good[0]


def test_total_order_special_values():
    # IEEE 754-2008 5.10: -NaN < -inf < -1 < -0 < +0 < denormal < 1 < +inf < +NaN
    qnan = np.frombuffer(np.uint32(0x7FC00000).tobytes(), F32)[0]
    nnan = np.frombuffer(np.uint32(0xFFC00000).tobytes(), F32)[0]
    den = np.frombuffer(np.uint32(0x00000001).tobytes(), F32)[0]
    ladder = [nnan, -np.inf, F32(-1), F32(-0.0), F32(0.0), den, F32(1), np.inf, qnan]
    key = T.total_order_key(np.array(ladder, dtype=F32))
    assert np.all(np.diff(key) > 0)
    # shuffled ladder: keeping k of them keeps the k highest rungs
    perm = np.array([4, 0, 8, 2, 6, 1, 7, 3, 5])
    row = np.array(ladder, dtype=F32)[perm]
    for k in range(1, 9):
        got = T.topk_select(row[None], np.array([9]), k)[0]
        kept_rungs = sorted(perm[got].tolist())
        assert kept_rungs == list(range(9 - k, 9)), k


def test_signed_zero_and_equal_bits():
    # -0 ranks below +0; identical patterns keep the lower position
    s = np.array([[-0.0, 0.0, -0.0, 0.0, 5.0]], dtype=F32)
    assert T.topk_select(s, np.array([5]), 2)[0].tolist() == [1, 4]
    assert T.topk_select(s, np.array([5]), 3)[0].tolist() == [1, 3, 4]
    assert T.topk_select(s, np.array([5]), 4)[0].tolist() == [0, 1, 3, 4]
    e = np.full((1, 10), 3.0, dtype=F32)
    assert T.topk_select(e, np.array([10]), 4)[0].tolist() == [0, 1, 2, 3]


def test_short_and_out_of_range_lengths():
    s = np.random.default_rng(3).standard_normal((4, 50)).astype(F32)
    out = T.topk_select(s, np.array([0, 7, 20, 99]), 20)
    assert np.all(out[0] == -1)
    assert out[1].tolist() == list(range(7)) + [-1] * 13
    assert out[2].tolist() == list(range(20))                   # len == k keeps every position
    assert np.array_equal(out[3], T.topk_select(s[3:4], np.array([50]), 20)[0])   # clamped to 50
    assert np.all(T.topk_select(s[:1], np.array([-5]), 3) == -1)


def test_positions_beyond_length_never_kept():
    s = np.zeros((1, 100), dtype=F32)
    s[0, 60:] = 1e30                                             # huge scores past the length
    out = T.topk_select(s, np.array([60]), 10)[0]
    assert out.tolist() == list(range(10))


def test_kept_set_is_an_upper_set_large():
    # at the decode's sizes: every kept score >= every dropped one, and equal scores split by position
    g = np.random.default_rng(4)
    s = np.round(g.standard_normal((2, 20000)) * 8).astype(F32)     # heavy ties
    out = T.topk_select(s, np.array([20000, 17000]), 512)
    for b, n in enumerate([20000, 17000]):
        kept = np.zeros(n, bool)
        kept[out[b]] = True
        assert kept.sum() == 512 and np.all(np.diff(out[b]) > 0)
        lo = s[b, :n][kept].min()
        assert np.all(s[b, :n][~kept] <= lo)
        border = np.flatnonzero(s[b, :n] == lo)
        assert np.all(kept[border][:int(kept[border].sum())]) and not np.any(kept[border][int(kept[border].sum()):])
