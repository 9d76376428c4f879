"""Oracle for top-k selection over indexer scores (the step that produces the top-k lists).

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this module:
only the tests and the benchmark's CPU baseline may call it.  It shares no code
with the CUDA library.

The pages give the indexer's output only as a count ("Inside the Decode
Performance Investigation", The Setup: index_topk = 512 positions per query,
and the per-step kernel inventory lists the indexer launches); the rule is not
written down.  Reading taken, the plainest one:

* Query b scores the positions 0 .. len_b - 1 of its request (len_b =
  seq_lens[b]); positions at or past len_b are not candidates.
* When len_b <= k every candidate is kept: the row is 0, 1, ..., len_b - 1
  followed by -1 padding (the padding value the decode skips).
* Otherwise the k candidates of largest score are kept.  Scores are ranked by
  IEEE 754-2008 totalOrder on binary32 (section 5.10): negative values below
  positive ones, -0 below +0, infinities at the ends of the finite range, NaNs
  beyond them by sign.  Scores with identical bit patterns are ranked by
  position, the lower position first.  With this order the kept set is unique.
* The kept positions are written in increasing position order (a canonical
  order; the decode does not depend on it).
"""
from __future__ import annotations

import numpy as np


def total_order_key(scores: np.ndarray) -> np.ndarray:
    """Signed int64 keys whose numeric order is IEEE totalOrder on the float32 bit patterns.

    From the definition: a value with the sign bit clear ranks by its magnitude
    bits (+0 lowest, then the positive subnormals and normals, +inf, +NaNs by
    payload); a value with the sign bit set ranks below every such value, and
    among themselves in reverse magnitude order (-0 highest of them).  So a
    positive pattern maps to its magnitude bits m >= 0 and a negative one to
    -m - 1 < 0.
    """
    bits = np.ascontiguousarray(scores, dtype=np.float32).view(np.uint32).astype(np.int64)
    mag = bits & 0x7FFFFFFF
    neg = (bits >> 31) == 1
    return np.where(neg, -mag - 1, mag)


def topk_select(scores: np.ndarray, seq_lens: np.ndarray, k: int) -> np.ndarray:
    """int32 [B][k]: per query the kept positions in increasing order, -1 padded.

    scores float32 [B][num_cols]; seq_lens int [B], each clamped to [0, num_cols].
    """
    scores = np.asarray(scores, dtype=np.float32)
    B, n_cols = scores.shape
    out = np.full((B, k), -1, dtype=np.int32)
    for b in range(B):
        n = int(min(max(int(seq_lens[b]), 0), n_cols))
        if n <= k:
            out[b, :n] = np.arange(n, dtype=np.int32)
            continue
        key = total_order_key(scores[b, :n])
        pos = np.arange(n)
        # lexsort: the last key is primary -> larger score first, then lower position
        order = np.lexsort((pos, -key))
        out[b] = np.sort(order[:k]).astype(np.int32)
    return out
