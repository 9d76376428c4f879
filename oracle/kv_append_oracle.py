"""Oracle for the FP8 KV append (the write side of the paged latent cache).

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this module:
only the tests may call it.  It shares no code with the CUDA library.

What it computes, written out from the definitions:

* E4M3 encoding (OCP 8-bit floating point, E4M3 variant: 1 sign bit, 4
  exponent bits with bias 7, 3 mantissa bits; normals (1 + m/8) * 2^(e - 7)
  for e = 1..15 except e = 15, m = 7 (NaN); subnormals m/8 * 2^-6; largest
  finite 448): round to nearest, ties to the code with an even mantissa,
  saturating finite values beyond 448 to 448; the sign is kept, also for
  values that round to zero.
* Per-token quantisation of the 512-dim latent in blocks of 128 dims
  ("Inside the Decode Performance Investigation", Task 1: FP8 latent KV with
  per-128-dim scales; the scale is amax / 448): scale = float32(amax / 448)
  (1 when the block is all zero), q = float32(x / scale), code = E4M3(q).  The
  two divisions are float32 round-to-nearest, the precision the kernel decides
  the codes in.
* The 656-byte record [512 codes | 4 x fp32 scale | 64 x bf16 rope], written
  at page block_table[r][t // 64], slot t % 64 for request r and logical
  position t; a token whose request, position or page is out of range is
  skipped.
"""
from __future__ import annotations

from typing import Optional

import numpy as np

PAGE_SIZE = 64
D_LATENT = 512
D_ROPE = 64
BLOCK = 128
RECORD_BYTES = 656
E4M3_MAX = 448.0


def _e4m3_magnitudes() -> np.ndarray:
    """Values of the codes 0x00..0x7E (all finite non-negative magnitudes), in code order."""
    vals = []
    for c in range(0x7F):
        e, m = c >> 3, c & 7
        vals.append(m / 8.0 * 2.0 ** -6 if e == 0 else (1 + m / 8.0) * 2.0 ** (e - 7))
    return np.array(vals, dtype=np.float64)


_MAGS = _e4m3_magnitudes()          # strictly increasing with the code


def e4m3_encode(x) -> np.ndarray:
    """float32/float64 array -> E4M3 codes (uint8): round to nearest even, saturating at 448."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    hi = np.searchsorted(_MAGS, a, side="left")          # first magnitude >= a
    hi = np.minimum(hi, len(_MAGS) - 1)
    lo = np.maximum(hi - 1, 0)
    d_lo = a - _MAGS[lo]
    d_hi = _MAGS[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo)
    code = np.where(a >= _MAGS[-1], len(_MAGS) - 1, code)  # saturate at 448
    code = np.where(a <= _MAGS[0], 0, code)                # exact zero
    neg = np.signbit(x)
    return (code.astype(np.uint8) | np.where(neg, 0x80, 0).astype(np.uint8)).astype(np.uint8)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float32 (the upper half of binary32)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def quantize_latent(latent: np.ndarray):
    """latent float32 [..., 512] -> (codes uint8 [..., 512], scales float32 [..., 4])."""
    x = np.asarray(latent, dtype=np.float32)
    blk = x.reshape(*x.shape[:-1], D_LATENT // BLOCK, BLOCK)
    amax = np.abs(blk).max(axis=-1, keepdims=True)
    scale = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
    q = (blk / scale).astype(np.float32)
    codes = e4m3_encode(q).reshape(x.shape)
    return codes, scale[..., 0]


def kv_append(kv_cache: np.ndarray, latent_bf16: np.ndarray, rope_bf16: np.ndarray, block_table: np.ndarray,
              positions: np.ndarray, requests: Optional[np.ndarray] = None) -> np.ndarray:
    """Return a copy of kv_cache (uint8 [pages, 64, 656]) with the new tokens' records written.

    latent_bf16 / rope_bf16: uint16 bf16 bit patterns [T, 512] / [T, 64]."""
    out = np.array(kv_cache, dtype=np.uint8, copy=True)
    T = latent_bf16.shape[0]
    codes, scales = quantize_latent(bf16_bits_to_f32(latent_bf16))
    num_req, max_pages = block_table.shape
    for i in range(T):
        r = int(requests[i]) if requests is not None else i
        t = int(positions[i])
        if r < 0 or r >= num_req or t < 0 or t // PAGE_SIZE >= max_pages:
            continue
        page = int(block_table[r, t // PAGE_SIZE])
        if page < 0 or page >= out.shape[0]:
            continue
        rec = out[page, t % PAGE_SIZE]
        rec[:D_LATENT] = codes[i]
        rec[D_LATENT:D_LATENT + 16] = scales[i].astype("<f4").view(np.uint8)
        rec[D_LATENT + 16:] = np.asarray(rope_bf16[i], dtype="<u2").view(np.uint8)
    return out
