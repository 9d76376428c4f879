"""Float64 CPU oracle for sparse-MLA decode over a paged FP8 latent cache.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this module:
only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may call it.  It shares no code with the CUDA library.

What it computes (plain definitions, written out step by step):

* a1  index -> address.  A top-k entry t of request b is a logical token
      position.  It is used when 0 <= t < seq_lens[b]; its page is
      block_table[b, t // 64], its slot t % 64.  Entries that fail the test,
      or whose page number is outside the cache, are skipped (-1 / padding).
      Source: "Inside the Decode Performance Investigation", Task 1 (attention
      stalls on scattered FP8 page-gathers); "The 64-Block Barrier", section
      "The Smoking Gun: Grid = (B, H)" (each block walks the 512 top-k tokens:
      gather, multiply, accumulate).
* a2  gather + dequantise.  Record layout [512 x E4M3 | 4 x fp32 scale |
      64 x bf16 rope]; k[d] = e4m3(code[d]) * scale[d // 128] for d < 512,
      k[512 + j] = rope[j]; v = k[:512].  Decoders are written here from the
      OCP FP8 E4M3 definition and the bf16 definition (upper half of binary32).
* a3  s_t = sm_scale * sum_{d<576} q[d] k_t[d].
* a4/a5  m = max_t s_t, lse = m + ln sum_t exp(s_t - m),
      out = sum_t exp(s_t - lse) v_t.  No valid token: out = 0, lse = -inf.
* a6  split partials: the same over a subset of the top-k positions.
* a7  log-sum-exp merge of partials ("The 64-Block Barrier", section "The
      Split-K Prescription": partial results combined with an online-softmax
      merge): lse = ln sum_s exp(lse_s); out = sum_s exp(lse_s - lse) out_s.
* pages' split heuristic (scheduler reference numbers): nsplit =
      ceil(256 / (B * 2)) capped at 16, grid = B * 2 * nsplit, and the wave
      count on the pages' 188-SM GPU ("Inside the Decode Performance
      Investigation", Task 1; "The Commit That Rewrote the Bottleneck",
      section "The Levers").

All floating-point arithmetic is float64.  Duplicated top-k entries count once
per occurrence.
"""
from __future__ import annotations

import math
from typing import List, Sequence, Tuple

import numpy as np

PAGE_SIZE = 64
D_LATENT = 512
D_ROPE = 64
D_QK = D_LATENT + D_ROPE
RECORD_BYTES = 656
SCALE_BLOCK = 128


# ----------------------------------------------------------------------------- decoders

def _e4m3_value(code: int) -> float:
    """OCP FP8 E4M3 ("fn"): 1 sign, 4 exponent (bias 7), 3 mantissa bits; no
    infinities; S.1111.111 is NaN; exponent field 0 encodes subnormals
    2^-6 * m/8."""
    s = -1.0 if (code >> 7) & 1 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return s * math.ldexp(m / 8.0, -6)
    return s * math.ldexp(1.0 + m / 8.0, e - 7)


E4M3_TABLE = np.array([_e4m3_value(c) for c in range(256)], dtype=np.float64)


def e4m3_to_f64(codes: np.ndarray) -> np.ndarray:
    return E4M3_TABLE[np.asarray(codes, dtype=np.uint8)]


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 is the upper 16 bits of an IEEE binary32."""
    b = np.asarray(bits).astype(np.uint32) & 0xFFFF
    with np.errstate(invalid="ignore"):
        return (b << np.uint32(16)).view(np.float32).astype(np.float64)


def f32_le_bytes_to_f64(b: np.ndarray) -> np.ndarray:
    """[..., 4k] little-endian bytes -> [..., k] float64."""
    b = np.ascontiguousarray(b, dtype=np.uint8)
    return b.view("<f4").astype(np.float64)


def decode_record(rec: np.ndarray) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """One or more 656-byte records -> (latent codes as values [..,512], scales [..,4], rope [..,64])."""
    rec = np.ascontiguousarray(rec, dtype=np.uint8)
    lat = e4m3_to_f64(rec[..., :D_LATENT])
    scales = f32_le_bytes_to_f64(rec[..., D_LATENT:D_LATENT + 16])
    rope_bits = np.ascontiguousarray(rec[..., D_LATENT + 16:]).view("<u2")
    rope = bf16_bits_to_f64(rope_bits)
    return lat, scales, rope


def dequantize_record(rec: np.ndarray) -> np.ndarray:
    """656-byte record(s) -> k [.., 576] float64 (latent * its block scale, then rope)."""
    lat, scales, rope = decode_record(rec)
    block_of_dim = np.arange(D_LATENT) // SCALE_BLOCK
    k_lat = lat * scales[..., block_of_dim]
    return np.concatenate([k_lat, rope], axis=-1)


def as_f64_q(q) -> np.ndarray:
    """q given as bf16 bit patterns (uint16/int16) or as real numbers."""
    a = np.asarray(q)
    if a.dtype in (np.uint16, np.int16):
        return bf16_bits_to_f64(a.view(np.uint16))
    return a.astype(np.float64)


# ----------------------------------------------------------------------------- a1: addresses

def gathered_rows(block_table, topk_idx, seq_lens, num_pages: int, page_size: int = PAGE_SIZE) -> np.ndarray:
    """Physical row (page * page_size + slot) of every top-k entry; -1 when skipped.

    Query b belongs to request b // s_q, s_q = (query rows) / (block-table rows): several queries of
    one request (each with its own top-k list and seq_lens entry) share its block-table row."""
    bt = np.asarray(block_table, dtype=np.int64)
    tk = np.asarray(topk_idx, dtype=np.int64)
    sl = np.asarray(seq_lens, dtype=np.int64)
    B, K = tk.shape
    s_q = B // bt.shape[0]
    rows = np.full((B, K), -1, dtype=np.int64)
    for b in range(B):
        for i in range(K):
            t = tk[b, i]
            if t < 0 or t >= sl[b]:
                continue
            lp = t // page_size
            if lp >= bt.shape[1]:
                continue
            page = bt[b // s_q, lp]
            if page < 0 or page >= num_pages:
                continue
            rows[b, i] = page * page_size + (t % page_size)
    return rows


# ----------------------------------------------------------------------------- a3..a5

def attend(q_heads: np.ndarray, k_rows: np.ndarray, sm_scale: float) -> Tuple[np.ndarray, np.ndarray]:
    """Softmax attention of H query rows over n key rows (k: [n, 576], v = k[:, :512]).

    Returns out [H, 512] and lse [H] (natural log, scores include sm_scale).
    """
    H = q_heads.shape[0]
    if k_rows.shape[0] == 0:
        return np.zeros((H, D_LATENT)), np.full(H, -np.inf)
    s = sm_scale * (q_heads @ k_rows.T)                    # [H, n]
    m = s.max(axis=1, keepdims=True)
    e = np.exp(s - m)
    l = e.sum(axis=1, keepdims=True)
    lse = (m + np.log(l))[:, 0]
    out = (e / l) @ k_rows[:, :D_LATENT]
    return out, lse


def sparse_mla_decode(q, kv_cache, block_table, topk_idx, seq_lens, sm_scale: float,
                      positions: Sequence[int] = None) -> Tuple[np.ndarray, np.ndarray]:
    """Full decode: out float64 [B, H, 512], lse float64 [B, H].

    ``positions`` restricts the top-k positions used (a split); None = all.
    """
    qf = as_f64_q(q)
    cache = np.asarray(kv_cache, dtype=np.uint8)
    num_pages = cache.shape[0]
    flat = cache.reshape(num_pages * PAGE_SIZE, RECORD_BYTES)
    rows = gathered_rows(block_table, topk_idx, seq_lens, num_pages)
    B, H, _ = qf.shape
    out = np.zeros((B, H, D_LATENT))
    lse = np.full((B, H), -np.inf)
    for b in range(B):
        r = rows[b] if positions is None else rows[b, list(positions)]
        r = r[r >= 0]
        k = dequantize_record(flat[r]) if r.size else np.zeros((0, D_QK))
        out[b], lse[b] = attend(qf[b], k, sm_scale)
    return out, lse


# ----------------------------------------------------------------------------- a6, a7

def split_positions(topk: int, nsplit: int) -> List[range]:
    """Contiguous top-k position ranges of ceil(topk / nsplit) entries (last one ragged)."""
    step = -(-topk // nsplit)
    return [range(min(s * step, topk), min((s + 1) * step, topk)) for s in range(nsplit)]


def split_partials(q, kv_cache, block_table, topk_idx, seq_lens, sm_scale, nsplit: int):
    """Per-split (out_s [B, nsplit, H, 512], lse_s [B, nsplit, H])."""
    qf = as_f64_q(q)
    B, H, _ = qf.shape
    K = np.asarray(topk_idx).shape[1]
    o = np.zeros((B, nsplit, H, D_LATENT))
    l = np.full((B, nsplit, H), -np.inf)
    for s, pos in enumerate(split_positions(K, nsplit)):
        o[:, s], l[:, s] = sparse_mla_decode(qf, kv_cache, block_table, topk_idx, seq_lens,
                                             sm_scale, positions=pos)
    return o, l


def combine(o_parts: np.ndarray, lse_parts: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """Merge partials over axis 1: o_parts [B, S, H, D], lse_parts [B, S, H]."""
    m = lse_parts.max(axis=1, keepdims=True)                       # [B,1,H]
    finite = np.isfinite(m)
    m_safe = np.where(finite, m, 0.0)
    w = np.where(np.isfinite(lse_parts), np.exp(lse_parts - m_safe), 0.0)   # [B,S,H]
    z = w.sum(axis=1, keepdims=True)
    lse = np.where(finite, m_safe + np.log(np.where(z > 0, z, 1.0)), -np.inf)[:, 0]
    wn = np.where(z > 0, w / np.where(z > 0, z, 1.0), 0.0)
    out = (wn[..., None] * o_parts).sum(axis=1)
    return out, lse


# ----------------------------------------------------------------------------- pages' split numbers

def pages_nsplit(B: int) -> int:
    """Split count of the pages' kernel: ceil(256 / (B * 2)), at most 16."""
    return min(16, -(-256 // (B * 2)))


def pages_grid(B: int, head_groups: int = 2) -> int:
    return B * head_groups * pages_nsplit(B)


def waves(ctas: int, slots: int) -> float:
    """Grid size in units of one full wave of resident CTAs."""
    return ctas / slots


def wave_efficiency(ctas: int, slots: int) -> float:
    """Fraction of launched CTA slots that do work: ctas / (ceil(ctas/slots) * slots)."""
    return ctas / (-(-ctas // slots) * slots)
