"""Seeded synthetic inputs for sparse-MLA paged decode.

This module only draws random inputs and lays them out in the cache format; it
holds none of the decode arithmetic (no dequantisation, no scores, no
softmax).  Both the CUDA path and the float64 oracle consume what it produces.

Cache format (one 656-byte record per token, pages of 64 tokens):

    bytes   0..511  latent, FP8 E4M3 codes (OCP "fn" variant)
    bytes 512..527  four little-endian fp32 scales, one per 128 latent dims
    bytes 528..655  64 bf16 rope values, little-endian

The latent is quantised per (token, 128-dim block) with scale = amax / 448
(scale = 1 for an all-zero block), codes = RNE(x / scale) via torch's
float8_e4m3fn cast.  That is the write side of the cache, which the decode
path only reads.

Workload recipes follow the sparse-MLA decode setting of the "Inside the
Decode Performance Investigation" page (Setup: 64 query heads,
index_topk = 512, contexts up to 512K) and the five synthetic configurations
listed in ``CONFIGS``.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional, Sequence

import torch

PAGE_SIZE = 64
D_LATENT = 512
D_ROPE = 64
D_QK = D_LATENT + D_ROPE          # 576
RECORD_BYTES = D_LATENT + 16 + 2 * D_ROPE   # 656
SCALE_BLOCK = 128
FP8_MAX = 448.0


@dataclasses.dataclass
class WorkloadSpec:
    """Shape and structure of one synthetic decode batch."""
    name: str
    B: int
    H: int
    topk: int
    ctx: Optional[int]                 # fixed context length, or None for the ragged draw
    pattern: str                       # "uniform", "recent_random" or "uniform_pad"
    seed: int
    outlier_channels: int = 0          # latent channels multiplied by 8
    pool_pages: Optional[int] = None   # physical pages in the cache (None: exactly what is used)
    ragged_lo: int = 64
    ragged_hi: int = 524288


# The five workloads.  "ragged" draws ctx = floor(64 * 8192**u), u ~ U[0,1)
# (log-uniform over 64..524288) and pads the top-k list with -1 when ctx < 512.
CONFIGS: Dict[str, WorkloadSpec] = {
    "tiny": WorkloadSpec("tiny", B=1, H=64, topk=64, ctx=256, pattern="uniform", seed=0),
    "bs1_ctx8k": WorkloadSpec("bs1_ctx8k", B=1, H=64, topk=512, ctx=8192,
                              pattern="recent_random", seed=1),
    "b32_ctx32k": WorkloadSpec("b32_ctx32k", B=32, H=64, topk=512, ctx=32768,
                               pattern="recent_random", seed=2, outlier_channels=5),
    "b80_ctx128k": WorkloadSpec("b80_ctx128k", B=80, H=64, topk=512, ctx=131072,
                                pattern="uniform", seed=3),
    "b96_ragged_h64": WorkloadSpec("b96_ragged_h64", B=96, H=64, topk=512, ctx=None,
                                   pattern="uniform_pad", seed=4, pool_pages=786432),
    "b96_ragged_h16": WorkloadSpec("b96_ragged_h16", B=96, H=16, topk=512, ctx=None,
                                   pattern="uniform_pad", seed=4, pool_pages=786432),
}


@dataclasses.dataclass
class Workload:
    """Device (or host) tensors for one decode call, plus the spec they came from."""
    spec: WorkloadSpec
    q: torch.Tensor            # bf16 [B, H, 576]
    kv_cache: torch.Tensor     # uint8 [num_pages, 64, 656]
    block_table: torch.Tensor  # int32 [B, max_pages_per_seq], -1 beyond a request's pages
    topk_idx: torch.Tensor     # int32 [B, topk], logical token positions, -1 = padding
    seq_lens: torch.Tensor     # int32 [B]
    sm_scale: float

    @property
    def B(self) -> int:
        return self.q.shape[0]

    @property
    def H(self) -> int:
        return self.q.shape[1]

    @property
    def topk(self) -> int:
        return self.topk_idx.shape[1]

    @property
    def num_pages(self) -> int:
        return self.kv_cache.shape[0]


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def draw_context_lengths(spec: WorkloadSpec, g: torch.Generator, device) -> List[int]:
    if spec.ctx is not None:
        return [spec.ctx] * spec.B
    u = torch.rand(spec.B, generator=g, device=device, dtype=torch.float64).cpu()
    span = spec.ragged_hi / spec.ragged_lo
    return [max(1, int(math.floor(spec.ragged_lo * span ** float(x)))) for x in u]


def quantize_latent_fp8(latent: torch.Tensor) -> (torch.Tensor, torch.Tensor):
    """Encode fp32 latent [..., 512] to E4M3 codes and per-128 fp32 scales.

    Write side of the cache: scale = amax / 448 per 128-dim block (1 when the
    block is all zero); codes = RNE(x / scale), clamped to +-448 first.
    """
    shp = latent.shape
    blk = latent.reshape(*shp[:-1], D_LATENT // SCALE_BLOCK, SCALE_BLOCK)
    amax = blk.abs().amax(dim=-1, keepdim=True)
    scale = torch.where(amax > 0, amax / FP8_MAX, torch.ones_like(amax))
    codes = (blk / scale).clamp_(-FP8_MAX, FP8_MAX).to(torch.float8_e4m3fn)
    return codes.view(torch.uint8).reshape(shp), scale.squeeze(-1).contiguous()


def pack_records(codes: torch.Tensor, scales: torch.Tensor, rope_bf16: torch.Tensor) -> torch.Tensor:
    """Lay out [.., 512] u8 codes, [.., 4] fp32 scales and [.., 64] bf16 rope as 656-byte records."""
    lead = codes.shape[:-1]
    sc_bytes = scales.contiguous().view(torch.uint8).reshape(*lead, 16)
    rope_bytes = rope_bf16.contiguous().view(torch.uint8).reshape(*lead, 2 * D_ROPE)
    return torch.cat([codes, sc_bytes, rope_bytes], dim=-1).contiguous()


def fill_kv_cache(num_pages: int, g: torch.Generator, device, outlier_channels: int = 0,
                  chunk_pages: int = 4096) -> torch.Tensor:
    """Random paged cache: latent N(0,1) (outlier channels x8), rope N(0,1) in bf16."""
    cache = torch.empty((num_pages, PAGE_SIZE, RECORD_BYTES), dtype=torch.uint8, device=device)
    mult = None
    if outlier_channels:
        ch = torch.randperm(D_LATENT, generator=g, device=device)[:outlier_channels]
        mult = torch.ones(D_LATENT, device=device)
        mult[ch] = 8.0
    for p0 in range(0, num_pages, chunk_pages):
        n = min(chunk_pages, num_pages - p0)
        lat = torch.randn((n, PAGE_SIZE, D_LATENT), generator=g, device=device, dtype=torch.float32)
        if mult is not None:
            lat.mul_(mult)
        codes, scales = quantize_latent_fp8(lat)
        rope = torch.randn((n, PAGE_SIZE, D_ROPE), generator=g, device=device,
                           dtype=torch.float32).to(torch.bfloat16)
        cache[p0:p0 + n] = pack_records(codes, scales, rope)
        del lat, codes, scales, rope
    return cache


def draw_block_table(ctx_lens: Sequence[int], pool_pages: int, g: torch.Generator, device) -> torch.Tensor:
    """Each request gets distinct physical pages drawn at random from the pool (shuffled order)."""
    pages = [(c + PAGE_SIZE - 1) // PAGE_SIZE for c in ctx_lens]
    total = sum(pages)
    if total > pool_pages:
        raise ValueError(f"pool of {pool_pages} pages cannot hold {total}")
    perm = torch.randperm(pool_pages, generator=g, device=device)[:total].to(torch.int32)
    maxp = max(max(pages), 1)
    bt = torch.full((len(ctx_lens), maxp), -1, dtype=torch.int32, device=device)
    off = 0
    for b, n in enumerate(pages):
        bt[b, :n] = perm[off:off + n]
        off += n
    return bt


def _uniform_without_replacement(lo: int, hi: int, k: int, g, device) -> torch.Tensor:
    """k distinct integers from [lo, hi), in random order."""
    n = hi - lo
    if k > n:
        raise ValueError("k > range")
    if n <= 4 * k or n <= 1 << 16:
        return torch.randperm(n, generator=g, device=device)[:k] + lo
    # sparse draw for large ranges: oversample, dedupe (keeping first occurrences), shuffle
    while True:
        cand = torch.randint(lo, hi, (2 * k + 64,), generator=g, device=device)
        uniq, inv = torch.unique(cand, sorted=True, return_inverse=True)
        if uniq.numel() < k:
            continue
        first = torch.full((uniq.numel(),), cand.numel(), device=device, dtype=torch.long)
        first.scatter_reduce_(0, inv, torch.arange(cand.numel(), device=device), reduce="amin")
        keep = uniq[torch.argsort(first)][:k]
        return keep[torch.randperm(k, generator=g, device=device)]


def draw_topk(ctx_lens: Sequence[int], topk: int, pattern: str, g, device) -> torch.Tensor:
    rows = []
    for c in ctx_lens:
        if pattern == "uniform":
            r = _uniform_without_replacement(0, c, topk, g, device)
        elif pattern == "recent_random":
            n_recent = topk // 2
            recent = torch.arange(c - n_recent, c, device=device)
            older = _uniform_without_replacement(0, c - n_recent, topk - n_recent, g, device)
            r = torch.cat([recent, older])
            r = r[torch.randperm(topk, generator=g, device=device)]
        elif pattern == "uniform_pad":
            if c >= topk:
                r = _uniform_without_replacement(0, c, topk, g, device)
            else:
                r = torch.cat([torch.arange(c, device=device),
                               torch.full((topk - c,), -1, device=device, dtype=torch.long)])
                r = r[torch.randperm(topk, generator=g, device=device)]
        else:
            raise ValueError(pattern)
        rows.append(r.to(torch.int32))
    return torch.stack(rows)


def make_workload(spec: WorkloadSpec, device="cpu", pool_pages: Optional[int] = None,
                  rotation: int = 0, kv_cache: Optional[torch.Tensor] = None) -> Workload:
    """Build the inputs of one decode call.

    ``rotation`` > 0 draws a fresh (q, top-k, block table) set over the same
    cache and context lengths: benchmarks cycle through rotations so that
    every timed call reads rows that are not in L2.  ``kv_cache`` reuses an
    existing cache (its page count becomes the pool).
    """
    g = _gen(device, spec.seed)
    ctx = draw_context_lengths(spec, g, device)
    used = sum((c + PAGE_SIZE - 1) // PAGE_SIZE for c in ctx)
    pool = max(used, spec.pool_pages or 0, pool_pages or 0)
    if kv_cache is None:
        kv_cache = fill_kv_cache(pool, g, device, spec.outlier_channels)
    else:
        pool = kv_cache.shape[0]
    gr = _gen(device, spec.seed * 1000003 + 7919 * (rotation + 1))
    bt = draw_block_table(ctx, pool, gr, device)
    topk = draw_topk(ctx, spec.topk, spec.pattern, gr, device)
    q = torch.randn((spec.B, spec.H, D_QK), generator=gr, device=device,
                    dtype=torch.float32).to(torch.bfloat16)
    seq = torch.tensor(ctx, dtype=torch.int32, device=device)
    return Workload(spec, q, kv_cache, bt, topk, seq, 1.0 / math.sqrt(D_QK))


def custom_spec(name: str, B: int, H: int, topk: int, ctx, pattern: str = "uniform",
                seed: int = 0, **kw) -> WorkloadSpec:
    """A workload outside the five named ones (used by tests for small ragged cases)."""
    return WorkloadSpec(name, B=B, H=H, topk=topk, ctx=ctx, pattern=pattern, seed=seed, **kw)


def make_custom(B: int, H: int, topk: int, ctx_lens: Sequence[int], seed: int, device="cpu",
                pattern: str = "uniform_pad", pool_pages: Optional[int] = None,
                outlier_channels: int = 0) -> Workload:
    """Inputs with explicit per-request context lengths (top-k padded with -1 when ctx < topk)."""
    g = _gen(device, seed)
    ctx = list(int(c) for c in ctx_lens)
    used = sum((c + PAGE_SIZE - 1) // PAGE_SIZE for c in ctx)
    pool = max(used, pool_pages or 0, 1)
    kv = fill_kv_cache(pool, g, device, outlier_channels)
    bt = draw_block_table(ctx, pool, g, device) if used else torch.full((B, 1), -1, dtype=torch.int32, device=device)
    rows = []
    for c in ctx:
        if c >= topk:
            r = _uniform_without_replacement(0, c, topk, g, device)
        else:
            r = torch.cat([torch.arange(c, device=device),
                           torch.full((topk - c,), -1, device=device, dtype=torch.long)])
            r = r[torch.randperm(topk, generator=g, device=device)]
        rows.append(r.to(torch.int32))
    topk_t = torch.stack(rows)
    q = torch.randn((B, H, D_QK), generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
    seq = torch.tensor(ctx, dtype=torch.int32, device=device)
    spec = WorkloadSpec("custom", B=B, H=H, topk=topk, ctx=None, pattern=pattern, seed=seed)
    return Workload(spec, q, kv, bt, topk_t, seq, 1.0 / math.sqrt(D_QK))


SCORE_PATTERNS = ("normal", "relu", "ties", "special")


def make_indexer_scores(B: int, num_cols: int, seed: int, device="cpu", pattern: str = "normal") -> torch.Tensor:
    """float32 [B, num_cols] stand-ins for the indexer's per-position scores.

    normal  standard normal (a continuous score, few ties)
    relu    max(0, normal): half the positions score exactly 0 (a ReLU-weighted indexer's zeros)
    ties    normal rounded to quarters: heavy ties at every rank
    special normal with about 1% of the entries replaced by +-0, +-inf, +-NaN and subnormals
    """
    g = _gen(device, seed)
    s = torch.randn((B, num_cols), generator=g, device=device, dtype=torch.float32)
    if pattern == "normal":
        return s
    if pattern == "relu":
        return torch.clamp_min(s, 0.0)
    if pattern == "ties":
        return torch.round(s * 4.0) / 4.0
    if pattern == "special":
        bits = torch.tensor([0x00000000, 0x80000000, 0x7F800000, 0xFF800000, 0x7FC00000, 0xFFC00000,
                             0x00000001, 0x807FFFFF], dtype=torch.int64, device=device)
        bits = torch.where(bits >= 2 ** 31, bits - 2 ** 32, bits).to(torch.int32)
        pick = torch.rand((B, num_cols), generator=g, device=device) < 0.01
        which = torch.randint(0, bits.numel(), (B, num_cols), generator=g, device=device)
        return torch.where(pick, bits[which].view(torch.float32), s)
    raise ValueError(f"unknown score pattern {pattern!r}")


def touched_pages(w: Workload, batch_index: Sequence[int]) -> torch.Tensor:
    """Physical pages referenced by the valid top-k entries of the given requests (sorted, unique)."""
    pages = []
    for b in batch_index:
        t = w.topk_idx[b].long()
        ok = (t >= 0) & (t < int(w.seq_lens[b]))
        lp = t[ok] // PAGE_SIZE
        pg = w.block_table[b].long()[lp]
        pages.append(pg[(pg >= 0) & (pg < w.num_pages)])
    if not pages:
        return torch.empty(0, dtype=torch.long)
    return torch.unique(torch.cat(pages))


def host_subset(w: Workload, batch_index: Sequence[int]):
    """Copy to host only what the given requests read: their q rows, top-k, seq_lens, and the
    pages their valid top-k entries touch, with block tables renumbered into the compact copy.

    Data movement only (no decode arithmetic); lets a CPU checker run on requests drawn from a
    multi-GB cache.  Returns (q, kv_pages, block_table, topk_idx, seq_lens) as host tensors.
    """
    idx = torch.as_tensor(list(batch_index), dtype=torch.long, device=w.q.device)
    pages = touched_pages(w, batch_index).to(w.kv_cache.device)
    kv = w.kv_cache.index_select(0, pages).cpu() if pages.numel() else torch.zeros((1, PAGE_SIZE, RECORD_BYTES), dtype=torch.uint8)
    remap = {int(p): i for i, p in enumerate(pages.cpu().tolist())}
    bt = w.block_table.index_select(0, idx).cpu().clone()
    flat = bt.view(-1)
    for i in range(flat.numel()):
        v = int(flat[i])
        flat[i] = remap.get(v, -1)
    return (w.q.index_select(0, idx).cpu(), kv, bt,
            w.topk_idx.index_select(0, idx).cpu(), w.seq_lens.index_select(0, idx).cpu())


def algorithmic_bytes(topk_idx: torch.Tensor, seq_lens: torch.Tensor, block_table: torch.Tensor,
                      H: int, num_pages: int) -> int:
    """Bytes one decode call must move at minimum: valid KV rows (656 B each), q (bf16),
    out (bf16), lse (fp32), the top-k list and one block-table entry per distinct page touched."""
    t = topk_idx.long()
    ok = (t >= 0) & (t < seq_lens.long().unsqueeze(1))
    n_valid = int(ok.sum())
    lp = torch.where(ok, t // PAGE_SIZE, torch.zeros_like(t))
    pages = torch.gather(block_table.long(), 1, lp)
    pages = torch.where(ok, pages, torch.full_like(pages, -1))
    distinct = 0
    for b in range(pages.shape[0]):
        u = torch.unique(pages[b])
        distinct += int((u >= 0).sum())
    B, K = topk_idx.shape
    return (n_valid * RECORD_BYTES + B * H * (D_QK * 2 + D_LATENT * 2 + 4)
            + B * K * 4 + 4 * distinct)


def algorithmic_flops(topk_idx: torch.Tensor, seq_lens: torch.Tensor, H: int) -> int:
    t = topk_idx.long()
    ok = (t >= 0) & (t < seq_lens.long().unsqueeze(1))
    return 2 * H * int(ok.sum()) * (D_QK + D_LATENT)
