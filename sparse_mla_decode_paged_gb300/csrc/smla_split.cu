// Split kernel (sm_103a): tcgen05 MMAs with TMEM accumulators, exact scores.
//
// One CTA per (partition s of the top-k list, group of NH heads, query b), NH = 16, 32 or 64 (a
// template parameter); the partition is walked in tiles of 128 top-k entries (MMA M = 128 tokens,
// N = NH heads).  ("The 64-Block Barrier", "The Split-K Prescription": dequantise, QK^T over 576
// dims, online softmax, PV over 512 dims, split-K.)
//
// Numerics.  A block scale is split as sc = mant * 2^e (e clamped to [-15, 7]; block 0: [-30, 7], so
// that its mant >= 1).  The K tile holds K' = code * 2^e in fp16, exact for every E4M3 code, and Q is
// fp16 (exact for bf16 inside the fp16 range), so each 128-dim block's MMA S_b = K'_b . Q_b^T is
// exact up to fp32 accumulation.  The rope rows are stored as rope / mant_0 and accumulate into
// S_0 (one fp16 rounding on the rope part); the softmax warps form  s = sum_b mant_b * S_b  in fp32
// as the four block accumulators complete.  PV reads the same K' with the mantissa moved onto the
// probabilities:  O_b^T += K'_b^T . (P * mant_b), the products P * mant_b rounded to fp16.
//
// Warp roles (12 warps, one CTA per SM):
//   gather (8 warps)   warp g owns tokens [16g, 16g + 16) of a tile.  Lanes 0..15 resolve index ->
//                      row through the block table (a1) in a four-stage pipeline: top-k entries of
//                      tile i + 4 and block-table entries of tile i + 3 in flight, the records of tile
//                      i + 3 bulk-prefetched into L2 while those of tile i + 1 are loaded into
//                      registers (all issued where they are written, so no load waits on another).
//                      Record bytes are read coalesced: one token's 512 code bytes per warp load,
//                      four tokens' rope bytes, sixteen tokens' scales.  Codes -> K' (fp16,
//                      128B-swizzled chunks of 64 dims), rope bf16 / mant_0 -> fp16, mantissas and
//                      validity to shared memory.  A warp signals its part of the tile (mbarrier)
//                      before it issues the next loads: a fence or barrier after them would wait for
//                      them.
//   MMA issue          one elected lane of softmax warp 0, from unrolled issuers whose descriptors
//                      are a base plus a compile-time offset: the 36 QK MMAs of a tile in one batch
//                      (block b into score buffer b, the rope into block 0's), then the PV MMAs.
//                      The issuing thread waits while the tensor core takes the MMAs (about as long
//                      as they run), so in launches of one tile per CTA (kOneTile) gather warp 0,
//                      which has no next tile to load, issues the QK instead, and every softmax warp
//                      reads each score buffer as it completes.
//   softmax (4 warps)  one token (TMEM lane) per thread, NH heads: scores accumulated from the score
//                      buffers as they complete, lazy running max (a head's reference moves only
//                      when a score exceeds it by more than 2^8; O and the row sums are then
//                      rescaled), P = exp2(s - m), row sums reduced over the warp.  PV: P * mant_0
//                      into the rope chunk, block 0's 8 MMAs; then P * mant_1..3 into chunks 0, 1
//                      and the rope chunk (free once block 0's PV is done) and the other 24 MMAs.
//   epilogue (all)     O / l from TMEM written straight to the [head][512] output rows (two dims per
//                      lane and store), lse.
//
// Shared memory: Q 9 * 128 * NH bytes (18, 36 or 72 KB) + K tile 144 KB + ~5 KB; TMEM: 8 * NH
// columns, O^T in 0 .. 4 NH - 1 (4 blocks x NH heads), score buffers in 4 NH .. 8 NH - 1.
#include <cuda_runtime.h>
#include <math_constants.h>

#include <atomic>
#include <mutex>

#include "smla_device.cuh"
#include "smla_ptx.cuh"
#include "smla_split_layout.cuh"

namespace smla {
namespace {

constexpr int kHeadsMax = 64;
constexpr int kThreads = 384;
constexpr int kSoftWarps = 4;
constexpr int kSoftThreads = 32 * kSoftWarps;     // warps 0..3: TMEM lane quadrants 0..3
constexpr int kGatherWarps = 8;
constexpr int kTokPerGatherWarp = kTile / kGatherWarps;   // 16
constexpr float kRescaleThreshold = 8.0f;         // log2 units: P <= 2^8
constexpr float kFp16Max = 65504.0f;
constexpr float kMaxScale = 16384.0f;             // P * mant <= 2^8 * 2^7 stays inside fp16

// Before tile 0 is converted the K tile is idle: it receives the raw bf16 Q of the head group (up to
// 64 x 1152 bytes at offset 0) and tile 0's raw E4M3 codes (128 x 512 bytes) by bulk copy.
constexpr uint32_t kRawQMax = kHeadsMax * kDQK * 2;          // 73728
constexpr uint32_t kRawLatOff = kRawQMax;
static_assert(kRawLatOff + kTile * kDLatent <= kKBytes, "raw staging inside the K tile");
constexpr uint32_t kGatherBar = 4;                           // named barrier of the gather warps

struct Misc {
  uint64_t q_raw;            // raw Q landed in the K tile (bulk copy)
  uint64_t raw0;             // tile 0's raw codes landed in the K tile (one arrival per token lane)
  uint64_t k_free0;          // raw Q read by every softmax warp: tile 0 may be written
  uint64_t q_ready;          // Q staged (one arrival per softmax warp)
  uint64_t tile_full;        // K tile and metadata of the tile written (one arrival per gather warp)
  uint64_t s_full[4];        // score buffer b holds block b of the tile (block 0 with the rope)
  uint64_t pv0_done;          // PV of block 0 complete: chunks 0, 1 and the rope chunk are free
  uint64_t pv_done;          // every PV MMA of the tile complete: the K tile is free
  uint64_t teardown;         // every MMA complete
  uint32_t tmem_slot;
  int abort;
  int range_err;
  alignas(16) float mant[4][kTile];
  unsigned char valid[kTile];
  alignas(16) float m_ref[kHeadsMax];    // reference max per head, log2 units
  alignas(16) float m_new[kHeadsMax];
  alignas(16) float alpha[kHeadsMax];
  alignas(16) float red[kSoftWarps][kHeadsMax];
  alignas(16) float linv[kHeadsMax];
  float lse_out[kHeadsMax];
  // merge inside a cluster of the query's partitions
  uint64_t merge_in;                     // peers' weighted rows of this CTA's head slice landed
  // (shared memory here is taken from the L1 that lands the record loads: kept small)
  alignas(16) float lse_in[kHeadsMax];   // lse of this CTA's L heads in every partition r: [r * L + i]
  alignas(16) float wts[kHeadsMax];      // merge weight of partition r for head i of this CTA: [r * L + i]
  float lse_merged[kHeadsMax / 2];
};

template <int NH>
constexpr size_t smem_bytes() { return 1024 + Cfg<NH>::kMiscOff + sizeof(Misc); }
static_assert(smem_bytes<64>() <= 232448, "shared memory per CTA");

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// sc = mant * 2^e, e = clamp(exponent(sc), -15, 7); returns mant (exact) and 2^e as fp16 bits.
__device__ __forceinline__ float pow2_split(float sc, uint32_t& p2) {
  const uint32_t bits = __float_as_uint(sc) & 0x7fffffffu;
  int e = (int)(bits >> 23) - 127;
  e = max(-15, min(7, e));
  const float mant = sc * __uint_as_float((uint32_t)(127 - e) << 23);
  p2 = e >= -14 ? (uint32_t)(e + 15) << 10 : 0x0200u;   // 2^-15 is an fp16 subnormal
  return mant;
}

// Block 0's scale, split so that mant >= 1 always (the rope is folded into block 0 as rope / mant):
// e = clamp(exponent(sc), -30, 7); 2^e as fp16 bits (subnormal below 2^-14, zero below 2^-24, where
// K' = code * 2^e is rounded or vanishes: such a block contributes below 2^-15 * 448 * |q|); sc == 0
// gives mant = 1 and 2^e = 0.
__device__ __forceinline__ float pow2_split_b0(float sc, uint32_t& p2) {
  const uint32_t bits = __float_as_uint(sc) & 0x7fffffffu;
  if (bits < 0x00800000u) {                  // zero or fp32-subnormal scale: the block contributes nothing
    p2 = 0;
    return 1.f;
  }
  int e = (int)(bits >> 23) - 127;
  e = max(-30, min(7, e));
  const float mant = sc * __uint_as_float((uint32_t)(127 - e) << 23);
  p2 = e >= -14 ? (uint32_t)(e + 15) << 10 : e >= -24 ? (1u << (e + 24)) : 0u;
  return mant;
}

// 2 bf16 -> 2 fp16 (saturating); flags values outside the fp16 range.
__device__ __forceinline__ uint32_t bf2_to_h2(uint32_t w, int& range_bad) {
  const float lo = __uint_as_float(w << 16), hi = __uint_as_float(w & 0xFFFF0000u);
  range_bad |= (fabsf(lo) > kFp16Max) | (fabsf(hi) > kFp16Max);
  return f32x2_to_f16x2_sat(lo, hi);
}

__device__ __forceinline__ uint4 bf8_to_h8(uint4 v, int& range_bad) {
  return make_uint4(bf2_to_h2(v.x, range_bad), bf2_to_h2(v.y, range_bad), bf2_to_h2(v.z, range_bad),
                    bf2_to_h2(v.w, range_bad));
}

// 2 bf16 times `f` (fp32) -> 2 fp16, rounded once (saturating; flags values outside the fp16 range).
__device__ __forceinline__ uint32_t bf2_scaled_to_h2(uint32_t w, float f, int& range_bad) {
  const float lo = __uint_as_float(w << 16) * f, hi = __uint_as_float(w & 0xFFFF0000u) * f;
  range_bad |= (fabsf(lo) > kFp16Max) | (fabsf(hi) > kFp16Max);
  return f32x2_to_f16x2_sat(lo, hi);
}

__device__ __forceinline__ uint4 bf8_scaled_to_h8(uint4 v, float f, int& range_bad) {
  return make_uint4(bf2_scaled_to_h2(v.x, f, range_bad), bf2_scaled_to_h2(v.y, f, range_bad),
                    bf2_scaled_to_h2(v.z, f, range_bad), bf2_scaled_to_h2(v.w, f, range_bad));
}

__device__ __forceinline__ int64_t shfl_i64(int64_t v, int src) {
  const int lo = __shfl_sync(0xffffffffu, (int)(v & 0xffffffff), src);
  const int hi = __shfl_sync(0xffffffffu, (int)(v >> 32), src);
  return (int64_t)(((uint64_t)(uint32_t)hi << 32) | (uint32_t)lo);
}

// Warp reduce-scatter over NH per-thread values.  Each level halves the values a lane keeps (the lane
// with the level's bit set keeps the upper half) until kR remain; levels left over reduce across the
// lane pair.  Afterwards lane l holds the reduction over the warp's 32 threads of heads
// kR l .. kR l + kR - 1 (NH >= 32), or of head l / 2 (NH = 16, on lanes l and l ^ 1).
template <bool kMax, int NH>
__device__ __forceinline__ void reduce_scatter(const float (&v)[NH], int lane, float (&out)[Cfg<NH>::kR]) {
  constexpr int R = Cfg<NH>::kR;
  float a[NH / 2];
  {
    const bool hi = lane & 16;
#pragma unroll
    for (int i = 0; i < NH / 2; ++i) {
      const float send = hi ? v[i] : v[NH / 2 + i];
      const float keep = hi ? v[NH / 2 + i] : v[i];
      const float r = __shfl_xor_sync(0xffffffffu, send, 16);
      a[i] = kMax ? fmaxf(keep, r) : keep + r;
    }
  }
  int span = NH / 2;
#pragma unroll
  for (int x = 8; x >= 1; x >>= 1) {
    if (span > R) {
      const int half = span / 2;
      const bool hi = lane & x;
#pragma unroll
      for (int i = 0; i < NH / 4; ++i) {
        if (i < half) {
          const float send = hi ? a[i] : a[half + i];
          const float keep = hi ? a[half + i] : a[i];
          const float r = __shfl_xor_sync(0xffffffffu, send, x);
          a[i] = kMax ? fmaxf(keep, r) : keep + r;
        }
      }
      span = half;
    } else {
      const float r = __shfl_xor_sync(0xffffffffu, a[0], x);
      a[0] = kMax ? fmaxf(a[0], r) : a[0] + r;
    }
  }
#pragma unroll
  for (int r = 0; r < R; ++r) out[r] = a[r];
}

// Head of value r a lane holds after reduce_scatter.
template <int NH>
__device__ __forceinline__ int rs_head(int lane, int r) {
  return NH >= 32 ? Cfg<NH>::kR * lane + r : lane >> 1;
}

struct Ctx {
  const SplitParams* p;
  Misc* ms;
  volatile int* abort;
  uint32_t q_base, k_base;   // shared addresses
  uint32_t tmem;
  int b, g, split, pos0, pos_end, n_tiles, hg_valid;
};

// ------------------------------------------------------------------------------------------ gather
template <int NH, bool kOneTile>
__device__ __forceinline__ void gather_role(const Ctx& x, int warp, int lane) {
  using C = Cfg<NH>;
  const SplitParams& p = *x.p;
  Misc& ms = *x.ms;
  const int gw = warp - kSoftWarps;
  const int tl = kTokPerGatherWarp * gw + (lane & 15);   // token resolved by this lane (lanes 16.. repeat)
  const int seq_len = __ldg(p.seq_lens + x.b);
  const int32_t* bt_row = p.block_table + (size_t)(x.b / p.q_per_req) * p.max_pages;   // the query's request
  const int32_t* tk_row = p.topk + (size_t)x.b * p.topk_n;
  const unsigned char* kv = p.kv;
  const int blk = lane >> 3;               // scale block of this lane's 16 latent dims
  int range_bad = 0;
  bool ok = true;

  // the block-table row of the query into L2 (one 128-byte line per gather lane, up to 32 KB), so the
  // page lookups after the top-k loads see L2 latency
  {
    const int pages = min(p.max_pages, (seq_len + kPageSize - 1) / kPageSize);
    const int line = 32 * gw + lane;
    if (line * 32 < pages) ptx::prefetch_l2_line(bt_row + line * 32);
  }

  // Index -> row (a1) in three stages.  A top-k entry t is used when 0 <= t < seq_len; its
  // logical page t / 64 must lie in the block-table row and the physical page in the cache, else
  // the entry is skipped and flagged.
  auto topk_load = [&](int j) -> int {
    const int pos = x.pos0 + j * kTile + tl;
    return (j < x.n_tiles && pos < x.pos_end) ? ptx::ldg_i32_now(tk_row + pos) : -1;
  };
  auto page_load = [&](int t) -> int {      // block-table entry of t (load issued here), or 0 when t reads none
    return entry_reads_table(t, seq_len, p.max_pages) ? ptx::ldg_i32_now(bt_row + (t >> 6)) : 0;
  };
  auto row_from = [&](int t, int page) -> int64_t {
    return row_from_page(t, page, seq_len, p.max_pages, p.num_pages, p.err);
  };
  // the row this lane resolved for its entry of tile j (the row whose record the tile loads), written
  // out when the caller asked for the resolved rows
  auto record_row = [&](int j, int64_t r) {
    const int pos = x.pos0 + j * kTile + tl;
    if (p.rows_out && lane < 16 && j < x.n_tiles && pos < x.pos_end) p.rows_out[(size_t)x.b * p.topk_n + pos] = r;
  };

  // Record bytes of the warp's 16 tokens: load k reads token 16 gw + k's 512 code bytes (one
  // contiguous segment per warp load, lane l: dims 16 l .. 16 l + 15); rope: four tokens x 128
  // bytes per load; scales: lanes 0..15, one token each.
  uint4 lat[16], rope[4], sc;
  auto load_side = [&](int64_t r_own) {
    const int64_t off_own = r_own >= 0 ? r_own * kRecordBytes : -1;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int64_t off = shfl_i64(off_own, 4 * k + (lane >> 3));
      rope[k] = off >= 0 ? ptx::ldg_stream(kv + off + 528 + 16 * (lane & 7)) : make_uint4(0, 0, 0, 0);
    }
    sc = off_own >= 0 ? ptx::ldg_stream(kv + off_own + 512) : make_uint4(0, 0, 0, 0);
  };
  auto load_tile = [&](int64_t r_own) {
    const int64_t off_own = r_own >= 0 ? r_own * kRecordBytes : -1;
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const int64_t off = shfl_i64(off_own, k);
      lat[k] = off >= 0 ? ptx::ldg_stream(kv + off + 16 * lane) : make_uint4(0, 0, 0, 0);
    }
    load_side(r_own);
  };

  // Records of tile i + 2 are prefetched into L2 when tile i's are loaded into registers, so the
  // register loads (which L1 can hold only ~28 KB of) see L2 latency.
  auto prefetch_row = [&](int64_t r) {
    if (lane < 16 && r >= 0) ptx::prefetch_l2_bulk(kv + r * kRecordBytes, kRecordBytes);
  };
  // prologue: tile 0 resolved and its records in flight, tiles 1 and 2 prefetched; tile 3's page and
  // tile 4's entries in flight
  const int t0 = topk_load(0);
  int t1 = topk_load(1), t2 = topk_load(2), t3 = topk_load(3);
  const int pg0 = page_load(t0);
  int pg1 = page_load(t1), pg2 = page_load(t2);
  int64_t row = row_from(t0, pg0);
  record_row(0, row);
  // tile 0's codes by bulk copy into the idle K tile (register loads are bound by the loads an SM
  // keeps in flight, which a cold first tile feels most); its rope and scales by register loads.  No
  // L2 prefetch of tile 0: the bulk copies fetch its lines.
  const uint32_t raw0 = x.k_base + kRawLatOff;
  if (lane < 16) {
    if (row >= 0) {
      ptx::mbar_arrive_expect_tx(&ms.raw0, kDLatent);
      ptx::bulk_g2s(raw0 + (uint32_t)tl * kDLatent, kv + row * kRecordBytes, kDLatent, &ms.raw0);
    } else {
      ptx::mbar_arrive(&ms.raw0);
    }
  }
  load_side(row);
  if (x.n_tiles > 1) prefetch_row(row_from(t1, pg1));
  if (x.n_tiles > 2) prefetch_row(row_from(t2, pg2));
  int pg3 = page_load(t3);
  int t4 = topk_load(4);

  for (int i = 0; i < x.n_tiles; ++i) {
    const bool valid = row >= 0;
    // the K tile is free once every PV MMA of the previous tile is done
    if (i > 0) ok = ptx::mbar_wait_warp(&ms.pv_done, (i - 1) & 1, x.abort, lane, p.wait_ns) && ok;
    if (i == 0) {
      // tile 0's codes from the raw copy into registers; the K tile is written only once every gather
      // warp has read its codes and every softmax warp its raw Q
      ok = ptx::mbar_wait_warp(&ms.raw0, 0, x.abort, lane, p.wait_ns) && ok;
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const int64_t rk = shfl_i64(row, k);
        lat[k] = (ok && rk >= 0) ? ptx::lds128(raw0 + (uint32_t)(kTokPerGatherWarp * gw + k) * kDLatent + 16u * lane)
                                 : make_uint4(0, 0, 0, 0);
      }
      ptx::named_bar_sync(kGatherBar, kGatherWarps * 32);
      ok = ptx::mbar_wait_warp(&ms.k_free0, 0, x.abort, lane, p.wait_ns) && ok;
    }
    if (ok) {
      const float s4[4] = {__uint_as_float(sc.x), __uint_as_float(sc.y), __uint_as_float(sc.z),
                           __uint_as_float(sc.w)};
      uint32_t e[4];
      float inv_m0 = 0.f;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float mt = q == 0 ? pow2_split_b0(s4[0], e[0]) : pow2_split(s4[q], e[q]);
        if (q == 0) inv_m0 = __frcp_rn(mt);
        if (lane < 16) ms.mant[q][tl] = valid ? mt : 0.f;
        if (valid) range_bad |= !(fabsf(s4[q]) <= kMaxScale);
      }
      if (lane < 16) ms.valid[tl] = valid;
      const uint32_t e01 = e[0] | (e[1] << 16), e23 = e[2] | (e[3] << 16);
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const uint32_t a01 = __shfl_sync(0xffffffffu, e01, k), a23 = __shfl_sync(0xffffffffu, e23, k);
        const uint32_t pair = blk < 2 ? a01 : a23;
        const uint32_t h = (blk & 1) ? (pair >> 16) : (pair & 0xFFFFu);
        const uint32_t m2 = h | (h << 16);
        const uint32_t w[4] = {lat[k].x, lat[k].y, lat[k].z, lat[k].w};
        uint32_t hv[8];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          hv[2 * q] = hmul2(e4m3x2_to_f16x2((uint16_t)(w[q] & 0xFFFFu)), m2);
          hv[2 * q + 1] = hmul2(e4m3x2_to_f16x2((uint16_t)(w[q] >> 16)), m2);
        }
        const uint32_t t = kTokPerGatherWarp * gw + k;
        const uint32_t cb = x.k_base + (lane >> 2) * kKChunk;
        const uint32_t u0 = 2 * (lane & 3), sw = (lane >> 2) & 1;
        const uint4 lo4 = make_uint4(hv[0], hv[1], hv[2], hv[3]), hi4 = make_uint4(hv[4], hv[5], hv[6], hv[7]);
        // units u0, u0 + 1 in an order that keeps every 8 lanes of a store on distinct banks
        ptx::sts128_async_only(cb + swz128(t, u0 + sw), sw ? hi4 : lo4);
        ptx::sts128_async_only(cb + swz128(t, u0 + 1 - sw), sw ? lo4 : hi4);
      }
      // the rope, divided by the token's block-0 mantissa: its MMAs accumulate into block 0's scores,
      // which the softmax scales by mant_0
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint32_t t = kTokPerGatherWarp * gw + 4 * k + (lane >> 3);
        const float f = __shfl_sync(0xffffffffu, inv_m0, 4 * k + (lane >> 3));
        ptx::sts128_async_only(x.k_base + kRopeChunk * kKChunk + swz128(t, lane & 7),
                               bf8_scaled_to_h8(rope[k], f, range_bad));
      }
    }
    // the tile is written: signal it, and only then put the next loads in flight (a fence or a
    // barrier after them would wait for them)
    ptx::fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(&ms.tile_full);
    // tile i + 1's records, tile i + 3's into L2, tile i + 4's pages, tile i + 5's entries
    row = row_from(t1, pg1);
    record_row(i + 1, row);
    if (i + 1 < x.n_tiles) load_tile(row);
    if (i + 3 < x.n_tiles) prefetch_row(row_from(t3, pg3));
    t1 = t2; pg1 = pg2;
    t2 = t3; pg2 = pg3;
    t3 = t4;
    pg3 = page_load(t4);
    t4 = topk_load(i + 5);
  }
  if (range_bad) ms.range_err = 1;
  if constexpr (kOneTile) {
    if (gw == 0) {
      // the tile's QK (one elected lane): latent block b into score buffer b, the rope (stored as
      // rope / mant_0) into buffer 0 after block 0, once every gather warp has written the tile
      ok = ptx::mbar_wait_warp(&ms.q_ready, 0, x.abort, lane, p.wait_ns) && ok;
      ok = ptx::mbar_wait_warp(&ms.tile_full, 0, x.abort, lane, p.wait_ns) && ok;
      if (ok) {
        ptx::tc_fence_after();
        if (ptx::elect_one()) {
          const uint64_t dK = desc_qk_operand(x.k_base), dQ = desc_qk_operand(x.q_base);
          issue_qk<NH, 0, 2>(x.tmem + C::kSCol, dK, dQ);
          issue_qk<NH, kRopeChunk, 1, true>(x.tmem + C::kSCol, dK, dQ);
          ptx::mma_commit(&ms.s_full[0]);
          issue_qk<NH, 2, 2>(x.tmem + C::kSCol + NH, dK, dQ);
          ptx::mma_commit(&ms.s_full[1]);
          issue_qk<NH, 4, 2>(x.tmem + C::kSCol + 2 * NH, dK, dQ);
          ptx::mma_commit(&ms.s_full[2]);
          issue_qk<NH, 6, 2>(x.tmem + C::kSCol + 3 * NH, dK, dQ);
          ptx::mma_commit(&ms.s_full[3]);
        }
        __syncwarp();
      }
      // the QK MMAs are complete when this commit arrives (one of the two teardown arrivals)
      if (ptx::elect_one()) ptx::mma_commit(&ms.teardown);
      __syncwarp();
    }
  }
}

// ------------------------------------------------------------------------------------------ softmax
template <int NH, bool kOneTile>
__device__ __forceinline__ void softmax_role(const Ctx& x, int warp, int lane) {
  using C = Cfg<NH>;
  constexpr int R = C::kR;
  const SplitParams& p = *x.p;
  Misc& ms = *x.ms;
  const int t = threadIdx.x;                 // token of the tile = TMEM lane
  const bool issue_warp = (warp == 0);       // one elected lane of warp 0 issues every MMA
  const uint32_t lane_q = (uint32_t)(32 * warp) << 16;
  int range_bad = 0;
  bool ok = true, mma_ok = true;

  {
    // Q head group -> fp16, 128B-swizzled, zero rows past the valid heads: NH rows x 72 16-byte units,
    // read from the raw bf16 rows the bulk copy put at the start of the K tile (unit id at 16 id)
    ok = ptx::mbar_wait_warp(&ms.q_raw, 0, x.abort, lane, p.wait_ns) && ok;
    constexpr int kUnits = NH * 72 / kSoftThreads;   // per thread: 9, 18 or 36
    constexpr int kBatch = kUnits < 18 ? kUnits : 18;
#pragma unroll 1
    for (int k0 = 0; k0 < kUnits; k0 += kBatch) {
      uint4 v[kBatch];
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        const int id = t + kSoftThreads * (k0 + k), n = id / 72;
        v[k] = (ok && n < x.hg_valid) ? ptx::lds128(x.k_base + 16u * (uint32_t)id) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        const int id = t + kSoftThreads * (k0 + k), n = id / 72, j = id % 72;
        ptx::sts128_async_only(x.q_base + chunked_offset(C::kQChunk, n, j), bf8_to_h8(v[k], range_bad));
      }
    }
    ptx::fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      ptx::mbar_arrive(&ms.k_free0);   // the raw Q is read: the gather warps may overwrite it
      ptx::mbar_arrive(&ms.q_ready);
    }
  }

  const float c2 = p.sm_scale * 1.4426950408889634f;
  float lsum[R];                             // this warp's row sums of the heads rs_head(lane, r)
#pragma unroll
  for (int r = 0; r < R; ++r) lsum[r] = 0.f;
  const uint32_t bufR = x.k_base + kRopeChunk * kKChunk, buf0 = x.k_base, buf1 = x.k_base + kKChunk;
  const uint64_t dK = desc_qk_operand(x.k_base), dQ = desc_qk_operand(x.q_base);
  const uint64_t dV = desc_v(x.k_base);      // K tile as the MN-major A of PV
  const uint64_t dBufR = desc_pm<NH>(bufR), dBuf0 = desc_pm<NH>(buf0), dBuf1 = desc_pm<NH>(buf1);

  for (int i = 0; i < x.n_tiles; ++i) {
    const uint32_t ph = i & 1;
    ok = ptx::mbar_wait_warp(&ms.tile_full, ph, x.abort, lane, p.wait_ns) && ok;
    const bool valid = ms.valid[t];
    float mant[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) mant[q] = ms.mant[q][t];
    // QK of latent block b into score buffer b, the rope (stored as rope / mant_0) into buffer 0
    // after block 0; all 36 MMAs in one batch (issued by gather warp 0 in one-tile launches)
    if (issue_warp && !kOneTile) {
      if (i == 0) mma_ok = mma_ok && ptx::mbar_wait_warp(&ms.q_ready, 0, x.abort, lane, p.wait_ns);
      mma_ok = mma_ok && ok;
      if (mma_ok) {
        ptx::tc_fence_after();
        if (ptx::elect_one()) {
          issue_qk<NH, 0, 2>(x.tmem + C::kSCol, dK, dQ);
          issue_qk<NH, kRopeChunk, 1, true>(x.tmem + C::kSCol, dK, dQ);
          ptx::mma_commit(&ms.s_full[0]);
          issue_qk<NH, 2, 2>(x.tmem + C::kSCol + NH, dK, dQ);
          ptx::mma_commit(&ms.s_full[1]);
          issue_qk<NH, 4, 2>(x.tmem + C::kSCol + 2 * NH, dK, dQ);
          ptx::mma_commit(&ms.s_full[2]);
          issue_qk<NH, 6, 2>(x.tmem + C::kSCol + 3 * NH, dK, dQ);
          ptx::mma_commit(&ms.s_full[3]);
        }
        __syncwarp();
      }
    }
    __syncwarp();
    float s[NH];
#pragma unroll
    for (int h = 0; h < NH; ++h) s[h] = 0.f;
    // scores s = sum_b mant_b S_b (the rope is inside S_0), buffers in the order they complete
#pragma unroll 1
    for (int bb = 0; bb < 4; ++bb) {
      ok = ptx::mbar_wait_warp(&ms.s_full[bb], ph, x.abort, lane, p.wait_ns) && ok;
      if (ok) {
        ptx::tc_fence_after();
        const float f = c2 * (bb == 0 ? mant[0] : bb == 1 ? mant[1] : bb == 2 ? mant[2] : mant[3]);
        const uint32_t sa = x.tmem + lane_q + C::kSCol + NH * bb;
        if constexpr (NH == 16) {
          uint32_t r0[16];
          ptx::tmem_ld16(sa, r0);
          ptx::tmem_wait_ld();
#pragma unroll
          for (int h = 0; h < 16; ++h) s[h] = fmaf(f, __uint_as_float(r0[h]), s[h]);
        } else {
#pragma unroll
          for (int hh = 0; hh < NH; hh += 64) {
            uint32_t r0[32], r1[32];
            ptx::tmem_ld32(sa + hh, r0);
            if (NH - hh > 32) ptx::tmem_ld32(sa + hh + 32, r1);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int h = 0; h < 32; ++h) {
              s[hh + h] = fmaf(f, __uint_as_float(r0[h]), s[hh + h]);
              if (NH - hh > 32) s[hh + 32 + h] = fmaf(f, __uint_as_float(r1[h]), s[hh + 32 + h]);
            }
          }
        }
      }
    }
#pragma unroll
    for (int h = 0; h < NH; ++h) s[h] = (ok && valid) ? s[h] : -CUDART_INF_F;
    bool need = false;
    if (i > 0) {
#pragma unroll
      for (int k = 0; k < NH / 4; ++k) {
        const float4 m = reinterpret_cast<const float4*>(ms.m_ref)[k];
        need |= (s[4 * k] > m.x + kRescaleThreshold) | (s[4 * k + 1] > m.y + kRescaleThreshold) |
                (s[4 * k + 2] > m.z + kRescaleThreshold) | (s[4 * k + 3] > m.w + kRescaleThreshold);
      }
      need = ptx::named_bar_or(3, kSoftThreads, need);
    }
    if (i == 0) {
      // first tile: a head's reference max is its tile max (no vote, nothing to rescale yet)
      float mx[R];
      reduce_scatter<true, NH>(s, lane, mx);
#pragma unroll
      for (int r = 0; r < R; ++r)
        if (NH >= 32 || (lane & 1) == 0) ms.red[warp][rs_head<NH>(lane, r)] = mx[r];
      ptx::named_bar_sync(2, kSoftThreads);
      if (warp == 0) {
        for (int h = lane; h < NH; h += 32)
          ms.m_ref[h] = fmaxf(fmaxf(ms.red[0][h], ms.red[1][h]), fmaxf(ms.red[2][h], ms.red[3][h]));
      }
      ptx::named_bar_sync(2, kSoftThreads);
    } else if (need) {
      // a head's reference max moves to its tile max when that exceeds it by more than the threshold
      float mx[R];
      reduce_scatter<true, NH>(s, lane, mx);
#pragma unroll
      for (int r = 0; r < R; ++r)
        if (NH >= 32 || (lane & 1) == 0) ms.red[warp][rs_head<NH>(lane, r)] = mx[r];
      ptx::named_bar_sync(2, kSoftThreads);
      if (warp == 0) {
        for (int h = lane; h < NH; h += 32) {
          const float tm = fmaxf(fmaxf(ms.red[0][h], ms.red[1][h]), fmaxf(ms.red[2][h], ms.red[3][h]));
          const float mo = ms.m_ref[h];
          const float mn = tm > mo + kRescaleThreshold ? tm : mo;
          ms.alpha[h] = mo == -CUDART_INF_F ? 0.f : ptx::ex2_approx(mo - mn);
          ms.m_new[h] = mn;
        }
      }
      ptx::named_bar_sync(2, kSoftThreads);
#pragma unroll
      for (int r = 0; r < R; ++r) lsum[r] *= ms.alpha[rs_head<NH>(lane, r)];
      if (i > 0 && ok) {
        // O of the previous tiles (their PV is complete: this tile's K was written after it)
#pragma unroll 1
        for (int c = 0; c < C::kChunks; ++c) {
          const uint32_t oa = x.tmem + lane_q + C::kChunkCols * c;
          const int h0 = (C::kChunkCols * c) % NH;
          if constexpr (NH == 16) {
            uint32_t r[16];
            ptx::tmem_ld16(oa, r);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int h = 0; h < 16; ++h) r[h] = __float_as_uint(__uint_as_float(r[h]) * ms.alpha[h]);
            ptx::tmem_st16(oa, r);
          } else {
            uint32_t r[32];
            ptx::tmem_ld32(oa, r);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int h = 0; h < 32; ++h) r[h] = __float_as_uint(__uint_as_float(r[h]) * ms.alpha[h0 + h]);
            ptx::tmem_st32(oa, r);
          }
        }
        ptx::tmem_wait_st();
      }
      ptx::named_bar_sync(2, kSoftThreads);
      if (warp == 0) {
        for (int h = lane; h < NH; h += 32) ms.m_ref[h] = ms.m_new[h];
      }
      ptx::named_bar_sync(2, kSoftThreads);
    }
    // P = exp2(s - m) (a head with no valid entry yet has m = -inf and P = 0), fp16 pairs
    uint32_t ph2[NH / 2];
#pragma unroll
    for (int k = 0; k < NH / 4; ++k) {
      const float4 m = reinterpret_cast<const float4*>(ms.m_ref)[k];
      const float mm[4] = {m.x, m.y, m.z, m.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int h = 4 * k + q;
        s[h] = mm[q] == -CUDART_INF_F ? 0.f : ptx::ex2_approx(s[h] - mm[q]);
      }
      ph2[2 * k] = f32x2_to_f16x2_sat(s[4 * k], s[4 * k + 1]);
      ph2[2 * k + 1] = f32x2_to_f16x2_sat(s[4 * k + 2], s[4 * k + 3]);
    }

    // PV: P * mant_0 into the rope chunk (free: the QK is complete), block 0's 8 MMAs; then P * mant
    // of blocks 1..3 into chunks 0 and 1 and the rope chunk (free once block 0's PV is done)
    auto write_pm = [&](int bb, uint32_t buf) {
      const float mb = bb == 0 ? mant[0] : bb == 1 ? mant[1] : bb == 2 ? mant[2] : mant[3];
      const uint32_t m2 = f32x2_to_f16x2_sat(mb, mb);
#pragma unroll
      for (int u = 0; u < C::kPUnits; ++u)
        ptx::sts128_async_only(buf + swz_row<C::kPRow>(t, u),
                               make_uint4(hmul2(ph2[4 * u], m2), hmul2(ph2[4 * u + 1], m2),
                                          hmul2(ph2[4 * u + 2], m2), hmul2(ph2[4 * u + 3], m2)));
    };
    write_pm(0, bufR);
    ptx::fence_proxy_async_smem();
    ptx::tc_fence_before();
    ptx::named_bar_sync(2, kSoftThreads);
    if (issue_warp) {
      mma_ok = mma_ok && ok;
      if (mma_ok) {
        ptx::tc_fence_after();
        if (ptx::elect_one()) {
          issue_pv<NH, 0>(x.tmem, dV, dBufR, i > 0);
          ptx::mma_commit(&ms.pv0_done);
        }
        __syncwarp();
      }
    }
    // row sums, while block 0's PV runs
    {
      float ps[R];
      reduce_scatter<false, NH>(s, lane, ps);
#pragma unroll
      for (int r = 0; r < R; ++r) lsum[r] += ps[r];
    }
    ok = ptx::mbar_wait_warp(&ms.pv0_done, ph, x.abort, lane, p.wait_ns) && ok;
    write_pm(1, buf0);
    write_pm(2, bufR);
    write_pm(3, buf1);
    ptx::fence_proxy_async_smem();
    ptx::named_bar_sync(2, kSoftThreads);
    if (issue_warp && mma_ok) {
      ptx::tc_fence_after();
      if (ptx::elect_one()) {
        issue_pv<NH, 1>(x.tmem, dV, dBuf0, i > 0);
        issue_pv<NH, 2>(x.tmem, dV, dBufR, i > 0);
        issue_pv<NH, 3>(x.tmem, dV, dBuf1, i > 0);
        ptx::mma_commit(&ms.pv_done);
      }
      __syncwarp();
    }
  }
  if (range_bad) ms.range_err = 1;
  if (issue_warp) {
    if (ptx::elect_one()) ptx::mma_commit(&ms.teardown);
    __syncwarp();
  }
#pragma unroll
  for (int r = 0; r < R; ++r)
    if (NH >= 32 || (lane & 1) == 0) ms.red[warp][rs_head<NH>(lane, r)] = lsum[r];
}

// ------------------------------------------------------------------------------------------ epilogue
// All 12 warps write O / l from TMEM straight to the output rows [head][512] (bf16, or fp32
// partials): warp w reads TMEM lane quadrant w % 4 (dims 32 (w % 4) .. of each 128-dim block) and the
// column chunks c = w / 4, w / 4 + 3, ... of O^T (chunks of 32 columns, 16 for NH = 16; block
// c * cols / NH).  Lanes 2j, 2j + 1 hold dims d, d + 1; for heads h, h + 1 the even lane writes row h
// and the odd lane row h + 1, two dims each.
template <int NH>
__device__ __forceinline__ void epilogue_write(const Ctx& x, int warp, int lane) {
  using C = Cfg<NH>;
  constexpr int kCols = C::kChunkCols;
  const SplitParams& p = *x.p;
  Misc& ms = *x.ms;
  const int quad = warp & 3;
  const uint32_t lane_q = (uint32_t)(32 * quad) << 16;
  const bool odd = lane & 1;
  const size_t head0 = (size_t)x.g * NH;
#pragma unroll 1
  for (int c = warp >> 2; c < C::kChunks; c += 3) {
    const int jb = (kCols * c) / NH, hb = (kCols * c) % NH;
    uint32_t r[kCols];
    if constexpr (kCols == 16) ptx::tmem_ld16(x.tmem + lane_q + kCols * c, r);
    else ptx::tmem_ld32(x.tmem + lane_q + kCols * c, r);
    float v[kCols];
#pragma unroll
    for (int k = 0; k < kCols / 4; ++k) {
      const float4 l4 = reinterpret_cast<const float4*>(ms.linv + hb)[k];
      v[4 * k] = l4.x; v[4 * k + 1] = l4.y; v[4 * k + 2] = l4.z; v[4 * k + 3] = l4.w;
    }
    ptx::tmem_wait_ld();
#pragma unroll
    for (int h = 0; h < kCols; ++h) v[h] *= __uint_as_float(r[h]);
    const int d0 = 128 * jb + 32 * quad + (lane & ~1);
#pragma unroll
    for (int h = 0; h < kCols; h += 2) {
      const float mine = odd ? v[h + 1] : v[h];
      const float other = __shfl_xor_sync(0xffffffffu, odd ? v[h] : v[h + 1], 1);
      const float lo = odd ? other : mine, hi = odd ? mine : other;   // dims d0, d0 + 1
      const int hl = hb + h + (odd ? 1 : 0);
      if (hl < x.hg_valid) {
        if (p.final_out) {
          uint16_t* dst = p.out + ((size_t)x.b * p.H + head0 + hl) * kDLatent + d0;
          *reinterpret_cast<uint32_t*>(dst) = f32x2_to_bf16x2(lo, hi);
        } else {
          float* dst = p.o_part + (((size_t)x.b * p.nsplit + x.split) * p.H + head0 + hl) * kDLatent + d0;
          *reinterpret_cast<float2*>(dst) = make_float2(lo, hi);
        }
      }
    }
  }
}

// O / l from TMEM: rows of heads outside [keep_lo, keep_lo + keep_n) go straight to global memory at dst
// (row h at dst + h * 512 elements: fp32, or fp16 when kHalf), rows inside it are staged in fp32 in shared
// memory at `stage` (row h - keep_lo, 2048 bytes each).  Warp w reads TMEM lane quadrant w % 4 and the
// column chunks w / 4, w / 4 + 3, ... of O^T (as epilogue_write); lanes 2j, 2j + 1 hold dims d, d + 1 and
// exchange one value per head pair, so each global store writes two dims of one row.
template <int NH, bool kHalf>
__device__ __forceinline__ void write_rows(const Ctx& x, int warp, int lane, void* dst, int rows, uint32_t stage,
                                           int keep_lo, int keep_n) {
  using C = Cfg<NH>;
  constexpr int kCols = C::kChunkCols;
  const Misc& ms = *x.ms;
  const int quad = warp & 3;
  const uint32_t lane_q = (uint32_t)(32 * quad) << 16;
  const bool odd = lane & 1;
#pragma unroll 1
  for (int c = warp >> 2; c < C::kChunks; c += 3) {
    const int jb = (kCols * c) / NH, hb = (kCols * c) % NH;
    uint32_t r[kCols];
    if constexpr (kCols == 16) ptx::tmem_ld16(x.tmem + lane_q + kCols * c, r);
    else ptx::tmem_ld32(x.tmem + lane_q + kCols * c, r);
    float v[kCols];
#pragma unroll
    for (int k = 0; k < kCols / 4; ++k) {
      const float4 l4 = reinterpret_cast<const float4*>(ms.linv + hb)[k];
      v[4 * k] = l4.x; v[4 * k + 1] = l4.y; v[4 * k + 2] = l4.z; v[4 * k + 3] = l4.w;
    }
    ptx::tmem_wait_ld();
#pragma unroll
    for (int h = 0; h < kCols; ++h) v[h] *= __uint_as_float(r[h]);
    const uint32_t d = 128 * jb + 32 * quad + lane;
    const int d0 = (int)(d & ~1u);
#pragma unroll
    for (int h = 0; h < kCols; h += 2) {
      const int h0 = hb + h;                  // a head pair lies inside or outside the kept range together
      if (h0 >= keep_lo && h0 < keep_lo + keep_n) {
        ptx::sts32f(stage + (uint32_t)(h0 - keep_lo) * 2048u + 4u * d, v[h]);
        ptx::sts32f(stage + (uint32_t)(h0 + 1 - keep_lo) * 2048u + 4u * d, v[h + 1]);
      } else {
        const float mine = odd ? v[h + 1] : v[h];
        const float other = __shfl_xor_sync(0xffffffffu, odd ? v[h] : v[h + 1], 1);
        const int hl = h0 + (odd ? 1 : 0);
        const float lo = odd ? other : mine, hi = odd ? mine : other;   // dims d0, d0 + 1
        if (hl < rows) {
          if constexpr (kHalf)
            *reinterpret_cast<uint32_t*>(static_cast<uint16_t*>(dst) + (size_t)hl * kDLatent + d0) =
                f32x2_to_f16x2_sat(lo, hi);
          else
            *reinterpret_cast<float2*>(static_cast<float*>(dst) + (size_t)hl * kDLatent + d0) = make_float2(lo, hi);
        }
      }
    }
  }
}

// Merge of the partitions inside the kernel ("The 64-Block Barrier", "The Split-K Prescription": the
// partial results combined by an online-softmax merge), for a launch whose nsplit CTAs of one (query,
// head group) form a thread-block cluster (rank = partition s).  CTA s owns the heads [s L, s L + L) of the
// group, L = NH / nsplit:
//   1. every CTA pushes its partition's lse of each head into the CTA that owns the head (distributed
//      shared memory), writes its normalised partial rows O_s / l_s of the other CTAs' heads into the workspace in
//      fp16 (a convex combination of dequantised latents, which stay inside the fp16 range; the rounding is
//      2^-11 relative against the 5e-3 output tolerance, and halves the exchange that bounds this step),
//      and stages those of its own heads in fp32 in shared memory; one cluster barrier (release / acquire)
//      makes all of it visible;
//   2. every CTA bulk-loads, for its own heads, the partial rows of every peer whose partition holds a
//      valid entry (a partition is empty for all heads or for none), and writes
//      out = sum_s exp(lse_s - lse) O_s / l_s (bf16) and lse = ln sum_s exp(lse_s) for them.
// A partition with no valid entry, or whose CTA gave up a wait, counts as lse = -inf (weight 0); every
// CTA takes the cluster barriers whatever happened, so no CTA waits on one that left.
template <int NH>
__device__ __forceinline__ void fused_merge(const Ctx& x, int warp, int lane, bool own_ok) {
  const SplitParams& p = *x.p;
  Misc& ms = *x.ms;
  const int S = p.nsplit, s = x.split, L = NH / S;
  const uint32_t stage = x.k_base;            // own rows at 0, then one L-row block per peer
  const int t = threadIdx.x;
  // 1. (the split cluster barrier started at kernel start completes here: every peer's shared memory exists)
  ptx::cluster_wait();
  const bool own_rows = own_ok && ms.lse_out[0] != -CUDART_INF_F;
  if (t < NH) {
    const float l = own_ok ? ms.lse_out[t] : -CUDART_INF_F;
    const int r = t / L, i = t % L;          // owner of head t and its index there
    ptx::st_cluster_f32(ptx::mapa(ptx::smem_u32(&ms.lse_in[s * L + i]), (uint32_t)r), l);
  }
  // the fp16 rows of partition r: [B][nsplit][H][512] fp16 in the workspace's partial area
  uint16_t* part16 = reinterpret_cast<uint16_t*>(p.o_part);
  if (own_rows)
    write_rows<NH, true>(x, warp, lane, part16 + (((size_t)x.b * S + s) * p.H + (size_t)x.g * NH) * kDLatent, NH,
                         stage, s * L, L);
  ptx::cluster_sync_all();
  // 2. the peers' rows of this CTA's heads (fp16, after the own fp32 rows)
  const uint32_t peers = stage + (uint32_t)L * 2048u;
  if (t == 0) {
    ptx::fence_proxy_async_global();
    uint32_t bytes = 0;
    for (int r = 0; r < S; ++r)
      if (r != s && ms.lse_in[r * L] != -CUDART_INF_F) bytes += (uint32_t)L * 1024u;
    if (bytes) {
      ptx::mbar_arrive_expect_tx(&ms.merge_in, bytes);
      for (int r = 0, k = 0; r < S; ++r) {
        if (r == s) continue;
        if (ms.lse_in[r * L] != -CUDART_INF_F) {
          const uint16_t* src = part16 + (((size_t)x.b * S + r) * p.H + (size_t)x.g * NH + (size_t)s * L) * kDLatent;
          ptx::bulk_g2s(peers + (uint32_t)(k * L) * 1024u, src, (uint32_t)L * 1024u, &ms.merge_in);
        }
        ++k;
      }
    } else {
      ptx::mbar_arrive(&ms.merge_in);
    }
  }
  if (t < L) {
    // merged lse and the weights of every partition for head s L + t
    float mx = -CUDART_INF_F;
    for (int r = 0; r < S; ++r) mx = fmaxf(mx, ms.lse_in[r * L + t]);
    float z = 0.f;
    if (mx != -CUDART_INF_F)
      for (int r = 0; r < S; ++r) z += expf(ms.lse_in[r * L + t] - mx);   // exp(-inf) = 0 for empty partitions
    const float lse = mx == -CUDART_INF_F ? -CUDART_INF_F : mx + logf(z);
    ms.lse_merged[t] = lse;
    for (int r = 0; r < S; ++r) {
      const float l = ms.lse_in[r * L + t];
      ms.wts[r * L + t] = (lse == -CUDART_INF_F || l == -CUDART_INF_F) ? 0.f : expf(l - lse);
    }
  }
  const bool in_ok = ptx::mbar_wait_bounded(&ms.merge_in, 0, x.abort, p.wait_ns);
  const bool ok = __syncthreads_and(in_ok) != 0;
  if (!ok) return;                           // flagged at teardown (abort)
  uint16_t* out = p.out + ((size_t)x.b * p.H + (size_t)x.g * NH + (size_t)s * L) * kDLatent;
  for (int id = t; id < L * (kDLatent / 4); id += kThreads) {
    const int i = id / (kDLatent / 4), j = id % (kDLatent / 4);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int r = 0, k = 0; r < S; ++r) {
      const float w = ms.wts[r * L + i];
      float4 v;
      if (r == s) {
        if (w == 0.f) continue;              // an empty partition: its rows are not read
        v = ptx::lds128f(stage + (uint32_t)i * 2048u + 16u * j);
      } else {
        const uint32_t row = peers + (uint32_t)(k * L + i) * 1024u;
        ++k;
        if (w == 0.f) continue;
        const uint2 hv = ptx::lds64(row + 8u * j);
        const float2 a = f16x2_to_f32x2(hv.x), b2 = f16x2_to_f32x2(hv.y);
        v = make_float4(a.x, a.y, b2.x, b2.y);
      }
      acc.x = fmaf(w, v.x, acc.x); acc.y = fmaf(w, v.y, acc.y);
      acc.z = fmaf(w, v.z, acc.z); acc.w = fmaf(w, v.w, acc.w);
    }
    reinterpret_cast<uint2*>(out + (size_t)i * kDLatent)[j] =
        make_uint2(f32x2_to_bf16x2(acc.x, acc.y), f32x2_to_bf16x2(acc.z, acc.w));
  }
  if (t < L) p.lse[(size_t)x.b * p.H + (size_t)x.g * NH + (size_t)s * L + t] = ms.lse_merged[t];
}

// kFused: the partitions of a (query, head group) form a cluster and merge inside the kernel; a separate
// instantiation, so that the other launches carry none of that code.  kOneTile: every partition holds at
// most one tile (gather warp 0 issues its QK); also a separate instantiation, as the extra issue path
// costs the multi-tile loop registers.
template <int NH, bool kFused, bool kOneTile>
__global__ void __launch_bounds__(kThreads, 1) split_kernel(const SplitParams p) {
  using C = Cfg<NH>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Misc& ms = *reinterpret_cast<Misc*>(base + C::kMiscOff);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the merge (launched as a programmatic dependent) may be scheduled now: it waits for this grid
  if (threadIdx.x == 0) ptx::griddep_launch_dependents();

  Ctx x;
  x.p = &p;
  x.ms = &ms;
  x.abort = &ms.abort;
  x.q_base = ptx::smem_u32(base);
  x.k_base = x.q_base + C::kKBase;
  x.split = blockIdx.x;
  x.g = blockIdx.y;
  x.b = blockIdx.z;
  x.pos0 = x.split * p.split_len;
  x.pos_end = min(x.pos0 + p.split_len, p.topk_n);
  x.n_tiles = x.pos_end > x.pos0 ? (x.pos_end - x.pos0 + kTile - 1) / kTile : 0;
  x.hg_valid = min(NH, p.H - NH * x.g);

  if (x.n_tiles == 0) {
    if constexpr (kFused) {
      // an empty partition still owns a head slice of the merge: weight 0 for its own rows
      if (threadIdx.x == 0) {
        ptx::mbar_init(&ms.merge_in, 1);
        ms.abort = 0;
        ptx::fence_mbar_init();
      }
      ptx::cluster_arrive_relaxed();
      __syncthreads();
      ptx::griddep_wait();
      fused_merge<NH>(x, warp, lane, false);
      if (threadIdx.x == 0 && ms.abort) {
        // the merge's bulk loads into this CTA land before it leaves (time limit only)
        volatile int no_abort = 0;
        ptx::mbar_wait_bounded(&ms.merge_in, 0, &no_abort, 100000000ull);
        if (p.err) atomicOr(p.err, SMLA_DEVERR_TIMEOUT);
      }
      __syncthreads();
      return;
    }
    // empty partition: out = 0, lse = -inf
    ptx::griddep_wait();
    for (int i = threadIdx.x; i < x.hg_valid * kDLatent; i += kThreads) {
      const size_t h = (size_t)x.g * NH + i / kDLatent;
      const int d = i % kDLatent;
      if (p.final_out) p.out[((size_t)x.b * p.H + h) * kDLatent + d] = 0;
      else p.o_part[(((size_t)x.b * p.nsplit + x.split) * p.H + h) * kDLatent + d] = 0.f;
    }
    if ((int)threadIdx.x < x.hg_valid) {
      const size_t h = (size_t)x.g * NH + threadIdx.x;
      if (p.final_out) p.lse[(size_t)x.b * p.H + h] = -CUDART_INF_F;
      else p.lse_part[((size_t)x.b * p.nsplit + x.split) * p.H + h] = -CUDART_INF_F;
    }
    return;
  }

  if (threadIdx.x == 0) {
    ptx::mbar_init(&ms.q_raw, 1);
    ptx::mbar_init(&ms.raw0, kGatherWarps * 16);
    ptx::mbar_init(&ms.k_free0, kSoftWarps);
    ptx::mbar_init(&ms.q_ready, kSoftWarps);
    ptx::mbar_init(&ms.tile_full, kGatherWarps);
    for (int bb = 0; bb < 4; ++bb) ptx::mbar_init(&ms.s_full[bb], 1);
    ptx::mbar_init(&ms.pv0_done, 1);
    ptx::mbar_init(&ms.pv_done, 1);
    ptx::mbar_init(&ms.teardown, kOneTile ? 2 : 1);   // one commit from each MMA-issuing thread
    ptx::mbar_init(&ms.merge_in, 1);
    ms.abort = 0;
    ms.range_err = 0;
    ptx::fence_mbar_init();
  }
  if (threadIdx.x < kHeadsMax) ms.m_ref[threadIdx.x] = -CUDART_INF_F;
  if (warp == 0) {
    ptx::tmem_alloc(&ms.tmem_slot, C::kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  x.tmem = ms.tmem_slot;
  if constexpr (kFused) ptx::cluster_arrive_relaxed();   // waited for before the merge writes into the peers
  // launched as a programmatic dependent: the setup above overlapped the previous kernel's tail;
  // nothing in global memory (inputs it may have written, partials it may still read) is touched
  // before that kernel has completed
  ptx::griddep_wait();
  if (threadIdx.x == 0) {
    // the head group's raw Q rows (contiguous, 1152 bytes each) into the idle K tile
    const uint32_t qbytes = (uint32_t)x.hg_valid * kDQK * 2;
    ptx::mbar_arrive_expect_tx(&ms.q_raw, qbytes);
    ptx::bulk_g2s(x.k_base, p.q + ((size_t)x.b * p.H + (size_t)x.g * NH) * kDQK, qbytes, &ms.q_raw);
  }

  if (warp >= kSoftWarps) gather_role<NH, kOneTile>(x, warp, lane);
  else softmax_role<NH, kOneTile>(x, warp, lane);

  // ------------------------------------------------------------------ epilogue
  bool ok = ptx::mbar_wait_warp(&ms.pv_done, (x.n_tiles - 1) & 1, x.abort, lane, p.wait_ns);
  ptx::tc_fence_after();
  __syncthreads();                           // row sums of the softmax warps are in ms.red
  if (threadIdx.x < NH) {
    const int h = threadIdx.x;
    const float L = ms.red[0][h] + ms.red[1][h] + ms.red[2][h] + ms.red[3][h];
    ms.linv[h] = L > 0.f ? 1.f / L : 0.f;
    ms.lse_out[h] = L > 0.f ? (ms.m_ref[h] + log2f(L)) * 0.6931471805599453f : -CUDART_INF_F;
  }
  __syncthreads();
  const bool out_ok = ok && !ms.abort;      // the same for every thread (any failed wait set ms.abort)
  if constexpr (kFused) {
    fused_merge<NH>(x, warp, lane, out_ok);
  } else if (out_ok) {
    epilogue_write<NH>(x, warp, lane);
    if ((int)threadIdx.x < x.hg_valid) {
      const int hl = threadIdx.x;
      const size_t h = (size_t)x.g * NH + hl;
      if (p.final_out) p.lse[(size_t)x.b * p.H + h] = ms.lse_out[hl];
      else p.lse_part[((size_t)x.b * p.nsplit + x.split) * p.H + h] = ms.lse_out[hl];
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (threadIdx.x == 0) {
    // every MMA has completed before TMEM is released (time limit only)
    volatile int no_abort = 0;
    bool drained = ptx::mbar_wait_bounded(&ms.teardown, 0, &no_abort, 100000000ull);
    if (ms.abort) {
      // a wait gave up: the first tile's bulk copies into shared memory may still be in flight, so they
      // are waited for (time limit only) before the CTA leaves
      drained = ptx::mbar_wait_bounded(&ms.q_raw, 0, &no_abort, 100000000ull) && drained;
      drained = ptx::mbar_wait_bounded(&ms.raw0, 0, &no_abort, 100000000ull) && drained;
      // the merge's bulk loads into this CTA (always armed in fused_merge) likewise
      if constexpr (kFused) drained = ptx::mbar_wait_bounded(&ms.merge_in, 0, &no_abort, 100000000ull) && drained;
    }
    if (p.err) {
      if (ms.abort || !drained) atomicOr(p.err, SMLA_DEVERR_TIMEOUT);
      if (ms.range_err) atomicOr(p.err, SMLA_DEVERR_RANGE);
    }
  }
  __syncthreads();
  if (warp == 0) ptx::tmem_dealloc(x.tmem, C::kTmemCols);
}

}  // namespace

bool split_shape_supported(int H, int topk) {
  return (H == 16 || H == 32 || H == 64 || H == 128) && topk >= 1 && topk <= kMaxTopk;
}

bool split_heads_supported(int nh) { return nh == 16 || nh == 32 || nh == 64; }

int split_ctas_per_unit() { return 1; }

bool split_fusable(int nsplit, int nh, int H) {
  return nsplit >= 2 && nsplit <= kMaxFusedSplit && nh % nsplit == 0 && nh <= H;
}

int split_ctas_per_sm(int H) {
  (void)H;
  return 1;
}

namespace {

constexpr int kMaxDevices = 64;

// Kernel attributes of split_kernel<NH, kFused, kOneTile> on the current device: set once per device (a
// per-device flag, read without a lock once set; the first call on a device configures it under the lock).
template <int NH, bool kFused, bool kOneTile>
cudaError_t configure_split_nh(int dev) {
  static std::atomic<bool> configured[kMaxDevices];
  static std::mutex mu;
  if (dev >= 0 && dev < kMaxDevices && configured[dev].load(std::memory_order_acquire)) return cudaSuccess;
  std::lock_guard<std::mutex> lock(mu);
  if (dev >= 0 && dev < kMaxDevices && configured[dev].load(std::memory_order_relaxed)) return cudaSuccess;
  cudaError_t e =
      cudaFuncSetAttribute(split_kernel<NH, kFused, kOneTile>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem_bytes<NH>());
  if (e != cudaSuccess) return e;
  // the smallest shared-memory carveout that holds the CTA: the rest of the SM's SRAM is L1, where the
  // record loads in flight land (about 28 KB at 64 heads per CTA, 60 KB at 16 or 32)
  int max_smem = 0;
  e = cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
  if (e != cudaSuccess) return e;
  const int pct = (int)((100 * (smem_bytes<NH>() + 1024) + max_smem - 1) / max_smem);
  e = cudaFuncSetAttribute(split_kernel<NH, kFused, kOneTile>, cudaFuncAttributePreferredSharedMemoryCarveout,
                           pct < 100 ? pct : 100);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < kMaxDevices) configured[dev].store(true, std::memory_order_release);
  return cudaSuccess;
}

template <int NH>
cudaError_t launch_split_nh(const SplitParams& p, cudaStream_t stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  // every partition holds at most one tile (the in-kernel merge keeps the general instantiation: with
  // both, the 64-head CTA spills registers)
  const bool one = !p.fused && p.split_len <= kTile;
  e = p.fused ? configure_split_nh<NH, true, false>(dev)
              : (one ? configure_split_nh<NH, false, true>(dev) : configure_split_nh<NH, false, false>(dev));
  if (e != cudaSuccess) return e;
  const int head_groups = (p.H + NH - 1) / NH;
  dim3 grid(p.nsplit, head_groups, p.B);
  // programmatic stream serialization: the CTAs may be scheduled, and set up, while the previous
  // kernel in the stream drains; they wait for it (griddep_wait) before touching global memory
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem_bytes<NH>();
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (p.fused) {
    // the partitions of a (query, head group) as one cluster: co-scheduled, they merge through each
    // other's shared memory and the workspace
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)p.nsplit;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
  }
  if (p.fused) return cudaLaunchKernelEx(&cfg, split_kernel<NH, true, false>, p);
  return one ? cudaLaunchKernelEx(&cfg, split_kernel<NH, false, true>, p)
             : cudaLaunchKernelEx(&cfg, split_kernel<NH, false, false>, p);
}

}  // namespace

cudaError_t launch_split(const SplitParams& p, cudaStream_t stream) {
  switch (p.nh) {
    case 16: return launch_split_nh<16>(p, stream);
    case 32: return launch_split_nh<32>(p, stream);
    case 64: return launch_split_nh<64>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace smla
