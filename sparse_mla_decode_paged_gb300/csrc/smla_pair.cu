// Split kernel on a pair of CTAs (a cluster of two SMs), tcgen05 MMAs with TMEM accumulators.
//
// One cluster per (partition s of the top-k list, group of 64 heads, query b).
// CTA c of the pair owns latent dims [256c, 256c + 256) (scale blocks 2c and
// 2c + 1) and rope dims [32c, 32c + 32); the partition is walked in tiles of
// 128 top-k entries (MMA M), double-buffered per CTA.
//
// Numerics (exact scores).  A block scale sc = mant * 2^e with mant in [1, 2)
// (e clamped to [-15, 7]).  The K tile holds V' = code * 2^e in fp16, which is
// exact for every E4M3 code; Q is fp16 (exact for bf16 inside the fp16 range).
// So the MMA S_b = V'_b . Q_b^T of each 128-dim block is exact up to fp32
// accumulation, and the score is  s = sum_b mant_b * S_b + S_rope  in fp32.
// PV uses V' too, with the mantissa moved onto the probabilities:
// O_b^T += V'_b^T . (P * mant_b) with P * mant_b rounded to fp16 (relative
// 2^-11 per term, averaged over the tile).  ("The 64-Block Barrier", "The
// Split-K Prescription": dequantise, QK^T over 576 dims, softmax, PV over 512.)
//
// Per tile, in each CTA:
//   gather warps (4)   index -> row through the block table; 16-byte loads of
//                      this CTA's 328 bytes of each record into registers, one
//                      token per thread, the next tile's loads in flight while
//                      the current one is converted; codes -> V' (fp16,
//                      128B-swizzled), rope bf16 -> fp16 (64B-swizzled),
//                      mantissas and validity to shared memory; lane 0 of the
//                      first gather warp then issues the 18 QK MMAs
//                      (M=128 tokens, N=64 heads) into three accumulators
//                      (block 2c, block 2c + 1, rope).
//   softmax warps (8)  one token (TMEM lane) and 32 heads per thread: partial
//                      score of this CTA's dims from TMEM, sent as fp32 into
//                      the other CTA's shared memory (DSMEM); the full score is
//                      own + other, identical in both CTAs, so both run the
//                      same softmax on all 128 x 64 scores and never need to
//                      agree on a running max.  The max is lazy: a head's
//                      reference max moves only when a score exceeds it by
//                      more than 2^8 (then O and the running sums are rescaled).
//                      P * mant for this CTA's two blocks is written (fp16)
//                      over the received partials; thread 0 issues the 16 PV
//                      MMAs and commits them to a barrier in both CTAs (the
//                      other CTA writes its next partials into this buffer).
//   epilogue           row sums reduced over the tokens, O / l for this CTA's
//                      256 dims straight from TMEM to global memory; CTA 0
//                      writes lse.
//
// Shared memory per CTA: Q 36 KB + 2 K slots x 72 KB + P/partials 32 KB +
// barriers ~ 222 KB, one CTA per SM; TMEM: O^T (2 x 64 columns) and two sets
// of three 64-column score accumulators (512 allocated).
#include <cuda_runtime.h>
#include <math_constants.h>

#include "smla_device.cuh"
#include "smla_ptx.cuh"

namespace smla {
namespace {

constexpr int kTile = 128;
constexpr int kHeads = 64;
constexpr int kThreads = 384;
constexpr int kSoftThreads = 256;          // warps 0..7
constexpr int kGatherThreads = 128;        // warps 8..11
constexpr int kSoftWarps = kSoftThreads / 32;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSCol = 128;            // score accumulators: 128 + 192 * parity + {0, 64, 128}
constexpr float kRescaleThreshold = 8.0f;  // log2 units: P <= 2^8
constexpr float kFp16Max = 65504.0f;
constexpr float kMaxScale = 16384.0f;      // P * mant <= 2^8 * 2^7 stays inside fp16

// shared-memory map (offsets from the 1024-aligned base)
constexpr uint32_t kQLat = 0;              // 4 chunks x (64 heads x 128 B), 128B swizzle
constexpr uint32_t kQChunk = kHeads * 128;
constexpr uint32_t kQRope = 4 * kQChunk;   // 64 heads x 64 B, 64B swizzle
constexpr uint32_t kSlot0 = kQRope + kHeads * 64;
constexpr uint32_t kKChunk = kTile * 128;  // 64 dims x 128 tokens
constexpr uint32_t kSlotRope = 4 * kKChunk;
constexpr uint32_t kSlotBytes = kSlotRope + kTile * 64;
constexpr uint32_t kPBase = kSlot0 + 2 * kSlotBytes;   // P * mant for blocks 2c, 2c+1 (128 tokens x 128 B each)
constexpr uint32_t kMiscOff = kPBase + 2 * kKChunk;
static_assert(kSlot0 % 1024 == 0 && kSlotBytes % 1024 == 0 && kPBase % 1024 == 0, "swizzle atoms");

constexpr uint32_t kIdescQK = ptx::idesc_f16(128, kHeads, 0, 0);
constexpr uint32_t kIdescPV = ptx::idesc_f16(128, kHeads, 1, 1);

struct PairMisc {
  uint64_t q_ready;          // Q staged (one arrival per softmax warp)
  uint64_t meta_full[2];     // slot metadata written (QK issuer, after the gather barrier)
  uint64_t s_full[2];        // QK of the slot's tile complete
  uint64_t s_free[2];        // scores read out of TMEM (one arrival per softmax warp)
  uint64_t pv_pair;          // PV of a tile complete in both CTAs (multicast commits)
  uint64_t part_full;        // the other CTA's partial scores arrived (one arrival per remote softmax warp)
  uint64_t teardown;         // every MMA of both issuers complete
  uint64_t exit_bar;         // the other CTA is done with this CTA's shared memory
  uint32_t tmem_slot;
  int abort;
  int range_err;
  alignas(16) float mant[2][2][kTile];   // [slot][block][token]
  unsigned char valid[2][kTile];
  alignas(16) float m_ref[kHeads];       // reference max per head, log2 units
  alignas(16) float m_new[kHeads];
  alignas(16) float alpha[kHeads];       // rescale factor of a max update
  alignas(16) float red[4][kHeads];
  alignas(16) float linv[kHeads];
  float lse_out[kHeads];
};

constexpr size_t kSmemBytes = 1024 + kMiscOff + sizeof(PairMisc);
static_assert(kSmemBytes <= 232448, "shared memory per CTA");

__device__ __forceinline__ uint32_t swz128(uint32_t row, uint32_t unit) {
  return row * 128u + ((unit ^ (row & 7u)) << 4);
}
__device__ __forceinline__ uint32_t swz64(uint32_t row, uint32_t unit) {
  return row * 64u + ((unit ^ ((row >> 1) & 3u)) << 4);
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// sc = mant * 2^e, e = clamp(exponent(sc), -15, 7); returns mant (exact) and 2^e as an fp16 pair.
__device__ __forceinline__ float pow2_split(float sc, uint32_t& p2) {
  const uint32_t bits = __float_as_uint(sc) & 0x7fffffffu;
  int e = (int)(bits >> 23) - 127;
  e = max(-15, min(7, e));
  const float mant = sc * __uint_as_float((uint32_t)(127 - e) << 23);
  const uint32_t h = e >= -14 ? (uint32_t)(e + 15) << 10 : 0x0200u;   // 2^-15 is an fp16 subnormal
  p2 = h | (h << 16);
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

// Order-preserving map of a float onto an unsigned key (for warp max with redux).
__device__ __forceinline__ uint32_t fkey(float f) {
  const uint32_t b = __float_as_uint(f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float fkey_inv(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}
__device__ __forceinline__ uint32_t redux_max(uint32_t v) {
  uint32_t r;
  asm volatile("redux.sync.max.u32 %0, %1, 0xffffffff;" : "=r"(r) : "r"(v));
  return r;
}

struct Ctx {
  const SplitParams* p;
  PairMisc* ms;
  volatile int* abort;
  uint32_t base;      // shared address of the aligned base
  uint32_t tmem;
  uint32_t c;         // rank in the pair
  int b, g, split, pos0, pos_end, n_tiles, hg_valid;
};

// ------------------------------------------------------------------------------------------ gather
__device__ __forceinline__ void gather_role(const Ctx& x, int warp, int lane) {
  const SplitParams& p = *x.p;
  PairMisc& ms = *x.ms;
  const int t = 32 * (warp - 8) + lane;
  const bool issuer = (warp == 8 && lane == 0);
  const int seq_len = __ldg(p.seq_lens + x.b);
  const int32_t* bt_row = p.block_table + (size_t)x.b * p.max_pages;
  const int32_t* tk_row = p.topk + (size_t)x.b * p.topk_n;
  const unsigned char* kv = p.kv + 256 * x.c;
  int range_bad = 0;
  bool ok = true, mma_ok = true;

  uint4 lat[16], rope[4];
  float2 sc = make_float2(0.f, 0.f);
  auto load_row = [&](int64_t r) {
    if (r >= 0) {
      const unsigned char* rec = kv + r * kRecordBytes;
#pragma unroll
      for (int k = 0; k < 16; ++k) lat[k] = __ldg(reinterpret_cast<const uint4*>(rec) + k);
      const unsigned char* rrec = p.kv + r * kRecordBytes + 528 + 64 * x.c;
#pragma unroll
      for (int k = 0; k < 4; ++k) rope[k] = __ldg(reinterpret_cast<const uint4*>(rrec) + k);
      sc = __ldg(reinterpret_cast<const float2*>(p.kv + r * kRecordBytes + 512 + 8 * x.c));
    }
  };
  auto topk_at = [&](int i) -> int {
    const int pos = x.pos0 + i * kTile + t;
    return pos < x.pos_end ? __ldg(tk_row + pos) : -1;
  };
  int64_t row = row_of(bt_row, topk_at(0), seq_len, p.max_pages, p.num_pages, p.err);
  int idx_next = x.n_tiles > 1 ? topk_at(1) : -1;
  load_row(row);

  for (int i = 0; i < x.n_tiles; ++i) {
    const int s = i & 1;
    const bool valid = row >= 0;
    // the next tile's block-table lookup overlaps this tile's conversion
    const int64_t row_next = (i + 1 < x.n_tiles) ? row_of(bt_row, idx_next, seq_len, p.max_pages, p.num_pages, p.err)
                                                 : -1;
    idx_next = (i + 2 < x.n_tiles) ? topk_at(i + 2) : -1;
    // slot s was last read by the PV of tile i - 2
    if (i >= 2) ok = ok && ptx::mbar_wait_bounded(&ms.pv_pair, (i - 2) & 1, x.abort);
    ok = __all_sync(0xffffffffu, ok);
    const uint32_t slot = x.base + kSlot0 + s * kSlotBytes;
    if (ok) {
      uint32_t p2[2];
      float mt[2];
      mt[0] = pow2_split(sc.x, p2[0]);
      mt[1] = pow2_split(sc.y, p2[1]);
      if (valid) range_bad |= !(fabsf(sc.x) <= kMaxScale) | !(fabsf(sc.y) <= kMaxScale);
      ms.mant[s][0][t] = valid ? mt[0] : 0.f;
      ms.mant[s][1][t] = valid ? mt[1] : 0.f;
      ms.valid[s][t] = valid;
#pragma unroll
      for (int k = 0; k < 16; ++k) {           // 16 codes: local dims [16k, 16k + 16), block k / 8
        const uint32_t w[4] = {lat[k].x, lat[k].y, lat[k].z, lat[k].w};
        const uint32_t m2 = p2[k >> 3];
        uint32_t hv[8];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          hv[2 * q] = valid ? hmul2(e4m3x2_to_f16x2((uint16_t)(w[q] & 0xFFFFu)), m2) : 0u;
          hv[2 * q + 1] = valid ? hmul2(e4m3x2_to_f16x2((uint16_t)(w[q] >> 16)), m2) : 0u;
        }
        const uint32_t cb = slot + (k >> 2) * kKChunk;
        const uint32_t uc = 2 * (k & 3);
        ptx::sts128_async_only(cb + swz128(t, uc), make_uint4(hv[0], hv[1], hv[2], hv[3]));
        ptx::sts128_async_only(cb + swz128(t, uc + 1), make_uint4(hv[4], hv[5], hv[6], hv[7]));
      }
#pragma unroll
      for (int k = 0; k < 4; ++k)
        ptx::sts128_async_only(slot + kSlotRope + swz64(t, k),
                               valid ? bf8_to_h8(rope[k], range_bad) : make_uint4(0, 0, 0, 0));
    }
    // registers are free again: the next tile's loads go out now
    row = row_next;
    if (i + 1 < x.n_tiles) load_row(row);
    ptx::fence_proxy_async_smem();
    ptx::named_bar_sync(1, kGatherThreads);
    if (issuer) {
      ptx::mbar_arrive(&ms.meta_full[s]);
      mma_ok = mma_ok && ok;
      if (i == 0) mma_ok = mma_ok && ptx::mbar_wait_bounded(&ms.q_ready, 0, x.abort);
      if (i >= 2) mma_ok = mma_ok && ptx::mbar_wait_bounded(&ms.s_free[s], ((i >> 1) - 1) & 1, x.abort);
      if (mma_ok) {
        ptx::tc_fence_after();
        const uint32_t dS = x.tmem + kSCol + 192 * s;
        const uint32_t qb = x.base + kQLat;
#pragma unroll
        for (int jj = 0; jj < 2; ++jj)
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            const int ch = 2 * jj + cc;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              ptx::mma_f16_ss(dS + 64 * jj, ptx::sw128_desc(slot + ch * kKChunk + 32 * kk, 16, 1024),
                              ptx::sw128_desc(qb + ch * kQChunk + 32 * kk, 16, 1024), kIdescQK, (cc | kk) != 0);
          }
#pragma unroll
        for (int kk = 0; kk < 2; ++kk)
          ptx::mma_f16_ss(dS + 128, ptx::sw64_desc(slot + kSlotRope + 32 * kk, 16, 512),
                          ptx::sw64_desc(x.base + kQRope + 32 * kk, 16, 512), kIdescQK, kk != 0);
        ptx::mma_commit(&ms.s_full[s]);
      }
    }
  }
  if (range_bad) ms.range_err = 1;
  if (issuer) ptx::mma_commit(&ms.teardown);
}

// ------------------------------------------------------------------------------------------ softmax
__device__ __forceinline__ void softmax_role(const Ctx& x, int warp, int lane) {
  const SplitParams& p = *x.p;
  PairMisc& ms = *x.ms;
  const int tid = threadIdx.x;
  const int quad = warp & 3, hh = warp >> 2;
  const int t = 32 * quad + lane;            // token of the tile = TMEM lane; dim within an O block
  const int hb = 32 * hh;                    // this thread's heads [hb, hb + 32)
  const bool issuer = (tid == 0);
  const uint32_t lane_q = (uint32_t)(32 * quad) << 16;
  int range_bad = 0;
  bool ok = true, mma_ok = true;

  // Q for this CTA's dims -> fp16, swizzled; zero rows past the valid heads
  {
    const uint16_t* qg = p.q + ((size_t)x.b * p.H + (size_t)x.g * kHeads) * kDQK;
    uint4 v[9];
#pragma unroll
    for (int k = 0; k < 9; ++k) {
      const int id = tid + kSoftThreads * k, n = id / 36, j = id % 36;
      const int col = j < 32 ? 256 * (int)x.c + 8 * j : 512 + 32 * (int)x.c + 8 * (j - 32);
      v[k] = n < x.hg_valid ? __ldg(reinterpret_cast<const uint4*>(qg + (size_t)n * kDQK + col))
                            : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int k = 0; k < 9; ++k) {
      const int id = tid + kSoftThreads * k, n = id / 36, j = id % 36;
      const uint32_t dst = j < 32 ? x.base + kQLat + (j >> 3) * kQChunk + swz128(n, j & 7)
                                  : x.base + kQRope + swz64(n, j - 32);
      ptx::sts128_async_only(dst, bf8_to_h8(v[k], range_bad));
    }
    ptx::fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(&ms.q_ready);
  }

  const float c2 = p.sm_scale * 1.4426950408889634f;
  const uint32_t own_p = x.base + kPBase + hh * kKChunk;               // partials for heads [hb, hb+32) land here
  const uint32_t peer_p = ptx::mapa(own_p, x.c ^ 1u);
  const uint32_t peer_part_full = ptx::mapa(ptx::smem_u32(&ms.part_full), x.c ^ 1u);
  float lsum[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) lsum[j] = 0.f;

  for (int i = 0; i < x.n_tiles; ++i) {
    const int s = i & 1;
    ok = ok && ptx::mbar_wait_bounded(&ms.meta_full[s], (i >> 1) & 1, x.abort) &&
         ptx::mbar_wait_bounded(&ms.s_full[s], (i >> 1) & 1, x.abort);
    ok = __all_sync(0xffffffffu, ok);
    ptx::tc_fence_after();
    const float mant0 = ms.mant[s][0][t], mant1 = ms.mant[s][1][t];
    const bool valid = ms.valid[s][t];
    float acc[32];
    if (ok) {
      const uint32_t sa = x.tmem + lane_q + kSCol + 192 * s + hb;
      uint32_t r[32];
      ptx::tmem_ld32(sa, r);
      ptx::tmem_wait_ld();
      const float f0 = mant0 * c2, f1 = mant1 * c2;
#pragma unroll
      for (int j = 0; j < 32; ++j) acc[j] = f0 * __uint_as_float(r[j]);
      ptx::tmem_ld32(sa + 64, r);
      ptx::tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < 32; ++j) acc[j] = fmaf(f1, __uint_as_float(r[j]), acc[j]);
      ptx::tmem_ld32(sa + 128, r);
      ptx::tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < 32; ++j) acc[j] = fmaf(c2, __uint_as_float(r[j]), acc[j]);
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j) acc[j] = 0.f;
    }
    ptx::tc_fence_before();
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(&ms.s_free[s]);

    // partial scores -> the other CTA (its buffer is free once both PVs of the previous tile are done)
    if (i > 0) ok = ok && ptx::mbar_wait_bounded(&ms.pv_pair, (i - 1) & 1, x.abort);
    ok = __all_sync(0xffffffffu, ok);
    if (ok) {
#pragma unroll
      for (int k = 0; k < 8; ++k)
        ptx::st_cluster128(peer_p + 128 * t + ((k ^ (t & 7)) << 4),
                           make_uint4(__float_as_uint(acc[4 * k]), __float_as_uint(acc[4 * k + 1]),
                                      __float_as_uint(acc[4 * k + 2]), __float_as_uint(acc[4 * k + 3])));
    }
    ptx::fence_acq_rel_cluster();
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive_cluster(peer_part_full);
    ok = ok && ptx::mbar_wait_cluster_bounded(&ms.part_full, i & 1, x.abort);
    ok = __all_sync(0xffffffffu, ok);

    // full scores (own + other: the same sum in both CTAs), in place of the partials
    if (ok) {
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint4 v = ptx::lds128(own_p + 128 * t + ((k ^ (t & 7)) << 4));
        acc[4 * k] += __uint_as_float(v.x);
        acc[4 * k + 1] += __uint_as_float(v.y);
        acc[4 * k + 2] += __uint_as_float(v.z);
        acc[4 * k + 3] += __uint_as_float(v.w);
      }
    }
    float* sx = acc;
#pragma unroll
    for (int j = 0; j < 32; ++j) sx[j] = (ok && valid) ? sx[j] : -CUDART_INF_F;
    bool need = false;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float4 v = reinterpret_cast<const float4*>(ms.m_ref)[hb / 4 + k];
      need |= (sx[4 * k] > v.x + kRescaleThreshold) | (sx[4 * k + 1] > v.y + kRescaleThreshold) |
              (sx[4 * k + 2] > v.z + kRescaleThreshold) | (sx[4 * k + 3] > v.w + kRescaleThreshold);
    }
    // every partial has been read once this barrier passes: the buffer may take P * mant
    need = ptx::named_bar_or(3, kSoftThreads, need);
    if (need) {
      // a head's reference max moves to its tile max when that exceeds it by more than the threshold
      float mine = 0.f;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float wmax = fkey_inv(redux_max(fkey(sx[j])));
        if (lane == j) mine = wmax;
      }
      ms.red[quad][hb + lane] = mine;
      ptx::named_bar_sync(2, kSoftThreads);
      if (quad == 0) {
        const int h = hb + lane;
        const float tm = fmaxf(fmaxf(ms.red[0][h], ms.red[1][h]), fmaxf(ms.red[2][h], ms.red[3][h]));
        const float mo = ms.m_ref[h];
        const float mn = tm > mo + kRescaleThreshold ? tm : mo;
        ms.alpha[h] = mo == -CUDART_INF_F ? 0.f : ptx::ex2_approx(mo - mn);
        ms.m_new[h] = mn;
      }
      ptx::named_bar_sync(2, kSoftThreads);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float4 a = reinterpret_cast<const float4*>(ms.alpha)[hb / 4 + k];
        lsum[4 * k] *= a.x; lsum[4 * k + 1] *= a.y; lsum[4 * k + 2] *= a.z; lsum[4 * k + 3] *= a.w;
      }
      if (i > 0 && ok) {
        // O columns of these heads (the previous PV is complete: waited above)
#pragma unroll 1
        for (int jb = 0; jb < 2; ++jb) {
          uint32_t r[32];
          const uint32_t oa = x.tmem + lane_q + 64 * jb + hb;
          ptx::tmem_ld32(oa, r);
          ptx::tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * ms.alpha[hb + j]);
          ptx::tmem_st32(oa, r);
        }
        ptx::tmem_wait_st();
      }
      ptx::named_bar_sync(2, kSoftThreads);
      if (quad == 0) ms.m_ref[hb + lane] = ms.m_new[hb + lane];
      ptx::named_bar_sync(2, kSoftThreads);
    }
    // P (lsum) and P * mant of this CTA's blocks, fp16, 128B-swizzled rows of 64 heads
    const uint32_t p0 = x.base + kPBase, p1 = p0 + kKChunk;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float4 ma = reinterpret_cast<const float4*>(ms.m_ref)[hb / 4 + 2 * u];
      const float4 mb = reinterpret_cast<const float4*>(ms.m_ref)[hb / 4 + 2 * u + 1];
      const float m[8] = {ma.x, ma.y, ma.z, ma.w, mb.x, mb.y, mb.z, mb.w};
      uint32_t w0[4], w1[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int j = 8 * u + 2 * q;
        // a head with no valid entry yet has m = -inf: its P is 0 (its scores are -inf too)
        const float pa = m[2 * q] == -CUDART_INF_F ? 0.f : ptx::ex2_approx(sx[j] - m[2 * q]);
        const float pb = m[2 * q + 1] == -CUDART_INF_F ? 0.f : ptx::ex2_approx(sx[j + 1] - m[2 * q + 1]);
        lsum[j] += pa;
        lsum[j + 1] += pb;
        w0[q] = f32x2_to_f16x2_sat(pa * mant0, pb * mant0);
        w1[q] = f32x2_to_f16x2_sat(pa * mant1, pb * mant1);
      }
      const uint32_t off = swz128(t, 4 * hh + u);
      ptx::sts128_async_only(p0 + off, make_uint4(w0[0], w0[1], w0[2], w0[3]));
      ptx::sts128_async_only(p1 + off, make_uint4(w1[0], w1[1], w1[2], w1[3]));
    }
    ptx::tc_fence_before();
    ptx::fence_proxy_async_smem();
    ptx::named_bar_sync(2, kSoftThreads);
    if (issuer) {
      mma_ok = mma_ok && ok;
      if (mma_ok) {
        ptx::tc_fence_after();
        const uint32_t slot = x.base + kSlot0 + s * kSlotBytes;
#pragma unroll
        for (int jb = 0; jb < 2; ++jb)
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk)
            ptx::mma_f16_ss(x.tmem + 64 * jb,
                            ptx::sw128_desc(slot + 2 * jb * kKChunk + kk * 2048, kKChunk, 1024),
                            // P spans one 64-head atom along N: its leading offset is never stepped
                            ptx::sw128_desc(p0 + jb * kKChunk + kk * 2048, 1024, 1024), kIdescPV,
                            (i > 0 || kk > 0) ? 1u : 0u);
        ptx::mma_commit_multicast(&ms.pv_pair, 0x3);
      }
    }
  }
  if (range_bad) ms.range_err = 1;
  if (issuer) ptx::mma_commit(&ms.teardown);

  // ------------------------------------------------------------------ epilogue
  if (x.n_tiles > 0) ok = ok && ptx::mbar_wait_bounded(&ms.pv_pair, (x.n_tiles - 1) & 1, x.abort);
  ok = __all_sync(0xffffffffu, ok);
  ptx::tc_fence_after();
  {
    float mine = 0.f;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      float v = lsum[j];
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
      if (lane == j) mine = v;
    }
    ms.red[quad][hb + lane] = mine;
  }
  ptx::named_bar_sync(2, kSoftThreads);
  if (quad == 0) {
    const int h = hb + lane;
    const float L = ms.red[0][h] + ms.red[1][h] + ms.red[2][h] + ms.red[3][h];
    ms.linv[h] = L > 0.f ? 1.f / L : 0.f;
    ms.lse_out[h] = L > 0.f ? (ms.m_ref[h] + log2f(L)) * 0.6931471805599453f : -CUDART_INF_F;
  }
  ptx::named_bar_sync(2, kSoftThreads);
  if (ok) {
    float li[32];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float4 v = reinterpret_cast<const float4*>(ms.linv)[hb / 4 + k];
      li[4 * k] = v.x; li[4 * k + 1] = v.y; li[4 * k + 2] = v.z; li[4 * k + 3] = v.w;
    }
#pragma unroll
    for (int jb = 0; jb < 2; ++jb) {
      uint32_t r[32];
      ptx::tmem_ld32(x.tmem + lane_q + 64 * jb + hb, r);
      ptx::tmem_wait_ld();
      const int d = 256 * (int)x.c + 128 * jb + t;
      const size_t hrow0 = (size_t)x.g * kHeads + hb;
      if (p.final_out) {
        uint16_t* o = p.out + ((size_t)x.b * p.H + hrow0) * kDLatent + d;
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (hb + j < x.hg_valid)
            o[(size_t)j * kDLatent] = (uint16_t)(f32x2_to_bf16x2(__uint_as_float(r[j]) * li[j], 0.f) & 0xFFFFu);
      } else {
        float* o = p.o_part + (((size_t)x.b * p.nsplit + x.split) * p.H + hrow0) * kDLatent + d;
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (hb + j < x.hg_valid) o[(size_t)j * kDLatent] = __uint_as_float(r[j]) * li[j];
      }
    }
    if (x.c == 0 && tid < x.hg_valid) {
      const size_t h = (size_t)x.g * kHeads + tid;
      if (p.final_out) p.lse[(size_t)x.b * p.H + h] = ms.lse_out[tid];
      else p.lse_part[((size_t)x.b * p.nsplit + x.split) * p.H + h] = ms.lse_out[tid];
    }
  }
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1) split_pair_kernel(const SplitParams p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  PairMisc& ms = *reinterpret_cast<PairMisc*>(base + kMiscOff);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  Ctx x;
  x.p = &p;
  x.ms = &ms;
  x.abort = &ms.abort;
  x.base = ptx::smem_u32(base);
  x.c = ptx::cluster_ctarank();
  x.split = blockIdx.x >> 1;
  x.g = blockIdx.y;
  x.b = blockIdx.z;
  x.pos0 = x.split * p.split_len;
  x.pos_end = min(x.pos0 + p.split_len, p.topk_n);
  x.n_tiles = x.pos_end > x.pos0 ? (x.pos_end - x.pos0 + kTile - 1) / kTile : 0;
  x.hg_valid = min(kHeads, p.H - kHeads * x.g);

  if (x.n_tiles == 0) {
    // empty partition (the same in both CTAs, which touch no shared memory of each other): out = 0,
    // lse = -inf for this CTA's dims
    for (int i = threadIdx.x; i < x.hg_valid * 256; i += kThreads) {
      const size_t h = (size_t)x.g * kHeads + i / 256;
      const int d = 256 * (int)x.c + i % 256;
      if (p.final_out) p.out[((size_t)x.b * p.H + h) * kDLatent + d] = 0;
      else p.o_part[(((size_t)x.b * p.nsplit + x.split) * p.H + h) * kDLatent + d] = 0.f;
    }
    if (x.c == 0 && (int)threadIdx.x < x.hg_valid) {
      const size_t h = (size_t)x.g * kHeads + threadIdx.x;
      if (p.final_out) p.lse[(size_t)x.b * p.H + h] = -CUDART_INF_F;
      else p.lse_part[((size_t)x.b * p.nsplit + x.split) * p.H + h] = -CUDART_INF_F;
    }
    return;
  }

  if (threadIdx.x == 0) {
    ptx::mbar_init(&ms.q_ready, kSoftWarps);
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(&ms.meta_full[s], 1);
      ptx::mbar_init(&ms.s_full[s], 1);
      ptx::mbar_init(&ms.s_free[s], kSoftWarps);
    }
    ptx::mbar_init(&ms.pv_pair, 2);
    ptx::mbar_init(&ms.part_full, kSoftWarps);
    ptx::mbar_init(&ms.teardown, 2);
    ptx::mbar_init(&ms.exit_bar, 1);
    ms.abort = 0;
    ms.range_err = 0;
    ptx::fence_mbar_init();
  }
  if (threadIdx.x < kHeads) ms.m_ref[threadIdx.x] = -CUDART_INF_F;
  if (warp == 0) {
    ptx::tmem_alloc(&ms.tmem_slot, kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  // barriers of both CTAs initialised before either CTA arrives remotely
  ptx::cluster_sync_all();
  ptx::tc_fence_after();
  x.tmem = ms.tmem_slot;

  if (warp >= kSoftWarps) gather_role(x, warp, lane);
  else softmax_role(x, warp, lane);

  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (threadIdx.x == 0) {
    // every MMA of both issuers has completed before TMEM is released (time limit only)
    volatile int no_abort = 0;
    if (!ptx::mbar_wait_bounded(&ms.teardown, 0, &no_abort, 100000000ull)) ms.abort = 1;
    // the other CTA writes into this CTA's shared memory and arrives on its barriers until it is
    // done: leave only after its exit arrival (time limit only)
    ptx::mbar_arrive_cluster(ptx::mapa(ptx::smem_u32(&ms.exit_bar), x.c ^ 1u));
    // (its own waits give up within about a second, so three seconds cover any state it can be in)
    volatile int no_abort2 = 0;
    if (!ptx::mbar_wait_cluster_bounded(&ms.exit_bar, 0, &no_abort2, 3000000000ull)) ms.abort = 1;
    if (p.err) {
      if (ms.abort) atomicOr(p.err, SMLA_DEVERR_TIMEOUT);
      if (ms.range_err) atomicOr(p.err, SMLA_DEVERR_RANGE);
    }
  }
  __syncthreads();
  if (warp == 0) ptx::tmem_dealloc(x.tmem, kTmemCols);
}

}  // namespace

bool split_shape_supported(int H, int topk) {
  return (H == 16 || H == 32 || H == 64 || H == 128) && topk >= 1 && topk <= kMaxTopk;
}

int split_heads_per_cta() { return kHeads; }

int split_ctas_per_unit() { return 2; }

int split_ctas_per_sm(int H) {
  (void)H;
  return 1;
}

cudaError_t launch_split_pair(const SplitParams& p, cudaStream_t stream) {
  static int configured_device = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_device != dev) {
    e = cudaFuncSetAttribute(split_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  const int head_groups = (p.H + kHeads - 1) / kHeads;
  dim3 grid(2 * p.nsplit, head_groups, p.B);
  split_pair_kernel<<<grid, kThreads, kSmemBytes, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace smla
