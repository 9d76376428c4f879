// Tensor-core split kernel (sm_103a): tcgen05 MMAs with TMEM accumulators.
//
// One CTA per (partition s of the top-k list, group of 64 heads, query b).
// The partition is walked in tiles of 128 top-k entries:
//
//   gather warps (8)   index -> row through the block table (a1); 16-byte
//                      loads of each 656-byte record into registers (warp w
//                      owns the 32 tokens of TMEM lane quadrant w % 4 and one
//                      half of the latent dims); dequantisation (a2):
//                      k = code * scale is split as K_hi = fp16(k) and
//                      K_lo = k - K_hi with packed fp16 error-free
//                      multiply-adds (scale = sc_h + s_r, both fp16); K_hi is
//                      stored 128B-swizzled into the K tile (9 chunks of 64
//                      dims), K_lo is written into TMEM in a second pass from
//                      the thread's own K_hi rows (codes recovered as
//                      e4m3(K_hi / scale)); bf16 rope to fp16 (exact).  The
//                      next tile's loads are issued between the two passes.
//   MMA (warp 0 lane 0) S^T[128 tok x 64 heads] = K_hi . Q^T from shared
//                      memory (36 MMAs M=128 N=64 K=16) plus the correction
//                      K_lo . Q^T with the A operand read from TMEM (two
//                      passes of 256 dims), so that the scores carry about
//                      2^-22 relative error (a3); then
//                      O^T[512 x 64] += V^T . P^T for the four 128-dim blocks
//                      (a5), V^T being the latent K_hi read MN-major.
//   softmax warps (4)  load Q once (fp16, swizzled); then one TMEM lane
//                      (token) per thread: per-head running max over the tile
//                      (warp reduce-scatter + shared memory), P = exp2(s - m)
//                      in fp16 written over the rope chunk (a4), lazy rescale
//                      of O when a head's max grows by more than 2^8, and the
//                      epilogue (a6): O / l and lse.
//
// QK of a tile, its softmax and its PV are sequential (one K tile), so the
// MMAs are issued by lane 0 of the first softmax warp between its softmax
// steps; no warp is spent on issue only.
//
// Shared memory: Q 72 KB (64 heads x 576 fp16) + K tile 144 KB (128 x 576
// fp16) + barriers: one CTA per SM, 12 warps (3 per SM sub-partition, 168
// registers per thread).  TMEM: O^T in columns 0..255, S^T in 256..319, K_lo
// in 320..447 (512 allocated).
// Sources: "The 64-Block Barrier" ("The Smoking Gun", "The Split-K
// Prescription"); "Inside the Decode Performance Investigation" (Task 1).
#include <cuda_runtime.h>
#include <math_constants.h>

#include "smla_device.cuh"
#include "smla_ptx.cuh"

namespace smla {
namespace {

constexpr int kTile = 128;                 // top-k entries per tile (MMA M)
constexpr int kHeads = 64;                 // heads per CTA (MMA N), zero rows past the valid heads
constexpr int kChunks = 9;                 // 576 dims / 64
constexpr int kQChunkBytes = kHeads * 128;               // 8 KB
constexpr int kKChunkBytes = kTile * 128;                // 16 KB
constexpr int kQBytes = kChunks * kQChunkBytes;          // 73728
constexpr int kKBytes = kChunks * kKChunkBytes;          // 147456
constexpr int kThreads = 384;
constexpr int kSoftmaxThreads = 128;       // warps 0..3 (TMEM lane quadrants 0..3); lane 0 of warp 0 issues MMAs
constexpr int kSoftmaxWarps = kSoftmaxThreads / 32;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSCol = 256;            // S^T
constexpr uint32_t kLoCol = 320;           // K_lo, 256 dims (128 columns) per pass
constexpr float kRescaleThreshold = 8.0f;  // log2 units: P stays <= 256
constexpr float kFp16Max = 65504.0f;
constexpr float kMaxScale = kFp16Max / 448.0f;   // largest block scale whose dequantised latent fits fp16

constexpr uint32_t kIdescQK = ptx::idesc_f16(128, kHeads, 0, 0);
constexpr uint32_t kIdescPV = ptx::idesc_f16(128, kHeads, 1, 1);

struct Misc {
  uint64_t q_ready, meta_ready, s_full, p_ready, pv_done, teardown, klo_free;
  uint64_t kv_ready[5];                    // latent blocks 0..3 (two chunks each), rope
  uint64_t klo_ready[2];                   // K_lo of dims 0..255, 256..511 written to TMEM
  uint64_t chunk_free[4];
  uint32_t tmem_slot;
  int abort;
  int need_rescale;
  int stop;
  int range_err;
  float red[4][kHeads];
  alignas(16) float m_used[kHeads];
  alignas(16) float alpha[kHeads];
  float lse_out[kHeads];
  alignas(16) float linv[kHeads];
  unsigned char valid[kTile];
};

constexpr size_t kSmemBytes = 1024 + kQBytes + kKBytes + sizeof(Misc);

__device__ __forceinline__ uint32_t swz(uint32_t row, uint32_t unit) {  // byte offset in a 128B-swizzled chunk
  return row * 128u + ((unit ^ (row & 7u)) << 4);
}

// fp16 pair factors of a block scale: sc_h = fp16(sc) and s_r = fp16(sc - sc_h), plus 1/sc in fp32.
struct ScaleSplit {
  uint32_t sch, sr;
  float inv;
};

__device__ __forceinline__ ScaleSplit split_scale(float sc) {
  const uint32_t h = f32x2_to_f16x2_sat(sc, sc);
  const float hf = f16x2_to_f32x2(h).x;
  const float r = sc - hf;                                   // exact in fp32
  return {h, f32x2_to_f16x2_sat(r, r), sc != 0.f ? 1.f / sc : 0.f};
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

__device__ __forceinline__ uint32_t hfma2(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t r;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
  return r;
}

__device__ __forceinline__ uint32_t hadd2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("add.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// Two codes c (as fp16, exact) times the scale: K_hi = fp16(c * sc) up to ~2^-22 relative.
__device__ __forceinline__ uint32_t k_hi2(uint32_t c, const ScaleSplit& sp) {
  return hfma2(c, sp.sch, hmul2(c, sp.sr));
}

// K_lo = c * sc - K_hi: fma(c, sc_h, -hi) is exact (the rounding error of a product fits the format),
// plus the small term c * s_r.
__device__ __forceinline__ uint32_t k_lo2(uint32_t c, uint32_t hi, const ScaleSplit& sp) {
  return hadd2(hfma2(c, sp.sch, hi ^ 0x80008000u), hmul2(c, sp.sr));
}

// The two E4M3 codes behind a K_hi pair: hi / sc is within 2^-10 of a code, far inside half an E4M3 step.
__device__ __forceinline__ uint32_t codes_of_hi(uint32_t hi, const ScaleSplit& sp) {
  const float2 f = f16x2_to_f32x2(hi);
  uint16_t e;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(e) : "f"(f.y * sp.inv), "f"(f.x * sp.inv));
  return e4m3x2_to_f16x2(e);
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

// Warp reduce-scatter over 64 per-thread values: afterwards lane l holds the
// reduction over the warp's 32 threads of columns 2l and 2l+1.
template <bool kMax>
__device__ __forceinline__ float2 reduce_scatter64(const float (&v)[64], int lane) {
  float a[32];
  {
    const bool hi = lane & 16;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const float send = hi ? v[i] : v[32 + i];
      const float keep = hi ? v[32 + i] : v[i];
      const float r = __shfl_xor_sync(0xffffffffu, send, 16);
      a[i] = kMax ? fmaxf(keep, r) : keep + r;
    }
  }
#pragma unroll
  for (int span = 16, x = 8; span >= 2; span >>= 1, x >>= 1) {
    const bool hi = lane & x;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if (i < span) {
        const float send = hi ? a[i] : a[span + i];
        const float keep = hi ? a[span + i] : a[i];
        const float r = __shfl_xor_sync(0xffffffffu, send, x);
        a[i] = kMax ? fmaxf(keep, r) : keep + r;
      }
    }
  }
  return make_float2(a[0], a[1]);
}

// Gather role of warps 4..11: H2 selects the half of the latent dims (and rope) the warp owns.
template <int H2>
__device__ __forceinline__ void gather_role(const SplitParams& p, Misc& ms, volatile int* abort, uint32_t tmem,
                                            uint32_t k_base, int warp, int lane, int b, int pos0, int pos_end,
                                            int n_tiles) {
    // ------------------------------------------------------------------ gather + dequantise
    const int quad = warp & 3;                 // TMEM lane quadrant this warp may access
    constexpr int h2 = H2;                     // latent dims [256 h2, 256 h2 + 256)
    const int t = 32 * quad + lane;            // token within the tile = TMEM lane
    const uint32_t lane_base = (uint32_t)(32 * quad) << 16;
    const unsigned char* kt = reinterpret_cast<const unsigned char*>(__cvta_shared_to_generic(k_base));
    const int seq_len = __ldg(p.seq_lens + b);
    const int32_t* bt_row = p.block_table + (size_t)b * p.max_pages;
    const int32_t* tk_row = p.topk + (size_t)b * p.topk_n;
    int range_bad = 0;

    uint4 lat[16], rope[4];
    float sc0 = 0.f, sc1 = 0.f;                // scales of latent blocks 2 h2, 2 h2 + 1
    auto load_row = [&](int64_t r) {
      if (r >= 0) {
        const unsigned char* rec = p.kv + r * kRecordBytes;
#pragma unroll
        for (int k = 0; k < 16; ++k) lat[k] = __ldg(reinterpret_cast<const uint4*>(rec + 256 * h2) + k);
#pragma unroll
        for (int k = 0; k < 4; ++k) rope[k] = __ldg(reinterpret_cast<const uint4*>(rec + 528 + 64 * h2) + k);
        const float2 sc = __ldg(reinterpret_cast<const float2*>(rec + 512 + 8 * h2));
        sc0 = sc.x;
        sc1 = sc.y;
      }
    };
    auto topk_at = [&](int i) -> int {
      const int pos = pos0 + i * kTile + t;
      return pos < pos_end ? __ldg(tk_row + pos) : -1;
    };
    int64_t row = row_of(bt_row, topk_at(0), seq_len, p.max_pages, p.num_pages, p.err);
    load_row(row);

    bool ok = true;
    for (int i = 0; ok && i < n_tiles; ++i) {
      const int t_next = (i + 1 < n_tiles) ? topk_at(i + 1) : -1;
      const bool valid = row >= 0;
      // latent blocks 2 h2 and 2 h2 + 1 (chunks 4 h2 .. 4 h2 + 3): K_hi into shared memory and, for the
      // first half of the dims, K_lo into TMEM lane t at once.  The K_lo columns take dims 256..511 only
      // after the first correction pass of this tile has read them (klo_free), so the second-half warps
      // write their K_lo in a second, cheap pass.  The previous tile's passes are complete once its PV
      // has freed a chunk.
      const ScaleSplit spb[2] = {split_scale(sc0), split_scale(sc1)};
      if (valid) range_bad |= !(fabsf(sc0) <= kMaxScale) | !(fabsf(sc1) <= kMaxScale);
#pragma unroll
      for (int jj = 0; jj < 2; ++jj) {
        const int j = 2 * h2 + jj;
        if (i > 0 && !__all_sync(0xffffffffu, ptx::mbar_wait_bounded(&ms.chunk_free[j], (i - 1) & 1, abort))) {
          ok = false;
          break;
        }
        if (jj == 0 && h2 == 0) ms.valid[t] = valid;
#pragma unroll
        for (int u = 0; u < 8; ++u) {            // 16-dim units of this block
          const int k = 8 * jj + u;
          const uint32_t w[4] = {lat[k].x, lat[k].y, lat[k].z, lat[k].w};
          uint32_t hv[8];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            hv[2 * q] = valid ? k_hi2(e4m3x2_to_f16x2((uint16_t)(w[q] & 0xFFFFu)), spb[jj]) : 0u;
            hv[2 * q + 1] = valid ? k_hi2(e4m3x2_to_f16x2((uint16_t)(w[q] >> 16)), spb[jj]) : 0u;
          }
          const int c = 2 * j + (u >> 2);         // chunk of this unit
          const uint32_t cb = k_base + c * kKChunkBytes;
          const int uc = u & 3;
          ptx::sts128(cb + swz(t, 2 * uc), make_uint4(hv[0], hv[1], hv[2], hv[3]));
          ptx::sts128(cb + swz(t, 2 * uc + 1), make_uint4(hv[4], hv[5], hv[6], hv[7]));
        }
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          if (jj == 0 && h2 == 0) ptx::mbar_arrive(&ms.meta_ready);
          ptx::mbar_arrive(&ms.kv_ready[j]);
        }
      }
      if (!ok) break;
      // rope chunk: free once the previous tile's PV is done (its P lives there)
      if (i > 0 && !__all_sync(0xffffffffu, ptx::mbar_wait_bounded(&ms.pv_done, (i - 1) & 1, abort))) {
        ok = false;
        break;
      }
      {
        const uint32_t cb = k_base + 8 * kKChunkBytes;
#pragma unroll
        for (int k = 0; k < 4; ++k)
          ptx::sts128(cb + swz(t, 4 * h2 + k), valid ? bf8_to_h8(rope[k], range_bad) : make_uint4(0, 0, 0, 0));
        // (bf8_to_h8 only runs for a used token, so its range check only counts those)
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&ms.kv_ready[4]);
      }
      // the codes of this tile are consumed: start the next tile's loads
      if (i + 1 < n_tiles) {
        row = row_of(bt_row, t_next, seq_len, p.max_pages, p.num_pages, p.err);
        load_row(row);
      }
      // K_lo into TMEM lane t from this thread's own K_hi rows: dims 0..255 at once (the previous
      // tile's correction passes are complete once its PV has freed a chunk), dims 256..511 once the
      // first correction pass of this tile has read the columns (klo_free)
      if (h2 == 1 && !__all_sync(0xffffffffu, ptx::mbar_wait_bounded(&ms.klo_free, i & 1, abort))) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
#pragma unroll
      for (int jj = 0; jj < 2; ++jj) {
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int c = 2 * (2 * h2 + jj) + (u >> 2);
          const uint32_t cb = k_base + c * kKChunkBytes;
          const uint4 h0 = *reinterpret_cast<const uint4*>(kt + (cb - k_base) + swz(t, 2 * (u & 3)));
          const uint4 h1 = *reinterpret_cast<const uint4*>(kt + (cb - k_base) + swz(t, 2 * (u & 3) + 1));
          const uint32_t hv[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
          uint32_t lo[8];
#pragma unroll
          for (int q = 0; q < 8; ++q) lo[q] = k_lo2(codes_of_hi(hv[q], spb[jj]), hv[q], spb[jj]);
          ptx::tmem_st8(tmem + lane_base + kLoCol + 64 * jj + 8 * u, lo);
        }
      }
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&ms.klo_ready[h2]);
    }
    if (range_bad) ms.range_err = 1;
}

__global__ void __launch_bounds__(kThreads, 1) split_tc_kernel(const SplitParams p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Misc& ms = *reinterpret_cast<Misc*>(base + kQBytes + kKBytes);
  volatile int* abort = &ms.abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int pos0 = split * p.split_len;
  const int pos_end = min(pos0 + p.split_len, p.topk_n);
  const int n_tiles = pos_end > pos0 ? (pos_end - pos0 + kTile - 1) / kTile : 0;
  const int hg_valid = min(kHeads, p.H - kHeads * g);
  const uint32_t q_base = ptx::smem_u32(base);
  const uint32_t k_base = q_base + kQBytes;
  const uint32_t p_base = k_base + 8 * kKChunkBytes;   // P over the rope chunk

  if (n_tiles == 0) {
    // empty partition: out = 0, lse = -inf
    for (int i = threadIdx.x; i < hg_valid * kDLatent; i += kThreads) {
      const int h = g * kHeads + i / kDLatent, d = i % kDLatent;
      if (p.final_out) p.out[((size_t)b * p.H + h) * kDLatent + d] = 0;
      else p.o_part[(((size_t)b * p.nsplit + split) * p.H + h) * kDLatent + d] = 0.f;
    }
    if (threadIdx.x < hg_valid) {
      const int h = g * kHeads + threadIdx.x;
      if (p.final_out) p.lse[(size_t)b * p.H + h] = -CUDART_INF_F;
      else p.lse_part[((size_t)b * p.nsplit + split) * p.H + h] = -CUDART_INF_F;
    }
    return;
  }

  if (threadIdx.x == 0) {
    // producer barriers count one arrival per warp (lane 0 after the warp's fences)
    ptx::mbar_init(&ms.q_ready, kSoftmaxWarps);
    ptx::mbar_init(&ms.meta_ready, 4);
    ptx::mbar_init(&ms.s_full, 1);
    ptx::mbar_init(&ms.p_ready, kSoftmaxWarps);
    ptx::mbar_init(&ms.pv_done, 1);
    ptx::mbar_init(&ms.teardown, 1);
    ptx::mbar_init(&ms.klo_free, 1);
    for (int c = 0; c < 4; ++c) ptx::mbar_init(&ms.kv_ready[c], 4);
    ptx::mbar_init(&ms.kv_ready[4], 8);
    ptx::mbar_init(&ms.klo_ready[0], 4);
    ptx::mbar_init(&ms.klo_ready[1], 4);
    for (int j = 0; j < 4; ++j) ptx::mbar_init(&ms.chunk_free[j], 1);
    ms.abort = 0;
    ms.need_rescale = 0;
    ms.stop = 0;
    ms.range_err = 0;
    ptx::fence_mbar_init();
  }
  if (threadIdx.x < kHeads) {
    ms.m_used[threadIdx.x] = -CUDART_INF_F;
    ms.alpha[threadIdx.x] = 1.f;
  }
  if (warp == 0) {
    ptx::tmem_alloc(&ms.tmem_slot, kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::fence_proxy_async_smem();
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = ms.tmem_slot;

  if (warp >= 4) {
    if (warp < 8) gather_role<0>(p, ms, abort, tmem, k_base, warp, lane, b, pos0, pos_end, n_tiles);
    else gather_role<1>(p, ms, abort, tmem, k_base, warp, lane, b, pos0, pos_end, n_tiles);
  } else {
    // ------------------------------------------------------------------ Q, MMA issue, softmax, epilogue
    // Every softmax warp runs the same sequence of named barriers; a failed wait
    // only stops the loop through ms.stop, which warp 0 publishes between the
    // two barriers of a tile, so all four warps leave at the same tile.
    const int t = threadIdx.x;                    // TMEM lane = token within the tile / dim within a block
    const bool issuer = (threadIdx.x == 0);
    int range_bad = 0;
    {
      // Q head group -> fp16, 128B-swizzled, zero rows past the valid heads
      const uint16_t* qg = p.q + ((size_t)b * p.H + (size_t)g * kHeads) * kDQK;
#pragma unroll 1
      for (int k0 = 0; k0 < 36; k0 += 18) {
        uint4 v[18];
#pragma unroll
        for (int k = 0; k < 18; ++k) {
          const int id = t + kSoftmaxThreads * (k0 + k);
          const int n = id / 72, j = id % 72;
          v[k] = n < hg_valid ? __ldg(reinterpret_cast<const uint4*>(qg + (size_t)n * kDQK) + j) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int k = 0; k < 18; ++k) {
          const int id = t + kSoftmaxThreads * (k0 + k);
          const int n = id / 72, j = id % 72;
          ptx::sts128_async_only(q_base + (j >> 3) * kQChunkBytes + swz(n, j & 7), bf8_to_h8(v[k], range_bad));
        }
      }
      ptx::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&ms.q_ready);
    }
    const float c2 = p.sm_scale * 1.4426950408889634f;
    const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
    float lsum0 = 0.f, lsum1 = 0.f;               // this warp's sums for heads 2*lane, 2*lane+1
    bool ok = true;
    bool mma_ok = true;                           // issuer only
    if (issuer) mma_ok = ptx::mbar_wait_bounded(&ms.q_ready, 0, abort);
    for (int i = 0; i < n_tiles; ++i) {
      const uint32_t ph = i & 1;
      if (issuer && mma_ok) {
        // QK: K_hi blocks 0, 1 | correction dims 0..255 | K_hi blocks 2, 3 | rope | correction dims 256..511
        const uint32_t dS = tmem + kSCol;
        for (int step = 0; mma_ok && step < 7; ++step) {
          if (step == 2 || step == 6) {
            const int pass = step == 2 ? 0 : 1;
            mma_ok = ptx::mbar_wait_bounded(&ms.klo_ready[pass], ph, abort);
            if (!mma_ok) break;
            ptx::tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 16; ++kk) {
              const int c = 4 * pass + (kk >> 2);
              const uint64_t db = ptx::sw128_desc(q_base + c * kQChunkBytes + (kk & 3) * 32, 16, 1024);
              ptx::mma_f16_ts(dS, tmem + kLoCol + 8 * kk, db, kIdescQK, 1u);
            }
            ptx::mma_commit(pass == 0 ? &ms.klo_free : &ms.s_full);
          } else {
            const int j = step < 2 ? step : step - 1;   // 0, 1, 2, 3, 4 (rope)
            mma_ok = ptx::mbar_wait_bounded(&ms.kv_ready[j], ph, abort);
            if (!mma_ok) break;
            ptx::tc_fence_after();
            const int c0 = j < 4 ? 2 * j : 8, nc = j < 4 ? 2 : 1;
            for (int cc = 0; cc < nc; ++cc) {
              const int c = c0 + cc;
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) {
                const uint64_t da = ptx::sw128_desc(k_base + c * kKChunkBytes + kk * 32, 16, 1024);
                const uint64_t db = ptx::sw128_desc(q_base + c * kQChunkBytes + kk * 32, 16, 1024);
                ptx::mma_f16_ss(dS, da, db, kIdescQK, (c | kk) != 0);   // the very first MMA overwrites S
              }
            }
          }
        }
      }
      ok = ptx::mbar_wait_bounded(&ms.meta_ready, ph, abort) && ptx::mbar_wait_bounded(&ms.s_full, ph, abort);
      ok = __all_sync(0xffffffffu, ok);
      ptx::tc_fence_after();
      float s[64];
      {
        const bool valid = ms.valid[t];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          uint32_t r[32];
          ptx::tmem_ld32(tmem + lane_base + kSCol + 32 * hh, r);
          ptx::tmem_wait_ld();
#pragma unroll
          for (int h = 0; h < 32; ++h) s[32 * hh + h] = valid ? __uint_as_float(r[h]) * c2 : -CUDART_INF_F;
        }
      }
      const float2 mx = reduce_scatter64<true>(s, lane);
      ms.red[warp][2 * lane] = mx.x;
      ms.red[warp][2 * lane + 1] = mx.y;
      ptx::named_bar_sync(1, kSoftmaxThreads);
      if (warp == 0) {
        bool resc = false;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int h = 2 * lane + e;
          const float mt = fmaxf(fmaxf(ms.red[0][h], ms.red[1][h]), fmaxf(ms.red[2][h], ms.red[3][h]));
          const float mo = ms.m_used[h];
          float mn = mo, a = 1.f;
          if (mt > mo + kRescaleThreshold) {      // also true when mo = -inf and mt is finite
            mn = mt;
            a = (mo == -CUDART_INF_F) ? 0.f : exp2f(mo - mn);
            resc |= (mo != -CUDART_INF_F);
          }
          ms.m_used[h] = mn;
          ms.alpha[h] = a;
        }
        const bool any = __any_sync(0xffffffffu, resc);
        if (lane == 0) {
          ms.need_rescale = any && i > 0;
          ms.stop = *abort || !ok;
        }
      }
      ptx::named_bar_sync(2, kSoftmaxThreads);
      if (ms.stop) {
        ok = false;
        break;
      }
      // P row of this token: 64 heads in fp16 (128 B), 128B-swizzled over the rope chunk
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const float4 ma = reinterpret_cast<const float4*>(ms.m_used)[2 * u];
        const float4 mb = reinterpret_cast<const float4*>(ms.m_used)[2 * u + 1];
        const float m[8] = {ma.x, ma.y, ma.z, ma.w, mb.x, mb.y, mb.z, mb.w};
        uint32_t w[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int h = 8 * u + 2 * q;
          // a head with no valid entry yet has m = -inf: its P is 0 (s is -inf there too)
          s[h] = (m[2 * q] == -CUDART_INF_F) ? 0.f : ptx::ex2_approx(s[h] - m[2 * q]);
          s[h + 1] = (m[2 * q + 1] == -CUDART_INF_F) ? 0.f : ptx::ex2_approx(s[h + 1] - m[2 * q + 1]);
          w[q] = f32x2_to_f16x2_sat(s[h], s[h + 1]);
        }
        ptx::sts128_async_only(p_base + swz(t, u), make_uint4(w[0], w[1], w[2], w[3]));
      }
      const float2 ps = reduce_scatter64<false>(s, lane);
      lsum0 = lsum0 * ms.alpha[2 * lane] + ps.x;
      lsum1 = lsum1 * ms.alpha[2 * lane + 1] + ps.y;
      if (ms.need_rescale) {
        for (int j = 0; j < 4; ++j) {
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            uint32_t r[32];
            const uint32_t ta = tmem + lane_base + 64 * j + 32 * hh;
            ptx::tmem_ld32(ta, r);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int q = 0; q < 32; ++q) r[q] = __float_as_uint(__uint_as_float(r[q]) * ms.alpha[32 * hh + q]);
            ptx::tmem_st32(ta, r);
          }
        }
        ptx::tmem_wait_st();
      }
      ptx::tc_fence_before();
      ptx::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&ms.p_ready);
      if (issuer && mma_ok) {
        // PV: O_j^T += V_j^T . P^T for the four 128-dim blocks
        mma_ok = ptx::mbar_wait_bounded(&ms.p_ready, ph, abort);
        if (mma_ok) {
          ptx::tc_fence_after();
          for (int j = 0; j < 4; ++j) {
#pragma unroll
            for (int kk = 0; kk < kTile / 16; ++kk) {
              const uint64_t da = ptx::sw128_desc(k_base + (2 * j) * kKChunkBytes + kk * 2048, kKChunkBytes, 1024);
              // P spans one 64-head atom along N, so its leading offset is never stepped; it is set
              // equal to the stride so that no reading of the two fields leaves the rope chunk.
              const uint64_t db = ptx::sw128_desc(p_base + kk * 2048, 1024, 1024);
              ptx::mma_f16_ss(tmem + 64 * j, da, db, kIdescPV, (i > 0 || kk > 0) ? 1u : 0u);
            }
            ptx::mma_commit(&ms.chunk_free[j]);
          }
          ptx::mma_commit(&ms.pv_done);
        }
      }
      __syncwarp();
    }
    if (range_bad) ms.range_err = 1;
    // epilogue: O / l, lse
    if (ok) ok = ptx::mbar_wait_bounded(&ms.pv_done, (n_tiles - 1) & 1, abort);
    ok = __all_sync(0xffffffffu, ok);
    ptx::tc_fence_after();
    ms.red[warp][2 * lane] = lsum0;
    ms.red[warp][2 * lane + 1] = lsum1;
    ptx::named_bar_sync(1, kSoftmaxThreads);
    if (warp == 0) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int h = 2 * lane + e;
        const float L = ms.red[0][h] + ms.red[1][h] + ms.red[2][h] + ms.red[3][h];
        ms.linv[h] = L > 0.f ? 1.f / L : 0.f;
        ms.lse_out[h] = L > 0.f ? (ms.m_used[h] + log2f(L)) * 0.6931471805599453f : -CUDART_INF_F;
      }
    }
    ptx::named_bar_sync(2, kSoftmaxThreads);
    if (ok) {
      // O / l staged as rows [head][512] (bf16 or fp32) over the K tile, which every MMA has finished
      // reading, then one bulk copy per head row
      const uint32_t elem = p.final_out ? 2u : 4u, row_bytes = 512u * elem;
      unsigned char* stage = base + kQBytes;
      for (int hh = 0; hh < 2; ++hh) {
        float li[32];
#pragma unroll
        for (int q = 0; q < 32; q += 4) {
          const float4 v = reinterpret_cast<const float4*>(ms.linv)[(32 * hh + q) / 4];
          li[q] = v.x; li[q + 1] = v.y; li[q + 2] = v.z; li[q + 3] = v.w;
        }
        for (int j = 0; j < 4; ++j) {
          const uint32_t d = 128u * j + t;
          uint32_t r[32];
          ptx::tmem_ld32(tmem + lane_base + 64 * j + 32 * hh, r);
          ptx::tmem_wait_ld();
          if (p.final_out) {
#pragma unroll
            for (int q = 0; q < 32; ++q) {
              const float o = __uint_as_float(r[q]) * li[q];
              *reinterpret_cast<uint16_t*>(stage + (32 * hh + q) * row_bytes + d * 2) =
                  (uint16_t)(f32x2_to_bf16x2(o, 0.f) & 0xFFFFu);
            }
          } else {
#pragma unroll
            for (int q = 0; q < 32; ++q)
              *reinterpret_cast<float*>(stage + (32 * hh + q) * row_bytes + d * 4) = __uint_as_float(r[q]) * li[q];
          }
        }
      }
      ptx::fence_proxy_async_smem();
      ptx::named_bar_sync(1, kSoftmaxThreads);
      if (t < hg_valid) {
        const size_t h = (size_t)g * kHeads + t;
        void* dst = p.final_out ? static_cast<void*>(p.out + ((size_t)b * p.H + h) * kDLatent)
                                : static_cast<void*>(p.o_part + (((size_t)b * p.nsplit + split) * p.H + h) * kDLatent);
        ptx::bulk_store(dst, k_base + t * row_bytes, row_bytes);
        ptx::bulk_commit();
        if (p.final_out) p.lse[(size_t)b * p.H + h] = ms.lse_out[t];
        else p.lse_part[((size_t)b * p.nsplit + split) * p.H + h] = ms.lse_out[t];
        ptx::bulk_wait_read();
      }
    }
    if (issuer) {
      // drain every MMA issued before the TMEM is released (time limit only)
      ptx::mma_commit(&ms.teardown);
      volatile int no_abort = 0;
      ptx::mbar_wait_bounded(&ms.teardown, 0, &no_abort, 100000000ull);
      if (!mma_ok) *abort = 1;
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (threadIdx.x == 0 && p.err) {
    if (ms.abort) atomicOr(p.err, SMLA_DEVERR_TIMEOUT);
    if (ms.range_err) atomicOr(p.err, SMLA_DEVERR_RANGE);
  }
  if (warp == 0) ptx::tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

bool split_shape_supported(int H, int topk) {
  return (H == 16 || H == 32 || H == 64 || H == 128) && topk >= 1 && topk <= kMaxTopk;
}

int split_heads_per_cta() { return kHeads; }

int split_ctas_per_sm(int H) {
  (void)H;
  return 1;
}

cudaError_t launch_split_tc(const SplitParams& p, cudaStream_t stream) {
  static int configured_device = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_device != dev) {
    e = cudaFuncSetAttribute(split_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  const int head_groups = (p.H + kHeads - 1) / kHeads;
  dim3 grid(p.nsplit, head_groups, p.B);
  split_tc_kernel<<<grid, kThreads, kSmemBytes, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace smla
