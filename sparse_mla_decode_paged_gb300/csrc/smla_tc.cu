// Tensor-core split kernel (sm_103a): tcgen05 MMAs with TMEM accumulators.
//
// One CTA per (partition s of the top-k list, group of 32 heads, query b).
// The partition is walked in tiles of 128 top-k entries:
//
//   gather warps (8)   index -> row through the block table (a1); 16-byte
//                      streaming loads of each 656-byte record into
//                      registers; the E4M3 latent codes are converted to fp16
//                      exactly (every E4M3 value is an fp16 value) and the bf16
//                      rope to fp16 (a2), stored 128B-swizzled into the K tile
//                      (9 chunks of 64 dims); the four fp32 scales of each
//                      token go to shared memory.  The next tile's loads are
//                      issued as soon as a tile is stored.
//   MMA (warp 0 lane 0) QK per scale block: S_b^T[128 tok x 32 heads] =
//                      K_b . Q_b^T for the four 128-dim latent blocks and the
//                      rope (a3), M=128 N=32, five fp32 TMEM accumulators;
//                      then O_j^T[128 dims x 32 heads] += V_j^T . P_j^T for the
//                      four dim blocks (a5), V_j^T being the same codes read
//                      MN-major and P_j = P scaled by the tokens' block-j scale.
//   softmax warps (4)  load Q once (fp16, swizzled); then one TMEM lane
//                      (token) per thread: exact score
//                      s = sum_b scale_b S_b + S_rope in fp32; per-head
//                      running max over the tile (warp reduce-scatter + shared
//                      memory), P = exp2(s - m) (a4), the four scaled P_j in
//                      fp16, lazy rescale of O when a head's max grows by more
//                      than 2^8, and the epilogue (a6): O / l and lse.
//
// Keeping the latent codes unscaled makes every product in QK exact, so the
// scores carry fp32 accumulation error only; the per-block scales enter in
// fp32 in the softmax and, for PV, through P_j.  P_j carries a per-CTA power
// of two F_j (fixed at the first tile with data) so that it sits in the fp16
// normal range; the epilogue divides it out.
//
// QK of a tile, its softmax and its PV are sequential (one K tile), so the
// MMAs are issued by lane 0 of the first softmax warp between its softmax
// steps; no warp is spent on issue only.
//
// Shared memory: Q 36 KB (32 heads x 576 fp16) + K tile 144 KB (128 x 576
// fp16) + P 32 KB (4 x 32 heads x 128 tokens fp16) + barriers: one CTA per
// SM, 12 warps.  TMEM: O^T in columns 0..127, S in 128..287 (512 allocated).
// Sources: "The 64-Block Barrier" ("The Smoking Gun", "The Split-K
// Prescription"); "Inside the Decode Performance Investigation" (Task 1).
#include <cuda_runtime.h>
#include <math_constants.h>

#include "smla_device.cuh"
#include "smla_ptx.cuh"

namespace smla {
namespace {

constexpr int kTile = 128;                 // top-k entries per tile (MMA M)
constexpr int kHeads = 32;                 // heads per CTA (MMA N), zero rows past the valid heads
constexpr int kChunks = 9;                 // 576 dims / 64
constexpr int kQChunkBytes = kHeads * 128;               // 4 KB
constexpr int kKChunkBytes = kTile * 128;                // 16 KB
constexpr int kPChunkBytes = kHeads * 128;               // 32 heads x 64 tokens
constexpr int kPBytes = 2 * kPChunkBytes;                // one P_j: 2 chunks of 64 tokens
constexpr int kQBytes = kChunks * kQChunkBytes;          // 36864
constexpr int kKBytes = kChunks * kKChunkBytes;          // 147456
constexpr int kPAllBytes = 4 * kPBytes;                  // 32768
// 12 warps = 3 per SM sub-partition, which leaves 168 registers per thread.
constexpr int kThreads = 384;
constexpr int kSoftmaxThreads = 128;       // warps 0..3 (TMEM lane quadrants 0..3); lane 0 of warp 0 issues MMAs
constexpr int kGatherThreads = 256;        // warps 4..11
constexpr int kGatherWarps = kGatherThreads / 32;
constexpr int kSoftmaxWarps = kSoftmaxThreads / 32;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSCol = 128;            // S_b at kSCol + 32 b, b = 0..4 (4 = rope)
constexpr float kRescaleThreshold = 8.0f;  // log2 units: P stays <= 256
constexpr float kFp16Max = 65504.0f;

constexpr uint32_t kIdescQK = ptx::idesc_f16(128, kHeads, 0, 0);
constexpr uint32_t kIdescPV = ptx::idesc_f16(128, kHeads, 1, 0);

struct Misc {
  uint64_t q_ready, meta_ready, s_full, p_ready, pv_done, teardown;
  uint64_t kv_ready[5];                    // latent blocks 0..3 (two chunks each), rope
  uint64_t chunk_free[4];
  uint32_t tmem_slot;
  int abort;
  int need_rescale;
  int stop;
  int range_err;
  int f_set;
  int scmax[4];                            // running max of the block scales (float bits, >= 0)
  float f[4];                              // power-of-two factor carried by P_j
  float red[4][kHeads];
  float m_used[kHeads];
  float alpha[kHeads];
  float lse_out[kHeads];
  float linv[kHeads];
  float sc[kTile][4];                      // block scales of the tile's tokens
  unsigned char valid[kTile];
};

constexpr size_t kSmemBytes = 1024 + kQBytes + kKBytes + kPAllBytes + sizeof(Misc);

__device__ __forceinline__ uint32_t swz(uint32_t row, uint32_t unit) {  // byte offset in a 128B-swizzled chunk
  return row * 128u + ((unit ^ (row & 7u)) << 4);
}

// 4 E4M3 codes -> 4 fp16 (exact).
__device__ __forceinline__ uint2 codes4(uint32_t w) {
  return make_uint2(e4m3x2_to_f16x2((uint16_t)(w & 0xFFFFu)), e4m3x2_to_f16x2((uint16_t)(w >> 16)));
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

__device__ __forceinline__ uint16_t f32_to_f16_sat(float x) {
  return (uint16_t)(f32x2_to_f16x2_sat(x, 0.f) & 0xFFFFu);
}

// Warp reduce-scatter over 32 per-thread values: afterwards lane l holds the
// reduction over the warp's 32 threads of column l.
template <bool kMax>
__device__ __forceinline__ float reduce_scatter32(const float (&v)[32], int lane) {
  float a[16];
  {
    const bool hi = lane & 16;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float send = hi ? v[i] : v[16 + i];
      const float keep = hi ? v[16 + i] : v[i];
      const float r = __shfl_xor_sync(0xffffffffu, send, 16);
      a[i] = kMax ? fmaxf(keep, r) : keep + r;
    }
  }
#pragma unroll
  for (int span = 8, x = 8; span >= 1; span >>= 1, x >>= 1) {
    const bool hi = lane & x;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (i < span) {
        const float send = hi ? a[i] : a[span + i];
        const float keep = hi ? a[span + i] : a[i];
        const float r = __shfl_xor_sync(0xffffffffu, send, x);
        a[i] = kMax ? fmaxf(keep, r) : keep + r;
      }
    }
  }
  return a[0];
}

__global__ void __launch_bounds__(kThreads, 1) split_tc_kernel(const SplitParams p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Misc& ms = *reinterpret_cast<Misc*>(base + kQBytes + kKBytes + kPAllBytes);
  volatile int* abort = &ms.abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int pos0 = split * p.split_len;
  const int pos_end = min(pos0 + p.split_len, p.topk_n);
  const int n_tiles = pos_end > pos0 ? (pos_end - pos0 + kTile - 1) / kTile : 0;
  const int hg_valid = min(kHeads, p.H - kHeads * g);
  const uint32_t q_base = ptx::smem_u32(base);
  const uint32_t k_base = q_base + kQBytes;
  const uint32_t p_base = k_base + kKBytes;

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
    ptx::mbar_init(&ms.meta_ready, kGatherWarps);
    ptx::mbar_init(&ms.s_full, 1);
    ptx::mbar_init(&ms.p_ready, kSoftmaxWarps);
    ptx::mbar_init(&ms.pv_done, 1);
    ptx::mbar_init(&ms.teardown, 1);
    for (int c = 0; c < 5; ++c) ptx::mbar_init(&ms.kv_ready[c], kGatherWarps);
    for (int j = 0; j < 4; ++j) ptx::mbar_init(&ms.chunk_free[j], 1);
    ms.abort = 0;
    ms.need_rescale = 0;
    ms.stop = 0;
    ms.range_err = 0;
    ms.f_set = 0;
    for (int j = 0; j < 4; ++j) {
      ms.scmax[j] = 0;
      ms.f[j] = 1.f;
    }
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
    // ------------------------------------------------------------------ gather + convert
    const int gid = threadIdx.x - kSoftmaxThreads;
    const int tl = gid >> 1, half = gid & 1;
    const int seq_len = __ldg(p.seq_lens + b);
    const int32_t* bt_row = p.block_table + (size_t)b * p.max_pages;
    const int32_t* tk_row = p.topk + (size_t)b * p.topk_n;
    int range_bad = 0;

    uint4 lat[16], rope[4], scv = make_uint4(0, 0, 0, 0);
    auto load_row = [&](int64_t r) {
      if (r >= 0) {
        const unsigned char* rec = p.kv + r * kRecordBytes;
#pragma unroll
        for (int k = 0; k < 16; ++k) lat[k] = ptx::ldg_stream(rec + 16 * (2 * k + half));
#pragma unroll
        for (int k = 0; k < 4; ++k) rope[k] = ptx::ldg_stream(rec + 528 + 16 * (2 * k + half));
        scv = ptx::ldg_stream(rec + 512);
      }
    };
    auto topk_at = [&](int i) -> int {
      const int pos = pos0 + i * kTile + tl;
      return pos < pos_end ? __ldg(tk_row + pos) : -1;
    };

    int64_t row = row_of(bt_row, topk_at(0), seq_len, p.max_pages, p.num_pages, p.err);
    load_row(row);

    bool ok = true;
    for (int i = 0; ok && i < n_tiles; ++i) {
      const int t_next = (i + 1 < n_tiles) ? topk_at(i + 1) : -1;
      const bool valid = row >= 0;
      // latent block j = chunks 2j, 2j+1; this thread owns units 4c+half and 4c+2+half of chunk c
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (i > 0 && !__all_sync(0xffffffffu, ptx::mbar_wait_bounded(&ms.chunk_free[j], (i - 1) & 1, abort))) {
          ok = false;
          break;
        }
        if (j == 0) {
          float sv[4] = {valid ? __uint_as_float(scv.x) : 0.f, valid ? __uint_as_float(scv.y) : 0.f,
                         valid ? __uint_as_float(scv.z) : 0.f, valid ? __uint_as_float(scv.w) : 0.f};
          if (half == 0) {
            ms.valid[tl] = valid;
            ms.sc[tl][0] = sv[0]; ms.sc[tl][1] = sv[1]; ms.sc[tl][2] = sv[2]; ms.sc[tl][3] = sv[3];
          }
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            float m = fabsf(sv[q]);
#pragma unroll
            for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
            sv[q] = m;
          }
          __syncwarp();
          if (lane == 0) {
#pragma unroll
            for (int q = 0; q < 4; ++q)
              if (sv[q] > 0.f) atomicMax(&ms.scmax[q], __float_as_int(sv[q]));
            ptx::mbar_arrive(&ms.meta_ready);
          }
        }
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const int c = 2 * j + cc;
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int k = 2 * c + e;                  // lat[] index: unit u = 2k + half
            const int uc = (2 * k + half) & 3;        // 16-dim unit within the chunk
            uint4 lo = make_uint4(0, 0, 0, 0), hi = make_uint4(0, 0, 0, 0);
            if (valid) {
              const uint2 a0 = codes4(lat[k].x), a1 = codes4(lat[k].y), a2 = codes4(lat[k].z), a3 = codes4(lat[k].w);
              lo = make_uint4(a0.x, a0.y, a1.x, a1.y);
              hi = make_uint4(a2.x, a2.y, a3.x, a3.y);
            }
            const uint32_t cb = k_base + c * kKChunkBytes;
            ptx::sts128(cb + swz(tl, 2 * uc), lo);
            ptx::sts128(cb + swz(tl, 2 * uc + 1), hi);
          }
        }
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&ms.kv_ready[j]);
      }
      if (!ok) break;
      // rope chunk: free once the previous tile's PV is done (all of its MMAs have completed)
      if (i > 0 && !__all_sync(0xffffffffu, ptx::mbar_wait_bounded(&ms.pv_done, (i - 1) & 1, abort))) {
        ok = false;
        break;
      }
      {
        const uint32_t cb = k_base + 8 * kKChunkBytes;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int r = 2 * k + half;
          ptx::sts128(cb + swz(tl, r), valid ? bf8_to_h8(rope[k], range_bad) : make_uint4(0, 0, 0, 0));
        }
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&ms.kv_ready[4]);
      }
      if (i + 1 < n_tiles) {
        row = row_of(bt_row, t_next, seq_len, p.max_pages, p.num_pages, p.err);
        load_row(row);
      }
    }
    if (range_bad) ms.range_err = 1;
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
      for (int k0 = 0; k0 < 18; k0 += 9) {
        uint4 v[9];
#pragma unroll
        for (int k = 0; k < 9; ++k) {
          const int id = t + kSoftmaxThreads * (k0 + k);
          const int n = id / 72, j = id % 72;
          v[k] = n < hg_valid ? __ldg(reinterpret_cast<const uint4*>(qg + (size_t)n * kDQK) + j) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int k = 0; k < 9; ++k) {
          const int id = t + kSoftmaxThreads * (k0 + k);
          const int n = id / 72, j = id % 72;
          ptx::sts128(q_base + (j >> 3) * kQChunkBytes + swz(n, j & 7), bf8_to_h8(v[k], range_bad));
        }
      }
      ptx::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&ms.q_ready);
    }
    const float c2 = p.sm_scale * 1.4426950408889634f;
    const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
    float lsum = 0.f;                             // this warp's sum for head `lane`
    bool ok = true;
    bool mma_ok = true;                           // issuer only
    if (issuer) mma_ok = ptx::mbar_wait_bounded(&ms.q_ready, 0, abort);
    for (int i = 0; i < n_tiles; ++i) {
      const uint32_t ph = i & 1;
      if (issuer && mma_ok) {
        // QK: latent block j (chunks 2j, 2j+1) into S_j, then the rope chunk into S_4
        for (int j = 0; mma_ok && j < 5; ++j) {
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
              // the first MMA into a block's accumulator overwrites it
              ptx::mma_f16_ss(tmem + kSCol + 32 * j, da, db, kIdescQK, (cc | kk) != 0);
            }
          }
        }
        if (mma_ok) ptx::mma_commit(&ms.s_full);
      }
      ok = ptx::mbar_wait_bounded(&ms.meta_ready, ph, abort) && ptx::mbar_wait_bounded(&ms.s_full, ph, abort);
      ok = __all_sync(0xffffffffu, ok);
      ptx::tc_fence_after();
      const float scb[4] = {ms.sc[t][0], ms.sc[t][1], ms.sc[t][2], ms.sc[t][3]};
      float s[32];
      {
        uint32_t r[32];
        ptx::tmem_ld32(tmem + lane_base + kSCol + 128, r);   // rope accumulator
        ptx::tmem_wait_ld();
#pragma unroll
        for (int h = 0; h < 32; ++h) s[h] = __uint_as_float(r[h]);
#pragma unroll
        for (int bb = 0; bb < 4; ++bb) {
          ptx::tmem_ld32(tmem + lane_base + kSCol + 32 * bb, r);
          ptx::tmem_wait_ld();
#pragma unroll
          for (int h = 0; h < 32; ++h) s[h] = fmaf(scb[bb], __uint_as_float(r[h]), s[h]);
        }
      }
      const bool valid = ms.valid[t];
#pragma unroll
      for (int h = 0; h < 32; ++h) s[h] = valid ? s[h] * c2 : -CUDART_INF_F;
      const float mx = reduce_scatter32<true>(s, lane);
      ms.red[warp][lane] = mx;
      ptx::named_bar_sync(1, kSoftmaxThreads);
      if (warp == 0) {
        const int h = lane;
        const float mt = fmaxf(fmaxf(ms.red[0][h], ms.red[1][h]), fmaxf(ms.red[2][h], ms.red[3][h]));
        const float mo = ms.m_used[h];
        float mn = mo, a = 1.f;
        bool resc = false;
        if (mt > mo + kRescaleThreshold) {        // also true when mo = -inf and mt is finite
          mn = mt;
          a = (mo == -CUDART_INF_F) ? 0.f : exp2f(mo - mn);
          resc = (mo != -CUDART_INF_F);
        }
        ms.m_used[h] = mn;
        ms.alpha[h] = a;
        const bool any = __any_sync(0xffffffffu, resc);
        // P_j factor: fixed at the first tile that holds data, so that F_j * max scale is in [0.5, 1)
        const bool set_now = !ms.f_set && (ms.scmax[0] | ms.scmax[1] | ms.scmax[2] | ms.scmax[3]) != 0;
        if (set_now && lane < 4) {
          const float mxs = __int_as_float(ms.scmax[lane]);
          int e = 0;
          if (mxs > 0.f) frexpf(mxs, &e);
          ms.f[lane] = ldexpf(1.f, -e);
        }
        __syncwarp();
        if (lane == 0) {
          if (set_now) ms.f_set = 1;
          ms.need_rescale = any && i > 0;
          ms.stop = *abort || !ok;
        }
      }
      ptx::named_bar_sync(2, kSoftmaxThreads);
      if (ms.stop) {
        ok = false;
        break;
      }
      // P = exp2(s - m), in place
#pragma unroll
      for (int h = 0; h < 32; ++h) {
        const float m = ms.m_used[h];
        s[h] = (m == -CUDART_INF_F) ? 0.f : exp2f(s[h] - m);
      }
      // P_j[h][t] = p * scale_j * F_j, K-major (rows = heads, 2 chunks of 64 tokens)
      {
        const uint32_t tok_off = (t >> 6) * kPChunkBytes + (t & 7) * 2;
        const uint32_t unit = (t & 63) >> 3;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float f = scb[j] * ms.f[j];
          range_bad |= !(f * 256.f <= kFp16Max);
          unsigned char* pj = base + kQBytes + kKBytes + j * kPBytes + tok_off;
#pragma unroll
          for (int h = 0; h < 32; ++h) *reinterpret_cast<uint16_t*>(pj + swz(h, unit)) = f32_to_f16_sat(s[h] * f);
        }
      }
      const float ps = reduce_scatter32<false>(s, lane);
      lsum = lsum * ms.alpha[lane] + ps;
      if (ms.need_rescale) {
        for (int j = 0; j < 4; ++j) {
          uint32_t r[32];
          const uint32_t ta = tmem + lane_base + 32 * j;
          ptx::tmem_ld32(ta, r);
          ptx::tmem_wait_ld();
#pragma unroll
          for (int q = 0; q < 32; ++q) r[q] = __float_as_uint(__uint_as_float(r[q]) * ms.alpha[q]);
          ptx::tmem_st32(ta, r);
        }
        ptx::tmem_wait_st();
      }
      ptx::tc_fence_before();
      ptx::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&ms.p_ready);
      if (issuer && mma_ok) {
        // PV: O_j^T += V_j^T . P_j^T for the four 128-dim blocks
        mma_ok = ptx::mbar_wait_bounded(&ms.p_ready, ph, abort);
        if (mma_ok) {
          ptx::tc_fence_after();
          for (int j = 0; j < 4; ++j) {
#pragma unroll
            for (int kk = 0; kk < kTile / 16; ++kk) {
              const uint64_t da = ptx::sw128_desc(k_base + (2 * j) * kKChunkBytes + kk * 2048, kKChunkBytes, 1024);
              const uint64_t db =
                  ptx::sw128_desc(p_base + j * kPBytes + (kk >> 2) * kPChunkBytes + (kk & 3) * 32, 16, 1024);
              ptx::mma_f16_ss(tmem + 32 * j, da, db, kIdescPV, (i > 0 || kk > 0) ? 1u : 0u);
            }
            ptx::mma_commit(&ms.chunk_free[j]);
          }
          ptx::mma_commit(&ms.pv_done);
        }
      }
      __syncwarp();
    }
    if (range_bad) ms.range_err = 1;
    // epilogue: O / (l F_j), lse
    if (ok) ok = ptx::mbar_wait_bounded(&ms.pv_done, (n_tiles - 1) & 1, abort);
    ok = __all_sync(0xffffffffu, ok);
    ptx::tc_fence_after();
    ms.red[warp][lane] = lsum;
    ptx::named_bar_sync(1, kSoftmaxThreads);
    if (warp == 0) {
      const int h = lane;
      const float L = ms.red[0][h] + ms.red[1][h] + ms.red[2][h] + ms.red[3][h];
      ms.linv[h] = L > 0.f ? 1.f / L : 0.f;
      ms.lse_out[h] = L > 0.f ? (ms.m_used[h] + log2f(L)) * 0.6931471805599453f : -CUDART_INF_F;
    }
    ptx::named_bar_sync(2, kSoftmaxThreads);
    if (ok) {
      for (int j = 0; j < 4; ++j) {
        const int d = 128 * j + t;
        const float finv = 1.f / ms.f[j];
        uint32_t r[32];
        ptx::tmem_ld32(tmem + lane_base + 32 * j, r);
        ptx::tmem_wait_ld();
#pragma unroll
        for (int q = 0; q < 32; ++q) {
          if (q < hg_valid) {
            const float o = __uint_as_float(r[q]) * (ms.linv[q] * finv);
            const size_t h = (size_t)g * kHeads + q;
            if (p.final_out) {
              p.out[((size_t)b * p.H + h) * kDLatent + d] = (uint16_t)(f32x2_to_bf16x2(o, 0.f) & 0xFFFFu);
            } else {
              p.o_part[(((size_t)b * p.nsplit + split) * p.H + h) * kDLatent + d] = o;
            }
          }
        }
      }
      if (t < hg_valid) {
        const size_t h = (size_t)g * kHeads + t;
        if (p.final_out) p.lse[(size_t)b * p.H + h] = ms.lse_out[t];
        else p.lse_part[((size_t)b * p.nsplit + split) * p.H + h] = ms.lse_out[t];
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
