// Scalar (CUDA-core, fp32) split kernel: one CTA per (partition, 16-head
// group, query).  Exact fp32 dequantisation and fp32 arithmetic throughout.
// It is the plain correctness baseline the tensor-core kernel is checked and
// timed against; the decode entry points use the tensor-core kernel.
#include <cuda_runtime.h>
#include <math_constants.h>

#include "smla_device.cuh"

namespace smla {
namespace {

constexpr int kHeadsPerCta = 16;
constexpr int kTile = 32;
constexpr int kThreads = 256;
constexpr int kKPitch = kDQK + 1;   // padded row: rows t and t+1 start in different banks

struct SimtSmem {
  float q[kHeadsPerCta][kDQK];
  float k[kTile][kKPitch];
  float s[kHeadsPerCta][kTile];
  long long row[kTile];
};

__global__ void __launch_bounds__(kThreads, 1) split_simt_kernel(SplitParams p) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  SimtSmem& sm = *reinterpret_cast<SimtSmem*>(smem_raw);
  const int split = blockIdx.x, hg = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x;
  const int h_local = tid / 16, lane16 = tid % 16;
  const int h = hg * kHeadsPerCta + h_local;
  const float kLog2e = 1.4426950408889634f;
  const float sl2 = p.sm_scale * kLog2e;        // scores kept in the log2 domain

  const int pos0 = split * p.split_len;
  const int pos1 = min(pos0 + p.split_len, p.topk_n);
  const int seq_len = __ldg(p.seq_lens + b);
  const int32_t* bt_row = p.block_table + (size_t)b * p.max_pages;
  const int32_t* tk_row = p.topk + (size_t)b * p.topk_n;

  for (int i = tid; i < kHeadsPerCta * kDQK; i += kThreads) {
    const int hh = i / kDQK, d = i % kDQK;
    sm.q[hh][d] = bf16_to_f32(p.q[((size_t)b * p.H + hg * kHeadsPerCta + hh) * kDQK + d]);
  }

  float acc[kDLatent / 16];
#pragma unroll
  for (int j = 0; j < kDLatent / 16; ++j) acc[j] = 0.f;
  float m_run = -CUDART_INF_F, l_run = 0.f;

  for (int t0 = pos0; t0 < pos1; t0 += kTile) {
    const int nt = min(kTile, pos1 - t0);
    __syncthreads();   // previous tile fully consumed
    if (tid < kTile) {
      long long r = -1;
      if (tid < nt) r = row_of(bt_row, __ldg(tk_row + t0 + tid), seq_len, p.max_pages, p.num_pages, p.err);
      sm.row[tid] = r;
    }
    __syncthreads();
    // gather + dequantise: 40 16-byte units per row (32 latent, 8 rope)
    for (int u = tid; u < kTile * 40; u += kThreads) {
      const int t = u / 40, c = u % 40;
      const long long r = sm.row[t];
      float* dst = &sm.k[t][c < 32 ? c * 16 : kDLatent + (c - 32) * 8];
      if (r < 0) {
        const int n = c < 32 ? 16 : 8;
        for (int i = 0; i < n; ++i) dst[i] = 0.f;
        continue;
      }
      const uint8_t* rec = p.kv + (size_t)r * kRecordBytes;
      const uint4 raw = __ldg(reinterpret_cast<const uint4*>(rec) + (c < 32 ? c : 33 + (c - 32)));
      const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
      if (c < 32) {
        const float sc = __ldg(reinterpret_cast<const float*>(rec + kDLatent) + c / 8);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 lo = f16x2_to_f32x2(e4m3x2_to_f16x2((uint16_t)(w[i] & 0xFFFF)));
          const float2 hi = f16x2_to_f32x2(e4m3x2_to_f16x2((uint16_t)(w[i] >> 16)));
          dst[4 * i + 0] = lo.x * sc;
          dst[4 * i + 1] = lo.y * sc;
          dst[4 * i + 2] = hi.x * sc;
          dst[4 * i + 3] = hi.y * sc;
        }
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          dst[2 * i + 0] = bf16_to_f32((uint16_t)(w[i] & 0xFFFF));
          dst[2 * i + 1] = bf16_to_f32((uint16_t)(w[i] >> 16));
        }
      }
    }
    __syncthreads();
    // scores: thread (h_local, lane16) -> tokens lane16 and lane16 + 16
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int t = lane16 + 16 * half;
      float dot = 0.f;
      for (int d = 0; d < kDQK; ++d) dot = fmaf(sm.q[h_local][d], sm.k[t][d], dot);
      sm.s[h_local][t] = (t < nt && sm.row[t] >= 0) ? dot * sl2 : -CUDART_INF_F;
    }
    __syncthreads();
    float m_tile = -CUDART_INF_F;
    for (int t = 0; t < kTile; ++t) m_tile = fmaxf(m_tile, sm.s[h_local][t]);
    const float m_new = fmaxf(m_run, m_tile);
    if (m_new == -CUDART_INF_F) continue;           // nothing valid yet for this head
    const float alpha = exp2f(m_run - m_new);        // m_run = -inf -> 0
    l_run *= alpha;
#pragma unroll
    for (int j = 0; j < kDLatent / 16; ++j) acc[j] *= alpha;
    for (int t = 0; t < kTile; ++t) {
      const float pt = exp2f(sm.s[h_local][t] - m_new);
      l_run += pt;
#pragma unroll
      for (int j = 0; j < kDLatent / 16; ++j) acc[j] = fmaf(pt, sm.k[t][lane16 + 16 * j], acc[j]);
    }
    m_run = m_new;
  }

  const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;
  const float lse_v = l_run > 0.f ? (m_run + log2f(l_run)) * 0.6931471805599453f : -CUDART_INF_F;
  if (p.final_out) {
    uint16_t* o = p.out + ((size_t)b * p.H + h) * kDLatent;
#pragma unroll
    for (int j = 0; j < kDLatent / 16; ++j) {
      const uint32_t two = f32x2_to_bf16x2(acc[j] * inv_l, 0.f);
      o[lane16 + 16 * j] = (uint16_t)(two & 0xFFFF);
    }
    if (lane16 == 0) p.lse[(size_t)b * p.H + h] = lse_v;
  } else {
    float* o = p.o_part + (((size_t)b * p.nsplit + split) * p.H + h) * kDLatent;
#pragma unroll
    for (int j = 0; j < kDLatent / 16; ++j) o[lane16 + 16 * j] = acc[j] * inv_l;
    if (lane16 == 0) p.lse_part[((size_t)b * p.nsplit + split) * p.H + h] = lse_v;
  }
}

}  // namespace

cudaError_t launch_split_simt(const SplitParams& p, cudaStream_t stream) {
  const size_t smem = sizeof(SimtSmem);
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(split_simt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  dim3 grid(p.nsplit, p.H / kHeadsPerCta, p.B);
  split_simt_kernel<<<grid, kThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace smla
