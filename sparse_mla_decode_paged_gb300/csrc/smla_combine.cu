// Log-sum-exp merge of split partials (a7) and the standalone index->address
// step (a1).
#include <cuda_runtime.h>
#include <math_constants.h>

#include "smla_device.cuh"
#include "smla_ptx.cuh"

namespace smla {
namespace {

constexpr int kCombineThreads = 128;   // 4 output dims per thread

// One CTA per (query, head): lse = ln sum_s exp(lse_s), out = sum_s exp(lse_s - lse) o_s.
// "The 64-Block Barrier", "The Split-K Prescription" (online-softmax merge).  Each thread puts its
// partial-row loads (up to kBatch partitions) in flight before the weights are known, so a call costs
// one round trip to the partials rather than two.
constexpr int kBatch = 8;

__global__ void __launch_bounds__(kCombineThreads) combine_kernel(int H, int nsplit,
                                                                  const float* __restrict__ o_part,
                                                                  const float* __restrict__ lse_part,
                                                                  uint16_t* __restrict__ out,
                                                                  float* __restrict__ lse) {
  const int bh = blockIdx.x;
  const int b = bh / H, h = bh % H;
  const int tid = threadIdx.x;
  __shared__ float w_s[kMaxCombineSplit];
  __shared__ float lse_s;
  // launched as a programmatic dependent of the split kernel: its partials are complete and visible
  // only after this wait (a no-op for an ordinary launch); the next split kernel may be scheduled now
  ptx::griddep_wait();
  if (tid == 0) ptx::griddep_launch_dependents();
  const float4* rows = reinterpret_cast<const float4*>(o_part + ((size_t)b * nsplit * H + h) * kDLatent) + tid;
  const size_t split_stride = (size_t)H * kDLatent / 4;      // float4s between partitions of a row
  float4 v[kBatch];
#pragma unroll
  for (int s = 0; s < kBatch; ++s) v[s] = s < nsplit ? __ldg(rows + s * split_stride) : make_float4(0.f, 0.f, 0.f, 0.f);
  if (tid < 32) {
    float m = -CUDART_INF_F;
    for (int s = tid; s < nsplit; s += 32) m = fmaxf(m, __ldg(lse_part + ((size_t)b * nsplit + s) * H + h));
#pragma unroll
    for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float z = 0.f;
    for (int s = tid; s < nsplit; s += 32) {
      const float l = __ldg(lse_part + ((size_t)b * nsplit + s) * H + h);
      const float w = (m == -CUDART_INF_F) ? 0.f : expf(l - m);   // exp(-inf) = 0 for empty partials
      w_s[s] = w;
      z += w;
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
    const float inv_z = z > 0.f ? 1.f / z : 0.f;
    __syncwarp();
    for (int s = tid; s < nsplit; s += 32) w_s[s] *= inv_z;
    if (tid == 0) lse_s = z > 0.f ? m + logf(z) : -CUDART_INF_F;
  }
  __syncthreads();
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s0 = 0; s0 < nsplit; s0 += kBatch) {
    if (s0 > 0) {
#pragma unroll
      for (int s = 0; s < kBatch; ++s)
        v[s] = s0 + s < nsplit ? __ldg(rows + (s0 + s) * split_stride) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int s = 0; s < kBatch; ++s) {
      if (s0 + s >= nsplit) break;
      const float w = w_s[s0 + s];
      if (w == 0.f) continue;          // a partition with no entry: its row is not read into the sum
      acc.x = fmaf(w, v[s].x, acc.x);
      acc.y = fmaf(w, v[s].y, acc.y);
      acc.z = fmaf(w, v[s].z, acc.z);
      acc.w = fmaf(w, v[s].w, acc.w);
    }
  }
  uint2 packed;
  packed.x = f32x2_to_bf16x2(acc.x, acc.y);
  packed.y = f32x2_to_bf16x2(acc.z, acc.w);
  reinterpret_cast<uint2*>(out + ((size_t)b * H + h) * kDLatent)[tid] = packed;
  if (tid == 0) lse[(size_t)b * H + h] = lse_s;
}

__global__ void gather_rows_kernel(const int32_t* __restrict__ bt, const int32_t* __restrict__ topk,
                                   const int32_t* __restrict__ seq_lens, int B, int topk_n, int max_pages,
                                   int64_t num_pages, int q_per_req, int64_t* __restrict__ rows) {
  const int64_t n = (int64_t)B * topk_n;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const int b = (int)(i / topk_n);
    rows[i] = row_of(bt + (size_t)(b / q_per_req) * max_pages, __ldg(topk + i), __ldg(seq_lens + b), max_pages, num_pages,
                     nullptr);
  }
}

}  // namespace

cudaError_t launch_combine(int B, int H, int nsplit, const float* o_part, const float* lse_part, uint16_t* out,
                           float* lse, cudaStream_t stream) {
  // programmatic stream serialization: the merge's CTAs may be scheduled while the split kernel
  // (which signals at its start) still runs; each waits for the split grid in griddep_wait
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(B * H);
  cfg.blockDim = dim3(kCombineThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, combine_kernel, H, nsplit, o_part, lse_part, out, lse);
}

cudaError_t launch_gather_rows(const int32_t* bt, const int32_t* topk, const int32_t* seq_lens, int B, int topk_n,
                               int max_pages, int64_t num_pages, int q_per_req, int64_t* rows, cudaStream_t stream) {
  const int64_t n = (int64_t)B * topk_n;
  const int threads = 256;
  const int blocks = (int)((n + threads - 1) / threads < 4096 ? (n + threads - 1) / threads : 4096);
  gather_rows_kernel<<<blocks, threads, 0, stream>>>(bt, topk, seq_lens, B, topk_n, max_pages, num_pages, q_per_req,
                                                      rows);
  return cudaGetLastError();
}

}  // namespace smla
