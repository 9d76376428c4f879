// FP8 KV append: the write side of the paged latent cache that the decode reads (the step before the
// hot path).  Each new token's 512-dim latent is quantised per 128-dim block to E4M3 with a float32
// scale amax / 448, its 64-dim rope copied as bf16, and the 656-byte record written at the page the
// block table gives for its position ("Inside the Decode Performance Investigation", Task 1: the
// paged FP8 latent cache with per-block scales; record layout [512 x E4M3 | 4 x fp32 | 64 x bf16]).
//
// One CTA of 128 threads per token: warp w quantises block w (4 values per lane), so the block amax
// is a warp reduction and each warp writes its 128 code bytes as one coalesced 128-byte store; lane 0
// of each warp writes the block's scale, threads 0..7 copy the rope.
#include <cuda_runtime.h>

#include "smla_device.cuh"
#include "smla_internal.h"

namespace smla {
namespace {

constexpr int kAppendThreads = 128;

// fp32 pair -> two E4M3 codes (round to nearest even, saturating to +-448), low byte = a.
__device__ __forceinline__ uint16_t f32x2_to_e4m3x2(float a, float b) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(b), "f"(a));
  return r;
}

__global__ void __launch_bounds__(kAppendThreads) kv_append_kernel(AppendParams p) {
  const int tok = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int req = p.requests ? __ldg(p.requests + tok) : tok;
  const int pos = __ldg(p.positions + tok);
  if (req < 0 || req >= p.num_requests || pos < 0 || (pos >> 6) >= p.max_pages) {
    if (threadIdx.x == 0 && p.err) atomicOr(p.err, SMLA_DEVERR_PAGE_RANGE);
    return;
  }
  const int page = __ldg(p.block_table + (size_t)req * p.max_pages + (pos >> 6));
  if (page < 0 || (int64_t)page >= p.num_pages) {
    if (threadIdx.x == 0 && p.err) atomicOr(p.err, SMLA_DEVERR_PAGE_RANGE);
    return;
  }
  unsigned char* rec = p.kv + ((int64_t)page * kPageSize + (pos & (kPageSize - 1))) * kRecordBytes;

  // latent: thread t holds dims 4t .. 4t + 3 (block t / 32 = its warp)
  const uint2 raw = __ldg(reinterpret_cast<const uint2*>(p.latent + (size_t)tok * kDLatent) + threadIdx.x);
  const float x[4] = {__uint_as_float(raw.x << 16), __uint_as_float(raw.x & 0xFFFF0000u),
                      __uint_as_float(raw.y << 16), __uint_as_float(raw.y & 0xFFFF0000u)};
  float amax = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
#pragma unroll
  for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float scale = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
  const uint16_t c01 = f32x2_to_e4m3x2(__fdiv_rn(x[0], scale), __fdiv_rn(x[1], scale));
  const uint16_t c23 = f32x2_to_e4m3x2(__fdiv_rn(x[2], scale), __fdiv_rn(x[3], scale));
  reinterpret_cast<uint32_t*>(rec)[threadIdx.x] = (uint32_t)c01 | ((uint32_t)c23 << 16);
  if (lane == 0) reinterpret_cast<float*>(rec + kDLatent)[warp] = scale;
  if (threadIdx.x < 8)
    reinterpret_cast<uint4*>(rec + kDLatent + 16)[threadIdx.x] =
        __ldg(reinterpret_cast<const uint4*>(p.rope + (size_t)tok * kDRope) + threadIdx.x);
}

}  // namespace

cudaError_t launch_kv_append(const AppendParams& p, cudaStream_t stream) {
  if (p.tokens == 0) return cudaSuccess;
  kv_append_kernel<<<p.tokens, kAppendThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace smla
