// Self-test of the tcgen05 building blocks used by the split kernel, laid out
// exactly as the kernel lays them out (32 heads per CTA):
//   - 128B-swizzled shared-memory fill of the K tile (128 rows x 9 chunks of
//     64 fp16) and of Q (32 rows x 9 chunks);
//   - QK: per 128-dim block b (chunks 2b, 2b+1) and the rope chunk 8,
//       S_b^T[128 x 32] = A_b[128 x 128] . Q_b[32 x 128]^T   (TMEM cols 128+32b)
//     K-major A and B, M=128, N=32;
//   - PV: O_j^T[128 x 32] = A[:, 128j:128j+128]^T . P_j        (TMEM cols 32j)
//     A read MN-major from the same tile, P_j K-major (rows = 32 heads,
//     2 chunks of 64 tokens), M=128, N=32, K=128;
//   - TMEM 32x32b loads.
// Shared memory is allocated at its maximum so that any misread stays inside it.
#include <cuda_runtime.h>
#include <stdint.h>

#include "smla_ptx.cuh"

using namespace smla;

namespace {

constexpr int kHeads = 32;
constexpr int kQChunk = kHeads * 128, kKChunk = 128 * 128, kPBytes = 2 * kHeads * 128;

__device__ __forceinline__ uint32_t swz(uint32_t row, uint32_t unit) { return row * 128u + ((unit ^ (row & 7u)) << 4); }

__global__ void __launch_bounds__(128, 1) selftest_kernel(const uint16_t* A, const uint16_t* Q, const uint16_t* P,
                                                           float* S_out, float* O_out, int* status) {
  extern __shared__ unsigned char raw[];
  unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  const uint32_t q_base = ptx::smem_u32(base), k_base = q_base + 9 * kQChunk, p_base = k_base + 9 * kKChunk;
  __shared__ uint64_t bar_s, bar_o;
  __shared__ uint32_t slot;
  __shared__ int abort_flag;
  const int t = threadIdx.x, warp = t >> 5;
  for (int id = t; id < 128 * 72; id += 128) {
    const int r = id / 72, j = id % 72;
    ptx::sts128(k_base + (j >> 3) * kKChunk + swz(r, j & 7), reinterpret_cast<const uint4*>(A)[id]);
  }
  for (int id = t; id < kHeads * 72; id += 128) {
    const int r = id / 72, j = id % 72;
    ptx::sts128(q_base + (j >> 3) * kQChunk + swz(r, j & 7), reinterpret_cast<const uint4*>(Q)[id]);
  }
  // P given as [4][128 tokens][32 heads]; stored K-major: P_j[h][token], 2 chunks of 64 tokens
  unsigned char* pb = base + 9 * kQChunk + 9 * kKChunk;
  for (int j = 0; j < 4; ++j)
    for (int h = 0; h < kHeads; ++h) {
      const uint32_t off = j * kPBytes + (t >> 6) * (kHeads * 128) + swz(h, (t & 63) >> 3) + (t & 7) * 2;
      *reinterpret_cast<uint16_t*>(pb + off) = P[(j * 128 + t) * kHeads + h];
    }
  if (t == 0) {
    ptx::mbar_init(&bar_s, 1);
    ptx::mbar_init(&bar_o, 1);
    abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0) {
    ptx::tmem_alloc(&slot, 512);
    ptx::tmem_relinquish();
  }
  ptx::fence_proxy_async_smem();
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = slot;
  if (t == 0) {
    for (int c = 0; c < 9; ++c) {
      const int blk = c < 8 ? c >> 1 : 4;
      for (int kk = 0; kk < 4; ++kk)
        ptx::mma_f16_ss(tmem + 128 + 32 * blk, ptx::sw128_desc(k_base + c * kKChunk + kk * 32, 16, 1024),
                        ptx::sw128_desc(q_base + c * kQChunk + kk * 32, 16, 1024),
                        ptx::idesc_f16(128, kHeads, 0, 0), ((c & 1) | kk) != 0);   // first MMA of a block clears it
    }
    ptx::mma_commit(&bar_s);
    for (int j = 0; j < 4; ++j)
      for (int kk = 0; kk < 8; ++kk)
        ptx::mma_f16_ss(tmem + 32 * j, ptx::sw128_desc(k_base + 2 * j * kKChunk + kk * 2048, kKChunk, 1024),
                        ptx::sw128_desc(p_base + j * kPBytes + (kk >> 2) * (kHeads * 128) + (kk & 3) * 32, 16, 1024),
                        ptx::idesc_f16(128, kHeads, 1, 0), kk != 0);
    ptx::mma_commit(&bar_o);
  }
  bool ok = ptx::mbar_wait_bounded(&bar_s, 0, &abort_flag);
  if (ok) ok = ptx::mbar_wait_bounded(&bar_o, 0, &abort_flag);
  ptx::tc_fence_after();
  const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
  uint32_t r[32];
  for (int blk = 0; blk < 5; ++blk) {
    ptx::tmem_ld32(tmem + lane_base + 128 + 32 * blk, r);
    ptx::tmem_wait_ld();
    for (int q = 0; q < 32; ++q) S_out[(blk * 128 + t) * kHeads + q] = __uint_as_float(r[q]);
  }
  for (int j = 0; j < 4; ++j) {
    ptx::tmem_ld32(tmem + lane_base + 32 * j, r);
    ptx::tmem_wait_ld();
    for (int q = 0; q < 32; ++q) O_out[(128 * j + t) * kHeads + q] = __uint_as_float(r[q]);
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (t == 0) *status = ok ? 0 : 1;
  if (warp == 0) ptx::tmem_dealloc(tmem, 512);
}

}  // namespace

extern "C" int tc_selftest(const void* A, const void* Q, const void* P, float* S, float* O, int* status) {
  const int smem = 226 * 1024;   // plus the static barriers, within the 227 KB opt-in limit
  if (cudaFuncSetAttribute(selftest_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return 1;
  selftest_kernel<<<1, 128, smem>>>(static_cast<const uint16_t*>(A), static_cast<const uint16_t*>(Q),
                                    static_cast<const uint16_t*>(P), S, O, status);
  if (cudaGetLastError() != cudaSuccess) return 2;
  return cudaDeviceSynchronize() == cudaSuccess ? 0 : 3;
}
