// Self-test of the tcgen05 building blocks used by the split kernel: the
// 128B-swizzled shared-memory fill, the K-major and MN-major smem
// descriptors, the kind::f16 instruction descriptor and the TMEM 32x32b
// loads.  One CTA computes, exactly as the split kernel lays things out,
//   S^T[128 x 64] = A[128 x 576] . Q[64 x 576]^T            (TMEM cols 256..319)
//   O^T[512 x 64] = A[:, 0:512]^T . P[128 x 64]             (TMEM cols 0..255)
// with P written over A's rope chunk after the first product.  Shared memory
// is allocated at its maximum so that any misread stays inside it.
#include <cuda_runtime.h>
#include <stdint.h>

#include "smla_ptx.cuh"

using namespace smla;

namespace {

constexpr int kQChunk = 64 * 128, kKChunk = 128 * 128;

__device__ __forceinline__ uint32_t swz(uint32_t row, uint32_t unit) { return row * 128u + ((unit ^ (row & 7u)) << 4); }

__global__ void __launch_bounds__(128, 1) selftest_kernel(const uint16_t* A, const uint16_t* Q, const uint16_t* P,
                                                           float* S_out, float* O_out, int variant, int* status) {
  extern __shared__ unsigned char raw[];
  unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  const uint32_t q_base = ptx::smem_u32(base), k_base = q_base + 9 * kQChunk;
  __shared__ uint64_t bar_s, bar_o;
  __shared__ uint32_t slot;
  __shared__ int abort_flag;
  const int t = threadIdx.x, warp = t >> 5;
  // fill A (128 rows x 72 units) and Q (64 rows x 72 units), 128B-swizzled per 64-dim chunk
  for (int id = t; id < 128 * 72; id += 128) {
    const int r = id / 72, j = id % 72;
    ptx::sts128(k_base + (j >> 3) * kKChunk + swz(r, j & 7), reinterpret_cast<const uint4*>(A)[id]);
  }
  for (int id = t; id < 64 * 72; id += 128) {
    const int r = id / 72, j = id % 72;
    ptx::sts128(q_base + (j >> 3) * kQChunk + swz(r, j & 7), reinterpret_cast<const uint4*>(Q)[id]);
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
  const uint32_t lbo_v = variant == 0 ? kKChunk : 1024, sbo_v = variant == 0 ? 1024 : kKChunk;
  if (t == 0) {
    for (int c = 0; c < 9; ++c)
      for (int kk = 0; kk < 4; ++kk)
        ptx::mma_f16_ss(tmem + 256, ptx::sw128_desc(k_base + c * kKChunk + kk * 32, 16, 1024),
                        ptx::sw128_desc(q_base + c * kQChunk + kk * 32, 16, 1024), ptx::idesc_f16(128, 64, 0, 0),
                        (c | kk) != 0);
    ptx::mma_commit(&bar_s);
  }
  bool ok = ptx::mbar_wait_bounded(&bar_s, 0, &abort_flag);
  ptx::tc_fence_after();
  // P over the rope chunk: row = token, 64 heads x fp16 = 128 B
  for (int u = 0; u < 8; ++u) ptx::sts128(k_base + 8 * kKChunk + swz(t, u), reinterpret_cast<const uint4*>(P)[t * 8 + u]);
  ptx::fence_proxy_async_smem();
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (t == 0 && ok) {
    for (int j = 0; j < 4; ++j)
      for (int kk = 0; kk < 8; ++kk)
        ptx::mma_f16_ss(tmem + 64 * j, ptx::sw128_desc(k_base + 2 * j * kKChunk + kk * 2048, lbo_v, sbo_v),
                        ptx::sw128_desc(k_base + 8 * kKChunk + kk * 2048, 1024, 1024), ptx::idesc_f16(128, 64, 1, 1),
                        kk != 0);
    ptx::mma_commit(&bar_o);
  }
  if (ok) ok = ptx::mbar_wait_bounded(&bar_o, 0, &abort_flag);
  ptx::tc_fence_after();
  const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
  uint32_t r[32];
  for (int hh = 0; hh < 2; ++hh) {
    ptx::tmem_ld32(tmem + lane_base + 256 + 32 * hh, r);
    ptx::tmem_wait_ld();
    for (int q = 0; q < 32; ++q) S_out[t * 64 + 32 * hh + q] = __uint_as_float(r[q]);
  }
  for (int j = 0; j < 4; ++j)
    for (int hh = 0; hh < 2; ++hh) {
      ptx::tmem_ld32(tmem + lane_base + 64 * j + 32 * hh, r);
      ptx::tmem_wait_ld();
      for (int q = 0; q < 32; ++q) O_out[(128 * j + t) * 64 + 32 * hh + q] = __uint_as_float(r[q]);
    }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (t == 0) *status = ok ? 0 : 1;
  if (warp == 0) ptx::tmem_dealloc(tmem, 512);
}

}  // namespace

extern "C" int tc_selftest(int variant, const void* A, const void* Q, const void* P, float* S, float* O, int* status) {
  const int smem = 226 * 1024;   // plus the static barriers, within the 227 KB opt-in limit
  if (cudaFuncSetAttribute(selftest_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return 1;
  selftest_kernel<<<1, 128, smem>>>(static_cast<const uint16_t*>(A), static_cast<const uint16_t*>(Q),
                                    static_cast<const uint16_t*>(P), S, O, variant, status);
  if (cudaGetLastError() != cudaSuccess) return 2;
  return cudaDeviceSynchronize() == cudaSuccess ? 0 : 3;
}
