// Self-test of the tcgen05 building blocks used by the split kernel, laid out
// exactly as the kernel lays them out (64 heads per CTA):
//   - 128B-swizzled shared-memory fill of the K tile (128 rows x 9 chunks of
//     64 fp16) and of Q (64 rows x 9 chunks);
//   - QK: S^T[128 x 64] = A[128 x 576] . Q[64 x 576]^T, K-major smem A and B,
//     M=128 N=64 (TMEM cols 256..319);
//   - correction: S^T += L[128 x 512] . Q[:, 0:512]^T with L taken from TMEM
//     (cols 320..447) in two passes of 256 dims, each written by tcgen05.st;
//   - PV: O^T[512 x 64] = A[:, 0:512]^T . P, A read MN-major from the same
//     tile, P MN-major over the rope chunk (TMEM cols 0..255);
//   - TMEM 32x32b loads and stores.
// Shared memory is allocated at its maximum so that any misread stays inside it.
#include <cuda_runtime.h>
#include <stdint.h>

#include "smla_ptx.cuh"

using namespace smla;

namespace {

constexpr int kHeads = 64;
constexpr int kQChunk = kHeads * 128, kKChunk = 128 * 128;

__device__ __forceinline__ uint32_t swz(uint32_t row, uint32_t unit) { return row * 128u + ((unit ^ (row & 7u)) << 4); }

__global__ void __launch_bounds__(128, 1) selftest_kernel(const uint16_t* A, const uint16_t* Q, const uint16_t* L,
                                                           const uint16_t* P, float* S_out, float* O_out,
                                                           int* status) {
  extern __shared__ unsigned char raw[];
  unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  const uint32_t q_base = ptx::smem_u32(base), k_base = q_base + 9 * kQChunk;
  __shared__ uint64_t bar[4];
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
  if (t == 0) {
    for (int i = 0; i < 4; ++i) ptx::mbar_init(&bar[i], 1);
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
  const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
  const uint32_t idesc_qk = ptx::idesc_f16(128, kHeads, 0, 0);
  bool ok = true;
  // QK from shared memory
  if (t == 0) {
    for (int c = 0; c < 9; ++c)
      for (int kk = 0; kk < 4; ++kk)
        ptx::mma_f16_ss(tmem + 256, ptx::sw128_desc(k_base + c * kKChunk + kk * 32, 16, 1024),
                        ptx::sw128_desc(q_base + c * kQChunk + kk * 32, 16, 1024), idesc_qk, (c | kk) != 0);
  }
  // correction from TMEM, two passes of 256 dims
  for (int pass = 0; pass < 2 && ok; ++pass) {
    if (pass == 1) {
      ok = ptx::mbar_wait_bounded(&bar[0], 0, &abort_flag);   // pass 0 MMAs done: TMEM L may be overwritten
      ptx::tc_fence_after();
    }
    for (int cb = 0; cb < 8; ++cb) {   // 8 x 16 columns = 256 fp16 of row t
      uint32_t r[16];
      for (int q = 0; q < 16; ++q) {
        const int d = pass * 256 + cb * 32 + 2 * q;
        r[q] = (uint32_t)L[t * 512 + d] | ((uint32_t)L[t * 512 + d + 1] << 16);
      }
      ptx::tmem_st16(tmem + lane_base + 320 + 16 * cb, r);
    }
    ptx::tmem_wait_st();
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (t == 0) {
      for (int kk = 0; kk < 16; ++kk) {
        const int c = pass * 4 + (kk >> 2);
        ptx::mma_f16_ts(tmem + 256, tmem + 320 + 8 * kk,
                        ptx::sw128_desc(q_base + c * kQChunk + (kk & 3) * 32, 16, 1024), idesc_qk, 1u);
      }
      ptx::mma_commit(&bar[pass]);
    }
  }
  if (ok) ok = ptx::mbar_wait_bounded(&bar[1], 0, &abort_flag);
  ptx::tc_fence_after();
  // P over the rope chunk: row = token, 64 heads x fp16 = 128 B (MN-major for the PV B operand)
  for (int u = 0; u < 8; ++u) ptx::sts128(k_base + 8 * kKChunk + swz(t, u), reinterpret_cast<const uint4*>(P)[t * 8 + u]);
  ptx::fence_proxy_async_smem();
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (t == 0 && ok) {
    for (int j = 0; j < 4; ++j)
      for (int kk = 0; kk < 8; ++kk)
        ptx::mma_f16_ss(tmem + 64 * j, ptx::sw128_desc(k_base + 2 * j * kKChunk + kk * 2048, kKChunk, 1024),
                        ptx::sw128_desc(k_base + 8 * kKChunk + kk * 2048, 1024, 1024), ptx::idesc_f16(128, kHeads, 1, 1),
                        kk != 0);
    ptx::mma_commit(&bar[2]);
  }
  if (ok) ok = ptx::mbar_wait_bounded(&bar[2], 0, &abort_flag);
  ptx::tc_fence_after();
  uint32_t r[32];
  for (int hh = 0; hh < 2; ++hh) {
    ptx::tmem_ld32(tmem + lane_base + 256 + 32 * hh, r);
    ptx::tmem_wait_ld();
    for (int q = 0; q < 32; ++q) S_out[t * kHeads + 32 * hh + q] = __uint_as_float(r[q]);
  }
  for (int j = 0; j < 4; ++j)
    for (int hh = 0; hh < 2; ++hh) {
      ptx::tmem_ld32(tmem + lane_base + 64 * j + 32 * hh, r);
      ptx::tmem_wait_ld();
      for (int q = 0; q < 32; ++q) O_out[(128 * j + t) * kHeads + 32 * hh + q] = __uint_as_float(r[q]);
    }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (t == 0) *status = ok ? 0 : 1;
  if (warp == 0) ptx::tmem_dealloc(tmem, 512);
}

}  // namespace

extern "C" int tc_selftest(const void* A, const void* Q, const void* L, const void* P, float* S, float* O,
                           int* status) {
  const int smem = 226 * 1024;   // plus the static barriers, within the 227 KB opt-in limit
  if (cudaFuncSetAttribute(selftest_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return 1;
  selftest_kernel<<<1, 128, smem>>>(static_cast<const uint16_t*>(A), static_cast<const uint16_t*>(Q),
                                    static_cast<const uint16_t*>(L), static_cast<const uint16_t*>(P), S, O, status);
  if (cudaGetLastError() != cudaSuccess) return 2;
  return cudaDeviceSynchronize() == cudaSuccess ? 0 : 3;
}
