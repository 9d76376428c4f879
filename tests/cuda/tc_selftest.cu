// Self-test of the split kernel's tcgen05 building blocks, using the kernel's own layout header
// (smla_split_layout.cuh: swizzled offsets, matrix descriptors, MMA issuers), for 16, 32 and 64
// heads per CTA:
//   - the K tile (128 tokens x 9 chunks of 64 fp16 dims) and Q (NH rows x 9 chunks), 128B-swizzled;
//   - QK as the kernel issues it: latent block b (chunks 2b, 2b + 1) into score buffer b, the rope
//     chunk accumulated into buffer 0 (S^T[128 x NH], TMEM columns 4 NH + NH b);
//   - PV as the kernel issues it: block 0 with its P * mant operand in the rope chunk, then blocks
//     1..3 with their operands in chunks 0, rope and 1 (written after block 0's PV completed), each
//     O^T_b[128 x NH] = K'_b^T . Pm_b with the K tile read MN-major and Pm MN-major with an NH * 2-byte
//     swizzle span (128, 64 or 32 bytes);
//   - TMEM 32x32b loads of 16 and 32 columns.
// Every wait is bounded (1 s of the global timer); a timeout sets *status and skips the rest.
#include <cuda_runtime.h>
#include <stdint.h>

#include "smla_ptx.cuh"
#include "smla_split_layout.cuh"

using namespace smla;

namespace {

template <int NH>
constexpr size_t selftest_smem() { return 1024 + Cfg<NH>::kQBytes + kKBytes; }

// Each thread reads its TMEM lane (token or dim) of `cols` consecutive columns from `col0` into dst.
template <int NH>
__device__ void read_cols(uint32_t tmem, uint32_t col0, int cols, float* dst) {
  const int warp = threadIdx.x >> 5;
  const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
  for (int c = 0; c < cols; c += (NH == 16 ? 16 : 32)) {
    if constexpr (NH == 16) {
      uint32_t r[16];
      ptx::tmem_ld16(tmem + lane_base + col0 + c, r);
      ptx::tmem_wait_ld();
      for (int h = 0; h < 16; ++h) dst[c + h] = __uint_as_float(r[h]);
    } else {
      uint32_t r[32];
      ptx::tmem_ld32(tmem + lane_base + col0 + c, r);
      ptx::tmem_wait_ld();
      for (int h = 0; h < 32; ++h) dst[c + h] = __uint_as_float(r[h]);
    }
  }
}

// Pm [128 tokens][NH] (fp16, row-major) into a P * mant buffer as the kernel lays it out.
template <int NH>
__device__ void write_pm(uint32_t buf, const uint16_t* pm) {
  using C = Cfg<NH>;
  const int t = threadIdx.x;
  for (int u = 0; u < C::kPUnits; ++u)
    ptx::sts128(buf + swz_row<C::kPRow>(t, u), reinterpret_cast<const uint4*>(pm + t * NH)[u]);
}

template <int NH>
__global__ void __launch_bounds__(128, 1) selftest_kernel(const uint16_t* K, const uint16_t* Q, const uint16_t* Pm,
                                                           float* S_out, float* O_out, int* status) {
  using C = Cfg<NH>;
  extern __shared__ unsigned char raw[];
  unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  const uint32_t q_base = ptx::smem_u32(base), k_base = q_base + C::kKBase;
  __shared__ uint64_t bar[6];
  __shared__ uint32_t slot;
  __shared__ int abort_flag;
  const int t = threadIdx.x, warp = t >> 5;
  for (int id = t; id < 128 * 72; id += 128)
    ptx::sts128(k_base + chunked_offset(kKChunk, id / 72, id % 72), reinterpret_cast<const uint4*>(K)[id]);
  for (int id = t; id < NH * 72; id += 128)
    ptx::sts128(q_base + chunked_offset(C::kQChunk, id / 72, id % 72), reinterpret_cast<const uint4*>(Q)[id]);
  if (t == 0) {
    for (int i = 0; i < 6; ++i) ptx::mbar_init(&bar[i], 1);
    abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0) {
    ptx::tmem_alloc(&slot, C::kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::fence_proxy_async_smem();
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = slot;
  const uint64_t dK = desc_qk_operand(k_base), dQ = desc_qk_operand(q_base), dV = desc_v(k_base);
  const uint32_t bufR = k_base + kRopeChunk * kKChunk, buf0 = k_base, buf1 = k_base + kKChunk;

  // QK exactly as the kernel issues it
  if (warp == 0) {
    if (ptx::elect_one()) {
      issue_qk<NH, 0, 2>(tmem + C::kSCol, dK, dQ);
      issue_qk<NH, kRopeChunk, 1, true>(tmem + C::kSCol, dK, dQ);
      ptx::mma_commit(&bar[0]);
      issue_qk<NH, 2, 2>(tmem + C::kSCol + NH, dK, dQ);
      ptx::mma_commit(&bar[1]);
      issue_qk<NH, 4, 2>(tmem + C::kSCol + 2 * NH, dK, dQ);
      ptx::mma_commit(&bar[2]);
      issue_qk<NH, 6, 2>(tmem + C::kSCol + 3 * NH, dK, dQ);
      ptx::mma_commit(&bar[3]);
    }
    __syncwarp();
  }
  bool ok = true;
  for (int b = 0; b < 4; ++b) ok = ok && ptx::mbar_wait_bounded(&bar[b], 0, &abort_flag);
  ptx::tc_fence_after();
  if (ok) {
    float v[NH];
    for (int b = 0; b < 4; ++b) {
      read_cols<NH>(tmem, C::kSCol + NH * b, NH, v);
      for (int h = 0; h < NH; ++h) S_out[((size_t)b * 128 + t) * NH + h] = v[h];
    }
  }

  // PV of block 0 with its operand in the rope chunk (free once the QK completed)
  write_pm<NH>(bufR, Pm);
  ptx::fence_proxy_async_smem();
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == 0 && ok) {
    if (ptx::elect_one()) {
      issue_pv<NH, 0>(tmem, dV, desc_pm<NH>(bufR), false);
      ptx::mma_commit(&bar[4]);
    }
    __syncwarp();
  }
  ok = ok && ptx::mbar_wait_bounded(&bar[4], 0, &abort_flag);
  // blocks 1..3 with their operands in chunks 0, rope and 1 (block 0's V is no longer read)
  write_pm<NH>(buf0, Pm + 1 * 128 * NH);
  write_pm<NH>(bufR, Pm + 2 * 128 * NH);
  write_pm<NH>(buf1, Pm + 3 * 128 * NH);
  ptx::fence_proxy_async_smem();
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == 0 && ok) {
    if (ptx::elect_one()) {
      issue_pv<NH, 1>(tmem, dV, desc_pm<NH>(buf0), false);
      issue_pv<NH, 2>(tmem, dV, desc_pm<NH>(bufR), false);
      issue_pv<NH, 3>(tmem, dV, desc_pm<NH>(buf1), false);
      ptx::mma_commit(&bar[5]);
    }
    __syncwarp();
  }
  ok = ok && ptx::mbar_wait_bounded(&bar[5], 0, &abort_flag);
  ptx::tc_fence_after();
  if (ok) {
    // O^T in chunks of kChunkCols columns, as the kernel's epilogue reads it: chunk c holds block
    // (kChunkCols c) / NH, heads (kChunkCols c) % NH ..; TMEM lane = dim within the block
    float v[C::kChunkCols];
    for (int c = 0; c < C::kChunks; ++c) {
      const int jb = (C::kChunkCols * c) / NH, hb = (C::kChunkCols * c) % NH;
      read_cols<NH>(tmem, C::kChunkCols * c, C::kChunkCols, v);
      for (int h = 0; h < C::kChunkCols; ++h) O_out[(size_t)(128 * jb + t) * NH + hb + h] = v[h];
    }
  }
  if (t == 0) *status = ok ? 0 : 1;
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == 0) ptx::tmem_dealloc(tmem, C::kTmemCols);
}

template <int NH>
int run(const uint16_t* K, const uint16_t* Q, const uint16_t* Pm, float* S, float* O, int* status) {
  const size_t smem = selftest_smem<NH>();
  if (cudaFuncSetAttribute(selftest_kernel<NH>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return 1;
  selftest_kernel<NH><<<1, 128, smem>>>(K, Q, Pm, S, O, status);
  if (cudaGetLastError() != cudaSuccess) return 2;
  return cudaDeviceSynchronize() == cudaSuccess ? 0 : 3;
}

}  // namespace

// K fp16 [128][576], Q fp16 [nh][576], Pm fp16 [4][128][nh]; S fp32 [4][128][nh], O fp32 [512][nh].
extern "C" int tc_selftest(int nh, const void* K, const void* Q, const void* Pm, float* S, float* O, int* status) {
  const uint16_t* k = static_cast<const uint16_t*>(K);
  const uint16_t* q = static_cast<const uint16_t*>(Q);
  const uint16_t* pm = static_cast<const uint16_t*>(Pm);
  switch (nh) {
    case 16: return run<16>(k, q, pm, S, O, status);
    case 32: return run<32>(k, q, pm, S, O, status);
    case 64: return run<64>(k, q, pm, S, O, status);
    default: return 4;
  }
}
