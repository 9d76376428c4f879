// Shared-memory and TMEM layouts of the split kernel's operands, and its MMA issuers.  Shared by the
// kernel and by the tcgen05 self-test, which checks these exact layouts against a host matmul.
//
// K tile: 128 tokens x 576 dims fp16 in 9 chunks of 64 dims (chunk c: dims 64c .. 64c + 63 for c < 8,
// the rope for c = 8), each chunk 128 rows of 128 bytes, 128B-swizzled (K-major for QK; the same bytes
// read MN-major as V^T for PV).  Q: NH rows x 576 dims fp16 in the same 9-chunk, 128B-swizzled form.
// TMEM (8 NH columns): O^T of latent block b in columns NH b .. NH b + NH - 1 (TMEM lane = dim within
// the block), score buffer b in columns 4 NH + NH b .. (lane = token, column = head).
#pragma once

#include <stdint.h>

#include "smla_ptx.cuh"

namespace smla {

constexpr int kTile = 128;                        // top-k entries per tile = MMA M
constexpr uint32_t kKChunk = kTile * 128;         // 128 tokens x 64 dims fp16
constexpr uint32_t kKBytes = 9 * kKChunk;         // 147456
constexpr uint32_t kRopeChunk = 8;

// Per head-group size NH: Q chunks of NH rows x 64 dims, TMEM columns, MMA N, and the P * mant
// buffers ([128 tokens][NH heads] fp16, MN-major with NH * 2-byte rows: a 128-, 64- or 32-byte
// swizzle span).
template <int NH>
struct Cfg {
  static_assert(NH == 16 || NH == 32 || NH == 64, "heads per CTA");
  static constexpr uint32_t kQChunk = NH * 128;
  static constexpr uint32_t kQBytes = 9 * kQChunk;
  static constexpr uint32_t kKBase = kQBytes;               // a multiple of 1024
  static constexpr uint32_t kMiscOff = kKBase + kKBytes;
  static constexpr uint32_t kTmemCols = 8 * NH;             // 128, 256, 512
  static constexpr uint32_t kSCol = 4 * NH;                 // score buffer b at 4 NH + NH b
  static constexpr uint32_t kIdescQK = ptx::idesc_f16(128, NH, 0, 0);
  static constexpr uint32_t kIdescPV = ptx::idesc_f16(128, NH, 1, 1);
  static constexpr int kPRow = 2 * NH;                      // bytes of one token's P * mant row
  static constexpr int kPUnits = NH / 8;                    // 16-byte units per row
  static constexpr uint32_t kPStep = 16 * kPRow;            // bytes of 16 tokens (one PV MMA's K)
  static constexpr int kR = NH >= 32 ? NH / 32 : 1;         // heads per lane after a reduce-scatter
  static constexpr int kChunkCols = NH >= 32 ? 32 : 16;     // TMEM columns per O^T chunk
  static constexpr int kChunks = 4 * NH / kChunkCols;       // O^T chunks
};

// Byte offset of 16-byte unit u of row r in a buffer of `row_bytes`-wide rows with the matching
// swizzle (128, 64 or 32 bytes): the unit index is XOR-ed with the row's bits above the span.
template <int kRowBytes>
__device__ __forceinline__ uint32_t swz_row(uint32_t row, uint32_t unit) {
  constexpr uint32_t mask = kRowBytes / 16 - 1;
  constexpr int shift = kRowBytes == 128 ? 0 : kRowBytes == 64 ? 1 : 2;
  return row * kRowBytes + ((unit ^ ((row >> shift) & mask)) << 4);
}

__device__ __forceinline__ uint32_t swz128(uint32_t row, uint32_t unit) {
  return row * 128u + ((unit ^ (row & 7u)) << 4);
}

// Byte offset of 16-byte unit u (dims 8u .. 8u + 7, u < 72) of row r of a 9-chunk operand whose chunks
// are `chunk_bytes` apart (the K tile: kKChunk; Q: Cfg<NH>::kQChunk).
__device__ __forceinline__ uint32_t chunked_offset(uint32_t chunk_bytes, uint32_t row, uint32_t unit) {
  return (unit >> 3) * chunk_bytes + swz128(row, unit & 7u);
}

// Matrix descriptors of the operands (shared addresses of the K tile, Q and a P * mant buffer):
//   K tile as the K-major A of QK and Q as the K-major B: 128-byte rows, 8-row groups 1024 bytes apart;
//   K tile as the MN-major A of PV (V^T): 64-dim chunks kKChunk apart along M, 8-token groups 1024 apart;
//   P * mant as the MN-major B of PV: one NH-head swizzle span along N (the leading offset is never
//   stepped), 8-token groups 8 * row bytes apart.
__device__ __forceinline__ uint64_t desc_qk_operand(uint32_t saddr) { return ptx::sw128_desc(saddr, 16, 1024); }
__device__ __forceinline__ uint64_t desc_v(uint32_t k_base) { return ptx::sw128_desc(k_base, kKChunk, 1024); }
template <int NH>
__device__ __forceinline__ uint64_t desc_pm(uint32_t buf) {
  return ptx::swz_desc(buf, 8 * Cfg<NH>::kPRow, 8 * Cfg<NH>::kPRow, Cfg<NH>::kPRow);
}

// MMA issue.  A descriptor's start address sits in its low 14 bits in 16-byte units, so the operand
// at byte offset o from a base is the base descriptor + o / 16 (shared addresses stay below 256 KB:
// no carry).  The issuers are unrolled with compile-time offsets: one thread issues every MMA, and
// rebuilding each descriptor on that thread costs more than the MMA itself.
//
// QK of chunks [ch0, ch0 + nch) into one score buffer.
template <int NH, int kCh0, int kNch, bool kAccumulate = false>
__device__ __forceinline__ void issue_qk(uint32_t d_tmem, uint64_t dK, uint64_t dQ) {
#pragma unroll
  for (int cc = 0; cc < kNch; ++cc)
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
      ptx::mma_f16_ss(d_tmem, dK + (uint64_t)(((kCh0 + cc) * kKChunk + 32 * kk) >> 4),
                      dQ + (uint64_t)(((kCh0 + cc) * Cfg<NH>::kQChunk + 32 * kk) >> 4), Cfg<NH>::kIdescQK,
                      (kAccumulate || cc != 0 || kk != 0) ? 1u : 0u);
}

// PV of latent block kB: O^T_b (+)= K'_b^T . (P * mant_b); A is the K tile read MN-major (dims of
// chunks 2b, 2b + 1), B the 16-token slices of the P * mant buffer.
template <int NH, int kB>
__device__ __forceinline__ void issue_pv(uint32_t tmem, uint64_t dV, uint64_t dBuf, bool accumulate) {
#pragma unroll
  for (int kk = 0; kk < kTile / 16; ++kk)
    ptx::mma_f16_ss(tmem + NH * kB, dV + (uint64_t)((2 * kB * kKChunk + kk * 2048) >> 4),
                    dBuf + (uint64_t)((kk * Cfg<NH>::kPStep) >> 4), Cfg<NH>::kIdescPV,
                    (accumulate || kk > 0) ? 1u : 0u);
}

}  // namespace smla
