// Device helpers shared by the library's kernels.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

#include "smla_internal.h"

namespace smla {

// Index -> address (a1).  Top-k entry t of a request is a logical position;
// used when 0 <= t < seq_len, row = block_table[t/64]*64 + t%64.  A used entry
// whose logical page is past the block-table row or whose physical page lies
// outside the cache is skipped and flagged.  ("Inside the Decode Performance
// Investigation", Task 1: scattered FP8 page-gathers.)
//
// The step is split in two so that a pipelined caller can put the block-table
// load in flight early and resolve the row later; every kernel that maps top-k
// entries to rows (the split kernel's gather warps and the row-gather entry
// point) goes through these two functions.
//
// Whether entry t reads the block table: a used entry whose logical page lies in the row.
__device__ __forceinline__ bool entry_reads_table(int t, int seq_len, int max_pages) {
  return t >= 0 && t < seq_len && (t >> 6) < max_pages;
}

// Row of entry t given its block-table entry `page` (any value when entry_reads_table(t) is false);
// -1 when the entry is skipped.  A used entry outside the table or the cache sets
// SMLA_DEVERR_PAGE_RANGE in *err (when err is not null).
__device__ __forceinline__ int64_t row_from_page(int t, int page, int seq_len, int max_pages, int64_t num_pages,
                                                 uint32_t* err) {
  if (t < 0 || t >= seq_len) return -1;
  if ((t >> 6) >= max_pages || page < 0 || (int64_t)page >= num_pages) {
    if (err) atomicOr(err, SMLA_DEVERR_PAGE_RANGE);
    return -1;
  }
  return (int64_t)page * kPageSize + (t & (kPageSize - 1));
}

// Both halves at once.
__device__ __forceinline__ int64_t row_of(const int32_t* __restrict__ bt_row, int t, int seq_len,
                                          int max_pages, int64_t num_pages, uint32_t* err) {
  const int page = entry_reads_table(t, seq_len, max_pages) ? __ldg(bt_row + (t >> 6)) : 0;
  return row_from_page(t, page, seq_len, max_pages, num_pages, err);
}

// Two E4M3 codes (low byte first) -> two fp16 (exact: every E4M3 value is an fp16 value).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t two) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(two));
  return r;
}

__device__ __forceinline__ float2 f16x2_to_f32x2(uint32_t h) {
  __half2 v = *reinterpret_cast<__half2*>(&h);
  return __half22float2(v);
}

__device__ __forceinline__ float bf16_to_f32(uint16_t b) {
  return __uint_as_float(((uint32_t)b) << 16);
}

// fp32 pair -> bf16x2, round to nearest even (low half = a).
__device__ __forceinline__ uint32_t f32x2_to_bf16x2(float a, float b) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(b), "f"(a));
  return r;
}

// fp32 pair -> fp16x2 with saturation to +-65504 (low half = a).
__device__ __forceinline__ uint32_t f32x2_to_f16x2_sat(float a, float b) {
  uint32_t r;
  asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(b), "f"(a));
  return r;
}

}  // namespace smla
