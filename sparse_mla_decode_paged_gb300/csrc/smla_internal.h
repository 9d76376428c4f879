// Internal declarations shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "sparse_mla.h"

namespace smla {

constexpr int kPageSize = 64;
constexpr int kDLatent = 512;
constexpr int kDRope = 64;
constexpr int kDQK = kDLatent + kDRope;   // 576
constexpr int kRecordBytes = 656;
constexpr int kMaxTopk = 2048;
constexpr int kMaxSplit = 16;
constexpr int kMaxBatch = 65535;      // decode queries per call (the split grid's z extent)
constexpr int kMaxCombineSplit = 64;
constexpr size_t kWorkspaceHeader = 256;
constexpr int kMaxFusedSplit = 8;      // partitions merged inside the split kernel (one portable cluster)

// Everything the split kernels need for one launch.
struct SplitParams {
  const uint16_t* q;          // bf16 [B][H][576]
  const uint8_t* kv;          // [num_pages][64][656]
  const int32_t* block_table; // [B][max_pages]
  const int32_t* topk;        // [B][topk]
  const int32_t* seq_lens;    // [B]
  float sm_scale;
  int B, H, topk_n, max_pages;
  int64_t num_pages;
  int nsplit;
  int nh;                     // heads per CTA (16, 32 or 64): H is split into ceil(H / nh) groups
  int q_per_req;              // queries per request: query b reads block-table row b / q_per_req
  int split_len;              // top-k positions per partition
  bool final_out;             // true: write out/lse directly (nsplit == 1); false: partials
  uint16_t* out;              // bf16 [B][H][512]
  float* lse;                 // [B][H]
  float* o_part;              // [B][nsplit][H][512]
  float* lse_part;            // [B][nsplit][H]
  uint32_t* err;              // device error word (may be null)
  bool fused;                 // nsplit > 1 merged inside the kernel: the nsplit CTAs of a (query, head
                              // group) form one cluster; o_part is their exchange area, out/lse the result
  int64_t* rows_out;          // [B][topk] or null: the row the gather warps resolved for each entry
  uint64_t wait_ns;           // time limit of each pipeline wait inside the kernel
};

// Host checks of a decode's dims (status code; SMLA_OK when the split kernel supports them).
int check_decode_dims(const smla_dims* d);

// Time limit of the split kernel's pipeline waits: kDefaultWaitNs unless a test set another one
// (sparse_mla_debug_set_wait_limit).
constexpr uint64_t kDefaultWaitNs = 1000000000ull;
uint64_t split_wait_limit_ns();

// Everything the KV append kernel needs for one launch.
struct AppendParams {
  const uint16_t* latent;     // bf16 [tokens][512]
  const uint16_t* rope;       // bf16 [tokens][64]
  const int32_t* block_table; // [num_requests][max_pages]
  const int32_t* requests;    // [tokens] request of each token, or null: token i belongs to request i
  const int32_t* positions;   // [tokens] logical position of each token in its request
  uint8_t* kv;                // [num_pages][64][656]
  int tokens, num_requests, max_pages;
  int64_t num_pages;
  uint32_t* err;              // device error word (may be null)
};

// Top-k selection (clusters of csize CTAs, chunk positions per CTA; a row spans at most one cluster).
constexpr int kTopkPortableCluster = 8;  // cluster sizes every launch supports
constexpr int kTopkMaxCluster = 16;      // with the non-portable cluster size attribute (rows past 8 chunks)
constexpr int kTopkMaxChunk = 65536;     // scores per CTA (chunk indexes are 16-bit)
constexpr int kTopkChunkAlign = 2048;    // chunks are multiples of this (16 warps x 128-entry steps)
constexpr int kTopkPackMaxRows = 2048;   // rows packed into clusters only for batches up to this size
struct TopkParams {
  const float* scores;        // [batch][stride]
  const int32_t* seq_lens;    // [batch]
  int32_t* out;               // [batch][k]
  uint32_t* err;              // device error word (may be null)
  int64_t stride;
  int num_cols, k, chunk, csize;
  int vec4;                   // scores 16-byte aligned and stride % 4 == 0: 16-byte loads
  int batch;                  // rows (set by launch_topk)
  int pack;                   // csize a power of two > 1: rows packed into clusters by their chunk count
  int pre8;                   // the top byte of every key kept in shared memory (set by launch_topk)
};
bool topk_plan(int batch, int num_cols, int sm_count, int forced_csize, int* csize, int* chunk);
size_t topk_smem_bytes(int chunk);
cudaError_t launch_topk(const TopkParams& p, int batch, cudaStream_t stream);

// Kernel launchers (return the launch error).
cudaError_t launch_split(const SplitParams& p, cudaStream_t stream);
size_t workspace_bytes_for(int B, int H, int nsplit);
cudaError_t launch_combine(int B, int H, int nsplit, const float* o_part, const float* lse_part,
                           uint16_t* out, float* lse, cudaStream_t stream);
cudaError_t launch_kv_append(const AppendParams& p, cudaStream_t stream);
cudaError_t launch_gather_rows(const int32_t* bt, const int32_t* topk, const int32_t* seq_lens,
                               int B, int topk_n, int max_pages, int64_t num_pages, int q_per_req,
                               int64_t* rows, cudaStream_t stream);

// Shape limits of the split kernel (checked on the host before any launch).
bool split_shape_supported(int H, int topk);
// Resident CTAs per SM of the split kernel for H heads (occupancy of its smem/threads).
int split_ctas_per_sm(int H);
// Heads per CTA the split kernel is built for (16, 32, 64).
bool split_heads_supported(int nh);
// CTAs per work unit (one unit per query, partition and head group).
int split_ctas_per_unit();
// Whether the split kernel merges nsplit partitions itself for nh heads per CTA and H heads (a cluster of
// nsplit CTAs, each owning nh / nsplit heads of the merge).
bool split_fusable(int nsplit, int nh, int H);

}  // namespace smla
