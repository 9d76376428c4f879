// C-ABI entry points: argument checks on the host, then kernel launches on
// the caller's stream.  No allocation, no synchronisation (except
// sparse_mla_read_errors).
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "smla_internal.h"

using namespace smla;

namespace {

std::atomic<uint64_t> g_wait_limit_ns{kDefaultWaitNs};

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

namespace smla {

uint64_t split_wait_limit_ns() { return g_wait_limit_ns.load(std::memory_order_relaxed); }

int check_decode_dims(const smla_dims* d) {
  if (!d) return SMLA_ERR_INVALID_ARG;
  if (d->batch < 1 || d->topk < 1 || d->max_pages_per_seq < 1 || d->num_pages < 1 || d->nsplit < 0)
    return SMLA_ERR_INVALID_ARG;
  if (d->heads_per_cta != 0 && !split_heads_supported(d->heads_per_cta)) return SMLA_ERR_INVALID_ARG;
  if (d->queries_per_request < 0 || (d->queries_per_request > 1 && d->batch % d->queries_per_request != 0))
    return SMLA_ERR_INVALID_ARG;
  if (d->merge < 0 || d->merge > 2) return SMLA_ERR_INVALID_ARG;
  if (d->page_size != kPageSize || d->d_latent != kDLatent || d->d_rope != kDRope) return SMLA_ERR_UNSUPPORTED;
  if (d->topk > kMaxTopk || d->nsplit > kMaxSplit || d->batch > kMaxBatch) return SMLA_ERR_UNSUPPORTED;
  if (!split_shape_supported(d->num_heads, d->topk)) return SMLA_ERR_UNSUPPORTED;
  return SMLA_OK;
}

}  // namespace smla

namespace {

int check_dims(const smla_dims* d) { return check_decode_dims(d); }

int check_inputs(const void* q, const void* kv, const int32_t* bt, const int32_t* topk, const int32_t* seq) {
  if (!q || !kv || !bt || !topk || !seq) return SMLA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(kv, 16) || !aligned(bt, 4) || !aligned(topk, 4) || !aligned(seq, 4))
    return SMLA_ERR_INVALID_ARG;
  return SMLA_OK;
}

constexpr int kMaxDevices = 64;

// SM count of the current device (queried once per device, then read from a per-device slot).
int sm_count_of_current_device(int* sms) {
  static std::atomic<int> cached[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SMLA_ERR_CUDA;
  if (dev >= 0 && dev < kMaxDevices) {
    const int c = cached[dev].load(std::memory_order_relaxed);
    if (c > 0) {
      *sms = c;
      return SMLA_OK;
    }
  }
  if (cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return SMLA_ERR_CUDA;
  if (dev >= 0 && dev < kMaxDevices) cached[dev].store(*sms, std::memory_order_relaxed);
  return SMLA_OK;
}

bool same_dims(const smla_dims& a, const smla_dims& b) {
  return a.batch == b.batch && a.num_heads == b.num_heads && a.topk == b.topk && a.page_size == b.page_size &&
         a.max_pages_per_seq == b.max_pages_per_seq && a.d_latent == b.d_latent && a.d_rope == b.d_rope &&
         a.nsplit == b.nsplit && a.num_pages == b.num_pages && a.heads_per_cta == b.heads_per_cta &&
         a.queries_per_request == b.queries_per_request && a.merge == b.merge;
}

// The scheduler's plan for dims with nsplit fixed (> 0) or chosen (0), on the current device.  The
// plan of the last call on this host thread is kept: a call with the same dims on a device with the
// same SM count reuses it.
int plan_on_current_device(const smla_dims* dims, int nsplit, smla_plan* plan) {
  struct Last {
    bool valid;
    int sms;
    smla_dims d;
    smla_plan plan;
  };
  thread_local Last last{};
  int sms = 0;
  const int st = sm_count_of_current_device(&sms);
  if (st != SMLA_OK) return st;
  smla_dims d = *dims;
  d.nsplit = nsplit;
  if (last.valid && last.sms == sms && same_dims(last.d, d)) {
    *plan = last.plan;
    return SMLA_OK;
  }
  const int r = sparse_mla_plan_for(&d, sms, plan);
  if (r == SMLA_OK) last = Last{true, sms, d, *plan};
  return r;
}

SplitParams make_params(const smla_dims* d, int nsplit, int nh, const void* q, const void* kv, const int32_t* bt,
                        const int32_t* topk, const int32_t* seq, float sm_scale) {
  SplitParams p{};
  p.q = static_cast<const uint16_t*>(q);
  p.kv = static_cast<const uint8_t*>(kv);
  p.block_table = bt;
  p.topk = topk;
  p.seq_lens = seq;
  p.sm_scale = sm_scale;
  p.B = d->batch;
  p.H = d->num_heads;
  p.topk_n = d->topk;
  p.max_pages = d->max_pages_per_seq;
  p.num_pages = d->num_pages;
  p.nsplit = nsplit;
  p.nh = nh;
  p.q_per_req = d->queries_per_request > 1 ? d->queries_per_request : 1;
  p.split_len = (d->topk + nsplit - 1) / nsplit;
  p.wait_ns = split_wait_limit_ns();
  return p;
}

// The whole decode (split kernel, then the merge when nsplit > 1); rows_out (may be null) receives the
// row the split kernel's gather warps resolved for every top-k entry.
int decode_impl(const smla_dims* dims, const void* q, const void* kv_cache, const int32_t* block_table,
                const int32_t* topk_idx, const int32_t* seq_lens, float sm_scale, void* out, float* lse,
                void* workspace, size_t workspace_bytes, int64_t* rows_out, cudaStream_t s) {
  int st = check_dims(dims);
  if (st != SMLA_OK) return st;
  st = check_inputs(q, kv_cache, block_table, topk_idx, seq_lens);
  if (st != SMLA_OK) return st;
  if (!out || !lse || !aligned(out, 16) || !aligned(lse, 4)) return SMLA_ERR_INVALID_ARG;
  if (rows_out && !aligned(rows_out, 8)) return SMLA_ERR_INVALID_ARG;
  // a fixed split count fixes the workspace size: checked before the device is queried for the plan
  if (dims->nsplit > 0) {
    const size_t need = workspace_bytes_for(dims->batch, dims->num_heads, dims->nsplit);
    if (!workspace || workspace_bytes < need || !aligned(workspace, 256)) return SMLA_ERR_WORKSPACE;
  }
  smla_plan plan;
  st = plan_on_current_device(dims, dims->nsplit, &plan);
  if (st != SMLA_OK) return st;
  const int nsplit = plan.nsplit;
  const size_t need = workspace_bytes_for(dims->batch, dims->num_heads, nsplit);
  if (!workspace || workspace_bytes < need || !aligned(workspace, 256)) return SMLA_ERR_WORKSPACE;
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  SplitParams p = make_params(dims, nsplit, plan.heads_per_cta, q, kv_cache, block_table, topk_idx, seq_lens,
                              sm_scale);
  p.err = reinterpret_cast<uint32_t*>(ws);
  p.out = static_cast<uint16_t*>(out);
  p.lse = lse;
  p.rows_out = rows_out;
  p.final_out = (nsplit == 1);
  p.fused = plan.fused != 0;
  if (nsplit > 1) {
    const size_t lse_bytes = ((size_t)dims->batch * nsplit * dims->num_heads * sizeof(float) + 255) / 256 * 256;
    p.lse_part = reinterpret_cast<float*>(ws + kWorkspaceHeader);
    p.o_part = reinterpret_cast<float*>(ws + kWorkspaceHeader + lse_bytes);
  }
  if (launch_split(p, s) != cudaSuccess) return SMLA_ERR_CUDA;
  if (nsplit > 1 && !p.fused &&
      launch_combine(dims->batch, dims->num_heads, nsplit, p.o_part, p.lse_part, p.out, lse, s) != cudaSuccess)
    return SMLA_ERR_CUDA;
  return SMLA_OK;
}

}  // namespace

extern "C" int sparse_mla_plan(const smla_dims* dims, int32_t device, smla_plan* plan) {
  if (!dims || !plan || device < 0) return SMLA_ERR_INVALID_ARG;
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) return SMLA_ERR_CUDA;
  return sparse_mla_plan_for(dims, sms, plan);
}

extern "C" int sparse_mla_split(const smla_dims* dims, int32_t nsplit, const void* q, const void* kv_cache,
                                const int32_t* block_table, const int32_t* topk_idx, const int32_t* seq_lens,
                                float sm_scale, float* o_part, float* lse_part, uint32_t* err_word,
                                smla_stream_t stream) {
  int st = check_dims(dims);
  if (st != SMLA_OK) return st;
  st = check_inputs(q, kv_cache, block_table, topk_idx, seq_lens);
  if (st != SMLA_OK) return st;
  if (nsplit < 1 || nsplit > kMaxCombineSplit) return SMLA_ERR_INVALID_ARG;
  if (nsplit > kMaxSplit) return SMLA_ERR_UNSUPPORTED;
  if (!o_part || !lse_part || !aligned(o_part, 16) || !aligned(lse_part, 4)) return SMLA_ERR_INVALID_ARG;
  if (err_word && !aligned(err_word, 4)) return SMLA_ERR_INVALID_ARG;
  smla_plan plan;
  st = plan_on_current_device(dims, nsplit, &plan);
  if (st != SMLA_OK) return st;
  SplitParams p = make_params(dims, nsplit, plan.heads_per_cta, q, kv_cache, block_table, topk_idx, seq_lens,
                              sm_scale);
  p.o_part = o_part;
  p.lse_part = lse_part;
  p.err = err_word;
  p.final_out = false;
  return launch_split(p, (cudaStream_t)stream) == cudaSuccess ? SMLA_OK : SMLA_ERR_CUDA;
}

extern "C" int sparse_mla_decode(const smla_dims* dims, const void* q, const void* kv_cache,
                                 const int32_t* block_table, const int32_t* topk_idx, const int32_t* seq_lens,
                                 float sm_scale, void* out, float* lse, void* workspace, size_t workspace_bytes,
                                 smla_stream_t stream) {
  return decode_impl(dims, q, kv_cache, block_table, topk_idx, seq_lens, sm_scale, out, lse, workspace,
                     workspace_bytes, nullptr, (cudaStream_t)stream);
}

extern "C" int sparse_mla_decode_rows(const smla_dims* dims, const void* q, const void* kv_cache,
                                      const int32_t* block_table, const int32_t* topk_idx, const int32_t* seq_lens,
                                      float sm_scale, void* out, float* lse, void* workspace,
                                      size_t workspace_bytes, int64_t* rows_out, smla_stream_t stream) {
  if (!rows_out) return SMLA_ERR_INVALID_ARG;
  return decode_impl(dims, q, kv_cache, block_table, topk_idx, seq_lens, sm_scale, out, lse, workspace,
                     workspace_bytes, rows_out, (cudaStream_t)stream);
}

extern "C" int sparse_mla_debug_set_wait_limit(uint64_t ns) {
  g_wait_limit_ns.store(ns ? ns : kDefaultWaitNs, std::memory_order_relaxed);
  return SMLA_OK;
}

extern "C" int sparse_mla_kv_append(const smla_append_dims* d, const void* latent, const void* rope,
                                    const int32_t* block_table, const int32_t* requests, const int32_t* positions,
                                    void* kv_cache, uint32_t* err_word, smla_stream_t stream) {
  if (!d) return SMLA_ERR_INVALID_ARG;
  if (d->tokens < 0 || d->num_requests < 1 || d->max_pages_per_seq < 1 || d->num_pages < 1)
    return SMLA_ERR_INVALID_ARG;
  if (d->page_size != kPageSize || d->d_latent != kDLatent || d->d_rope != kDRope) return SMLA_ERR_UNSUPPORTED;
  if (d->tokens > 0) {
    if (!latent || !rope || !block_table || !positions || !kv_cache) return SMLA_ERR_INVALID_ARG;
    if (!aligned(latent, 16) || !aligned(rope, 16) || !aligned(kv_cache, 16) || !aligned(block_table, 4) ||
        !aligned(positions, 4) || (requests && !aligned(requests, 4)))
      return SMLA_ERR_INVALID_ARG;
  }
  if (err_word && !aligned(err_word, 4)) return SMLA_ERR_INVALID_ARG;
  AppendParams p{};
  p.latent = static_cast<const uint16_t*>(latent);
  p.rope = static_cast<const uint16_t*>(rope);
  p.block_table = block_table;
  p.requests = requests;
  p.positions = positions;
  p.kv = static_cast<uint8_t*>(kv_cache);
  p.tokens = d->tokens;
  p.num_requests = d->num_requests;
  p.max_pages = d->max_pages_per_seq;
  p.num_pages = d->num_pages;
  p.err = err_word;
  return launch_kv_append(p, (cudaStream_t)stream) == cudaSuccess ? SMLA_OK : SMLA_ERR_CUDA;
}

extern "C" int sparse_mla_topk_select(const smla_topk_dims* d, const float* scores, const int32_t* seq_lens,
                                      int32_t* topk_idx, uint32_t* err_word, smla_stream_t stream) {
  if (!d) return SMLA_ERR_INVALID_ARG;
  if (d->batch < 0 || d->num_cols < 1 || d->row_stride < d->num_cols || d->k < 1 || d->cluster_ctas < 0 ||
      d->cluster_ctas > kTopkMaxCluster)
    return SMLA_ERR_INVALID_ARG;
  if (d->k > kMaxTopk || d->num_cols > kTopkMaxCluster * kTopkMaxChunk) return SMLA_ERR_UNSUPPORTED;
  if (d->batch > 0) {
    if (!scores || !seq_lens || !topk_idx) return SMLA_ERR_INVALID_ARG;
    if (!aligned(scores, 4) || !aligned(seq_lens, 4) || !aligned(topk_idx, 4)) return SMLA_ERR_INVALID_ARG;
  }
  if (err_word && !aligned(err_word, 4)) return SMLA_ERR_INVALID_ARG;
  if (d->batch == 0) return SMLA_OK;
  int sms = 0;
  const int st = sm_count_of_current_device(&sms);
  if (st != SMLA_OK) return st;
  TopkParams p{};
  if (!topk_plan(d->batch, d->num_cols, sms, d->cluster_ctas, &p.csize, &p.chunk)) return SMLA_ERR_UNSUPPORTED;
  p.scores = scores;
  p.seq_lens = seq_lens;
  p.out = topk_idx;
  p.err = err_word;
  p.stride = d->row_stride;
  p.num_cols = d->num_cols;
  p.k = d->k;
  p.vec4 = aligned(scores, 16) && d->row_stride % 4 == 0;
  return launch_topk(p, d->batch, (cudaStream_t)stream) == cudaSuccess ? SMLA_OK : SMLA_ERR_CUDA;
}

extern "C" int sparse_mla_topk_plan_for(const smla_topk_dims* d, int32_t sm_count, int32_t* cluster_ctas,
                                        int32_t* chunk_positions) {
  if (!d || !cluster_ctas || !chunk_positions || sm_count < 1) return SMLA_ERR_INVALID_ARG;
  if (d->batch < 0 || d->num_cols < 1 || d->row_stride < d->num_cols || d->k < 1 || d->cluster_ctas < 0 ||
      d->cluster_ctas > kTopkMaxCluster)
    return SMLA_ERR_INVALID_ARG;
  if (d->k > kMaxTopk || d->num_cols > kTopkMaxCluster * kTopkMaxChunk) return SMLA_ERR_UNSUPPORTED;
  int c = 0, ch = 0;
  if (!topk_plan(d->batch > 0 ? d->batch : 1, d->num_cols, sm_count, d->cluster_ctas, &c, &ch))
    return SMLA_ERR_UNSUPPORTED;
  *cluster_ctas = c;
  *chunk_positions = ch;
  return SMLA_OK;
}

extern "C" int sparse_mla_combine(int32_t batch, int32_t num_heads, int32_t nsplit, const float* o_part,
                                  const float* lse_part, void* out, float* lse, smla_stream_t stream) {
  if (batch < 1 || num_heads < 1 || nsplit < 1 || nsplit > kMaxCombineSplit) return SMLA_ERR_INVALID_ARG;
  if (!o_part || !lse_part || !out || !lse) return SMLA_ERR_INVALID_ARG;
  if (!aligned(o_part, 16) || !aligned(out, 8) || !aligned(lse_part, 4) || !aligned(lse, 4))
    return SMLA_ERR_INVALID_ARG;
  return launch_combine(batch, num_heads, nsplit, o_part, lse_part, static_cast<uint16_t*>(out), lse,
                        (cudaStream_t)stream) == cudaSuccess
             ? SMLA_OK
             : SMLA_ERR_CUDA;
}

extern "C" int sparse_mla_gather_rows(const smla_dims* dims, const int32_t* block_table, const int32_t* topk_idx,
                                      const int32_t* seq_lens, int64_t* rows_out, smla_stream_t stream) {
  if (!dims) return SMLA_ERR_INVALID_ARG;
  if (dims->batch < 1 || dims->topk < 1 || dims->max_pages_per_seq < 1 || dims->num_pages < 1)
    return SMLA_ERR_INVALID_ARG;
  if (dims->page_size != kPageSize) return SMLA_ERR_UNSUPPORTED;
  if (!block_table || !topk_idx || !seq_lens || !rows_out || !aligned(rows_out, 8)) return SMLA_ERR_INVALID_ARG;
  return launch_gather_rows(block_table, topk_idx, seq_lens, dims->batch, dims->topk, dims->max_pages_per_seq,
                            dims->num_pages, dims->queries_per_request > 1 ? dims->queries_per_request : 1, rows_out,
                            (cudaStream_t)stream) == cudaSuccess
             ? SMLA_OK
             : SMLA_ERR_CUDA;
}

extern "C" int sparse_mla_clear_errors(void* workspace, smla_stream_t stream) {
  if (!workspace) return SMLA_ERR_INVALID_ARG;
  return cudaMemsetAsync(workspace, 0, sizeof(uint32_t), (cudaStream_t)stream) == cudaSuccess ? SMLA_OK
                                                                                            : SMLA_ERR_CUDA;
}

extern "C" int sparse_mla_read_errors(const void* workspace, uint32_t* flags, smla_stream_t stream) {
  if (!workspace || !flags) return SMLA_ERR_INVALID_ARG;
  if (cudaMemcpyAsync(flags, workspace, sizeof(uint32_t), cudaMemcpyDeviceToHost, (cudaStream_t)stream) !=
      cudaSuccess)
    return SMLA_ERR_CUDA;
  return cudaStreamSynchronize((cudaStream_t)stream) == cudaSuccess ? SMLA_OK : SMLA_ERR_CUDA;
}

extern "C" const char* sparse_mla_status_string(int status) {
  switch (status) {
    case SMLA_OK: return "ok";
    case SMLA_ERR_INVALID_ARG: return "invalid argument";
    case SMLA_ERR_UNSUPPORTED: return "unsupported shape";
    case SMLA_ERR_WORKSPACE: return "workspace missing or too small";
    case SMLA_ERR_CUDA: return "CUDA error";
    default: return "unknown status";
  }
}
