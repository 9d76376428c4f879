// Decode entry point that allocates nothing: the split partials and the device
// error word live in a fixed-size file-scope device array instead of a
// caller-provided workspace.
//
// Some callers cannot allocate device memory at all: plugins hosted by an
// engine that owns the whole device memory pool and hands out no workspace,
// code that runs while a stream is being captured into a CUDA graph (a
// cudaMalloc there would break the capture), and host paths that must not
// risk the implicit device synchronisation of cudaMalloc/cudaFree.  This
// entry point serves them with the same kernels as sparse_mla_decode.
//
// The array is part of the library image: every GPU that loads the library
// holds kNoAllocScratchBytes of it until the process exits.  In host code the
// name g_noalloc_scratch is only a host-side stand-in, not a device address, so
// the device address is looked up with cudaGetSymbolAddress, once per device,
// with that device current, on the first call on that device.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "smla_internal.h"

namespace smla {
namespace {

constexpr size_t kNoAllocScratchBytes = 32u << 20;   // 32 MiB
static_assert(kNoAllocScratchBytes == SMLA_NOALLOC_SCRATCH_BYTES, "the header states the scratch size");
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once per device).
int scratch_of_current_device(void** ptr) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SMLA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return SMLA_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *ptr = g_scratch_ptr[dev];
  return SMLA_OK;
}

}  // namespace
}  // namespace smla

using namespace smla;

extern "C" int sparse_mla_decode_noalloc(const smla_dims* dims, const void* q, const void* kv_cache,
                                         const int32_t* block_table, const int32_t* topk_idx,
                                         const int32_t* seq_lens, float sm_scale, void* out, float* lse,
                                         smla_stream_t stream) {
  // the same dims checks (and status codes) as sparse_mla_decode, before any size is computed
  const int dst = check_decode_dims(dims);
  if (dst != SMLA_OK) return dst;
  // the split count decides the scratch size; fix it here so the size check and the call agree
  smla_dims d = *dims;
  if (d.nsplit == 0) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SMLA_ERR_CUDA;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return SMLA_ERR_CUDA;
    smla_plan plan;
    const int st = sparse_mla_plan_for(&d, sms, &plan);
    if (st != SMLA_OK) return st;
    d.nsplit = plan.nsplit;
  }
  const size_t need = sparse_mla_workspace_size(&d, d.nsplit);
  if (need == 0) return SMLA_ERR_INVALID_ARG;
  if (need > kNoAllocScratchBytes) return SMLA_ERR_WORKSPACE;
  void* scratch = nullptr;
  const int st = scratch_of_current_device(&scratch);
  if (st != SMLA_OK) return st;
  // the error word must start clear for this call; the partials are fully rewritten by the split kernel
  if (cudaMemsetAsync(scratch, 0, sizeof(uint32_t), (cudaStream_t)stream) != cudaSuccess) return SMLA_ERR_CUDA;
  return sparse_mla_decode(&d, q, kv_cache, block_table, topk_idx, seq_lens, sm_scale, out, lse, scratch,
                           kNoAllocScratchBytes, stream);
}

extern "C" int sparse_mla_noalloc_read_errors(uint32_t* flags, smla_stream_t stream) {
  if (!flags) return SMLA_ERR_INVALID_ARG;
  void* scratch = nullptr;
  const int st = scratch_of_current_device(&scratch);
  if (st != SMLA_OK) return st;
  // the error word is the array's first 4 bytes (the workspace header of the last call)
  if (cudaMemcpyAsync(flags, scratch, sizeof(uint32_t), cudaMemcpyDeviceToHost, (cudaStream_t)stream) != cudaSuccess)
    return SMLA_ERR_CUDA;
  return cudaStreamSynchronize((cudaStream_t)stream) == cudaSuccess ? SMLA_OK : SMLA_ERR_CUDA;
}
