// kvq_noalloc.cu -- kvq_paged_decode_noalloc: the paged decode for callers that
// cannot allocate device memory.
//
// kvq_paged_decode needs a caller-provided workspace for its split-K partials
// whenever a request spans more than one partition.  Some callers cannot
// provide one: code that runs where allocating is not allowed or not possible
// (inside a custom allocator or memory-pool callback that must not re-enter
// the allocator, a plugin that a host framework hands only its input and
// output buffers, a runtime that fixes its device memory budget at start-up
// and forbids cudaMalloc afterwards).  For them this file keeps a fixed scratch
// array in the library itself and runs the same two launches on it.
//
// The array is a file-scope __device__ variable, so every GPU that loads the
// library holds it (kNoAllocScratchBytes) until the process exits.  In host
// code its name is only a host-side stand-in for the symbol, never a device
// address; the device address comes from cudaGetSymbolAddress, looked up once
// per device (with that device current) the first time the entry point runs
// on it and cached.
#include <cuda_runtime.h>

#include <atomic>
#include <cstddef>
#include <cstdint>

#include "kvq.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;   // 16 MiB
constexpr int kMaxDevices = 64;

std::atomic<void *> g_scratch_address[kMaxDevices];

}  // namespace

static __device__ __align__(256) unsigned char g_decode_scratch[kNoAllocScratchBytes];

namespace {

// Device address of g_decode_scratch on the current device.
cudaError_t scratch_address(void **ptr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < kMaxDevices) {
    void *p = g_scratch_address[dev].load(std::memory_order_acquire);
    if (p != nullptr) {
      *ptr = p;
      return cudaSuccess;
    }
  }
  void *p = nullptr;
  e = cudaGetSymbolAddress(&p, g_decode_scratch);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < kMaxDevices) g_scratch_address[dev].store(p, std::memory_order_release);
  *ptr = p;
  return cudaSuccess;
}

}  // namespace

extern "C" kvq_status kvq_paged_decode_noalloc(
    const kvq_cache *cache, const void *q, int32_t num_requests, int32_t rows_per_request,
    int32_t num_q_heads, const int32_t *block_tables, int32_t max_blocks_per_req,
    const int32_t *context_lens, int32_t max_context_len, float sm_scale,
    int32_t partition_tokens, void *out, int32_t *err_flags, kvq_stream_t stream) {
  if (cache == nullptr) return KVQ_ERR_INVALID_ARGUMENT;
  // 0 both when no scratch is needed and for invalid arguments, which
  // kvq_paged_decode below rejects with its own status
  const size_t need = kvq_paged_decode_workspace_size(
      num_requests, rows_per_request, num_q_heads, cache->num_kv_heads, cache->head_dim,
      cache->block_size, max_context_len, partition_tokens);
  if (need > kNoAllocScratchBytes) return KVQ_ERR_WORKSPACE_TOO_SMALL;
  void *scratch = nullptr;
  if (need > 0 && scratch_address(&scratch) != cudaSuccess) return KVQ_ERR_CUDA;
  return kvq_paged_decode(cache, q, num_requests, rows_per_request, num_q_heads, block_tables,
                          max_blocks_per_req, context_lens, max_context_len, sm_scale,
                          partition_tokens, out, scratch, need, err_flags, stream);
}
