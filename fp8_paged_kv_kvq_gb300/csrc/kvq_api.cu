// kvq_api.cu -- the C ABI of libkvq (declared in include/kvq.h): host-side
// argument validation, shape decisions and the kernel launches.  Nothing here
// allocates, synchronises or reads device memory.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>

#include "kvq.h"
#include "kvq_internal.h"

namespace {

constexpr int32_t kAbiVersion = 3;
constexpr int32_t kMaxRowsPerKvHead = 128;
constexpr int32_t kMaxPartitionTokens = 1 << 20;

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

std::atomic<uint32_t> g_call_tag{0};

bool is_pow2(int64_t x) { return x > 0 && (x & (x - 1)) == 0; }

int32_t log2_exact(int64_t x) {
  int32_t l = 0;
  while ((int64_t(1) << l) < x) ++l;
  return l;
}

int current_sm_count() {
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return 152;
  }
  int v = cached[dev].load(std::memory_order_relaxed);
  if (v > 0) return v;
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    n = 152;
  }
  cached[dev].store(n, std::memory_order_relaxed);
  return n;
}

kvq_status check_cache(const kvq_cache *c, bool need_block_size) {
  if (c == nullptr) return KVQ_ERR_INVALID_ARGUMENT;
  if (c->num_slots < 0 || c->num_kv_heads <= 0 || c->head_dim <= 0)
    return KVQ_ERR_INVALID_ARGUMENT;
  if (c->head_dim != kvq::kHeadDimAbi) return KVQ_ERR_UNSUPPORTED;
  if (c->num_slots > 0 &&
      (c->k_codes == nullptr || c->v_codes == nullptr || c->k_scales == nullptr ||
       c->v_scales == nullptr))
    return KVQ_ERR_INVALID_ARGUMENT;
  if (!aligned(c->k_codes, 16) || !aligned(c->v_codes, 16) || !aligned(c->k_scales, 4) ||
      !aligned(c->v_scales, 4))
    return KVQ_ERR_MISALIGNED;
  if (need_block_size) {
    if (c->block_size <= 0) return KVQ_ERR_INVALID_ARGUMENT;
    if (!is_pow2(c->block_size)) return KVQ_ERR_UNSUPPORTED;
  }
  return KVQ_OK;
}

kvq_status from_cuda(cudaError_t e) { return e == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA; }

// Tokens per partition, a power of two in [256, 8192] (up to 32768 for the
// tcgen05 kernel).  9..32 stacked rows per KV head on pages of 16..128 tokens
// with KV heads in groups of 4 go to the tcgen05 kernel (one CTA per SM, with
// a per-CTA setup and epilogue): the longest P within its 512 pages that
// still gives ~6 waves of CTAs.  Long contexts (>= 64K tokens) on pages of
// >= 16 tokens with KV heads in groups of 4 suit the page-major kernel (one
// CTA per 4 heads, partition and request): the largest P with at least ~12
// such CTAs per SM.  Otherwise (one CTA per KV head, partition and request)
// the largest P with 2P <= N H ctx / (4 SMs).
int32_t heuristic_partition(int32_t num_requests, int32_t num_kv_heads, int32_t block_size,
                            int32_t max_context_len, int64_t rows) {
  const int64_t sms = current_sm_count();
  const int64_t n = num_requests > 0 ? num_requests : 1;
  const int64_t h = num_kv_heads > 0 ? num_kv_heads : 1;
  const int64_t ctx = max_context_len > 0 ? max_context_len : 1;
  int32_t p = 256;
  if (rows > 8 && rows <= 32 && block_size >= 16 && block_size <= 128 && h % 4 == 0) {
    const int64_t cap = std::min<int64_t>(32768, 512 * static_cast<int64_t>(block_size));
    while (int64_t(p) * 2 <= cap && n * h * ((ctx + 2 * p - 1) / (2 * p)) >= 6 * sms) p *= 2;
    return p;
  }
  if (ctx >= 65536 && block_size >= 16 && h % 4 == 0) {
    const int64_t target = n * (h / 4) * ctx / (12 * sms);
    while (p < 8192 && int64_t(p) * 2 <= target) p *= 2;
    return p;
  }
  const int64_t target = n * h * ctx / (sms * 4);
  while (p < 8192 && int64_t(p) * 2 <= target) p *= 2;
  return p;
}

// Validates the decode arguments shared by the partials and combine calls and
// fills the shape.
kvq_status make_shape(const kvq_cache *cache, int32_t num_requests, int32_t rows_per_request,
                      int32_t num_q_heads, int32_t max_blocks_per_req,
                      int32_t max_context_len, int32_t partition_tokens, kvq::AttnShape *s) {
  kvq_status st = check_cache(cache, true);
  if (st != KVQ_OK) return st;
  if (num_requests < 0 || rows_per_request < 1 || num_q_heads < 1 || max_blocks_per_req < 0 ||
      max_context_len < 0 || partition_tokens < 0)
    return KVQ_ERR_INVALID_ARGUMENT;
  if (num_q_heads % cache->num_kv_heads != 0) return KVQ_ERR_INVALID_ARGUMENT;
  if (partition_tokens % 64 != 0 || partition_tokens > kMaxPartitionTokens)
    return KVQ_ERR_INVALID_ARGUMENT;
  const int32_t G = num_q_heads / cache->num_kv_heads;
  const int64_t M = static_cast<int64_t>(rows_per_request) * G;
  // more than 8 stacked rows per KV head with the partition size left to the
  // library: the rows-on-M tensor-core kernel (no partitions, up to
  // kRowsMaxRows rows: verify and chunked prefill).  An explicit partition
  // size keeps 9..32 rows on the partitioned tcgen05 kernel.
  const bool rows_path = partition_tokens == 0 && M > 8 && M <= kvq::kRowsMaxRows &&
                         cache->block_size >= 16 && cache->num_kv_heads % 4 == 0 &&
                         num_requests <= kvq::kRowsMaxRequests;
  if (M > kMaxRowsPerKvHead && !rows_path) return KVQ_ERR_UNSUPPORTED;
  if (num_requests > 65535) return KVQ_ERR_UNSUPPORTED;
  s->num_requests = num_requests;
  s->rows_per_request = rows_per_request;
  s->num_q_heads = num_q_heads;
  s->group = G;
  s->rows = static_cast<int32_t>(M);
  s->row_groups = static_cast<int32_t>((M + 31) / 32);
  s->max_blocks_per_req = max_blocks_per_req;
  s->max_context_len = max_context_len;
  s->partition_tokens = partition_tokens > 0
                            ? partition_tokens
                            : heuristic_partition(num_requests, cache->num_kv_heads,
                                                  cache->block_size, max_context_len, M);
  const int64_t np = (static_cast<int64_t>(max_context_len) + s->partition_tokens - 1) /
                     s->partition_tokens;
  if (np > 65535) return KVQ_ERR_UNSUPPORTED;
  s->num_partitions = np > 0 ? static_cast<int32_t>(np) : 1;
  if (static_cast<int64_t>(cache->num_kv_heads) * s->row_groups > 0x7FFFFFFF)
    return KVQ_ERR_UNSUPPORTED;
  s->log2_block = log2_exact(cache->block_size);
  s->sms = current_sm_count();
  s->stream = 0;
  s->num_kv_heads = cache->num_kv_heads;
  s->rows_kernel = rows_path ? 1 : 0;
  if (rows_path) {
    s->num_partitions = 1;
    return KVQ_OK;
  }
  // With the partition size left to the library, batches of <= 8 stacked rows
  // whose page-major partition grid would be small (under ~3 waves) go to the
  // load-balanced kernel, which splits the batch's tokens evenly over a
  // persistent grid.  It loads the scale planes by TMA; for planes that are
  // not 16-byte aligned the partitioned kernels run instead, with partitions
  // long enough to fit the same workspace (<= kStreamSlots of them).
  if (partition_tokens == 0 && kvq::attn_stream_shape_ok(cache->num_kv_heads, *s)) {
    const int64_t page_ctas = static_cast<int64_t>(cache->num_kv_heads / 4) * s->num_partitions *
                              num_requests;
    if (page_ctas < 9LL * s->sms) {
      const bool aligned16 = aligned(cache->k_scales, 16) && aligned(cache->v_scales, 16);
      if (aligned16) {
        s->stream = 1;
        s->num_partitions = kvq::kStreamSlots;
      } else {
        const int64_t need = (static_cast<int64_t>(max_context_len) + kvq::kStreamSlots - 1) /
                             kvq::kStreamSlots;
        const int64_t p64 = (need + 63) / 64 * 64;
        if (p64 > s->partition_tokens) s->partition_tokens = static_cast<int32_t>(p64);
        const int64_t np2 = (static_cast<int64_t>(max_context_len) + s->partition_tokens - 1) /
                            s->partition_tokens;
        s->num_partitions = np2 > 0 ? static_cast<int32_t>(np2) : 1;
      }
    }
  }
  return KVQ_OK;
}

size_t workspace_for(const kvq::AttnShape &s) {
  if (s.rows_kernel) return kvq::attn_rows_workspace_bytes(s, s.num_kv_heads);
  const int64_t rows_total =
      static_cast<int64_t>(s.num_requests) * s.rows_per_request * s.num_q_heads;
  if (s.stream)
    return kvq::attn_stream_pieces_bytes(s.num_requests, s.num_kv_heads) +
           kvq::attn_workspace_bytes(rows_total, kvq::kStreamSlots);
  return kvq::attn_workspace_bytes(rows_total, s.num_partitions);
}

}  // namespace

namespace kvq {

uint32_t next_call_tag() {
  uint32_t t = g_call_tag.fetch_add(1, std::memory_order_relaxed) + 1;
  while (t == 0) t = g_call_tag.fetch_add(1, std::memory_order_relaxed) + 1;
  return t;
}

}  // namespace kvq

extern "C" {

const char *kvq_status_string(kvq_status status) {
  switch (status) {
    case KVQ_OK: return "ok";
    case KVQ_ERR_INVALID_ARGUMENT: return "invalid argument";
    case KVQ_ERR_UNSUPPORTED: return "unsupported shape or parameter";
    case KVQ_ERR_MISALIGNED: return "misaligned pointer or stride";
    case KVQ_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case KVQ_ERR_CUDA: return "CUDA error";
  }
  return "unknown status";
}

int32_t kvq_abi_version(void) { return kAbiVersion; }

size_t kvq_cache_bytes(int64_t num_slots, int32_t num_kv_heads, int32_t head_dim) {
  if (num_slots < 0 || num_kv_heads < 0 || head_dim < 0) return 0;
  return 2u * static_cast<size_t>(num_slots) * static_cast<size_t>(num_kv_heads) *
         (static_cast<size_t>(head_dim) + sizeof(float));
}

kvq_status kvq_quantize_scatter(const kvq_cache *cache, const void *k, int64_t k_token_stride,
                                const void *v, int64_t v_token_stride, int64_t num_tokens,
                                const int64_t *slot_ids, int32_t *err_flags,
                                kvq_stream_t stream) {
  kvq_status st = check_cache(cache, false);
  if (st != KVQ_OK) return st;
  if (num_tokens < 0 || k_token_stride < 0 || v_token_stride < 0)
    return KVQ_ERR_INVALID_ARGUMENT;
  if (num_tokens == 0) return KVQ_OK;
  if (k == nullptr || v == nullptr || slot_ids == nullptr) return KVQ_ERR_INVALID_ARGUMENT;
  if (!aligned(k, 16) || !aligned(v, 16) || (k_token_stride % 8) != 0 ||
      (v_token_stride % 8) != 0 || !aligned(slot_ids, 8) || !aligned(err_flags, 4))
    return KVQ_ERR_MISALIGNED;
  // rows (token, K/V, head) are numbered in 32 bits
  if (num_tokens > (int64_t(1) << 31) / (2 * cache->num_kv_heads) - 32) return KVQ_ERR_UNSUPPORTED;
  return from_cuda(kvq::launch_quantize_scatter(*cache, k, k_token_stride, v, v_token_stride,
                                                num_tokens, slot_ids, err_flags,
                                                reinterpret_cast<cudaStream_t>(stream)));
}

int32_t kvq_paged_decode_partition_tokens(int32_t num_requests, int32_t rows_per_request,
                                          int32_t num_q_heads, int32_t num_kv_heads,
                                          int32_t block_size, int32_t max_context_len) {
  const int64_t rows = (num_kv_heads > 0 && num_q_heads % num_kv_heads == 0 && rows_per_request > 0)
                           ? static_cast<int64_t>(rows_per_request) * (num_q_heads / num_kv_heads)
                           : 1;
  return heuristic_partition(num_requests, num_kv_heads, block_size, max_context_len, rows);
}

size_t kvq_paged_decode_workspace_size(int32_t num_requests, int32_t rows_per_request,
                                       int32_t num_q_heads, int32_t num_kv_heads,
                                       int32_t head_dim, int32_t block_size,
                                       int32_t max_context_len, int32_t partition_tokens) {
  kvq_cache c{};
  c.num_slots = 0;
  c.num_kv_heads = num_kv_heads;
  c.head_dim = head_dim;
  c.block_size = block_size;
  kvq::AttnShape s;
  if (make_shape(&c, num_requests, rows_per_request, num_q_heads, 1, max_context_len,
                 partition_tokens, &s) != KVQ_OK)
    return 0;
  return workspace_for(s);
}

namespace {

// kvq_paged_decode_partials, with a decode step's new rows stored first when
// `append` is given (inside the load-balanced kernel where the shape takes it)
kvq_status decode_partials(const kvq_cache *cache, const void *q, int32_t num_requests,
                                     int32_t rows_per_request, int32_t num_q_heads,
                                     const int32_t *block_tables, int32_t max_blocks_per_req,
                                     const int32_t *context_lens, int32_t max_context_len,
                                     float sm_scale, int32_t partition_tokens, void *out,
                                     void *workspace, size_t workspace_bytes,
                                     int32_t *err_flags, kvq_stream_t stream,
                                     const kvq::AppendRows *append) {
  kvq::AttnShape s;
  kvq_status st = make_shape(cache, num_requests, rows_per_request, num_q_heads,
                             max_blocks_per_req, max_context_len, partition_tokens, &s);
  if (st != KVQ_OK) return st;
  if (!std::isfinite(sm_scale)) return KVQ_ERR_INVALID_ARGUMENT;
  if (num_requests == 0) return KVQ_OK;
  if (q == nullptr || out == nullptr || block_tables == nullptr || context_lens == nullptr)
    return KVQ_ERR_INVALID_ARGUMENT;
  if (!aligned(q, 16) || !aligned(out, 16) || !aligned(block_tables, 4) ||
      !aligned(context_lens, 4) || !aligned(workspace, 16) || !aligned(err_flags, 4))
    return KVQ_ERR_MISALIGNED;
  const size_t need = workspace_for(s);
  if (need > 0 && (workspace == nullptr || workspace_bytes < need))
    return KVQ_ERR_WORKSPACE_TOO_SMALL;
  // the rows-on-M kernel loads the scale planes by TMA (16-byte aligned) and
  // numbers slots in 32 bits; other caches of <= 128 stacked rows run the
  // partitioned kernels with one partition per request (no workspace)
  if (s.rows_kernel && !kvq::attn_rows_supported(*cache, s)) {
    if (s.rows > kMaxRowsPerKvHead) return KVQ_ERR_UNSUPPORTED;
    s.rows_kernel = 0;
    s.partition_tokens = std::max<int32_t>(64, (max_context_len + 63) / 64 * 64);
    s.num_partitions = 1;
  }
  return from_cuda(kvq::launch_attn_partials(*cache, s, q, block_tables, context_lens, sm_scale,
                                             out, workspace, err_flags,
                                             reinterpret_cast<cudaStream_t>(stream), append));
}

}  // namespace

kvq_status kvq_paged_decode_partials(const kvq_cache *cache, const void *q, int32_t num_requests,
                                     int32_t rows_per_request, int32_t num_q_heads,
                                     const int32_t *block_tables, int32_t max_blocks_per_req,
                                     const int32_t *context_lens, int32_t max_context_len,
                                     float sm_scale, int32_t partition_tokens, void *out,
                                     void *workspace, size_t workspace_bytes,
                                     int32_t *err_flags, kvq_stream_t stream) {
  return decode_partials(cache, q, num_requests, rows_per_request, num_q_heads, block_tables,
                         max_blocks_per_req, context_lens, max_context_len, sm_scale,
                         partition_tokens, out, workspace, workspace_bytes, err_flags, stream,
                         nullptr);
}

kvq_status kvq_paged_decode_append_partials(
    const kvq_cache *cache, const void *k_new, int64_t k_token_stride, const void *v_new,
    int64_t v_token_stride, const void *q, int32_t num_requests, int32_t rows_per_request,
    int32_t num_q_heads, const int32_t *block_tables, int32_t max_blocks_per_req,
    const int32_t *context_lens, int32_t max_context_len, float sm_scale,
    int32_t partition_tokens, void *out, void *workspace, size_t workspace_bytes,
    int32_t *err_flags, kvq_stream_t stream) {
  kvq_status st = check_cache(cache, true);
  if (st != KVQ_OK) return st;
  if (num_requests > 0) {
    if (k_new == nullptr || v_new == nullptr || k_token_stride < 0 || v_token_stride < 0 ||
        rows_per_request < 1)
      return KVQ_ERR_INVALID_ARGUMENT;
    if (!aligned(k_new, 16) || !aligned(v_new, 16) || (k_token_stride % 8) != 0 ||
        (v_token_stride % 8) != 0)
      return KVQ_ERR_MISALIGNED;
    // rows (token, K/V, head) of the store are numbered in 32 bits
    if (static_cast<int64_t>(num_requests) * rows_per_request >
        (int64_t(1) << 31) / (2 * cache->num_kv_heads) - 32)
      return KVQ_ERR_UNSUPPORTED;
  }
  const kvq::AppendRows append{k_new, k_token_stride, v_new, v_token_stride};
  return decode_partials(cache, q, num_requests, rows_per_request, num_q_heads, block_tables,
                         max_blocks_per_req, context_lens, max_context_len, sm_scale,
                         partition_tokens, out, workspace, workspace_bytes, err_flags, stream,
                         &append);
}

kvq_status kvq_paged_decode_combine(const kvq_cache *cache, int32_t num_requests,
                                    int32_t rows_per_request, int32_t num_q_heads,
                                    int32_t max_blocks_per_req, const int32_t *context_lens,
                                    int32_t max_context_len, int32_t partition_tokens,
                                    void *out, void *workspace, size_t workspace_bytes,
                                    kvq_stream_t stream) {
  kvq::AttnShape s;
  kvq_status st = make_shape(cache, num_requests, rows_per_request, num_q_heads,
                             max_blocks_per_req, max_context_len, partition_tokens, &s);
  if (st != KVQ_OK) return st;
  if (num_requests == 0 || s.rows_kernel || s.num_partitions <= 1) return KVQ_OK;
  if (out == nullptr || context_lens == nullptr) return KVQ_ERR_INVALID_ARGUMENT;
  if (!aligned(out, 16) || !aligned(context_lens, 4) || !aligned(workspace, 16))
    return KVQ_ERR_MISALIGNED;
  const size_t need = workspace_for(s);
  if (workspace == nullptr || workspace_bytes < need) return KVQ_ERR_WORKSPACE_TOO_SMALL;
  return from_cuda(kvq::launch_attn_combine(s, context_lens, out, workspace,
                                            reinterpret_cast<cudaStream_t>(stream)));
}

kvq_status kvq_paged_decode(const kvq_cache *cache, const void *q, int32_t num_requests,
                            int32_t rows_per_request, int32_t num_q_heads,
                            const int32_t *block_tables, int32_t max_blocks_per_req,
                            const int32_t *context_lens, int32_t max_context_len,
                            float sm_scale, int32_t partition_tokens, void *out,
                            void *workspace, size_t workspace_bytes, int32_t *err_flags,
                            kvq_stream_t stream) {
  kvq_status st = kvq_paged_decode_partials(
      cache, q, num_requests, rows_per_request, num_q_heads, block_tables, max_blocks_per_req,
      context_lens, max_context_len, sm_scale, partition_tokens, out, workspace,
      workspace_bytes, err_flags, stream);
  if (st != KVQ_OK) return st;
  return kvq_paged_decode_combine(cache, num_requests, rows_per_request, num_q_heads,
                                  max_blocks_per_req, context_lens, max_context_len,
                                  partition_tokens, out, workspace, workspace_bytes, stream);
}

kvq_status kvq_paged_decode_append(const kvq_cache *cache, const void *k_new,
                                   int64_t k_token_stride, const void *v_new,
                                   int64_t v_token_stride, const void *q, int32_t num_requests,
                                   int32_t rows_per_request, int32_t num_q_heads,
                                   const int32_t *block_tables, int32_t max_blocks_per_req,
                                   const int32_t *context_lens, int32_t max_context_len,
                                   float sm_scale, int32_t partition_tokens, void *out,
                                   void *workspace, size_t workspace_bytes, int32_t *err_flags,
                                   kvq_stream_t stream) {
  kvq_status st = kvq_paged_decode_append_partials(
      cache, k_new, k_token_stride, v_new, v_token_stride, q, num_requests, rows_per_request,
      num_q_heads, block_tables, max_blocks_per_req, context_lens, max_context_len, sm_scale,
      partition_tokens, out, workspace, workspace_bytes, err_flags, stream);
  if (st != KVQ_OK) return st;
  return kvq_paged_decode_combine(cache, num_requests, rows_per_request, num_q_heads,
                                  max_blocks_per_req, context_lens, max_context_len,
                                  partition_tokens, out, workspace, workspace_bytes, stream);
}

kvq_status kvq_quantize_scatter_unscaled(const kvq_cache *cache, int32_t code_format,
                                         const void *k, int64_t k_token_stride, const void *v,
                                         int64_t v_token_stride, int64_t num_tokens,
                                         const int64_t *slot_ids, int32_t *err_flags,
                                         kvq_stream_t stream) {
  if (code_format != KVQ_CODES_E4M3 && code_format != KVQ_CODES_E5M2)
    return KVQ_ERR_INVALID_ARGUMENT;
  kvq_status st = check_cache(cache, false);
  if (st != KVQ_OK) return st;
  if (num_tokens < 0 || k_token_stride < 0 || v_token_stride < 0)
    return KVQ_ERR_INVALID_ARGUMENT;
  if (num_tokens == 0) return KVQ_OK;
  if (k == nullptr || v == nullptr || slot_ids == nullptr) return KVQ_ERR_INVALID_ARGUMENT;
  if (!aligned(k, 16) || !aligned(v, 16) || (k_token_stride % 8) != 0 ||
      (v_token_stride % 8) != 0 || !aligned(slot_ids, 8) || !aligned(err_flags, 4))
    return KVQ_ERR_MISALIGNED;
  if (num_tokens > (int64_t(1) << 31) / (2 * cache->num_kv_heads) - 32) return KVQ_ERR_UNSUPPORTED;
  return from_cuda(kvq::launch_quantize_unscaled(*cache, code_format, k, k_token_stride, v,
                                                 v_token_stride, num_tokens, slot_ids, err_flags,
                                                 reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"

namespace {

// The shape of a kvq_paged_decode_codes call: the rows-on-M kernel for every
// row count.
kvq_status make_codes_shape(const kvq_cache *cache, int32_t num_requests,
                            int32_t rows_per_request, int32_t num_q_heads,
                            int32_t max_blocks_per_req, int32_t max_context_len,
                            kvq::AttnShape *s) {
  if (cache != nullptr && cache->num_kv_heads > 0 && num_q_heads > 0 && rows_per_request > 0 &&
      num_q_heads % cache->num_kv_heads == 0 &&
      static_cast<int64_t>(rows_per_request) * (num_q_heads / cache->num_kv_heads) > kvq::kRowsMaxRows)
    return KVQ_ERR_UNSUPPORTED;
  // the common checks (cache, sizes, GQA) as for one query row with a fixed
  // partition size; then the shape is switched to the rows-on-M kernel
  if (rows_per_request < 1) return KVQ_ERR_INVALID_ARGUMENT;
  kvq_status st = make_shape(cache, num_requests, 1, num_q_heads, max_blocks_per_req,
                             max_context_len, 64, s);
  if (st != KVQ_OK) return st;
  if (cache->block_size < 16 || cache->num_kv_heads % 4 != 0 ||
      num_requests > kvq::kRowsMaxRequests)
    return KVQ_ERR_UNSUPPORTED;
  const int64_t M = static_cast<int64_t>(rows_per_request) * s->group;
  s->rows_per_request = rows_per_request;
  s->rows = static_cast<int32_t>(M);
  s->row_groups = static_cast<int32_t>((M + 31) / 32);
  s->rows_kernel = 1;
  s->stream = 0;
  s->num_partitions = 1;
  return KVQ_OK;
}

}  // namespace

extern "C" {

size_t kvq_paged_decode_codes_workspace_size(int32_t num_requests, int32_t rows_per_request,
                                             int32_t num_q_heads, int32_t num_kv_heads,
                                             int32_t head_dim, int32_t block_size,
                                             int32_t max_context_len) {
  kvq_cache c{};
  c.num_slots = 0;
  c.num_kv_heads = num_kv_heads;
  c.head_dim = head_dim;
  c.block_size = block_size;
  kvq::AttnShape s;
  if (make_codes_shape(&c, num_requests, rows_per_request, num_q_heads, 1, max_context_len, &s) !=
      KVQ_OK)
    return 0;
  return kvq::attn_rows_workspace_bytes(s, num_kv_heads);
}

kvq_status kvq_paged_decode_codes(const kvq_cache *cache, int32_t code_format, const void *q,
                                  int32_t num_requests, int32_t rows_per_request,
                                  int32_t num_q_heads, const int32_t *block_tables,
                                  int32_t max_blocks_per_req, const int32_t *context_lens,
                                  int32_t max_context_len, float sm_scale, void *out,
                                  void *workspace, size_t workspace_bytes, int32_t *err_flags,
                                  kvq_stream_t stream) {
  if (code_format != KVQ_CODES_E4M3 && code_format != KVQ_CODES_E5M2)
    return KVQ_ERR_INVALID_ARGUMENT;
  kvq::AttnShape s;
  kvq_status st = make_codes_shape(cache, num_requests, rows_per_request, num_q_heads,
                                   max_blocks_per_req, max_context_len, &s);
  if (st != KVQ_OK) return st;
  if (!std::isfinite(sm_scale)) return KVQ_ERR_INVALID_ARGUMENT;
  if (num_requests == 0) return KVQ_OK;
  if (q == nullptr || out == nullptr || block_tables == nullptr || context_lens == nullptr)
    return KVQ_ERR_INVALID_ARGUMENT;
  if (!aligned(q, 16) || !aligned(out, 16) || !aligned(block_tables, 4) ||
      !aligned(context_lens, 4) || !aligned(workspace, 16) || !aligned(err_flags, 4))
    return KVQ_ERR_MISALIGNED;
  if (!kvq::attn_rows_supported(*cache, s)) return KVQ_ERR_UNSUPPORTED;
  const size_t need = kvq::attn_rows_workspace_bytes(s, cache->num_kv_heads);
  if (workspace == nullptr || workspace_bytes < need) return KVQ_ERR_WORKSPACE_TOO_SMALL;
  return from_cuda(kvq::launch_attn_rows(*cache, s, q, block_tables, context_lens, sm_scale, out,
                                         workspace, err_flags,
                                         reinterpret_cast<cudaStream_t>(stream), code_format));
}

kvq_status kvq_dequant_rows(const kvq_cache *cache, const int64_t *slot_ids, int64_t n,
                            int32_t out_dtype, void *out_k, void *out_v, int32_t *err_flags,
                            kvq_stream_t stream) {
  kvq_status st = check_cache(cache, false);
  if (st != KVQ_OK) return st;
  if (n < 0 || (out_dtype != 0 && out_dtype != 1)) return KVQ_ERR_INVALID_ARGUMENT;
  if (n == 0 || (out_k == nullptr && out_v == nullptr)) return KVQ_OK;
  if (slot_ids == nullptr) return KVQ_ERR_INVALID_ARGUMENT;
  if (!aligned(slot_ids, 8) || !aligned(out_k, 16) || !aligned(out_v, 16) ||
      !aligned(err_flags, 4))
    return KVQ_ERR_MISALIGNED;
  if ((n + 7) / 8 > 0x7FFFFFFF) return KVQ_ERR_UNSUPPORTED;
  return from_cuda(kvq::launch_dequant_rows(*cache, slot_ids, n, out_dtype, out_k, out_v,
                                            err_flags, reinterpret_cast<cudaStream_t>(stream)));
}

size_t kvq_index_cache_bytes(int64_t num_slots, int32_t format, int32_t dim) {
  if (num_slots < 0 || dim <= 0 || dim % 32 != 0) return 0;
  if (format == KVQ_INDEX_FP8) return static_cast<size_t>(num_slots) * (dim + 4);
  if (format == KVQ_INDEX_MXFP4) return static_cast<size_t>(num_slots) * (dim / 2 + dim / 32);
  return 0;
}

}  // extern "C"

namespace {

kvq_status check_index_cache(const kvq_index_cache *c) {
  if (c == nullptr) return KVQ_ERR_INVALID_ARGUMENT;
  if (c->num_slots < 0 || c->dim <= 0) return KVQ_ERR_INVALID_ARGUMENT;
  if (c->format != KVQ_INDEX_FP8 && c->format != KVQ_INDEX_MXFP4) return KVQ_ERR_INVALID_ARGUMENT;
  if (c->dim != kvq::kHeadDimAbi) return KVQ_ERR_UNSUPPORTED;
  if (c->num_slots > 0) {
    if (c->codes == nullptr) return KVQ_ERR_INVALID_ARGUMENT;
    if (c->format == KVQ_INDEX_FP8 && c->scales == nullptr) return KVQ_ERR_INVALID_ARGUMENT;
    if (c->format == KVQ_INDEX_MXFP4 && c->exponents == nullptr) return KVQ_ERR_INVALID_ARGUMENT;
  }
  if (!aligned(c->codes, 16) || !aligned(c->scales, 4)) return KVQ_ERR_MISALIGNED;
  return KVQ_OK;
}

}  // namespace

extern "C" {

kvq_status kvq_index_quantize_scatter(const kvq_index_cache *cache, const void *x,
                                      int64_t x_token_stride, int64_t num_tokens,
                                      const int64_t *slot_ids, int32_t *err_flags,
                                      kvq_stream_t stream) {
  kvq_status st = check_index_cache(cache);
  if (st != KVQ_OK) return st;
  if (num_tokens < 0 || x_token_stride < 0) return KVQ_ERR_INVALID_ARGUMENT;
  if (num_tokens == 0) return KVQ_OK;
  if (x == nullptr || slot_ids == nullptr) return KVQ_ERR_INVALID_ARGUMENT;
  if (!aligned(x, 16) || (x_token_stride % 8) != 0 || !aligned(slot_ids, 8) ||
      !aligned(err_flags, 4))
    return KVQ_ERR_MISALIGNED;
  if ((num_tokens + 31) / 32 > 0x7FFFFFFF) return KVQ_ERR_UNSUPPORTED;
  return from_cuda(kvq::launch_index_quantize_scatter(*cache, x, x_token_stride, num_tokens,
                                                      slot_ids, err_flags,
                                                      reinterpret_cast<cudaStream_t>(stream)));
}

kvq_status kvq_index_dequant_rows(const kvq_index_cache *cache, const int64_t *slot_ids,
                                  int64_t n, int32_t out_dtype, void *out, int32_t *err_flags,
                                  kvq_stream_t stream) {
  kvq_status st = check_index_cache(cache);
  if (st != KVQ_OK) return st;
  if (n < 0 || (out_dtype != 0 && out_dtype != 1)) return KVQ_ERR_INVALID_ARGUMENT;
  if (n == 0) return KVQ_OK;
  if (slot_ids == nullptr || out == nullptr) return KVQ_ERR_INVALID_ARGUMENT;
  if (!aligned(slot_ids, 8) || !aligned(out, 16) || !aligned(err_flags, 4))
    return KVQ_ERR_MISALIGNED;
  if ((n + 3) / 4 > 0x7FFFFFFF) return KVQ_ERR_UNSUPPORTED;
  return from_cuda(kvq::launch_index_dequant_rows(*cache, slot_ids, n, out_dtype, out, err_flags,
                                                  reinterpret_cast<cudaStream_t>(stream)));
}

kvq_status kvq_index_scores(const kvq_index_cache *cache, int32_t block_size, const void *q,
                            int32_t num_requests, int32_t rows_per_request,
                            int32_t num_index_heads, const int32_t *block_tables,
                            int32_t max_blocks_per_req, const int32_t *context_lens,
                            int32_t max_context_len, float *out, int32_t *err_flags,
                            kvq_stream_t stream) {
  kvq_status st = check_index_cache(cache);
  if (st != KVQ_OK) return st;
  if (block_size <= 0 || num_requests < 0 || rows_per_request < 1 || num_index_heads < 1 ||
      max_blocks_per_req < 0 || max_context_len < 0)
    return KVQ_ERR_INVALID_ARGUMENT;
  if (!is_pow2(block_size) || block_size < 16 ||
      !kvq::index_scores_supported(rows_per_request, num_index_heads))
    return KVQ_ERR_UNSUPPORTED;
  if (num_requests > 65535) return KVQ_ERR_UNSUPPORTED;
  if (num_requests == 0 || max_context_len == 0) return KVQ_OK;
  if (q == nullptr || block_tables == nullptr || context_lens == nullptr || out == nullptr)
    return KVQ_ERR_INVALID_ARGUMENT;
  if (!aligned(q, 16) || !aligned(block_tables, 4) || !aligned(context_lens, 4) ||
      !aligned(out, 4) || !aligned(err_flags, 4) || !aligned(cache->scales, 16) ||
      !aligned(cache->exponents, 16))
    return KVQ_ERR_MISALIGNED;
  return from_cuda(kvq::launch_index_scores(
      *cache, log2_exact(block_size), q, num_requests, rows_per_request, num_index_heads,
      block_tables, max_blocks_per_req, context_lens, max_context_len, out, err_flags,
      current_sm_count(), reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
