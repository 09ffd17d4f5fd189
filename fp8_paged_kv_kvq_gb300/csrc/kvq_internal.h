// kvq_internal.h -- launchers shared between the C-ABI layer (kvq_api.cu) and
// the kernel translation units.  Not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "kvq.h"

namespace kvq {

// Launches `kernel` with programmatic stream serialization, so that its launch
// overlaps the drain of the previous kernel in the stream; every kernel
// launched this way calls grid_dependency_wait() before its first access to
// global memory (read or write), so it sees everything earlier work on the
// stream wrote -- also when that work let its dependents launch early -- and
// overwrites nothing that work still reads.
template <typename... KArgs, typename... Args>
cudaError_t launch_overlapped(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

// The only head_dim the kernels implement; the ABI refuses any other.
constexpr int32_t kHeadDimAbi = 128;

// Shape of one paged attention call after host-side validation.
struct AttnShape {
  int32_t num_requests;
  int32_t rows_per_request;   // R
  int32_t num_q_heads;        // Hq
  int32_t group;              // G = Hq / H
  int32_t rows;               // M = R * G
  int32_t row_groups;         // ceil(M / 32)
  int32_t max_blocks_per_req;
  int32_t max_context_len;
  int32_t partition_tokens;   // P, multiple of 64
  int32_t num_partitions;     // ceil(max_context_len / P), >= 1
  int32_t log2_block;
  int32_t sms;                // SMs of the current device
  int32_t stream;             // 1: the load-balanced kernel (partials in stream slots)
  int32_t rows_kernel;        // 1: the rows-on-M tcgen05 kernel (no combine launch)
  int32_t num_kv_heads;
};

// A nonzero tag per launch of a kernel that counts pieces with tagged
// tickets (ticket_take): a ticket word left by another call, or any other
// content of the workspace, carries another tag and is restarted.
uint32_t next_call_tag();

// The load-balanced decode kernel's workspace: the piece count of each
// (request, group of 4 KV heads) as int32, then partials in kStreamSlots slots
// per output row.
constexpr int32_t kStreamSlots = 16;
// A segment (the chunks of one request and head group) is charged this many
// extra chunks at its start, so a CTA whose range crosses into a new segment
// (a second query preparation, during which its ring stands full) gets
// correspondingly less work.
constexpr int32_t kStreamSwitchChunks = 5;
constexpr int32_t kStreamMaxRequests = 1024;
// New rows per request that the load-balanced kernel stores itself (a decode
// step's store fused into its attention); more take the store's own launch.
constexpr int32_t kStreamNewRows = 2;
size_t attn_stream_pieces_bytes(int32_t num_requests, int32_t num_kv_heads);

// Whether a shape suits the load-balanced kernel (apart from the cache's
// scale alignment): at most 8 stacked rows, pages of >= 16 tokens, KV heads in
// groups of 4, at most kStreamMaxRequests requests, a segment's block ids
// within its window.
bool attn_stream_shape_ok(int32_t num_kv_heads, const AttnShape &s);
// The step's new K and V rows for a store fused into the attention: row
// r * R + i (token pitch k_stride / v_stride elements, heads 128 elements
// apart) goes to position L_r - R + i of request r.
struct AppendRows {
  const void *k;
  int64_t k_stride;
  const void *v;
  int64_t v_stride;
};
cudaError_t launch_attn_partials_stream(const kvq_cache &c, const AttnShape &s, const void *q,
                                        const int32_t *block_tables,
                                        const int32_t *context_lens, float sm_scale, void *out,
                                        void *workspace, int32_t *err_flags,
                                        cudaStream_t stream, const AppendRows *append = nullptr);
cudaError_t launch_attn_combine_stream(const AttnShape &s, void *out, void *workspace,
                                       cudaStream_t stream);

// Workspace carve-up: partial outputs [rows_total][num_partitions][128] fp32,
// then (max, denominator) pairs [rows_total][num_partitions][2] fp32.
size_t attn_workspace_bytes(int64_t rows_total, int32_t num_partitions);

cudaError_t launch_quantize_scatter(const kvq_cache &c, const void *k, int64_t k_stride,
                                    const void *v, int64_t v_stride, int64_t num_tokens,
                                    const int64_t *slot_ids, int32_t *err_flags,
                                    cudaStream_t stream);
// The quantize-scatter of a decode step's new rows, slots from the block
// tables: token r R + i to position L_r - R + i of request r (skipped when
// negative; a page id out of range is skipped and flagged).
cudaError_t launch_quantize_positions(const kvq_cache &c, const void *k, int64_t k_stride,
                                     const void *v, int64_t v_stride, int32_t num_requests,
                                     int32_t rows_per_request, const int32_t *block_tables,
                                     int32_t max_blocks_per_req, const int32_t *context_lens,
                                     int32_t ctx_limit, int32_t log2_block, int32_t *err_flags,
                                     cudaStream_t stream);

cudaError_t launch_dequant_rows(const kvq_cache &c, const int64_t *slot_ids, int64_t n,
                                int32_t out_dtype, void *out_k, void *out_v,
                                int32_t *err_flags, cudaStream_t stream);

cudaError_t launch_index_quantize_scatter(const kvq_index_cache &c, const void *x,
                                          int64_t x_stride, int64_t num_tokens,
                                          const int64_t *slot_ids, int32_t *err_flags,
                                          cudaStream_t stream);

cudaError_t launch_index_dequant_rows(const kvq_index_cache &c, const int64_t *slot_ids,
                                      int64_t n, int32_t out_dtype, void *out,
                                      int32_t *err_flags, cudaStream_t stream);

// Stacked index scorer: R * H <= 16 query vectors per request, H in {1,2,4,8}.
bool index_scores_supported(int32_t rows_per_request, int32_t num_index_heads);
cudaError_t launch_index_scores(const kvq_index_cache &c, int32_t log2_block, const void *q,
                                int32_t num_requests, int32_t rows_per_request,
                                int32_t num_index_heads, const int32_t *block_tables,
                                int32_t max_blocks_per_req, const int32_t *context_lens,
                                int32_t max_context_len, float *out, int32_t *err_flags,
                                int32_t sms, cudaStream_t stream);

cudaError_t launch_attn_partials(const kvq_cache &c, const AttnShape &s, const void *q,
                                 const int32_t *block_tables, const int32_t *context_lens,
                                 float sm_scale, void *out, void *workspace,
                                 int32_t *err_flags, cudaStream_t stream,
                                 const AppendRows *append = nullptr);

// Tensor map over one code plane [num_slots, H, 128] uint8: boxes of `rows`
// slots of one head, 128-byte swizzled in shared memory.
bool encode_code_tensor_map(CUtensorMap *map, const uint8_t *codes, int64_t num_slots, int H,
                            int rows);

// Tensor map over one scale plane [num_slots, H] fp32: boxes of 4 heads x `rows`
// slots (H a multiple of 4, the plane 16-byte aligned).
bool encode_scale_tensor_map(CUtensorMap *map, const float *scales, int64_t num_slots, int H,
                             int rows);

// Tensor map over one code plane [num_slots, H, 128] uint8 ordered (128 bytes,
// slots, heads): boxes of 16 slots x 4 heads, 128-byte swizzled per head.
bool encode_code_tensor_map_strided(CUtensorMap *map, const uint8_t *codes, int64_t num_slots,
                                    int H);

// The page-major partials kernel for at most 8 stacked rows per KV head
// (pages of >= 16 tokens, KV heads a multiple of 4).
bool attn_page_supported(const kvq_cache &c, const AttnShape &s);
cudaError_t launch_attn_partials_page(const kvq_cache &c, const AttnShape &s, const void *q,
                                      const int32_t *block_tables, const int32_t *context_lens,
                                      float sm_scale, void *out, float *o_part, float2 *ml_part,
                                      int32_t *err_flags, cudaStream_t stream);

// The rows-on-M tcgen05 kernel for more than 8 stacked rows per KV head
// (verify, chunked prefill): a persistent grid of one CTA per SM over the
// batch's 128-token chunks, units cut by a range boundary merged by their last
// piece.  Its workspace: a ticket per (request, KV head, 128-row tile), then
// the pieces' partials, two slots per CTA.
constexpr int32_t kRowsMaxRequests = 1024;
constexpr int32_t kRowsSwitch = 3;          // chunk charge per unit start
constexpr int32_t kRowsMaxRows = 8192;      // stacked rows per KV head
int32_t attn_rows_per_tile(int32_t rows);
bool attn_rows_supported(const kvq_cache &c, const AttnShape &s);
size_t attn_rows_workspace_bytes(const AttnShape &s, int32_t num_kv_heads);
cudaError_t launch_attn_rows(const kvq_cache &c, const AttnShape &s, const void *q,
                             const int32_t *block_tables, const int32_t *context_lens,
                             float sm_scale, void *out, void *workspace, int32_t *err_flags,
                             cudaStream_t stream, int32_t code_format = KVQ_CODES_E4M3);

// The unscaled store of the codec ablation: codes = e4m3 or e5m2 cast of each
// value, scales 1.
cudaError_t launch_quantize_unscaled(const kvq_cache &c, int32_t code_format, const void *k,
                                     int64_t k_stride, const void *v, int64_t v_stride,
                                     int64_t num_tokens, const int64_t *slot_ids,
                                     int32_t *err_flags, cudaStream_t stream);

// The tcgen05 partials kernel for 9..32 stacked rows per KV head.
bool attn_tc_supported(const kvq_cache &c, const AttnShape &s);
cudaError_t launch_attn_partials_tc(const kvq_cache &c, const AttnShape &s, const void *q,
                                    const int32_t *block_tables, const int32_t *context_lens,
                                    float sm_scale, void *out, float *o_part, float2 *ml_part,
                                    int32_t *err_flags, cudaStream_t stream);

// The partials kernel for at most 8 stacked rows per KV head (block size >= 8).
bool attn_skinny_supported(const kvq_cache &c, const AttnShape &s);
cudaError_t launch_attn_partials_skinny(const kvq_cache &c, const AttnShape &s, const void *q,
                                        const int32_t *block_tables, const int32_t *context_lens,
                                        float sm_scale, void *out, float *o_part,
                                        float2 *ml_part, int32_t *err_flags,
                                        cudaStream_t stream);

cudaError_t launch_attn_combine(const AttnShape &s, const int32_t *context_lens, void *out,
                                void *workspace, cudaStream_t stream);

}  // namespace kvq
