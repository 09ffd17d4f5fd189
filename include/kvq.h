/*
 * kvq.h -- C ABI of libkvq: an FP8 E4M3 paged KV cache with one FP32 scale per
 * (token, KV head) row, for NVIDIA GB300 (sm_103a).
 *
 * What the operations compute, and where that is defined:
 *
 *  - Row format.  ROCm/ATOM PR #2655 "fix(qwen4-exp): register the QSA FP8
 *    scale planes for KV offload", PR description (K/V bullet), and
 *    FlashML-org/FreeToken PR #354 "feat(kvcache): store the KV cache as fp8
 *    e4m3 codes", PR description: every cached (token, KV head) row, of K as of
 *    V, is held as head_dim E4M3 bytes and a single symmetric fp32 scale,
 *        scale = amax(|x|) / 448,   code_d = e4m3_rne(x_d / scale),
 *    so the row's largest element maps to +-448 and nothing saturates.  The
 *    code bytes sit in a plain uint8 buffer shaped like the 16-bit cache
 *    ([num_slots, num_kv_heads, head_dim]); the scales in a sidecar
 *    [num_slots, num_kv_heads] fp32.  Division and rounding are IEEE binary32,
 *    round-to-nearest-even; |x / scale| >= 448 saturates to 448; an all-zero
 *    row stores scale 0 and codes 0x00; a NaN code is never written.
 *
 *  - Attention.  ATOM PR #2655, PR description (K/V bullet): attention runs
 *    on the E4M3 tiles; a token's key scale is applied to its score after the
 *    code dot product and its value scale to its probability ahead of PV.  With G = Hq / H query
 *    heads per KV head (query head hq reads KV head hq / G), for request r with
 *    context length L and R query rows (R = 1: decode; R > 1: the rows of a
 *    multi-token verify whose last R tokens are already cached, as in the
 *    stacked MTP-verify rows of ATOM PR #2655), row i sees cached tokens
 *    j < L - R + 1 + i and
 *        s_j  = sm_scale * k_scale_j * sum_d q_d * e4m3(kc_{j,d})
 *        out  = sum_j (p_j * v_scale_j) * e4m3(vc_j) / sum_j p_j,
 *        p_j  = exp(s_j - max_j s_j).
 *    A row that sees no token outputs zeros.
 *
 * Conventions for every entry point:
 *  - Pointers named as device memory must be device (or managed) memory of the
 *    current CUDA device; the caller owns every buffer.  The library never
 *    allocates, never synchronises and never reads device data on the host, so
 *    each call is asynchronous on `stream` and can be captured in a CUDA graph.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).
 *  - Ordering on the stream.  Every kernel of the library is launched with
 *    programmatic stream serialization, so it may start while the previous
 *    kernel on `stream` is still draining; before its first access to global
 *    memory (inputs, cache, workspace, outputs, err_flags) each kernel waits
 *    until that kernel has completed and its writes are visible
 *    (griddepcontrol.wait).  Only the launch and the shared-memory set-up
 *    overlap.  Inputs written by earlier work on the stream -- also by a
 *    kernel of the caller's that lets its dependents launch early -- are
 *    therefore read after that work has finished; no extra synchronisation is
 *    needed.
 *  - Arguments are validated on the host before anything is launched; a
 *    violation returns a status and launches nothing.  A launch failure returns
 *    KVQ_ERR_CUDA.  Unsupported shapes are refused, never silently handled by
 *    a slower path.
 *  - Errors that depend on device data (an out-of-range slot id, block id or
 *    context length) cannot be seen on the host: the offending write or read is
 *    skipped and a bit is OR-ed into the optional device word `err_flags`
 *    (KVQ_ERRF_*); read it after the stream completes.  Outputs that depend on
 *    skipped data are unspecified but every access stays inside the buffers.
 *  - head_dim must be 128.  Alignment: code buffers, q, out, k, v and the
 *    workspace 16 bytes; token strides of k and v multiples of 8 elements;
 *    slot ids 8 bytes; scales, block tables and context lengths 4 bytes.
 */
#ifndef KVQ_H
#define KVQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;                      /* the type cudaStream_t points to */
typedef struct CUstream_st *kvq_stream_t;

typedef enum kvq_status {
    KVQ_OK = 0,
    KVQ_ERR_INVALID_ARGUMENT = 1,        /* null pointer, negative size, bad shape     */
    KVQ_ERR_UNSUPPORTED = 2,             /* valid but not implemented (e.g. head_dim)  */
    KVQ_ERR_MISALIGNED = 3,              /* a pointer or stride breaks the alignment   */
    KVQ_ERR_WORKSPACE_TOO_SMALL = 4,     /* workspace_bytes below the required size    */
    KVQ_ERR_CUDA = 5                     /* a CUDA call or kernel launch failed        */
} kvq_status;

/* Bits OR-ed into *err_flags by the kernels. */
#define KVQ_ERRF_SLOT_RANGE 1            /* slot id >= num_slots (write/read skipped)  */
#define KVQ_ERRF_BLOCK_RANGE 2           /* block id outside [0, num_slots/block_size) */
#define KVQ_ERRF_CONTEXT_RANGE 4         /* context length < 0, > max_context_len or
                                            > max_blocks_per_req * block_size          */
#define KVQ_ERRF_WAIT_TIMEOUT 8          /* a bounded in-kernel wait for an async copy
                                            gave up; that CTA's outputs are not written */

/* The cache: codes and scales always travel together (ATOM PR #2655,
 * "Motivation": a restore that drops the scale planes decodes rows under the
 * wrong scales).  All four arrays are device memory owned by the caller.
 *   k_codes, v_codes   uint8 [num_slots, num_kv_heads, head_dim]
 *   k_scales, v_scales fp32  [num_slots, num_kv_heads]
 * Slot s of a paged cache belongs to block s / block_size. */
typedef struct kvq_cache {
    uint8_t *k_codes;
    uint8_t *v_codes;
    float *k_scales;
    float *v_scales;
    int64_t num_slots;
    int32_t num_kv_heads;
    int32_t head_dim;
    int32_t block_size;                  /* a power of two; used by the decode only */
} kvq_cache;

/* Text for a status code (static storage). */
const char *kvq_status_string(kvq_status status);

/* ABI version of this header (incremented on any signature change). */
int32_t kvq_abi_version(void);

/* Bytes of codes plus scales for a cache of this size, K and V together:
 * 2 * num_slots * num_kv_heads * (head_dim + 4).  FreeToken PR #354, PR
 * description: the pool counts codes plus the scale sidecar.  Returns 0 for a
 * negative argument. */
size_t kvq_cache_bytes(int64_t num_slots, int32_t num_kv_heads, int32_t head_dim);

/* Fused quantize + scatter of K and V rows into the cache (one launch).
 * FreeToken PR #354, PR description (fused quantize+scatter, one launch under
 * CUDA graph capture, slot ids as a device tensor) and fix commit "give the V
 * tensor its own row pitch in the fp8 KV store" (K and V each have a pitch).
 *   k, v            device bf16; token t's row for KV head h starts at element
 *                   t*k_token_stride + h*head_dim of k (v: v_token_stride); the
 *                   head_dim elements of a row are contiguous.  Either may be a
 *                   strided view of a fused qkv projection output.
 *   k_token_stride, v_token_stride   in elements, multiples of 8, >= 0
 *   num_tokens      rows to store (0 launches nothing)
 *   slot_ids        device int64 [num_tokens]; id < 0 skips the token (padding);
 *                   id >= num_slots skips it and sets KVQ_ERRF_SLOT_RANGE.
 *                   Ids must be unique (two tokens writing one slot race).
 *   err_flags       device int32, optional (NULL)
 * Writes codes and scales of every valid token's K and V rows. */
kvq_status kvq_quantize_scatter(const kvq_cache *cache,
                                const void *k, int64_t k_token_stride,
                                const void *v, int64_t v_token_stride,
                                int64_t num_tokens, const int64_t *slot_ids,
                                int32_t *err_flags, kvq_stream_t stream);

/* Tokens per split-K partition that kvq_paged_decode uses when passed 0 and
 * the shape takes a partitioned kernel: a power of two in [256, 8192] (up to
 * 32768 for 9..32 stacked rows per KV head) chosen from the batch shape and
 * the current device's SM count (152 is assumed when no device is visible);
 * always a multiple of 64.  With 0, shapes of <= 8 stacked rows per KV head
 * whose partition grid would be small, and every shape of more than 8 stacked
 * rows per KV head (rows_per_request * num_q_heads / num_kv_heads; pages of
 * >= 16 tokens, KV heads a multiple of 4), instead split the batch's tokens
 * evenly over a persistent grid and use no fixed partitions. */
int32_t kvq_paged_decode_partition_tokens(int32_t num_requests, int32_t rows_per_request,
                                          int32_t num_q_heads, int32_t num_kv_heads,
                                          int32_t block_size, int32_t max_context_len);

/* Workspace bytes kvq_paged_decode needs for this shape (0 when every request
 * fits one partition).  With fixed partitions: num_requests*rows_per_request*
 * num_q_heads * ceil(max_context_len / partition) * (head_dim + 2) * 4, each
 * of the two parts rounded up to 256.  With partition_tokens 0 the library's
 * own split decides (see kvq_paged_decode_partition_tokens): for <= 8 stacked
 * rows per KV head one piece count per (request, group of 4 KV heads) plus
 * 16 pieces of partial results per output row; for the rows-on-M kernel one 64-bit
 * counter per (request, KV head, 128-row tile) plus two pieces of partial
 * results per SM.  Returns 0 for invalid arguments. */
size_t kvq_paged_decode_workspace_size(int32_t num_requests, int32_t rows_per_request,
                                       int32_t num_q_heads, int32_t num_kv_heads,
                                       int32_t head_dim, int32_t block_size,
                                       int32_t max_context_len, int32_t partition_tokens);

/* Paged GQA decode / multi-row verify attention over the FP8 cache, split-K
 * over partitions of the context (flash-decoding) followed by a combine launch
 * when any request spans more than one partition.
 *   q               device bf16 [num_requests*rows_per_request, num_q_heads,
 *                   head_dim], contiguous; row r*rows_per_request + i is query
 *                   row i of request r.
 *   rows_per_request R >= 1; the stacked rows per KV head, R * (num_q_heads /
 *                   num_kv_heads), at most 128 with a fixed partition size and
 *                   at most 8192 with partition_tokens 0 (a verify step, a
 *                   chunk of prefill: tiles of up to 128 rows each read the
 *                   head's codes once; more than 128 need a cache whose scale
 *                   planes are 16-byte aligned and fewer than 2^31 slots).
 *   num_q_heads     a multiple of cache->num_kv_heads
 *   block_tables    device int32 [num_requests, max_blocks_per_req]: physical
 *                   block of each logical block of the request
 *   context_lens    device int32 [num_requests]: cached tokens per request,
 *                   the R query tokens included
 *   max_context_len host bound on every context length (sizes the grid, so a
 *                   captured graph stays valid while lengths stay below it)
 *   sm_scale        softmax scale applied to q.k (e.g. 1/sqrt(head_dim))
 *   partition_tokens tokens per split-K partition, a multiple of 64 in
 *                   [64, 1<<20]; 0 = kvq_paged_decode_partition_tokens()
 *   out             device bf16, same shape as q (written, round-to-nearest)
 *   workspace       device, >= kvq_paged_decode_workspace_size(...) bytes
 *                   (may be NULL when that size is 0); needs no
 *                   initialisation: every byte a call reads was written by
 *                   the same call, and the piece counters of the rows-on-M
 *                   kernel carry the tag of the call that wrote them, so
 *                   whatever the buffer held before is ignored.
 *   err_flags       device int32, optional
 * Calls that share a workspace must not run concurrently. */
kvq_status kvq_paged_decode(const kvq_cache *cache, const void *q,
                            int32_t num_requests, int32_t rows_per_request,
                            int32_t num_q_heads, const int32_t *block_tables,
                            int32_t max_blocks_per_req, const int32_t *context_lens,
                            int32_t max_context_len, float sm_scale,
                            int32_t partition_tokens, void *out, void *workspace,
                            size_t workspace_bytes, int32_t *err_flags,
                            kvq_stream_t stream);

/* The two launches of kvq_paged_decode, exposed so a caller can time or
 * schedule them separately.  kvq_paged_decode_partials takes kvq_paged_decode's
 * arguments and makes the split-K launch: requests that fit one partition get
 * their final output written to `out`, the others leave per-partition partials
 * (running max, denominator, unnormalised output) in the workspace.
 * kvq_paged_decode_combine merges those partials into `out`; it must follow
 * kvq_paged_decode_partials on the same stream with the same shape, partition
 * size and workspace, and does nothing when no request spans two partitions. */
kvq_status kvq_paged_decode_partials(const kvq_cache *cache, const void *q,
                                     int32_t num_requests, int32_t rows_per_request,
                                     int32_t num_q_heads, const int32_t *block_tables,
                                     int32_t max_blocks_per_req,
                                     const int32_t *context_lens, int32_t max_context_len,
                                     float sm_scale, int32_t partition_tokens, void *out,
                                     void *workspace, size_t workspace_bytes,
                                     int32_t *err_flags, kvq_stream_t stream);

kvq_status kvq_paged_decode_combine(const kvq_cache *cache, int32_t num_requests,
                                    int32_t rows_per_request, int32_t num_q_heads,
                                    int32_t max_blocks_per_req, const int32_t *context_lens,
                                    int32_t max_context_len, int32_t partition_tokens,
                                    void *out, void *workspace, size_t workspace_bytes,
                                    kvq_stream_t stream);

/* One decode step: the store of the step's new rows and the attention that
 * reads them.  kvq_paged_decode_append_partials does what
 * kvq_quantize_scatter of the new rows (slots from the block tables, below)
 * followed by kvq_paged_decode_partials does, with the same arguments and
 * results; kvq_paged_decode_append adds kvq_paged_decode_combine.  The store
 * follows the cache format of the pages (FreeToken PR #354 "feat(kvcache):
 * store the KV cache as fp8 e4m3 codes"; ROCm/ATOM PR #2655, K/V bullet) bit
 * for bit; fusing it with the attention is this library's own step: where the
 * shape takes the load-balanced kernel (kvq_paged_decode_partition_tokens) and
 * rows_per_request is at most 2, the CTA that streams a chunk holding new
 * positions quantises those rows once the chunk has landed in its shared
 * memory, writes their codes and scales over the slots' old contents there
 * (the attention reads the new rows from that copy) and stores them to the
 * cache, so the store costs no launch of its own and the copy never waits
 * for it; other shapes make the store's launch first.
 *   k_new, v_new    device bf16; row r*rows_per_request + i (token pitch
 *                   k_token_stride / v_token_stride elements, multiples of 8,
 *                   16-byte aligned; head h at element h*head_dim) is new token
 *                   i of request r, stored at position
 *                   context_lens[r] - rows_per_request + i of its block table
 *                   (the lengths count the new tokens).  Rows whose position is
 *                   negative are not stored; a position whose page id is outside
 *                   the cache is skipped and sets KVQ_ERRF_BLOCK_RANGE.
 * Other arguments as for kvq_paged_decode. */
kvq_status kvq_paged_decode_append_partials(const kvq_cache *cache, const void *k_new,
                                            int64_t k_token_stride, const void *v_new,
                                            int64_t v_token_stride, const void *q,
                                            int32_t num_requests, int32_t rows_per_request,
                                            int32_t num_q_heads, const int32_t *block_tables,
                                            int32_t max_blocks_per_req,
                                            const int32_t *context_lens, int32_t max_context_len,
                                            float sm_scale, int32_t partition_tokens, void *out,
                                            void *workspace, size_t workspace_bytes,
                                            int32_t *err_flags, kvq_stream_t stream);

kvq_status kvq_paged_decode_append(const kvq_cache *cache, const void *k_new,
                                   int64_t k_token_stride, const void *v_new,
                                   int64_t v_token_stride, const void *q, int32_t num_requests,
                                   int32_t rows_per_request, int32_t num_q_heads,
                                   const int32_t *block_tables, int32_t max_blocks_per_req,
                                   const int32_t *context_lens, int32_t max_context_len,
                                   float sm_scale, int32_t partition_tokens, void *out,
                                   void *workspace, size_t workspace_bytes, int32_t *err_flags,
                                   kvq_stream_t stream);

/* kvq_paged_decode for callers that cannot allocate device memory.  The pages
 * have no counterpart to this entry point; it exists for code that must not or
 * cannot call cudaMalloc where it decodes (inside an allocator or memory-pool
 * callback that must not re-enter the allocator, a plugin handed only its
 * input and output buffers, a runtime that fixes its device memory budget at
 * start-up).  Arguments and results are those of kvq_paged_decode without the
 * workspace: the split-K scratch is a fixed 16 MiB array inside the library,
 * which every GPU that loads the library holds until the process exits.
 *  - A shape whose kvq_paged_decode_workspace_size exceeds 16 MiB (16777216
 *    bytes) is refused with KVQ_ERR_WORKSPACE_TOO_SMALL before any launch.
 *  - The first call on a device looks up the array's device address (once per
 *    device, with that device current) and caches it; make that first call
 *    before any stream capture on the device.
 *  - All calls share the one array and it keeps the last call's contents.
 *    Nothing in it needs to start at zero: every byte a call reads was
 *    written by the same call, and its piece counters carry the call's tag.
 *    Calls that overlap on the GPU (on different streams, or from several
 *    host threads) race on the array and give wrong results; order them on
 *    one stream or with events. */
kvq_status kvq_paged_decode_noalloc(const kvq_cache *cache, const void *q,
                                    int32_t num_requests, int32_t rows_per_request,
                                    int32_t num_q_heads, const int32_t *block_tables,
                                    int32_t max_blocks_per_req, const int32_t *context_lens,
                                    int32_t max_context_len, float sm_scale,
                                    int32_t partition_tokens, void *out, int32_t *err_flags,
                                    kvq_stream_t stream);

/* ------------------------------------------------------------------------ */
/* The codec ablation.  sgl-project/sglang-jax #1776 "feat(dsa): implement fp8
 * KV cache (e4m3) with a bf16 indexer cache", design points and accuracy
 * tests: a cache of O(1) values cast to fp8 with no scale at all, e4m3
 * preferred to e5m2 for its extra mantissa bit (worst-case relative rounding
 * error about 6 % against 12.5 %; attention error against a bf16 cache about
 * twice as large for e5m2).  These two calls store and read such caches, so
 * the three (per-row-scaled e4m3, unscaled e4m3, unscaled e5m2) can be
 * compared on the same kernels. */
#define KVQ_CODES_E4M3 0                 /* 1 sign, 4 exponent (bias 7), 3 mantissa */
#define KVQ_CODES_E5M2 1                 /* 1 sign, 5 exponent (bias 15), 2 mantissa */

/* Quantize + scatter with no scale: code_d = cast(x_d), round-to-nearest-even,
 * saturating at the format's largest finite magnitude (448 for e4m3, 57344 for
 * e5m2; no infinity or NaN code from a finite input), the sign of a zero code
 * taken from its input.  Both scale planes of every stored row are set to 1, so
 * kvq_paged_decode_codes (and, for e4m3, kvq_paged_decode and
 * kvq_dequant_rows) read the codes' own values.  Arguments and errors as for
 * kvq_quantize_scatter; code_format KVQ_CODES_E4M3 or KVQ_CODES_E5M2, anything
 * else KVQ_ERR_INVALID_ARGUMENT. */
kvq_status kvq_quantize_scatter_unscaled(const kvq_cache *cache, int32_t code_format,
                                         const void *k, int64_t k_token_stride,
                                         const void *v, int64_t v_token_stride,
                                         int64_t num_tokens, const int64_t *slot_ids,
                                         int32_t *err_flags, kvq_stream_t stream);

/* Workspace bytes kvq_paged_decode_codes needs (the rows-on-M split: one
 * 64-bit counter per (request, KV head, 128-row tile) plus two pieces of
 * partial results per SM); 0 for invalid arguments. */
size_t kvq_paged_decode_codes_workspace_size(int32_t num_requests, int32_t rows_per_request,
                                             int32_t num_q_heads, int32_t num_kv_heads,
                                             int32_t head_dim, int32_t block_size,
                                             int32_t max_context_len);

/* kvq_paged_decode over a cache whose codes are in `code_format`: scores use
 * e4m3(kc) or e5m2(kc) times the key scale, values e4m3(vc) or e5m2(vc) times
 * the value scale (1 for the unscaled caches).  Always the rows-on-M
 * tensor-core kernel (1 to 8192 stacked rows per KV head), so both formats run
 * the same code; it needs KV heads in groups of 4, pages of >= 16 tokens,
 * 16-byte aligned scale planes and fewer than 2^31 slots (else
 * KVQ_ERR_UNSUPPORTED).  Other arguments as for kvq_paged_decode with
 * partition_tokens 0; the workspace needs no initialisation. */
kvq_status kvq_paged_decode_codes(const kvq_cache *cache, int32_t code_format, const void *q,
                                  int32_t num_requests, int32_t rows_per_request,
                                  int32_t num_q_heads, const int32_t *block_tables,
                                  int32_t max_blocks_per_req, const int32_t *context_lens,
                                  int32_t max_context_len, float sm_scale, void *out,
                                  void *workspace, size_t workspace_bytes, int32_t *err_flags,
                                  kvq_stream_t stream);

/* Dequantise whole rows back to real values: out = fl32(e4m3(c) * scale), one
 * IEEE multiply, or that value rounded once more to bf16 (nearest-even).
 * sglang-jax #1776 "feat(dsa): implement fp8 KV cache (e4m3) with a bf16
 * indexer cache", Modifications: a consumer upcasts the cached block before it
 * is used.
 *   slot_ids    device int64 [n]; an id outside [0, num_slots) gives a zero row
 *               (ids >= num_slots also set KVQ_ERRF_SLOT_RANGE)
 *   out_dtype   0 = fp32, 1 = bf16
 *   out_k, out_v device [n, num_kv_heads, head_dim] of out_dtype; either may be
 *               NULL to skip that half
 *   err_flags   device int32, optional */
kvq_status kvq_dequant_rows(const kvq_cache *cache, const int64_t *slot_ids, int64_t n,
                            int32_t out_dtype, void *out_k, void *out_v,
                            int32_t *err_flags, kvq_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Compressed index keys.  ATOM PR #2655, PR description, index-key bullet:
 * index keys are cached either as FP8 with one FP32 scale per row -- the K/V
 * row format above -- or as MXFP4: two E2M1 codes per byte plus one E8M0
 * exponent per 32 dims, the exponent large enough that no element of the group
 * overflows; the FP4 codes are decoded by bit manipulation.  One row of `dim` values per token (one index head):
 *   FP8    codes uint8 [num_slots, dim] (e4m3) and scales fp32 [num_slots]:
 *          scale = amax / 448, code_d = e4m3_rne(x_d / scale), as for K/V.
 *   MXFP4  codes uint8 [num_slots, dim / 2]: element 2i in the low nibble of
 *          byte i, element 2i + 1 in the high nibble, each an E2M1 code (1 sign,
 *          2 exponent bits with bias 1, 1 mantissa bit; magnitudes 0, 0.5, 1,
 *          1.5, 2, 3, 4, 6); exponents uint8 [num_slots, dim / 32]: byte X + 127
 *          for the group scale 2^X, X the smallest integer with the group's
 *          amax <= 6 * 2^X, clamped to [-127, 127] (-127 for an all-zero
 *          group); code = the E2M1 value nearest x / 2^X, ties to the even
 *          mantissa bit, carrying the sign of x.
 * dim must be 128; alignment as for the K/V cache (codes 16 bytes, x rows 16
 * bytes with a token stride of a multiple of 8 elements, slot ids 8). */
#define KVQ_INDEX_FP8 0
#define KVQ_INDEX_MXFP4 1

typedef struct kvq_index_cache {
    uint8_t *codes;                      /* see above, per format                   */
    float *scales;                       /* FP8: [num_slots] fp32; MXFP4: unused    */
    uint8_t *exponents;                  /* MXFP4: [num_slots, dim/32]; FP8: unused */
    int64_t num_slots;
    int32_t format;                      /* KVQ_INDEX_FP8 or KVQ_INDEX_MXFP4        */
    int32_t dim;                         /* 128                                     */
} kvq_index_cache;

/* Bytes of an index-key cache: FP8 num_slots * (dim + 4); MXFP4 num_slots *
 * (dim / 2 + dim / 32).  0 for an invalid argument. */
size_t kvq_index_cache_bytes(int64_t num_slots, int32_t format, int32_t dim);

/* Quantise index-key rows and scatter them to slots (one launch, capturable).
 *   x               device bf16; token t's row starts at element t*x_token_stride
 *   x_token_stride  in elements, a multiple of 8, >= 0
 *   num_tokens      rows (0 launches nothing)
 *   slot_ids        device int64 [num_tokens]: as for kvq_quantize_scatter
 *   err_flags       device int32, optional */
kvq_status kvq_index_quantize_scatter(const kvq_index_cache *cache, const void *x,
                                      int64_t x_token_stride, int64_t num_tokens,
                                      const int64_t *slot_ids, int32_t *err_flags,
                                      kvq_stream_t stream);

/* Index-key rows back to real values: FP8 fl32(e4m3(c) * scale); MXFP4
 * fl32(e2m1(c) * 2^X); out_dtype 1 rounds that once more to bf16.
 *   slot_ids  device int64 [n]; an id outside [0, num_slots) gives a zero row
 *             (ids >= num_slots also set KVQ_ERRF_SLOT_RANGE)
 *   out       device [n, dim] of out_dtype (0 = fp32, 1 = bf16) */
kvq_status kvq_index_dequant_rows(const kvq_index_cache *cache, const int64_t *slot_ids,
                                  int64_t n, int32_t out_dtype, void *out,
                                  int32_t *err_flags, kvq_stream_t stream);

/* Stacked index scores over the compressed index keys (one launch, capturable).
 * ATOM PR #2655, PR description: the decode-time scorer there multiplies all
 * R query rows x H index heads of a request against each cached index key in
 * a single matrix product, so every key is loaded once per step; each head's
 * dot product is clipped at zero (ReLU) and the clipped values are added.  For request r, row i
 * and token t < L_r - R + 1 + i (row i sees the context up to and including
 * its own position, as in verify):
 *     out[r*R + i][t] = sum_h max(0, sum_d q[r][i][h][d] * khat_t[d]),
 * khat_t the dequantised key of token t (FP8: e4m3(c) * scale; MXFP4:
 * e2m1(c) * 2^X), read through the request's block table.  Every other entry
 * of the row, up to max_context_len, is -inf.
 *   cache            index keys, paged in blocks of block_size slots; its scale
 *                    (FP8) or exponent (MXFP4) plane 16-byte aligned
 *   block_size       tokens per block, a power of two >= 16
 *   q                device bf16 [num_requests, rows_per_request,
 *                    num_index_heads, dim], 16-byte aligned
 *   rows_per_request R >= 1;  num_index_heads H in {1, 2, 4, 8}; R * H <= 16
 *   block_tables     device int32 [num_requests, max_blocks_per_req]
 *   context_lens     device int32 [num_requests]: L_r, in [0, min(max_context_len,
 *                    max_blocks_per_req * block_size)]; outside that range it is
 *                    clamped and KVQ_ERRF_CONTEXT_RANGE set
 *   out              device fp32 [num_requests * R, max_context_len]
 *   err_flags        device int32, optional: KVQ_ERRF_BLOCK_RANGE for a block id
 *                    outside [0, num_slots / block_size) (the scores of that
 *                    block's tokens are then unspecified), KVQ_ERRF_CONTEXT_RANGE
 *                    as above, KVQ_ERRF_WAIT_TIMEOUT if a bounded in-kernel wait
 *                    for a copy gave up
 * Accuracy: the dots are f16 products accumulated in fp32 (both key formats
 * and the bf16 query, scaled by a power of two, are exact in f16 except for
 * parts below 2^-24 of a vector's largest element); each score is within
 * 1e-5 * sum_h sum_d |q_hd * khat_d| of the exact value. */
kvq_status kvq_index_scores(const kvq_index_cache *cache, int32_t block_size, const void *q,
                            int32_t num_requests, int32_t rows_per_request,
                            int32_t num_index_heads, const int32_t *block_tables,
                            int32_t max_blocks_per_req, const int32_t *context_lens,
                            int32_t max_context_len, float *out, int32_t *err_flags,
                            kvq_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_H */
