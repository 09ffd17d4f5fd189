// kvq_attention_stream.cu -- paged decode attention for up to 8 stacked query
// rows per KV head over a whole batch, load-balanced: a persistent grid that
// splits the batch's work into equal contiguous ranges, FP8 cache.
//
// Same method and per-chunk arithmetic as kvq_attention_skinny.cu (ROCm/ATOM
// PR #2655 "fix(qwen4-exp): register the QSA FP8 scale planes for KV offload",
// PR description, K/V bullet: per-token key scale on the score after the code
// dot, per-token value scale on the probability ahead of PV; transposed tiles S^T = K Q^T on FP8
// tensor cores with Q as two e4m3 pieces (exact for elements >= 2^-9 of the row's
// largest, off by <= 2^-17 of it below), O^T = V^T P^T on f16 tensor
// cores) and the page-major loads of kvq_attention_page.cu (one TMA box of 16
// slots x 4 KV heads per K and V chunk, 4-head scale boxes, a producer warp and
// a 3-deep ring), with the work split by tokens instead of fixed partitions:
//
//  * The batch's work is the sequence of 16-token chunks ordered (request r,
//    group g of 4 KV heads, chunk c): request r holds C_r = ceil(L_r / 16)
//    chunks per group, at global chunk index (H/4) * sum_{r' < r} C_r' +
//    g * C_r + c (plus a charge of a few positions per segment start).  The
//    (3 per SM) grid splits it into contiguous ranges whatever the context
//    lengths (no partition tails, no waves): weighted 135 : 128 : 121 over the
//    grid's three thirds by block index, the measured ratio of their streaming
//    rates when all three run together, or, for batches whose smallest
//    weighted range would cut a (request, group) into more than 16 pieces,
//    equal ranges of max(ceil(total / grid), ceil(C_max / 15)).
//  * A CTA walks its range segment by segment (a segment: its chunks of one
//    (request, head group)).  The producer warp stages the next segment's
//    block ids in shared memory and streams the chunks through the ring
//    without stopping at segment ends; each head warp stages the next
//    segment's query rows and context length by cp.async while the current
//    segment runs, turns them into query pieces at the switch, runs the
//    chunks and writes either the final row (a segment that is the whole
//    request) or its (max, denominator, output) to partial slot
//    b - first CTA of the (request, group).
//  * The CTA holding a segment's first chunk writes the segment's piece count
//    into the workspace (0 for a request with no cached token); the combine
//    kernel (one warp per output row) reads it with all of the row's slots
//    in one memory round trip.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>

#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {

namespace {

constexpr int kStHeads = 4;                          // KV heads per CTA = compute warps
constexpr int kStThreads = (kStHeads + 1) * 32;      // + the producer warp
constexpr int kChunk = 16;                           // tokens per stage
constexpr int kStStages = 3;
constexpr int kStRows = 8;                           // stacked query rows per KV head
constexpr int kStMaxPages = 520;                     // block ids of one segment
constexpr float kStLazyRescale = 8.0f;
// Range weights of the grid's three thirds (blockIdx / (grid / 3)): with three
// CTAs per SM, CTAs of the first third stream ~10 % faster than those of the
// last whatever work they hold (a per-CTA timer trace of the decode batch, also
// with the work order reversed), so equal ranges leave the last third ~4.5 us
// behind.
constexpr int64_t kStW0 = 135, kStW1 = 128, kStW2 = 121, kStWSum = kStW0 + kStW1 + kStW2;

// shared memory from a 1024-byte aligned base; a stage is
// [K: head][row][128 B] | [V: head][row][128 B] | K scales [row][head] | V scales
constexpr int kStCodeBytes = kStHeads * kChunk * kHeadDim;            // 8 KiB
constexpr int kStScBytes = kChunk * kStHeads * 4;                     // 256 B
constexpr int kStStageBytes = ((2 * kStCodeBytes + 2 * kStScBytes) + 1023) / 1024 * 1024;
constexpr int kOffStQ = kStStages * kStStageBytes;                    // [head][2][8][128]
constexpr int kOffStRowExp = kOffStQ + kStHeads * 2 * kStRows * kHeadDim;
// a decode step's new rows stored by this kernel: at most kStNewRows per request
constexpr int kStNewRows = kStreamNewRows;
constexpr int kOffStNew = kOffStRowExp + kStHeads * kStRows * 4;       // [head][row][K|V][256 B]
constexpr int kOffStSlot = kOffStNew + kStHeads * kStNewRows * 2 * 2 * kHeadDim;   // int64 [stage]
constexpr int kOffStLen = kOffStSlot + kStStages * 8;                  // [head][4] int32
constexpr int kOffStSplit = kOffStLen + kStHeads * 16;   // int64: x_begin, x_end, B, total
constexpr int kOffStPre = kOffStSplit + 32;                            // [N + 1] int32
constexpr int kOffStBt = kOffStPre + (kStreamMaxRequests + 1 + 3) / 4 * 16;
constexpr int kOffStBar = kOffStBt + 2 * kStMaxPages * 4;     // two segments' block ids
constexpr int kOffStAbort = kOffStBar + 2 * kStStages * 8;
constexpr int kStSmem = kOffStAbort + 16 + 1024;

struct StParams {
  uint32_t num_blocks;        // < 2^31 (slots < 2^31)
  int32_t H;
  int32_t log2_bs;
  const uint16_t *q;
  uint16_t *out;
  const int32_t *block_tables;
  int32_t max_blocks;
  const int32_t *context_lens;
  int32_t ctx_limit;
  int32_t N, R, Hq, G, M;
  float qk_scale;             // sm_scale * log2(e)
  int32_t cmax;               // ceil(max context / 16)
  float *o_part;              // [rows][kStreamSlots][128]
  float2 *ml_part;            // [rows][kStreamSlots]
  int32_t *pieces;            // [N][H / 4]: pieces of each (request, head group)
  int32_t *err_flags;
  // the step's new rows (k_new == nullptr: none; R <= kStNewRows): row
  // r * R + i of request r goes to position L_r - R + i, stored by the CTA
  // that streams its chunk
  const uint16_t *k_new;
  const uint16_t *v_new;
  int64_t k_stride, v_stride;  // token pitch, elements
  uint8_t *k_codes;
  uint8_t *v_codes;
  float *k_scales;
  float *v_scales;
};

__device__ __forceinline__ float st_ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Bounded wait that also gives up once another warp raised the abort flag.
__device__ __forceinline__ bool st_wait(uint32_t bar, uint32_t parity, volatile int *abort) {
  for (int i = 0; i < (1 << 19); ++i) {
    if (mbar_try_wait_sleep(bar, parity, 2000u)) return true;
    if ((i & 15) == 15 && *abort) return false;
  }
  *abort = 1;
  return false;
}

// In the work sequence a segment (request r, head group g) spans
// V_r = C_r + kStreamSwitchChunks positions: the charge for starting it, then
// its C_r chunks; pre[r] is the sum of V over the requests before r.  The
// CTA's part of the segment holding position x (x < x_end): request r (the
// largest with (H/4) pre[r] <= x, so V_r > 0), head group g, its first chunk
// c0 and chunk count n (0 when the range ends inside the charge), the
// segment's C, the position of its first chunk, and the position where the
// CTA's range continues.
struct Segment {
  int r, g, c0, n, C;
  int64_t base, next;
};

__device__ __forceinline__ Segment locate(const int32_t *pre, int N, int hg, int64_t x,
                                          int64_t x_end) {
  int lo = 0, hi = N - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (static_cast<int64_t>(hg) * pre[mid] <= x) lo = mid;
    else hi = mid - 1;
  }
  Segment s;
  s.r = lo;
  const int V = pre[lo + 1] - pre[lo];
  s.C = V - kStreamSwitchChunks;
  // positions stay below 2^31 (attn_stream_shape_ok), so 32-bit division
  const int64_t off = x - static_cast<int64_t>(hg) * pre[lo];
  s.g = static_cast<int>(static_cast<uint32_t>(off) / static_cast<uint32_t>(V));
  const int64_t start = static_cast<int64_t>(hg) * pre[lo] + static_cast<int64_t>(s.g) * V;
  s.base = start + kStreamSwitchChunks;
  const int64_t end = start + V < x_end ? start + V : x_end;
  const int64_t xs = x > s.base ? x : s.base;
  s.next = end;
  if (xs >= end) {
    s.c0 = 0;
    s.n = 0;
  } else {
    s.c0 = static_cast<int>(xs - s.base);
    s.n = static_cast<int>(end - xs);
  }
  return s;
}

// The split of the work sequence (total positions) over the grid: CTA b
// takes [start(b), start(b + 1)).  Weighted (B == 0): the grid's thirds get
// ranges in the ratio kStW0 : kStW1 : kStW2, every range at least b_min long;
// else equal ranges of B positions (CTAs past the end idle).  owner(x) is the
// CTA whose range holds position x.
struct StSplit {
  int64_t total;
  int64_t B;
  int64_t cls;                         // CTAs per third of the grid

  __host__ __device__ int64_t wpre(int64_t b) const {   // weights of CTAs < b
    const int64_t b0 = b < cls ? b : cls;
    const int64_t b1 = b < cls ? 0 : (b < 2 * cls ? b - cls : cls);
    const int64_t b2 = b < 2 * cls ? 0 : b - 2 * cls;
    return kStW0 * b0 + kStW1 * b1 + kStW2 * b2;
  }
  __host__ __device__ int64_t start(int64_t b) const {
    if (B > 0) return b * B < total ? b * B : total;
    return total * wpre(b) / (kStWSum * cls);
  }
  __host__ __device__ int64_t owner(int64_t x) const {   // 0 <= x < total
    if (B > 0) return x / B;
    // the largest b with start(b) <= x, i.e. wpre(b) <= y
    const int64_t y = ((x + 1) * kStWSum * cls - 1) / total;
    const int64_t w1 = kStW0 * cls, w2 = w1 + kStW1 * cls;
    const int64_t b = y < w1 ? y / kStW0 : (y < w2 ? cls + (y - w1) / kStW1 : 2 * cls + (y - w2) / kStW2);
    return b < 3 * cls - 1 ? b : 3 * cls - 1;
  }
};

// b_min: the shortest range that cuts no segment of <= cmax chunks into more
// than kStreamSlots pieces.
__host__ __device__ inline StSplit make_split(int64_t total, int64_t grid, int64_t cmax) {
  const int64_t b_min0 = (cmax + kStreamSlots - 2) / (kStreamSlots - 1);
  const int64_t b_min = b_min0 > 1 ? b_min0 : 1;
  StSplit sp;
  sp.total = total;
  sp.cls = grid / 3;
  sp.B = 0;
  // every weighted range is at least floor(total kStW2 / (kStWSum cls)) long
  if (grid % 3 != 0 || sp.cls == 0 || total * kStW2 / (kStWSum * sp.cls) < b_min) {
    const int64_t B = (total + grid - 1) / grid;
    sp.B = B > b_min ? B : b_min;
  }
  return sp;
}

// The step's new rows of one chunk, one warp for KV head h (tile w of the
// stage): each row quantised with the store's codec (one row per warp pass,
// 4 elements a lane), put into the stage's code tile (row tr of the 128-byte
// swizzled tile) and scale column, and stored to the cache at slot0 + tr
// (slot0 < 0: a page id out of range, nothing stored).  Rare (a chunk per
// segment end): rolled loops keep the chunk loop free of spills.
__device__ __forceinline__ void patch_new_rows(const StParams &p, uint8_t *stage, int w, int h,
                                            int lane, int L, int j0, const uint8_t *newb,
                                            int64_t slot0) {
  uint8_t *kbm = stage + w * kChunk * kHeadDim;
  uint8_t *vbm = kbm + kStCodeBytes;
  float *ksm = reinterpret_cast<float *>(stage + 2 * kStCodeBytes) + w;
  float *vsm = ksm + kStScBytes / 4;
#pragma unroll 1
  for (int i = 0; i < p.R; ++i) {
    const int pos = L - p.R + i;
    if (pos < j0 || pos >= j0 + kChunk) continue;
    const int tr = pos - j0;
#pragma unroll 1
    for (int kv = 0; kv < 2; ++kv) {
      const uint2 v = *reinterpret_cast<const uint2 *>(newb + (2 * i + kv) * 2 * kHeadDim + 8 * lane);
      uint32_t mg = __vmaxu2(v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) mg = __vmaxu2(mg, __shfl_xor_sync(0xFFFFFFFFu, mg, off));
      const float amax = __uint_as_float(max(mg & 0xFFFFu, mg >> 16) << 16);
      uint32_t word = 0u;
      float sc = 0.0f;
      if (amax != 0.0f) {
        sc = row_scale(amax);
        word = (sc >= kMarksteinMinScale) ? encode4<true>(v.x, v.y, sc, __frcp_rn(sc))
                                          : encode4<false>(v.x, v.y, sc, 0.0f);
      }
      *reinterpret_cast<uint32_t *>((kv ? vbm : kbm) + tr * kHeadDim +
                                    (((lane >> 2) ^ (tr & 7)) << 4) + 4 * (lane & 3)) = word;
      if (lane == 0) (kv ? vsm : ksm)[4 * tr] = sc;
      if (slot0 >= 0) {
        const int64_t row = (slot0 + tr) * p.H + h;
        *reinterpret_cast<uint32_t *>((kv ? p.v_codes : p.k_codes) + row * kHeadDim + 4 * lane) = word;
        if (lane == 0) (kv ? p.v_scales : p.k_scales)[row] = sc;
      }
    }
  }
}

__global__ void __launch_bounds__(kStThreads, 3)
attn_stream_kernel(const StParams p, const __grid_constant__ CUtensorMap tmap_k,
                   const __grid_constant__ CUtensorMap tmap_v,
                   const __grid_constant__ CUtensorMap tmap_ks,
                   const __grid_constant__ CUtensorMap tmap_vs) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int g8 = lane >> 2;            // fragment row group
  const int c4 = lane & 3;             // fragment thread in group

  int32_t *pre = reinterpret_cast<int32_t *>(smem + kOffStPre);
  int32_t *bt_s = reinterpret_cast<int32_t *>(smem + kOffStBt);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + kOffStBar);
  uint64_t *empty = full + kStStages;
  volatile int *abort_s = reinterpret_cast<volatile int *>(smem + kOffStAbort);
  float *row_exp = reinterpret_cast<float *>(smem + kOffStRowExp);

  // The launch overlaps the previous kernel's drain; every global access
  // (context lengths, block tables, queries, the cache, the workspace, the
  // outputs) comes after the wait, so whatever a previous kernel wrote is
  // visible and whatever it still reads is not overwritten.
  allow_dependents_launch();
  grid_dependency_wait();
  const int N = p.N;
  if (warp == 0) {
    // positions per request (its chunks plus the segment charge) and their
    // prefix: pre[r] is the sum of V over the requests before r
    int carry = 0;
    for (int r0 = 0; r0 < N; r0 += 32) {
      const int r = r0 + lane;
      int L = (r < N) ? p.context_lens[r] : 0;
      if (L < 0 || L > p.ctx_limit) {
        if (blockIdx.x == 0 && p.err_flags) atomicOr(p.err_flags, KVQ_ERRF_CONTEXT_RANGE);
        L = L < 0 ? 0 : p.ctx_limit;
      }
      const int c = (L + kChunk - 1) / kChunk;
      int v = (c > 0) ? c + kStreamSwitchChunks : 0;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int t = __shfl_up_sync(0xFFFFFFFFu, v, off);
        if (lane >= off) v += t;
      }
      if (r < N) pre[r + 1] = carry + v;
      carry += __shfl_sync(0xFFFFFFFFu, v, 31);
    }
    if (lane == 0) {
      pre[0] = 0;
      // the split and this CTA's range, once (64-bit divisions by every
      // thread of the SM's three CTAs would hold up the range's first copy)
      const StSplit sp = make_split(static_cast<int64_t>(p.H / kStHeads) * carry, gridDim.x, p.cmax);
      int64_t *sx = reinterpret_cast<int64_t *>(smem + kOffStSplit);
      sx[0] = sp.start(blockIdx.x);
      sx[1] = sp.start(blockIdx.x + 1);
      sx[2] = sp.B;
      sx[3] = sp.total;
    }
  }
  if (tid == 0) {
    for (int s = 0; s < kStStages; ++s) {
      mbar_init(smem_addr(&full[s]), 1);
      mbar_init(smem_addr(&empty[s]), kStHeads);
    }
    *abort_s = 0;
    fence_mbarrier_init();
    fence_proxy_async_smem();
  }
  __syncthreads();
  const int hg = p.H / kStHeads;
  const int64_t *sx = reinterpret_cast<const int64_t *>(smem + kOffStSplit);
  const int64_t x_begin = sx[0];
  const int64_t x_end = sx[1];
  // requests with no cached token: no pieces (the combine writes zero rows)
  for (int r = blockIdx.x; r < N; r += gridDim.x)
    if (pre[r + 1] == pre[r])
      for (int g = tid; g < hg; g += kStThreads) p.pieces[static_cast<int64_t>(r) * hg + g] = 0;
  if (x_begin >= x_end) return;

  if (warp == kStHeads) {
    // ---------------------------------------------------------- producer
    uint32_t u = 0;                    // chunks issued (lane 0's count)
    bool bad = false, stop = false;
    // a segment's block ids into one of two shared-memory buffers (all lanes,
    // cp.async): the first segment's up front, each next one's while the
    // current segment is issued, so a segment change costs no memory round
    // trip in the issue loop
    auto stage_ids = [&](const Segment &sg, int buf) {
      const int p0 = (kChunk * sg.c0) >> p.log2_bs;
      const int np = ((kChunk * (sg.c0 + sg.n) - 1) >> p.log2_bs) - p0 + 1;
      const int32_t *bt = p.block_tables + static_cast<int64_t>(sg.r) * p.max_blocks + p0;
      for (int i = lane; i < np && i < kStMaxPages; i += 32)
        cp_async_4(bt_s + buf * kStMaxPages + i, bt + i, 4u);
      cp_async_commit();
    };
    Segment sg = locate(pre, N, hg, x_begin, x_end);
    if (sg.n > 0) stage_ids(sg, 0);
    int buf = 0;
    while (sg.n > 0 && !stop) {
      cp_async_wait<0>();              // this segment's ids (issued a segment ago)
      __syncwarp();
      Segment nx;
      nx.n = 0;
      if (sg.next < x_end) {
        nx = locate(pre, N, hg, sg.next, x_end);
        if (nx.n > 0) stage_ids(nx, buf ^ 1);
      }
      const int32_t *ids = bt_s + buf * kStMaxPages;
      const int p0 = (kChunk * sg.c0) >> p.log2_bs;
      if (lane == 0) {
        for (int k = 0; k < sg.n; ++k, ++u) {
          const int st = u % kStStages;
          if (u >= kStStages &&
              !st_wait(smem_addr(&empty[st]), ((u / kStStages) - 1) & 1, abort_s)) {
            stop = true;
            break;
          }
          uint8_t *sb = smem + st * kStStageBytes;
          const uint32_t fb = smem_addr(&full[st]);
          const int j = kChunk * (sg.c0 + k);        // chunks lie within a page (bs >= 16)
          const int pi = (j >> p.log2_bs) - p0;
          const uint32_t blk = (pi < kStMaxPages) ? static_cast<uint32_t>(ids[pi]) : 0xFFFFFFFFu;
          uint32_t bytes = 0;
          int64_t *stage_slot = reinterpret_cast<int64_t *>(smem + kOffStSlot);
          stage_slot[st] = -1;                       // read after the stage's full barrier
          if (blk >= p.num_blocks) {                 // also every negative id
            bad = true;
          } else {
            const int z = static_cast<int>((blk << p.log2_bs) | (j & ((1 << p.log2_bs) - 1)));
            stage_slot[st] = z;
            const int h0 = kStHeads * sg.g;
            tma_load_3d(smem_addr(sb), &tmap_k, 0, z, h0, fb);
            tma_load_3d(smem_addr(sb + kStCodeBytes), &tmap_v, 0, z, h0, fb);
            tma_load_2d(smem_addr(sb + 2 * kStCodeBytes), &tmap_ks, h0, z, fb);
            tma_load_2d(smem_addr(sb + 2 * kStCodeBytes + kStScBytes), &tmap_vs, h0, z, fb);
            bytes = 2u * kStCodeBytes + 2u * kStScBytes;
          }
          mbar_arrive_expect_tx(fb, bytes);
        }
      }
      stop = __shfl_sync(0xFFFFFFFFu, stop ? 1 : 0, 0) != 0;
      sg = nx;
      buf ^= 1;
    }
    if (lane == 0) {
      if (bad && p.err_flags) atomicOr(p.err_flags, KVQ_ERRF_BLOCK_RANGE);
      // copies still in flight (after an abort) land before the CTA leaves
      for (uint32_t v = (u > kStStages ? u - kStStages : 0); v < u; ++v)
        mbar_wait_sleep_bounded(smem_addr(&full[v % kStStages]), (v / kStStages) & 1);
    }
    return;
  }

  // ------------------------------------------------------------ head warps
  const int w = warp;
  // [2][8][128]: the query pieces; while they sit in registers, the next
  // segment's raw query rows [8][256 B] land here
  uint8_t *plane = smem + kOffStQ + w * 2 * kStRows * kHeadDim;
  float *rexp = row_exp + w * kStRows;
  int32_t *len_s = reinterpret_cast<int32_t *>(smem + kOffStLen) + 4 * w;
  // the step's new rows of this warp's head, [row][K|V][256 B] bf16
  uint8_t *newb = smem + kOffStNew + w * kStNewRows * 2 * 2 * kHeadDim;
  const int64_t *stage_slot = reinterpret_cast<const int64_t *>(smem + kOffStSlot);
  // a segment's query rows of this warp's head (16-byte cp.async, row m at
  // m * 256) and its request's context length into shared memory
  auto stage_q = [&](const Segment &sg) {
    const int h = kStHeads * sg.g + w;
    for (int c = lane; c < p.M * 16; c += 32) {
      const int m = c >> 4, i = m / p.G, gq = m - i * p.G;
      const uint16_t *src =
          p.q + ((static_cast<int64_t>(sg.r) * p.R + i) * p.Hq + h * p.G + gq) * kHeadDim + 8 * (c & 15);
      cp_async_16(plane + m * 2 * kHeadDim + 16 * (c & 15), src, 16u);
    }
    if (lane == 0) cp_async_4(len_s, p.context_lens + sg.r, 4u);
    cp_async_commit();
  };
  // the step's new rows of a segment whose part in this range reaches its
  // last two chunks (the rows' positions L - R .. L - 1 lie there)
  auto stage_new = [&](const Segment &sg) {
    if (p.k_new == nullptr || sg.c0 + sg.n + 1 < sg.C) return;
    const int h = kStHeads * sg.g + w;
    for (int c = lane; c < p.R * 2 * 16; c += 32) {
      const int i = c >> 5, kv = (c >> 4) & 1, piece = c & 15;
      const int64_t t = static_cast<int64_t>(sg.r) * p.R + i;
      const uint16_t *src = (kv ? p.v_new + t * p.v_stride : p.k_new + t * p.k_stride) +
                            h * kHeadDim + 8 * piece;
      cp_async_16(newb + (2 * i + kv) * 2 * kHeadDim + 16 * piece, src, 16u);
    }
    cp_async_commit();
  };
  Segment sg = locate(pre, N, hg, x_begin, x_end);
  if (sg.n > 0) stage_q(sg);
  // this lane's ldmatrix row address within a head's K tile, per k-step
  const int ld_row = (lane & 7) + 8 * ((lane >> 3) & 1);
  uint32_t ld_off[4];
#pragma unroll
  for (int s2 = 0; s2 < 4; ++s2)
    ld_off[s2] = ld_row * kHeadDim + (((2 * s2 + (lane >> 4)) ^ (lane & 7)) << 4);
  uint32_t u = 0;                      // chunks consumed
  bool timed_out = false;
  bool first_seg = true;
  while (sg.n > 0 && !timed_out) {
    const int r = sg.r;
    const int h = kStHeads * sg.g + w;
    cp_async_wait<0>();                // this segment's rows (staged a segment ago)
    __syncwarp();
    int L = *len_s;
    L = L < 0 ? 0 : (L > p.ctx_limit ? p.ctx_limit : L);
    // exponents and the two e4m3 pieces of each element, q = 2^e (p1 + p2);
    // rows past M get zero pieces
    {
      uint2 vq[kStRows];
#pragma unroll
      for (int m = 0; m < kStRows; ++m)
        vq[m] = (m < p.M) ? *reinterpret_cast<const uint2 *>(plane + m * 2 * kHeadDim + 8 * lane)
                          : make_uint2(0u, 0u);
      __syncwarp();                    // every lane holds its rows before the pieces overwrite them
#pragma unroll
      for (int m = 0; m < kStRows; ++m) {
        uint32_t c1w = 0u, c2w = 0u;
        float rx = 0.0f;
        if (m < p.M) {
          const uint2 v = vq[m];
          float amax = fmaxf(fmaxf(fabsf(bf16_lo(v.x)), fabsf(bf16_hi(v.x))),
                             fmaxf(fabsf(bf16_lo(v.y)), fabsf(bf16_hi(v.y))));
#pragma unroll
          for (int off = 16; off > 0; off >>= 1)
            amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, off));
          const int ex = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFFu);
          int e = (ex == 0) ? -126 : ex - 127 - 7;
          e = e < -126 ? -126 : (e > 126 ? 126 : e);
          rx = (amax == 0.0f) ? 0.0f : __int_as_float((127 + e) << 23);   // 2^e
          if (rx != 0.0f) {
            const float inv = __int_as_float((254u << 23) - __float_as_uint(rx));
            const float xs[4] = {bf16_lo(v.x) * inv, bf16_hi(v.x) * inv, bf16_lo(v.y) * inv,
                                 bf16_hi(v.y) * inv};
            e4m3_pieces4(xs, c1w, c2w);
          }
        }
        if (lane == 0) rexp[m] = rx;
        *reinterpret_cast<uint32_t *>(plane + m * kHeadDim + 4 * lane) = c1w;
        *reinterpret_cast<uint32_t *>(plane + kStRows * kHeadDim + m * kHeadDim + 4 * lane) = c2w;
      }
      __syncwarp();
    }
    // B fragments for k-step s2: b0 = dims 32 s2 + 4c + 0..3, b1 = + 16, row g
    uint32_t qb[4][2][2];
#pragma unroll
    for (int s2 = 0; s2 < 4; ++s2)
#pragma unroll
      for (int pc = 0; pc < 2; ++pc) {
        const uint8_t *qr = plane + pc * kStRows * kHeadDim + g8 * kHeadDim + 32 * s2 + 4 * c4;
        qb[s2][pc][0] = *reinterpret_cast<const uint32_t *>(qr);
        qb[s2][pc][1] = *reinterpret_cast<const uint32_t *>(qr + 16);
      }
    // the next segment's rows land in the planes while this one runs
    if (sg.next < x_end) {
      const Segment nx = locate(pre, N, hg, sg.next, x_end);
      if (nx.n > 0) {
        __syncwarp();                  // every lane has read its pieces
        stage_q(nx);
      }
    }
    stage_new(sg);
    // this thread's rows: n = 2c + e
    int vis[2];
    float rowf[2], m_run[2], l_run[2], thr[2], ms[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int n = 2 * c4 + e;
      vis[e] = (n < p.M) ? (L - p.R + 1 + n / p.G) : 0;
      rowf[e] = (n < p.M) ? rexp[n] * p.qk_scale : 0.0f;
      m_run[e] = -INFINITY;
      l_run[e] = 0.0f;
      thr[e] = -INFINITY;
      ms[e] = 0.0f;
    }
    float o[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int e = 0; e < 4; ++e) o[i][e] = 0.0f;
    int ev = -1000;
    float vbound = -1.0f, vnorm = 1.0f;

    for (int k = 0; k < sg.n; ++k, ++u) {
      const int st = u % kStStages;
      if (!st_wait(smem_addr(&full[st]), (u / kStStages) & 1, abort_s)) {
        timed_out = true;
        break;
      }
      const uint8_t *sbase = smem + st * kStStageBytes;
      const uint8_t *kb = sbase + w * kChunk * kHeadDim;
      const uint8_t *vb = sbase + kStCodeBytes + w * kChunk * kHeadDim;
      const float *ksv = reinterpret_cast<const float *>(sbase + 2 * kStCodeBytes) + w;
      const float *vsv = reinterpret_cast<const float *>(sbase + 2 * kStCodeBytes + kStScBytes) + w;
      const int j0 = kChunk * (sg.c0 + k);
      if (p.k_new != nullptr && j0 + kChunk > L - p.R) {
        // the step's new rows in this chunk (the copy brought whatever the
        // slots held)
        cp_async_wait<0>();
        __syncwarp();
        patch_new_rows(p, smem + st * kStStageBytes, w, h, lane, L, j0, newb, stage_slot[st]);
        fence_proxy_async_smem();      // before a later copy refills the stage
        __syncwarp();
      }

      // ---- S^T = K Q^T (K fragments by ldmatrix), two accumulation chains
      float sacc[4] = {0.f, 0.f, 0.f, 0.f}, sacc2[4] = {0.f, 0.f, 0.f, 0.f};
      {
        const uint32_t kbase = smem_addr(kb);
#pragma unroll
        for (int s2 = 0; s2 < 4; ++s2) {
          uint32_t a[4];
          ldsm_x4(kbase + ld_off[s2], a);
          mma_e4m3_16832(sacc, a, qb[s2][0][0], qb[s2][0][1]);
          mma_e4m3_16832(sacc2, a, qb[s2][1][0], qb[s2][1][1]);
        }
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) sacc[e] += sacc2[e];

      // ---- scale, mask.  sacc: [tok g][row 2c], [g][2c+1], [g+8][2c], [g+8][2c+1]
      const float ks_lo = ksv[4 * g8], ks_hi = ksv[4 * (g8 + 8)];
      float vs_lo = vsv[4 * g8], vs_hi = vsv[4 * (g8 + 8)];
      float xs[4];
      xs[0] = sacc[0] * ks_lo * rowf[0];
      xs[1] = sacc[1] * ks_lo * rowf[1];
      xs[2] = sacc[2] * ks_hi * rowf[0];
      xs[3] = sacc[3] * ks_hi * rowf[1];
      if (j0 + kChunk > min(vis[0], vis[1])) {      // some token of the chunk is masked
        xs[0] = (j0 + g8 < vis[0]) ? xs[0] : -INFINITY;
        xs[1] = (j0 + g8 < vis[1]) ? xs[1] : -INFINITY;
        xs[2] = (j0 + g8 + 8 < vis[0]) ? xs[2] : -INFINITY;
        xs[3] = (j0 + g8 + 8 < vis[1]) ? xs[3] : -INFINITY;
        // slots past the context end hold whatever they held
        vs_lo = (j0 + g8 < L) ? vs_lo : 0.0f;
        vs_hi = (j0 + g8 + 8 < L) ? vs_hi : 0.0f;
      }
      // ---- online softmax, lazily: the warp reductions and the rescale run
      // only when a lane's score passes its row's threshold or a value scale
      // passes the bound 2^ev (the same updates as reducing every chunk)
      const bool need = xs[0] > thr[0] || xs[2] > thr[0] || xs[1] > thr[1] || xs[3] > thr[1] ||
                        vs_lo > vbound || vs_hi > vbound;
      if (__any_sync(0xFFFFFFFFu, need)) {
        float mx0 = fmaxf(xs[0], xs[2]), mx1 = fmaxf(xs[1], xs[3]);
        float vmax = fmaxf(vs_lo, vs_hi);
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          mx0 = fmaxf(mx0, __shfl_xor_sync(0xFFFFFFFFu, mx0, off));
          mx1 = fmaxf(mx1, __shfl_xor_sync(0xFFFFFFFFu, mx1, off));
          vmax = fmaxf(vmax, __shfl_xor_sync(0xFFFFFFFFu, vmax, off));
        }
        float fac[2] = {1.0f, 1.0f};
        bool grow = false;
        {
          const float mxs[2] = {mx0, mx1};
#pragma unroll
          for (int e = 0; e < 2; ++e)
            if (mxs[e] > m_run[e] + kStLazyRescale) {
              fac[e] = st_ex2(m_run[e] - mxs[e]);
              m_run[e] = mxs[e];
              grow = true;
            }
        }
        float vfac = 1.0f;
        bool vgrow = false;
        {
          const uint32_t bits = __float_as_uint(vmax);
          const int ex = static_cast<int>((bits >> 23) & 0xFFu);
          int ec = (ex == 0) ? -126 : ex - 127 + ((bits & 0x7FFFFFu) != 0u ? 1 : 0);
          ec = ec > 126 ? 126 : ec;
          if (ec > ev) {
            const int d = ev - ec;
            vfac = (d >= -126) ? __int_as_float((127 + d) << 23) : 0.0f;
            ev = ec;
            vgrow = true;
          }
        }
        if (__any_sync(0xFFFFFFFFu, grow) || vgrow) {
          l_run[0] *= fac[0];
          l_run[1] *= fac[1];
          const float f0 = fac[0] * vfac, f1 = fac[1] * vfac;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            o[i][0] *= f0;
            o[i][1] *= f1;
            o[i][2] *= f0;
            o[i][3] *= f1;
          }
        }
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          thr[e] = m_run[e] + kStLazyRescale;
          ms[e] = (m_run[e] == -INFINITY) ? 0.0f : m_run[e];
        }
        vbound = __int_as_float((127 + ev) << 23);      // 2^ev, ev in [-126, 126]
        vnorm = __int_as_float((127 - ev) << 23);
      }
      const float p0 = st_ex2(xs[0] - ms[0]), p1 = st_ex2(xs[1] - ms[1]);
      const float p2 = st_ex2(xs[2] - ms[0]), p3 = st_ex2(xs[3] - ms[1]);
      l_run[0] += p0 + p2;
      l_run[1] += p1 + p3;
      const float wl = vs_lo * vnorm, wh = vs_hi * vnorm;
      // row 2c: (tok g, tok g+8); row 2c+1: (tok g, tok g+8)
      const uint32_t X = pack_f16x2(p0 * wl, p2 * wh);
      const uint32_t Y = pack_f16x2(p1 * wl, p3 * wh);
      // B = P^T: this lane (column = row g) needs tokens 2c, 2c+1 (b0) and
      // 2c+8, 2c+9 (b1) of row g, held by lanes 4*(2c) + g/2 and 4*(2c+1) + g/2
      const int la = 8 * c4 + (g8 >> 1), lb = la + 4;
      const uint32_t xa = __shfl_sync(0xFFFFFFFFu, X, la), ya = __shfl_sync(0xFFFFFFFFu, Y, la);
      const uint32_t xb = __shfl_sync(0xFFFFFFFFu, X, lb), yb = __shfl_sync(0xFFFFFFFFu, Y, lb);
      const uint32_t va = (g8 & 1) ? ya : xa;      // (tok 2c,   tok 2c+8)
      const uint32_t vc = (g8 & 1) ? yb : xb;      // (tok 2c+1, tok 2c+9)
      const uint32_t pb0 = prmt(va, vc, 0x5410u);
      const uint32_t pb1 = prmt(va, vc, 0x7632u);

      // ---- O^T += V^T P^T.  m-tile i, row g -> dim 16g + 2i, row g+8 -> 16g +
      // 2i + 1; this lane reads dims 16g..16g+15 of tokens 2c, 2c+1, 2c+8, 2c+9
      uint32_t wa[4], wb[4], wc[4], wd[4];
      {
        const int ta = 2 * c4, tb = ta + 1, tc = ta + 8, td = ta + 9;
        const uint4 A = *reinterpret_cast<const uint4 *>(vb + ta * kHeadDim + ((g8 ^ (ta & 7)) << 4));
        const uint4 Bv = *reinterpret_cast<const uint4 *>(vb + tb * kHeadDim + ((g8 ^ (tb & 7)) << 4));
        const uint4 C = *reinterpret_cast<const uint4 *>(vb + tc * kHeadDim + ((g8 ^ (tc & 7)) << 4));
        const uint4 Dv = *reinterpret_cast<const uint4 *>(vb + td * kHeadDim + ((g8 ^ (td & 7)) << 4));
        wa[0] = A.x; wa[1] = A.y; wa[2] = A.z; wa[3] = A.w;
        wb[0] = Bv.x; wb[1] = Bv.y; wb[2] = Bv.z; wb[3] = Bv.w;
        wc[0] = C.x; wc[1] = C.y; wc[2] = C.z; wc[3] = C.w;
        wd[0] = Dv.x; wd[1] = Dv.y; wd[2] = Dv.z; wd[3] = Dv.w;
        // tokens at or past the context end hold whatever the slot held (a
        // NaN code would poison the PV product even times p = 0)
        const int lim = L - j0;
        if (lim < kChunk) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            wa[e] = (ta < lim) ? wa[e] : 0u;
            wb[e] = (tb < lim) ? wb[e] : 0u;
            wc[e] = (tc < lim) ? wc[e] : 0u;
            wd[e] = (td < lim) ? wd[e] : 0u;
          }
        }
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t sel = (i & 1) ? 0x7362u : 0x5140u;
        const uint32_t xab = prmt(wa[i >> 1], wb[i >> 1], sel);
        const uint32_t xcd = prmt(wc[i >> 1], wd[i >> 1], sel);
        const uint32_t a[4] = {e4m3x2_to_f16x2(xab), e4m3x2_to_f16x2(xab >> 16),
                               e4m3x2_to_f16x2(xcd), e4m3x2_to_f16x2(xcd >> 16)};
        mma_f16_16816(o[i], a, pb0, pb1);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&empty[st]));

    }
    timed_out = __any_sync(0xFFFFFFFFu, timed_out);
    if (timed_out) {
      cp_async_wait<0>();              // the next segment's rows land before the CTA leaves
      break;
    }

    // ---- the segment's (max, denominator, O) for this head's rows
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      float l = l_run[e];
      l += __shfl_xor_sync(0xFFFFFFFFu, l, 4);
      l += __shfl_xor_sync(0xFFFFFFFFu, l, 8);
      l += __shfl_xor_sync(0xFFFFFFFFu, l, 16);
      l_run[e] = l;
    }
    const float vsc = (ev == -1000) ? 0.0f : __int_as_float((127 + ev) << 23);   // undo 2^-ev
    const bool direct = (sg.c0 == 0 && sg.n == sg.C);
    // the piece slot of a cut segment: the CTA's index among those holding it
    // (0 for every segment after the range's first, which starts inside it)
    int slot = 0;
    if (first_seg && !direct) {
      StSplit sp;
      sp.B = sx[2];
      sp.total = sx[3];
      sp.cls = gridDim.x / 3;
      slot = static_cast<int>(blockIdx.x - sp.owner(sg.base));
    }
    if (sg.c0 == 0 && w == 0 && lane == 0) {
      // this CTA holds the segment's first chunk: its piece count
      int n_pieces = 1;
      if (!direct) {
        StSplit sp;
        sp.B = sx[2];
        sp.total = sx[3];
        sp.cls = gridDim.x / 3;
        n_pieces = static_cast<int>(sp.owner(sg.base + sg.C - 1) - blockIdx.x) + 1;
      }
      p.pieces[static_cast<int64_t>(r) * hg + sg.g] = n_pieces;
    }
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int n = 2 * c4 + e;
      if (n >= p.M) continue;
      const int i = n / p.G, gq = n - i * p.G;
      const int64_t orow = (static_cast<int64_t>(r) * p.R + i) * p.Hq + h * p.G + gq;
      if (direct) {
        const float inv = (l_run[e] > 0.0f) ? vsc / l_run[e] : 0.0f;
        uint32_t pk[8];
#pragma unroll
        for (int t = 0; t < 8; ++t) pk[t] = pack_bf16x2(o[t][e] * inv, o[t][2 + e] * inv);
        uint4 *dst = reinterpret_cast<uint4 *>(p.out + orow * kHeadDim + 16 * g8);
        dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
      } else {
        const int64_t sl = orow * kStreamSlots + slot;
        float4 *dst = reinterpret_cast<float4 *>(p.o_part + sl * kHeadDim + 16 * g8);
#pragma unroll
        for (int t = 0; t < 4; ++t)
          dst[t] = make_float4(o[2 * t][e] * vsc, o[2 * t][2 + e] * vsc, o[2 * t + 1][e] * vsc,
                               o[2 * t + 1][2 + e] * vsc);
        if (g8 == 0) p.ml_part[sl] = make_float2(m_run[e], l_run[e]);
      }
    }
    first_seg = false;
    if (sg.next < x_end) {
      sg = locate(pre, N, hg, sg.next, x_end);
    } else {
      sg.n = 0;
    }
  }
  cp_async_wait<0>();                  // new rows staged for a chunk past the range's end
  if (timed_out && lane == 0 && p.err_flags) atomicOr(p.err_flags, KVQ_ERRF_WAIT_TIMEOUT);
}

// ---------------------------------------------------------------------------
// Combine for the stream layout: one warp per output row and one row per CTA
// (CTAs of one warp fit into whatever the decode kernel's CTAs free as they
// finish: 1, 2, 4, 8 and 16 rows per CTA measured 60.8, 61.0, 61.1, 61.0 and
// 61.2 us per decode step).
struct StCombineParams {
  int32_t R, Hq, G, H;
  int64_t rows_total;
  const int32_t *pieces;
  const float *o_part;
  const float2 *ml_part;
  uint16_t *out;
};

constexpr int kStCombineRows = 1;

__global__ void __launch_bounds__(kStCombineRows * 32)
attn_combine_stream_kernel(const StCombineParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kStCombineRows + (threadIdx.x >> 5);
  allow_dependents_launch();
  if (row >= p.rows_total) return;
  grid_dependency_wait();              // the piece counts and the partials (any global read)
  const int r = static_cast<int>(row / (static_cast<int64_t>(p.R) * p.Hq));
  const int qh = static_cast<int>(row % p.Hq);
  const int g = (qh / p.G) / kStHeads;
  // one memory round trip: the row's piece count and all of its slots,
  // whether or not the pieces exist (a slot past the count holds whatever
  // an earlier call left and is not used)
  const int n = p.pieces[static_cast<int64_t>(r) * (p.H / kStHeads) + g];
  const float2 *ml = p.ml_part + row * kStreamSlots;
  const float4 *op = reinterpret_cast<const float4 *>(p.o_part + row * kStreamSlots * kHeadDim) +
                     lane;
  float2 v[kStreamSlots];
  float4 o[kStreamSlots];
#pragma unroll
  for (int k = 0; k < kStreamSlots; ++k) {
    v[k] = ml[k];
    o[k] = op[k * (kHeadDim / 4)];
  }
  if (n == 1) return;                  // written by the partials kernel
  // n == 0: a request with no cached token gets a zero row
  float m_w = -INFINITY, lsum = 0.0f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int k = 0; k < kStreamSlots; ++k) {
    // no piece, or a piece that saw no visible token
    if (k >= n || v[k].x == -INFINITY) continue;
    const float mn = fmaxf(m_w, v[k].x);
    const float a = st_ex2(m_w - mn), b = st_ex2(v[k].x - mn);
    lsum = lsum * a + v[k].y * b;
    acc.x = acc.x * a + o[k].x * b;
    acc.y = acc.y * a + o[k].y * b;
    acc.z = acc.z * a + o[k].z * b;
    acc.w = acc.w * a + o[k].w * b;
    m_w = mn;
  }
  const float inv = (lsum > 0.0f) ? 1.0f / lsum : 0.0f;
  const uint2 packed = make_uint2(pack_bf16x2(acc.x * inv, acc.y * inv),
                                  pack_bf16x2(acc.z * inv, acc.w * inv));
  *reinterpret_cast<uint2 *>(p.out + row * kHeadDim + 4 * lane) = packed;
}

}  // namespace

size_t attn_stream_pieces_bytes(int32_t num_requests, int32_t num_kv_heads) {
  return (static_cast<size_t>(num_requests) * (num_kv_heads / kStHeads) * 4 + 255) / 256 * 256;
}

bool attn_stream_shape_ok(int32_t num_kv_heads, const AttnShape &s) {
  const int bs = 1 << s.log2_block;
  const int64_t sms = s.sms > 0 ? s.sms : 152;
  const int64_t cmax = (static_cast<int64_t>(s.max_context_len) + kChunk - 1) / kChunk;
  const int64_t hg = num_kv_heads / kStHeads;
  // chunks per CTA stay within the block-id window of one segment, whichever
  // split the kernel takes for the batch's actual lengths (at most total_ub
  // positions): equal ranges of max(ceil(total / grid), b_min), or weighted
  // ranges of at most ceil(total kStW0 / (kStWSum grid / 3)) + 1
  const int64_t total_ub = s.num_requests * hg * (cmax + kStreamSwitchChunks);
  const int64_t grid = 3 * sms;
  const int64_t per_cta = (total_ub + grid - 1) / grid;
  const int64_t per_cta_w = (total_ub * kStW0 + kStWSum * sms - 1) / (kStWSum * sms) + 1;
  const int64_t b_min = (cmax + kStreamSlots - 2) / (kStreamSlots - 1);
  int64_t b = per_cta > b_min ? per_cta : b_min;
  b = b > per_cta_w ? b : per_cta_w;
  return s.rows <= kStRows && bs >= kChunk && num_kv_heads % kStHeads == 0 &&
         s.num_requests >= 1 && s.num_requests <= kStreamMaxRequests &&
         total_ub < (int64_t(1) << 31) && b * kChunk / bs + 2 <= kStMaxPages;
}

cudaError_t launch_attn_partials_stream(const kvq_cache &c, const AttnShape &s, const void *q,
                                        const int32_t *block_tables,
                                        const int32_t *context_lens, float sm_scale, void *out,
                                        void *workspace, int32_t *err_flags,
                                        cudaStream_t stream, const AppendRows *append) {
  const int64_t rows_total =
      static_cast<int64_t>(s.num_requests) * s.rows_per_request * s.num_q_heads;
  StParams p;
  p.k_new = static_cast<const uint16_t *>(append ? append->k : nullptr);
  p.v_new = static_cast<const uint16_t *>(append ? append->v : nullptr);
  p.k_stride = append ? append->k_stride : 0;
  p.v_stride = append ? append->v_stride : 0;
  p.k_codes = c.k_codes;
  p.v_codes = c.v_codes;
  p.k_scales = c.k_scales;
  p.v_scales = c.v_scales;
  p.num_blocks = static_cast<uint32_t>(c.num_slots >> s.log2_block);
  p.H = c.num_kv_heads;
  p.log2_bs = s.log2_block;
  p.q = static_cast<const uint16_t *>(q);
  p.out = static_cast<uint16_t *>(out);
  p.block_tables = block_tables;
  p.max_blocks = s.max_blocks_per_req;
  p.context_lens = context_lens;
  const int64_t cap = static_cast<int64_t>(s.max_blocks_per_req) << s.log2_block;
  p.ctx_limit = static_cast<int32_t>(cap < s.max_context_len ? cap : s.max_context_len);
  p.N = s.num_requests;
  p.R = s.rows_per_request;
  p.Hq = s.num_q_heads;
  p.G = s.group;
  p.M = s.rows;
  p.qk_scale = sm_scale * 1.4426950408889634f;
  p.cmax = static_cast<int32_t>((static_cast<int64_t>(p.ctx_limit) + kChunk - 1) / kChunk);
  p.pieces = static_cast<int32_t *>(workspace);
  char *parts = static_cast<char *>(workspace) + attn_stream_pieces_bytes(s.num_requests, c.num_kv_heads);
  const size_t o = static_cast<size_t>(rows_total) * kStreamSlots * kHeadDim * sizeof(float);
  p.o_part = reinterpret_cast<float *>(parts);
  p.ml_part = reinterpret_cast<float2 *>(parts + (o + 255) / 256 * 256);
  p.err_flags = err_flags;
  CUtensorMap mk, mv, mks, mvs;
  if (!encode_code_tensor_map_strided(&mk, c.k_codes, c.num_slots, c.num_kv_heads) ||
      !encode_code_tensor_map_strided(&mv, c.v_codes, c.num_slots, c.num_kv_heads) ||
      !encode_scale_tensor_map(&mks, c.k_scales, c.num_slots, c.num_kv_heads, kChunk) ||
      !encode_scale_tensor_map(&mvs, c.v_scales, c.num_slots, c.num_kv_heads, kChunk))
    return cudaErrorInvalidValue;
  static std::atomic<uint64_t> configured{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = (dev >= 0 && dev < 64) ? (uint64_t(1) << dev) : 0;
  if (bit == 0 || !(configured.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(attn_stream_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kStSmem);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit, std::memory_order_acq_rel);
  }
  if (c.num_slots >= (int64_t(1) << 31)) return cudaErrorInvalidValue;
  const int grid = 3 * (s.sms > 0 ? s.sms : 152);
  return launch_overlapped(attn_stream_kernel, dim3(grid), dim3(kStThreads), kStSmem, stream,
                           p, mk, mv, mks, mvs);
}

cudaError_t launch_attn_combine_stream(const AttnShape &s, void *out, void *workspace,
                                       cudaStream_t stream) {
  StCombineParams p;
  p.R = s.rows_per_request;
  p.Hq = s.num_q_heads;
  p.G = s.group;
  p.H = s.num_q_heads / s.group;
  p.rows_total = static_cast<int64_t>(s.num_requests) * s.rows_per_request * s.num_q_heads;
  p.pieces = static_cast<const int32_t *>(workspace);
  const char *parts = static_cast<const char *>(workspace) +
                      attn_stream_pieces_bytes(s.num_requests, s.num_q_heads / s.group);
  const size_t o = static_cast<size_t>(p.rows_total) * kStreamSlots * kHeadDim * sizeof(float);
  p.o_part = reinterpret_cast<const float *>(parts);
  p.ml_part = reinterpret_cast<const float2 *>(parts + (o + 255) / 256 * 256);
  p.out = static_cast<uint16_t *>(out);
  const int64_t ctas = (p.rows_total + kStCombineRows - 1) / kStCombineRows;
  return launch_overlapped(attn_combine_stream_kernel, dim3(static_cast<unsigned>(ctas)),
                           dim3(kStCombineRows * 32), 0, stream, p);
}

}  // namespace kvq
