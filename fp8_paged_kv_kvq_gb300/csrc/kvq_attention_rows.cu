// kvq_attention_rows.cu -- paged attention over the FP8 cache for many stacked
// query rows per KV head (multi-token verify, chunked prefill) on the
// 5th-generation tensor cores, with the query rows on the MMA's M side.
//
// The method is the one of the other attention kernels (ROCm/ATOM PR #2655
// "fix(qwen4-exp): register the QSA FP8 scale planes for KV offload", PR
// description, K/V bullet: each token's key scale multiplies its score after
// the code dot product and its value scale its probability ahead of PV; the
// verify rows of a request that share a KV head are stacked so its codes are
// read once per verify).  sgl-project/sglang-jax #1776 "feat(dsa): implement
// fp8 KV cache (e4m3) with a bf16 indexer cache", Modifications: a prefill
// chunk attends causally over the cached blocks, the probabilities are never
// rounded to fp8.  Laid out for sm_103a:
//
//  * A unit of work is (request, KV head, tile of up to 128 stacked rows) over
//    the tokens its last row sees, in 128-token chunks.  The batch's chunks,
//    ordered (request, head, tile, chunk) with a small charge per unit start,
//    are split into equal contiguous ranges over a persistent grid of one CTA
//    per SM, so every CTA streams the same bytes whatever the lengths.  A
//    unit cut by a range boundary is finished by the CTA whose piece lands
//    last (a tagged ticket per unit), which merges the pieces' (max,
//    denominator, output) from the workspace; no second launch.
//  * The stacked rows fill the 128 TMEM lanes.  With RC rows per tile (32, 64
//    or 128) the tile is replicated 128 / RC times on M; copy c takes the
//    tokens [c RC, c RC + RC) of each chunk, so every softmax thread owns one
//    (row, token slice) with its own running max, denominator and value bound
//    -- no cross-thread reduction per chunk -- and the copies' partial results
//    are merged once per unit in shared memory.
//  * S = Q K^T: M = 128 rows x N = 128 tokens x K = 128, kind::f8f6f4, A = the
//    query tile as two e4m3 pieces (q = 2^e (p1 + p2), exact for elements >=
//    2^-9 of the row's largest, off by at most 2^-17 of it below), the second
//    piece accumulating onto the first, B = the K code tile straight from the
//    TMA ring (K-major, 128-byte swizzle).  O += P V: M = 128 x N = 128 dims x
//    K = 128 tokens, kind::f16, A = P'' = p v_scale 2^-E read from TMEM (the
//    softmax writes it there as f16), B = the V codes converted exactly to f16
//    (MN-major, 128-byte swizzle) by four converter warps.
//  * Warp roles (512 threads): 0-3 and 4-7 two softmax groups (each covering
//    TMEM lane quarters 0-3), group g taking the chunks s with s & 1 == g
//    under references of its own and accumulating into O buffer g; 8-11 V
//    conversion; 12 TMA (block ids fetched ahead by cp.async, one 3-D box per
//    page and plane, one 2-D box of 4 heads' scales per page and plane); 13
//    QK^T MMAs and 14 PV MMAs (one lane each: the two chains of tensor-core
//    work run side by side); 15 idle.  TMEM layouts: see RwCols.
//  * Every wait is bounded; a role that gives up raises a shared abort flag,
//    the softmax warps agree on it at their barriers, copies and MMAs in
//    flight complete, the CTA frees its tensor memory (KVQ_ERRF_WAIT_TIMEOUT).
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <climits>

#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {

namespace {

constexpr int kRwTok = 128;                  // tokens per chunk
constexpr int kRwStages = 5;                 // code ring depth
constexpr int kRwSoftWarps = 4;             // warps of a chunk group (one per lane quarter)
constexpr int kRwGroups = 2;                 // chunk groups: chunk s goes to group s & 1
constexpr int kRwGroupWarps = kRwGroups * kRwSoftWarps;   // warps 0-7
constexpr int kRwWarpTma = kRwGroupWarps;                   // warp 8
constexpr int kRwWarpMma = kRwWarpTma + 1;                  // warp 9: QK^T issuer
constexpr int kRwWarpPv = kRwWarpMma + 1;                   // warp 10: PV issuer
constexpr int kRwThreads = (kRwWarpPv + 1) * 32;

constexpr int kRwIdAhead = 4;                // chunks whose block ids are in flight
constexpr int kRwMaxPagesPerChunk = 8;       // block size >= 16
constexpr float kRwLazy = 14.0f;             // log2 of the largest unnormalised p
constexpr float kRwOvershoot = 4.0f;         // a moved reference sits this far above the max

// TMEM, tiles of 128 rows: S buffer b at columns 128 b .. 128 b + 127; once
// the softmax has read S of chunk s it writes P'' of chunk s into the first 64
// columns of the same buffer (f16 pairs, the PV MMA's A operand).  O buffer b
// at 256 + 128 b: the PV of chunk s accumulates into O buffer s & 1, the
// buffer of the softmax group that takes chunk s, so a reference move of that
// group rescales only its own buffer -- last written by PV(s - 2), complete
// before QK(s) was issued: no wait for an MMA in flight.  The epilogue adds
// the two with their references.
constexpr uint32_t kColS = 0;
constexpr uint32_t kColO = 256;
constexpr uint32_t kRwTmemCols = 512;
// Tiles of at most 64 rows read only their own slice's S columns, which they
// can take in before computing P'': there S is one buffer (columns 0 .. 127)
// and P'' has two of its own (b at 128 + 64 b), whose columns outside a lane's
// slice stay zero for the whole launch.  QK(s + 1) then waits only for the
// softmax to have read S(s) -- not for PV(s) -- and a chunk's P'' store
// writes just its slice's columns.
template <int RC>
struct RwCols {
  static constexpr bool kSplitP = RC < 128;
  __device__ static uint32_t S(int sb) { return kSplitP ? kColS : kColS + 128u * sb; }
  __device__ static uint32_t P(int sb) { return kSplitP ? 128u + 64u * sb : kColS + 128u * sb; }
};

// shared memory, offsets from a 1024-byte aligned base
constexpr int kCodeBytes = kRwTok * kHeadDim;                 // one plane of a chunk
constexpr int kStageBytes = 2 * kCodeBytes;                   // K codes | V codes
constexpr int kScBytes = kRwTok * 16;                         // [token][4 heads] fp32
constexpr int kVfBytes = kRwTok * kHeadDim * 2;               // f16 V operand = a stage
constexpr int kQBytes = 128 * kHeadDim;                       // one e4m3 piece, 128 rows
constexpr int kOffSc = kRwStages * kStageBytes;
constexpr int kOffQ = kOffSc + kRwStages * 2 * kScBytes;       // also the merge scratch
constexpr int kOffTs = kOffQ + 2 * kQBytes;                   // [warp][K | V][128] fp32
constexpr int kOffIds = kOffTs + kRwGroupWarps * 2 * kRwTok * 4;
constexpr int kOffRowf = kOffIds + (kRwIdAhead + 1) * kRwMaxPagesPerChunk * 4;
// [group][128 lanes] (m, l, E, -): over the scale buffers, which only the
// chunk loop uses (the epilogue starts once both groups have left it)
constexpr int kOffMl = kOffTs;
constexpr int kOffPre = kOffRowf + 128 * 4;
constexpr int kOffBar = kOffPre + (kRowsMaxRequests + 4) * 4;
constexpr int kBarKvFull = 0;
constexpr int kBarKvEmpty = kBarKvFull + kRwStages;
constexpr int kBarSFull = kBarKvEmpty + kRwStages;
// chunk s is ready for its PV once its P'' is in TMEM (softmax warps, which
// have also finished reading its S) and its V operand converted (converters)
// tiles of at most 64 rows: S(s) has been read (the single S buffer is free)
constexpr int kBarSFree = kBarSFull + 2;
constexpr int kBarReady = kBarSFree + 2;
constexpr int kBarPvDone = kBarReady + 2;
constexpr int kBarQReady = kBarPvDone + 2;
constexpr int kBarOFree = kBarQReady + 1;
constexpr int kNumBars = kBarOFree + 1;
constexpr int kOffMisc = kOffBar + kNumBars * 8;              // tmem base, abort, ticket
constexpr int kRwSmem = kOffMisc + 64 + 1024;

static_assert(kVfBytes == kStageBytes, "a stage holds its chunk's V operand after conversion");
static_assert(kOffSc % 1024 == 0 && kOffQ % 1024 == 0,
              "operand buffers need 1024-byte alignment");
static_assert(kOffBar % 8 == 0, "barrier alignment");
static_assert(kRwSmem <= 227 * 1024, "shared memory budget");

// S = Q K^T: M = 128 rows, N = 128 tokens, both operands K-major; A (the
// query pieces) e4m3, B (the key codes) e4m3 or, for a cache of e5m2 codes,
// e5m2 (B format field, bits 10-12: 1)
constexpr uint32_t kIdescQK = mma_idesc(128, kRwTok, false, false);
constexpr uint32_t kIdescQK_e5m2 = kIdescQK | (1u << 10);
// O = P V: M = 128 rows, N = 128 dims, A (TMEM) K-major, B MN-major
constexpr uint32_t kIdescPV = mma_idesc(128, kHeadDim, false, true);

struct RwParams {
  uint32_t num_blocks;       // < 2^31
  int32_t H;
  int32_t log2_bs;
  int32_t box;               // rows of a TMA box: min(block size, 128)
  const uint16_t *q;
  uint16_t *out;
  const int32_t *block_tables;
  int32_t max_blocks;
  const int32_t *context_lens;
  int32_t ctx_limit;
  int32_t N, R, Hq, G, M;
  int32_t T;                 // row tiles per (request, KV head)
  float qk_scale;            // sm_scale * log2(e)
  float *o_part;             // [grid][2][rows per tile][128]
  float2 *ml_part;           // [grid][2][rows per tile]
  unsigned long long *tickets;  // [N * H * T]: (call tag, pieces landed)
  uint32_t tag;              // this call's tag (nonzero)
  int32_t *err_flags;
};

__device__ __forceinline__ float rw_ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Bounded wait that also gives up once another role raised the abort flag.
// One out-of-line copy for the whole kernel: inlined (and unrolled) at every
// wait it would multiply the code the warps' loops have to keep in the
// instruction cache.
__device__ __noinline__ bool rw_wait(uint32_t bar, uint32_t parity, volatile int *abort) {
#pragma unroll 1
  for (int i = 0; i < (1 << 19); ++i) {
    if (mbar_try_wait_sleep(bar, parity, 2000u)) return true;
    if ((i & 15) == 15 && *abort) return false;
  }
  *abort = 1;
  return false;
}

// The same with the common case inline: a phase already complete costs one
// try_wait, not a call (which, at this kernel's register load, saves and
// restores live registers around it).
__device__ __forceinline__ bool rw_wait_fast(uint32_t bar, uint32_t parity, volatile int *abort) {
  return mbar_try_wait(bar, parity) || rw_wait(bar, parity, abort);
}

// Barrier over the softmax warps that also ORs a flag across them.
__device__ __forceinline__ bool soft_barrier_or(bool flag) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n"
      " bar.red.or.pred q, 1, %2, p;\n selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r) : "r"(flag ? 1u : 0u), "n"(kRwGroups * kRwSoftWarps * 32) : "memory");
  return r != 0;
}

__device__ __forceinline__ void soft_barrier() {
  named_barrier(1, kRwGroups * kRwSoftWarps * 32);
}

// Barrier over group 0's warps (the unit's final merge).
__device__ __forceinline__ void group0_barrier() { named_barrier(2, kRwSoftWarps * 32); }



// Smallest e in [-126, 126] with 2^e >= v (v >= 0 given as its bits).
__device__ __forceinline__ int rw_pow2_ceil(uint32_t bits) {
  const int ex = static_cast<int>((bits >> 23) & 0xFFu);
  int e = (ex == 0) ? -126 : ex - 127 + ((bits & 0x7FFFFFu) != 0u ? 1 : 0);
  return e > 126 ? 126 : e;
}

__device__ __forceinline__ float pow2f(int e) {    // e in [-126, 127]
  return __int_as_float((127 + e) << 23);
}

__device__ __forceinline__ float pow2f_down(int d) {   // 2^d for d <= 0, 0 below 2^-126
  return d < -126 ? 0.0f : pow2f(d);
}

// ---------------------------------------------------------------------------
// Work layout.  Unit (r, h, t): the rows [128 t, 128 t + 128) of the stacked
// rows m = i G + g (query row i, query head h G + g) of request r; it reads the
// tokens its last row sees.  In the work sequence it spans V = C + kRowsSwitch
// positions (C its chunks) or none when C = 0; request r's units take
// W_r = H sum_t V_rt positions from pre[r] on, ordered (h, t).

struct Geo {
  int32_t R, G, M, T, H, ctx_limit;
};

__device__ __forceinline__ int clamp_len(int L, int lim) { return L < 0 ? 0 : (L > lim ? lim : L); }

// Tokens the last row of tile t sees, and the tile's chunk count.
__device__ __forceinline__ int tile_tokens(const Geo &g, int L, int t) {
  const int m_last = min(g.M, 128 * (t + 1)) - 1;
  const int v = L - g.R + 1 + m_last / g.G;
  return v < 0 ? 0 : (v > L ? L : v);
}

__device__ __forceinline__ int tile_positions(const Geo &g, int L, int t) {
  const int c = (tile_tokens(g, L, t) + kRwTok - 1) / kRwTok;
  return c > 0 ? c + kRowsSwitch : 0;
}

struct Seg {
  int r, h, t, L;
  int C, c0, n;          // the unit's chunks, the CTA's first chunk and count
  int vis;               // tokens the unit reads
  int64_t first;         // position of the unit's first chunk
  int64_t next;          // where the CTA's range continues
};

__device__ __forceinline__ Seg locate_rows(const int32_t *pre, const int32_t *context_lens, const Geo g, int N,
                           int64_t x, int64_t x_end) {
  int lo = 0, hi = N - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (pre[mid] <= x) lo = mid;
    else hi = mid - 1;
  }
  Seg s;
  s.r = lo;
  s.L = clamp_len(context_lens[lo], g.ctx_limit);
  int S = 0;
  for (int t = 0; t < g.T; ++t) S += tile_positions(g, s.L, t);
  const int64_t off = x - pre[lo];
  s.h = static_cast<int>(off / S);
  int rem = static_cast<int>(off - static_cast<int64_t>(s.h) * S);
  int acc = 0, t = 0;
  for (; t < g.T - 1; ++t) {
    const int v = tile_positions(g, s.L, t);
    if (rem < acc + v) break;
    acc += v;
  }
  s.t = t;
  s.vis = tile_tokens(g, s.L, t);
  s.C = (s.vis + kRwTok - 1) / kRwTok;
  const int64_t start = pre[lo] + static_cast<int64_t>(s.h) * S + acc;
  s.first = start + kRowsSwitch;
  const int64_t uend = start + (s.C > 0 ? s.C + kRowsSwitch : 0);
  const int64_t end = uend < x_end ? uend : x_end;
  const int64_t xs = x > s.first ? x : s.first;
  s.next = end > x ? end : x + 1;
  if (xs >= end) {
    s.c0 = 0;
    s.n = 0;
  } else {
    s.c0 = static_cast<int>(xs - s.first);
    s.n = static_cast<int>(end - xs);
  }
  return s;
}

// The first segment with chunks at or after position x (n = 0 when the range
// has none left).  Out of line: it runs once per segment, and its code stays
// out of the roles' hot loops.
__device__ __noinline__ Seg next_segment(const int32_t *pre, const int32_t *cl, const Geo g, int N,
                                         int64_t x, int64_t x_end) {
  while (x < x_end) {
    const Seg sg = locate_rows(pre, cl, g, N, x, x_end);
    if (sg.n > 0) return sg;
    x = sg.next;
  }
  Seg e;
  e.r = e.h = e.t = e.L = e.C = e.c0 = e.n = e.vis = 0;
  e.first = e.next = x_end;
  return e;
}

// Walks the chunks of a CTA's range in order (its state in registers).
struct ChunkWalk {
  Seg sg;
  int k;                 // chunk within the segment
  int seg;               // segment index
  int64_t x_end;
  bool valid;
  __device__ __forceinline__ void start(const int32_t *pre, const int32_t *cl, const Geo g, int N,
                                        int64_t xb, int64_t xe) {
    x_end = xe;
    seg = 0;
    k = 0;
    sg = next_segment(pre, cl, g, N, xb, xe);
    valid = sg.n > 0;
  }
  __device__ __forceinline__ void advance_segment(const int32_t *pre, const int32_t *cl,
                                                  const Geo g, int N) {
    sg = next_segment(pre, cl, g, N, sg.next, x_end);
    valid = sg.n > 0;
    k = 0;
    ++seg;
  }
  __device__ __forceinline__ void next(const int32_t *pre, const int32_t *cl, const Geo g, int N) {
    if (!valid) return;
    if (++k < sg.n) return;
    advance_segment(pre, cl, g, N);
  }
};

// ---------------------------------------------------------------------------
// Softmax pieces.  A softmax thread owns TMEM lane L (row L % RC of the tile,
// copy L / RC) and the chunk's token slice [copy RC, copy RC + RC).  The hot
// loop below is kept compact (16 tokens per trip, not unrolled over the
// slice) and the rare or once-per-unit steps live in functions of their own:
// the kernel's warps run four different loops side by side, and their code
// has to stay in the SM's instruction cache.

// A move of one thread's references in the middle of a chunk: the new
// references, the factor that takes exponentials under the old score
// reference to the new (the denominator's terms) and the one for P'' (which
// also carries 2^-E).
struct RwMove {
  float m;
  int e;
  float fl, fp;
};
__device__ __forceinline__ RwMove rows_move(float gmx, float gvmax, float m_ref, int E) {
  RwMove r;
  r.m = (gmx > m_ref + kRwLazy) ? gmx + kRwOvershoot : m_ref;
  const int e_need = rw_pow2_ceil(__float_as_uint(gvmax));
  r.e = e_need > E ? min(e_need + 2, 126) : E;
  r.fl = (m_ref == -INFINITY) ? 0.0f : rw_ex2(m_ref - r.m);
  r.fp = r.fl * pow2f_down(E - r.e);
  return r;
}

// An f16 pair times f, through f32 (f may lie below the f16 range).
__device__ __forceinline__ uint32_t scale_f16x2(uint32_t w, float f) {
  float lo, hi;
  asm("{\n .reg .f16 l, h;\n mov.b32 {l, h}, %2;\n cvt.f32.f16 %0, l;\n"
      " cvt.f32.f16 %1, h;\n}\n" : "=f"(lo), "=f"(hi) : "r"(w));
  return pack_f16x2(lo * f, hi * f);
}

// One 16-token group of a row's slice.  Scores in log2 units relative to the
// present reference, u = S k_scale rowf - m (pairs of f32: the arithmetic
// runs on the f32x2 path), the value scales beside them, unseen tokens
// (j >= lim; only a unit's last chunk has them, hence the warp-uniform
// `masked`) at -inf with weight 0, and the group's maxima.
struct RwGroup {
  uint64_t u[8], vw[8];
  float gmx, gvm;
};
__device__ __forceinline__ void rows_group_u(const float (&x)[16], const float *ks,
                                             const float *vs, int g, float rowf, float ms,
                                             int lim, bool masked, RwGroup &gr) {
  const uint64_t rf = pack_f32x2(rowf, rowf), nms = pack_f32x2(-ms, -ms);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float4 k4 = reinterpret_cast<const float4 *>(ks)[4 * g + q];
    const float4 v4 = reinterpret_cast<const float4 *>(vs)[4 * g + q];
    gr.u[2 * q] = fma_f32x2(mul_f32x2(pack_f32x2(x[4 * q], x[4 * q + 1]), pack_f32x2(k4.x, k4.y)),
                            rf, nms);
    gr.u[2 * q + 1] = fma_f32x2(
        mul_f32x2(pack_f32x2(x[4 * q + 2], x[4 * q + 3]), pack_f32x2(k4.z, k4.w)), rf, nms);
    gr.vw[2 * q] = pack_f32x2(v4.x, v4.y);
    gr.vw[2 * q + 1] = pack_f32x2(v4.z, v4.w);
  }
  if (masked) {
    // (their scales may be stale: the selects also drop a NaN product)
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float a, b, va, vb;
      unpack_f32x2(gr.u[i], a, b);
      unpack_f32x2(gr.vw[i], va, vb);
      const bool s0 = 16 * g + 2 * i < lim, s1 = 16 * g + 2 * i + 1 < lim;
      gr.u[i] = pack_f32x2(s0 ? a : -INFINITY, s1 ? b : -INFINITY);
      gr.vw[i] = pack_f32x2(s0 ? va : 0.0f, s1 ? vb : 0.0f);
    }
  }
  float mx = -INFINITY, vm = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    float a, b, va, vb;
    unpack_f32x2(gr.u[i], a, b);
    unpack_f32x2(gr.vw[i], va, vb);
    mx = fmaxf(mx, fmaxf(a, b));
    vm = fmaxf(vm, fmaxf(va, vb));
  }
  gr.gmx = mx;
  gr.gvm = vm;
}

// Whether a row of the warp has to move its references before the group's
// exponentials (a score past the headroom, or a value scale past 2^E).
__device__ __forceinline__ bool rows_group_over(const RwGroup &gr, float m_ref, int E) {
  const float thr = (m_ref == -INFINITY) ? -INFINITY : kRwLazy;
  return __any_sync(0xFFFFFFFFu, gr.gmx > thr || gr.gvm > pow2f(E));
}

// Moves this thread's references for the group (rows whose references hold
// get factor 1) and shifts the group's u to the new score reference; returns
// the factor for P'' already produced, after scaling the denominators.
__device__ __forceinline__ float rows_group_move(RwGroup &gr, float &m_ref, int &E, float &lsum,
                                                 float &lchunk) {
  const float ms = (m_ref == -INFINITY) ? 0.0f : m_ref;
  const RwMove mv = rows_move(gr.gmx + ms, gr.gvm, m_ref, E);
  lsum *= mv.fl;
  lchunk *= mv.fl;
  m_ref = mv.m;
  E = mv.e;
  const float ms_new = (m_ref == -INFINITY) ? 0.0f : m_ref;
  const uint64_t d = pack_f32x2(ms - ms_new, ms - ms_new), one = pack_f32x2(1.0f, 1.0f);
#pragma unroll
  for (int i = 0; i < 8; ++i) gr.u[i] = fma_f32x2(gr.u[i], one, d);
  return mv.fp;
}

// The group's P'' = 2^u v_scale 2^-E as f16 pairs, and its share of the
// denominator added to lchunk.
__device__ __forceinline__ void rows_group_p(const RwGroup &gr, int E, float &lchunk,
                                             uint32_t *w8) {
  const uint64_t vn = pack_f32x2(pow2f(-E), pow2f(-E));
  uint64_t lc = pack_f32x2(0.0f, 0.0f);
  const uint64_t one = pack_f32x2(1.0f, 1.0f);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    float a, b;
    unpack_f32x2(gr.u[i], a, b);
    const uint64_t pp = pack_f32x2(rw_ex2(a), rw_ex2(b));
    lc = fma_f32x2(pp, one, lc);
    float w0, w1;
    unpack_f32x2(mul_f32x2(pp, mul_f32x2(gr.vw[i], vn)), w0, w1);
    w8[i] = pack_f16x2(w0, w1);
  }
  float l0, l1;
  unpack_f32x2(lc, l0, l1);
  lchunk += l0 + l1;
}

// P'' = p v_scale 2^-E of this thread's slice (RC <= 64 tokens), packed as f16
// pairs into pk, and its share of the denominator.  The slice's S columns are
// read first and the warp announces it on sfree (the next chunk's QK^T may
// then overwrite them).  The slice goes in groups of 16 tokens (32-token
// slices: both groups under one decision); a row whose scores pass its
// reference's headroom, or whose value scales pass the bound 2^E, moves its
// references before the group's exponentials and brings the P'' already
// packed and the denominators under the new ones, so no exponential is
// computed twice.  (One decision for both groups of a 32-token slice lets
// their exponentials interleave: verify 904 vs 907 us.)
template <int RC>
__device__ __forceinline__ void rows_chunk_p(uint32_t scol, uint32_t sfree, int lane,
                                            const float *ks, const float *vs, int lim, float rowf,
                                            float &m_ref, int &E, float &lchunk, float &lsum,
                                            uint32_t (&pk)[RC / 2]) {
  float xs[RC];
#pragma unroll
  for (int c = 0; c < RC; c += 32) {
    float x32[32];
    tmem_ld32(scol + c, x32);
#pragma unroll
    for (int i = 0; i < 32; ++i) xs[c + i] = x32[i];
  }
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(sfree);
  const bool masked = __any_sync(0xFFFFFFFFu, lim < RC);
  if constexpr (RC == 32) {
    // both 16-token groups' scores first, one reference decision for the
    // slice, then both groups' exponentials side by side
    const float ms = (m_ref == -INFINITY) ? 0.0f : m_ref;
    RwGroup g0, g1;
    {
      float x[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) x[i] = xs[i];
      rows_group_u(x, ks, vs, 0, rowf, ms, lim, masked, g0);
#pragma unroll
      for (int i = 0; i < 16; ++i) x[i] = xs[16 + i];
      rows_group_u(x, ks, vs, 1, rowf, ms, lim, masked, g1);
    }
    RwGroup all;
    all.gmx = fmaxf(g0.gmx, g1.gmx);
    all.gvm = fmaxf(g0.gvm, g1.gvm);
    if (rows_group_over(all, m_ref, E)) {
      const RwMove mv = rows_move(all.gmx + ms, all.gvm, m_ref, E);
      lsum *= mv.fl;
      lchunk *= mv.fl;
      m_ref = mv.m;
      E = mv.e;
      const float ms_new = (m_ref == -INFINITY) ? 0.0f : m_ref;
      const uint64_t d = pack_f32x2(ms - ms_new, ms - ms_new), one = pack_f32x2(1.0f, 1.0f);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        g0.u[i] = fma_f32x2(g0.u[i], one, d);
        g1.u[i] = fma_f32x2(g1.u[i], one, d);
      }
    }
    rows_group_p(g0, E, lchunk, &pk[0]);
    rows_group_p(g1, E, lchunk, &pk[8]);
  } else {
#pragma unroll
    for (int g = 0; g < RC / 16; ++g) {
      float x[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) x[i] = xs[16 * g + i];
      RwGroup gr;
      rows_group_u(x, ks, vs, g, rowf, (m_ref == -INFINITY) ? 0.0f : m_ref, lim, masked, gr);
      if (rows_group_over(gr, m_ref, E)) {
        const float f = rows_group_move(gr, m_ref, E, lsum, lchunk);
#pragma unroll
        for (int i = 0; i < 8 * g; ++i) pk[i] = scale_f16x2(pk[i], f);
      }
      rows_group_p(gr, E, lchunk, &pk[8 * g]);
    }
  }
}

// The O rows of one buffer brought to this thread's present references
// (factor 2^(ref_o - m) 2^(e_o - E); rows of the warp already there multiply
// by 1).  The buffer must have no MMA in flight.
__device__ __forceinline__ void rows_rescale_o(uint32_t ocol, float f) {
#pragma unroll 1
  for (int c = 0; c < 128; c += 32) {
    float o[32];
    tmem_ld32(ocol + c, o);
#pragma unroll
    for (int i = 0; i < 32; ++i) o[i] *= f;
    tmem_st32(ocol + c, o);
  }
  tmem_wait_st();
}

// The P'' columns [pcol, pcol + ncols) of this thread's lane times f (the
// warp's rows whose references stayed put have f = 1).
__device__ __noinline__ void rows_rescale_p(uint32_t pcol, int ncols, float f) {
#pragma unroll 1
  for (int c = 0; c < ncols; c += 8) {
    uint32_t w[8];
    tmem_ld8u(pcol + c, w);
#pragma unroll
    for (int i = 0; i < 8; ++i) w[i] = scale_f16x2(w[i], f);
    tmem_st8u(pcol + c, w);
  }
}

// P'' of a whole 128-token chunk for one row (RC = 128, one copy), 32 tokens
// (two 16-token groups under one decision, their exponentials interleaved:
// prefill 2.20 vs 2.34 ms with a decision per group) at a time, stored 16
// columns at a time over the S columns of tokens already read (groups g, g + 1
// put their P'' in columns [8 g, 8 g + 16), whose S values the groups up to
// g + 1 have consumed).  A row that outgrows its references moves them
// before the pair's exponentials and brings the P'' already stored, the
// chunk's denominator share and the running denominator under the new ones,
// so no S value is needed twice and nothing is held in registers across the
// chunk.
__device__ __forceinline__ void rows_chunk_p_direct(uint32_t scol, const float *ks,
                                                    const float *vs, int lim, float rowf,
                                                    float &m_ref, int &E, float &lchunk,
                                                    float &lsum) {
  const bool masked = __any_sync(0xFFFFFFFFu, lim < 128);
#pragma unroll
  for (int g = 0; g < 8; g += 2) {
    // two groups per decision: both groups' scores, one reference check,
    // then both groups' exponentials side by side
    float x[32];
    tmem_ld32(scol + 16 * g, x);
    const float ms = (m_ref == -INFINITY) ? 0.0f : m_ref;
    RwGroup g0, g1;
    {
      float y[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) y[i] = x[i];
      rows_group_u(y, ks, vs, g, rowf, ms, lim, masked, g0);
#pragma unroll
      for (int i = 0; i < 16; ++i) y[i] = x[16 + i];
      rows_group_u(y, ks, vs, g + 1, rowf, ms, lim, masked, g1);
    }
    RwGroup both;
    both.gmx = fmaxf(g0.gmx, g1.gmx);
    both.gvm = fmaxf(g0.gvm, g1.gvm);
    if (rows_group_over(both, m_ref, E)) {
      const RwMove mv = rows_move(both.gmx + ms, both.gvm, m_ref, E);
      lsum *= mv.fl;
      lchunk *= mv.fl;
      m_ref = mv.m;
      E = mv.e;
      const float ms_new = (m_ref == -INFINITY) ? 0.0f : m_ref;
      const uint64_t d = pack_f32x2(ms - ms_new, ms - ms_new), one = pack_f32x2(1.0f, 1.0f);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        g0.u[i] = fma_f32x2(g0.u[i], one, d);
        g1.u[i] = fma_f32x2(g1.u[i], one, d);
      }
      if (g > 0) rows_rescale_p(scol, 8 * g, mv.fp);
    }
    uint32_t w16[16];
    rows_group_p(g0, E, lchunk, &w16[0]);
    rows_group_p(g1, E, lchunk, &w16[8]);
    tmem_st16u(scol + 8 * g, w16);
  }
}

// The unit's query tile (rows m < rows_here of tile row0, every copy) as two
// e4m3 pieces per element in the K-major 128-byte swizzled layout, and each
// row's factor 2^e sm_scale log2(e).  The 8 softmax warps take every 8th row;
// the rows are fetched into registers while the previous unit's epilogue
// runs (the tile's space is its scratch) and stored afterwards.
struct QArgs {
  const uint16_t *q;
  int32_t R, Hq, G;
  float qk_scale;
};

template <int RC>
struct QRows {
  uint2 v[RC / kRwGroupWarps];                  // this warp's rows, 4 bf16 per lane
};

template <int RC>
__device__ __forceinline__ void rows_fetch_q(QRows<RC> &f, const QArgs p, int r, int h,
                                             int row0, int rows_here, int warp, int lane) {
#pragma unroll
  for (int i = 0; i < RC / kRwGroupWarps; ++i) {
    const int m = warp + kRwGroupWarps * i;
    f.v[i] = make_uint2(0u, 0u);
    if (m < rows_here) {
      const int ma = row0 + m, ir = ma / p.G, gq = ma - ir * p.G;
      f.v[i] = *reinterpret_cast<const uint2 *>(
          p.q + ((static_cast<int64_t>(r) * p.R + ir) * p.Hq + h * p.G + gq) * kHeadDim +
          4 * lane);
    }
  }
}

template <int RC>
__device__ __forceinline__ void rows_store_q(const QRows<RC> &f, float qk_scale, uint8_t *smem,
                                             float *rowf_s, int warp, int lane) {
  constexpr int kCopies = 128 / RC;
#pragma unroll 1
  for (int i = 0; i < RC / kRwGroupWarps; ++i) {
    const int m = warp + kRwGroupWarps * i;
    const uint2 v = f.v[i];
    float amax = fmaxf(fmaxf(fabsf(bf16_lo(v.x)), fabsf(bf16_hi(v.x))),
                       fmaxf(fabsf(bf16_lo(v.y)), fabsf(bf16_hi(v.y))));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
      amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, off));
    const int ex = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFFu);
    int e = (ex == 0) ? -126 : ex - 127 - 7;
    e = e < -126 ? -126 : (e > 126 ? 126 : e);
    const float rx = (amax == 0.0f) ? 0.0f : pow2f(e);          // 2^e
    uint32_t c1w = 0u, c2w = 0u;
    if (rx != 0.0f) {
      const float inv = pow2f(-e);
      const float xs[4] = {bf16_lo(v.x) * inv, bf16_hi(v.x) * inv, bf16_lo(v.y) * inv,
                           bf16_hi(v.y) * inv};
      e4m3_pieces4(xs, c1w, c2w);
    }
    if (lane == 0) rowf_s[m] = rx * qk_scale;
#pragma unroll
    for (int c = 0; c < kCopies; ++c) {
      const int row = c * RC + m;
      const int off = row * kHeadDim + (((lane >> 2) ^ (row & 7)) << 4) + 4 * (lane & 3);
      *reinterpret_cast<uint32_t *>(smem + kOffQ + off) = c1w;
      *reinterpret_cast<uint32_t *>(smem + kOffQ + kQBytes + off) = c2w;
    }
  }
}

// Two codes (bytes 0 and 1 of w16) to their exact f16 values: e4m3 through
// the hardware conversion; e5m2 is the top byte of an f16, so a byte shift.
template <int kFmt>
__device__ __forceinline__ uint32_t codes2_to_f16x2(uint32_t w16) {
  if (kFmt == KVQ_CODES_E5M2) return prmt(w16, 0u, 0x1404u);
  return e4m3x2_to_f16x2(w16);
}

template <int RC, int kFmt>
__global__ void __launch_bounds__(kRwThreads, 1)
attn_rows_kernel(const RwParams p, const __grid_constant__ CUtensorMap tm_kc,
                 const __grid_constant__ CUtensorMap tm_vc,
                 const __grid_constant__ CUtensorMap tm_ks,
                 const __grid_constant__ CUtensorMap tm_vs) {
  constexpr int kCopies = 128 / RC;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;

  int32_t *pre = reinterpret_cast<int32_t *>(smem + kOffPre);
  const uint32_t bar0 = smem_addr(smem + kOffBar);
  auto BAR = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kOffMisc);
  volatile int *abort_s = reinterpret_cast<volatile int *>(smem + kOffMisc + 4);
  int *ticket_s = reinterpret_cast<int *>(smem + kOffMisc + 8);
  float *rowf_s = reinterpret_cast<float *>(smem + kOffRowf);

  // The launch overlaps the previous kernel's drain; every global access comes
  // after the wait.
  allow_dependents_launch();
  grid_dependency_wait();

  const Geo geo{p.R, p.G, p.M, p.T, p.H, p.ctx_limit};
  const int N = p.N;
  if (warp == 0) {
    int carry = 0;
    for (int r0 = 0; r0 < N; r0 += 32) {
      const int r = r0 + lane;
      int W = 0;
      if (r < N) {
        int L = p.context_lens[r];
        if (L < 0 || L > p.ctx_limit) {
          if (blockIdx.x == 0 && p.err_flags) atomicOr(p.err_flags, KVQ_ERRF_CONTEXT_RANGE);
          L = clamp_len(L, p.ctx_limit);
        }
        for (int t = 0; t < p.T; ++t) W += tile_positions(geo, L, t);
        W *= p.H;
      }
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int v = __shfl_up_sync(0xFFFFFFFFu, W, off);
        if (lane >= off) W += v;
      }
      if (r < N) pre[r + 1] = carry + W;
      carry += __shfl_sync(0xFFFFFFFFu, W, 31);
    }
    if (lane == 0) pre[0] = 0;
  }
  if (tid == 32) {
    for (int s = 0; s < kRwStages; ++s) {
      mbar_init(BAR(kBarKvFull + s), 1);
      mbar_init(BAR(kBarKvEmpty + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(BAR(kBarSFull + b), 1);
      mbar_init(BAR(kBarSFree + b), kRwSoftWarps);
      // P'' from the owner group, V from the other one (tiles of 128 rows)
      // or from the owner too
      mbar_init(BAR(kBarReady + b), (RC == 128 ? 2 : 1) * kRwSoftWarps);
      mbar_init(BAR(kBarPvDone + b), 1);
    }
    mbar_init(BAR(kBarQReady), kRwGroupWarps);
    mbar_init(BAR(kBarOFree), kRwGroups * kRwSoftWarps);
    *abort_s = 0;
    fence_mbarrier_init();
  }
  if (warp == kRwWarpTma) {
    tmem_alloc(smem_addr(tmem_slot), kRwTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int64_t total = pre[N];
  const int64_t B = total > 0 ? (total + gridDim.x - 1) / gridDim.x : 1;
  const int64_t x_begin = static_cast<int64_t>(blockIdx.x) * B;
  const int64_t x_end = total < x_begin + B ? total : x_begin + B;

  if (warp == kRwWarpTma) {
    // ---------------------------------------------------------------- TMA
    // Block ids of chunk u + kRwIdAhead are fetched (lanes < pages, cp.async,
    // one commit group per chunk) while chunk u is issued.
    int32_t *ids = reinterpret_cast<int32_t *>(smem + kOffIds);
    const int npg = p.box < kRwTok ? kRwTok / p.box : 1;
    ChunkWalk fw, iw;
    fw.start(pre, p.context_lens, geo, N, x_begin, x_end);
    iw = fw;
    auto fetch = [&](const ChunkWalk &w, int slot) {
      if (w.valid && lane < npg) {
        const int j = (w.sg.c0 + w.k) * kRwTok + lane * p.box;     // first token of the box
        const bool need = j < w.sg.vis;
        const int32_t *src = p.block_tables + static_cast<int64_t>(w.sg.r) * p.max_blocks +
                             (need ? (j >> p.log2_bs) : 0);
        cp_async_4(ids + slot * kRwMaxPagesPerChunk + lane, src, need ? 4u : 0u);
      }
      cp_async_commit();
    };
    for (int a = 0; a < kRwIdAhead; ++a) {
      fetch(fw, a % (kRwIdAhead + 1));
      fw.next(pre, p.context_lens, geo, N);
    }
    uint32_t u = 0;
    bool bad = false, stop = false;
    // a unit's codes are read once when a (request, KV head) has one tile of
    // rows; with several tiles each re-reads them, and L2 should keep them
    const uint64_t pol = p.T == 1 ? l2_policy_evict_first() : l2_policy_evict_normal();
    for (; iw.valid && !stop; ++u) {
      fetch(fw, (u + kRwIdAhead) % (kRwIdAhead + 1));
      fw.next(pre, p.context_lens, geo, N);
      cp_async_wait<kRwIdAhead>();
      __syncwarp();
      if (lane == 0) {
        const int b = u % kRwStages;
        if (u >= kRwStages &&
            !rw_wait_fast(BAR(kBarKvEmpty + b), ((u / kRwStages) - 1) & 1, abort_s)) {
          stop = true;
        } else {
          const uint32_t kdst = smem_addr(smem + b * kStageBytes);
          const uint32_t vdst = kdst + kCodeBytes;
          const uint32_t ksd = smem_addr(smem + kOffSc + b * 2 * kScBytes);
          const uint32_t vsd = ksd + kScBytes;
          const uint32_t fb = BAR(kBarKvFull + b);
          const int32_t *cid = ids + (u % (kRwIdAhead + 1)) * kRwMaxPagesPerChunk;
          const int j0 = (iw.sg.c0 + iw.k) * kRwTok;
          const int h = iw.sg.h;
          uint32_t bytes = 0;
          for (int i = 0; i < npg; ++i) {
            const int j = j0 + i * p.box;
            if (j >= iw.sg.vis) break;
            const uint32_t blk = static_cast<uint32_t>(cid[i]);
            if (blk >= p.num_blocks) {
              bad = true;
              continue;
            }
            const int z = static_cast<int>((blk << p.log2_bs) | (j & ((1 << p.log2_bs) - 1)));
            // codes read once go first, so the scale lines (each 32-byte
            // sector holds 8 heads' scales of a slot, wanted by 8 units at
            // different times) stay in L2 longer
            tma_load_3d_hint(kdst + i * p.box * kHeadDim, &tm_kc, 0, h, z, fb, pol);
            tma_load_3d_hint(vdst + i * p.box * kHeadDim, &tm_vc, 0, h, z, fb, pol);
            tma_load_2d(ksd + i * p.box * 16, &tm_ks, h & ~3, z, fb);
            tma_load_2d(vsd + i * p.box * 16, &tm_vs, h & ~3, z, fb);
            bytes += 2u * p.box * kHeadDim + 2u * p.box * 16u;
          }
          mbar_arrive_expect_tx(fb, bytes);
        }
      }
      stop = __shfl_sync(0xFFFFFFFFu, stop ? 1 : 0, 0) != 0;
      iw.next(pre, p.context_lens, geo, N);
    }
    cp_async_wait<0>();
    if (lane == 0) {
      if (bad && p.err_flags) atomicOr(p.err_flags, KVQ_ERRF_BLOCK_RANGE);
      // copies still in flight (after an abort) land before the CTA leaves
      const uint32_t issued = stop ? u - 1 : u;
      for (uint32_t v = (issued > kRwStages ? issued - kRwStages : 0); v < issued; ++v)
        mbar_wait_sleep_bounded(BAR(kBarKvFull + v % kRwStages), (v / kRwStages) & 1);
    }
  } else if (warp == kRwWarpMma) {
    // ------------------------------------------------------------ QK^T MMA
    if (lane == 0) {
      constexpr uint32_t kQK = kFmt == KVQ_CODES_E5M2 ? kIdescQK_e5m2 : kIdescQK;
      const uint32_t q0 = smem_addr(smem + kOffQ);
      uint32_t last_bar = 0, last_par = 0;
      bool any = false;
      ChunkWalk w;
      w.start(pre, p.context_lens, geo, N, x_begin, x_end);
      for (int s = 0; w.valid; ++s) {
        const int b = s % kRwStages, sb = s & 1;
        // a new unit's query tile (written once the last unit's softmax and
        // merge are done)
        if (w.k == 0 && !rw_wait_fast(BAR(kBarQReady), w.seg & 1, abort_s)) break;
        if (!rw_wait_fast(BAR(kBarKvFull + b), (s / kRwStages) & 1, abort_s)) break;
        if constexpr (RwCols<RC>::kSplitP) {
          // the one S buffer is free once the softmax has read S(s - 1)
          if (s >= 1 &&
              !rw_wait_fast(BAR(kBarSFree + ((s - 1) & 1)), ((s - 1) >> 1) & 1, abort_s))
            break;
        } else {
          // S buffer s & 1 holds P of chunk s - 2 until that chunk's PV is done
          if (s >= 2 && !rw_wait_fast(BAR(kBarPvDone + sb), ((s >> 1) - 1) & 1, abort_s)) break;
        }
        tc_fence_after();
        const uint64_t kd = smem_desc(smem_addr(smem + b * kStageBytes), 16, 1024, kSmemSwizzle128);
        const uint64_t qa = smem_desc(q0, 16, 1024, kSmemSwizzle128);
        const uint64_t qb = smem_desc(q0 + kQBytes, 16, 1024, kSmemSwizzle128);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          tc_mma_e4m3(tmem + RwCols<RC>::S(sb), qa + 2 * kk, kd + 2 * kk, kQK, kk != 0);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          tc_mma_e4m3(tmem + RwCols<RC>::S(sb), qb + 2 * kk, kd + 2 * kk, kQK, 1u);
        tc_commit(BAR(kBarSFull + sb));
        last_bar = BAR(kBarSFull + sb);
        last_par = (s >> 1) & 1;
        any = true;
        w.next(pre, p.context_lens, geo, N);
      }
      // every MMA issued has completed before the tensor memory is freed
      if (any) mbar_wait_sleep_bounded(last_bar, last_par);
    }
  } else if (warp == kRwWarpPv) {
    // -------------------------------------------------------------- PV MMA
    if (lane == 0) {
      const uint32_t st0 = smem_addr(smem);
      uint32_t last_bar = 0, last_par = 0;
      bool any = false;
      ChunkWalk w;
      w.start(pre, p.context_lens, geo, N, x_begin, x_end);
      for (int s = 0; w.valid; ++s) {
        const int cb = s & 1;
        const bool first = w.k == 0;
        const bool fresh = w.k < 2;              // the unit's first PV into O buffer cb
        // P'' and the V operand of chunk s; a new unit's O once the last
        // unit's rows have been read back
        if (!rw_wait_fast(BAR(kBarReady + cb), (s >> 1) & 1, abort_s)) break;
        if (first && w.seg >= 1 && !rw_wait_fast(BAR(kBarOFree), (w.seg - 1) & 1, abort_s)) break;
        tc_fence_after();
        // the chunk's stage holds its V operand, converted in place
        const uint64_t bd = smem_desc(st0 + (s % kRwStages) * kStageBytes, kVfBytes / 2, 1024,
                                      kSmemSwizzle128);
#pragma unroll
        for (int kk = 0; kk < kRwTok / 16; ++kk)
          tc_mma_f16_tmem_a(tmem + kColO + 128 * cb, tmem + RwCols<RC>::P(cb) + 8 * kk,
                            bd + (2048 >> 4) * kk, kIdescPV, (fresh && kk == 0) ? 0u : 1u);
        tc_commit(BAR(kBarPvDone + cb));
        tc_commit(BAR(kBarKvEmpty + s % kRwStages));   // the stage is free again
        last_bar = BAR(kBarPvDone + cb);
        last_par = (s >> 1) & 1;
        any = true;
        w.next(pre, p.context_lens, geo, N);
      }
      if (any) mbar_wait_sleep_bounded(last_bar, last_par);
    }
  } else if (warp < kRwGroupWarps) {
    // ------------------------------------------------ chunk groups: softmax
    // Group gp = warp / 4 takes the chunks s with s & 1 == gp: their P'' (a
    // thread owns TMEM lane L of quarter warp % 4: row L % RC of the tile,
    // copy L / RC, tokens [copy RC, copy RC + RC) of each chunk) and O buffer
    // gp, under references of its own; the groups' partial rows are merged
    // once per unit.  While one group works on chunk s, the other has chunk
    // s + 1.
    const int gp = warp / kRwSoftWarps, q4 = warp % kRwSoftWarps;
    const int L32 = 32 * q4 + lane;             // this thread's TMEM lane
    const int copy = L32 / RC;                  // its token slice [copy RC, copy RC + RC)
    const int mrow = L32 % RC;                  // its row within the tile
    const uint32_t tl = tmem + (static_cast<uint32_t>(32 * q4) << 16);
    float4 *ml_s = reinterpret_cast<float4 *>(smem + kOffMl);
    bool aborted = false;
    if constexpr (RwCols<RC>::kSplitP) {
      // this group's P'' buffer zero in this lane: a chunk writes only its
      // slice's columns
      float z[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) z[i] = 0.0f;
#pragma unroll
      for (int c = 0; c < 64; c += 32) tmem_st32(tl + RwCols<RC>::P(gp) + c, z);
      tmem_wait_st();
    }
    ChunkWalk w;
    w.start(pre, p.context_lens, geo, N, x_begin, x_end);
    const QArgs qa{p.q, p.R, p.Hq, p.G, p.qk_scale};
    QRows<RC> qrows;
    if (w.valid)
      rows_fetch_q<RC>(qrows, qa, w.sg.r, w.sg.h, 128 * w.sg.t, min(p.M - 128 * w.sg.t, RC),
                       warp, lane);
    int s = 0;                                  // chunks consumed (both groups')
    while (w.valid) {
      const Seg sg = w.sg;
      const int r = sg.r, h = sg.h;
      const int row0 = 128 * sg.t;              // the tile's first stacked row
      const int rows_here = min(p.M - row0, RC);
      // ---- the unit's query tile (fetched ahead): rows m < rows_here of the
      //      tile, every copy (the previous unit's MMAs reading Q and its
      //      merge are finished)
      rows_store_q<RC>(qrows, p.qk_scale, smem, rowf_s, warp, lane);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR(kBarQReady));
      if (soft_barrier_or(aborted || *abort_s)) {
        aborted = true;
        break;
      }
      // ---- this thread's row
      const bool row_ok = mrow < rows_here;
      const int ma = row0 + mrow;
      const int vis = row_ok ? min(sg.L, sg.L - p.R + 1 + ma / p.G) : 0;   // tokens it sees
      const float rowf = rowf_s[mrow];
      float m_ref = -INFINITY, lsum = 0.0f;
      int E = -126;
      // ---- chunk s's V codes -> f16 in place in its stage, the chunk's PV
      //      operand (thread L converts token L): MN-major, 128-byte swizzle,
      //      dims 64j.. in block j -- block 0 over the K codes (read by
      //      QK^T(s), complete), block 1 over the V codes, where token t's 128
      //      bytes of dims 64..127 land exactly on its own 128 code bytes (t*128
      //      = (t/8)*1024 + (t%8)*128), read before anything is written.
      //      Within a block token t sits at (t/8)*1024 + (t%8)*128, the chunk of
      //      dims 8c'.. at (c' ^ (t % 8)).  Tokens past the unit's range get
      //      zeros: their rows hold stale codes, and a NaN code would poison the
      //      product even at p = 0.
      auto convert_v = [&](int sc_, int kc_) {
        const int tv = L32;
        const bool valid = (sg.c0 + kc_) * kRwTok + tv < sg.vis;
        uint8_t *stg = smem + (sc_ % kRwStages) * kStageBytes;
        uint4 w4[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          w4[c] = make_uint4(0u, 0u, 0u, 0u);
          if (valid)
            w4[c] = *reinterpret_cast<const uint4 *>(stg + kCodeBytes + tv * kHeadDim +
                                                      ((c ^ (tv & 7)) << 4));
        }
        uint8_t *vf = stg + (tv >> 3) * 1024 + (tv & 7) * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 lo = make_uint4(
              codes2_to_f16x2<kFmt>(w4[c].x & 0xFFFFu), codes2_to_f16x2<kFmt>(w4[c].x >> 16),
              codes2_to_f16x2<kFmt>(w4[c].y & 0xFFFFu), codes2_to_f16x2<kFmt>(w4[c].y >> 16));
          const uint4 hi = make_uint4(
              codes2_to_f16x2<kFmt>(w4[c].z & 0xFFFFu), codes2_to_f16x2<kFmt>(w4[c].z >> 16),
              codes2_to_f16x2<kFmt>(w4[c].w & 0xFFFFu), codes2_to_f16x2<kFmt>(w4[c].w >> 16));
          uint8_t *blk = vf + (c >> 2) * (kVfBytes / 2);
          const int c0 = (2 * c) & 7;
          *reinterpret_cast<uint4 *>(blk + ((c0 ^ (tv & 7)) << 4)) = lo;
          *reinterpret_cast<uint4 *>(blk + (((c0 + 1) ^ (tv & 7)) << 4)) = hi;
        }
        fence_proxy_async_smem();
      };
      int mine = 0;                             // this group's chunks of the unit so far
      const int s_first = s;
      for (int k = 0; k < sg.n; ++k, ++s) {
        if ((s & 1) != gp) {
          // ---- tiles of 128 rows: the other group's chunk's V operand, while
          //      that group runs its (long) softmax; its PV waits for both.
          //      (Smaller tiles: the owner converts, after its softmax.)
          if constexpr (RC < 128) continue;
          const int b = s % kRwStages;
          bool ok = rw_wait_fast(BAR(kBarKvFull + b), (s / kRwStages) & 1, abort_s);
          ok = ok && rw_wait_fast(BAR(kBarSFull + (s & 1)), (s >> 1) & 1, abort_s);
          if (__any_sync(0xFFFFFFFFu, !ok)) {
            aborted = true;
            break;
          }
          tc_fence_after();
          convert_v(s, k);
          __syncwarp();
          if (lane == 0) mbar_arrive(BAR(kBarReady + (s & 1)));
          continue;
        }
        const int b = s % kRwStages, sb = gp;
        const int j0 = (sg.c0 + k) * kRwTok + copy * RC;   // this slice's first token
        // the stage's data, and S(s) -- QK^T(s) has completed, so the
        // stage's K codes are no longer needed
        bool ok = rw_wait_fast(BAR(kBarKvFull + b), (s / kRwStages) & 1, abort_s);
        ok = ok && rw_wait_fast(BAR(kBarSFull + sb), (s >> 1) & 1, abort_s);
        if (__any_sync(0xFFFFFFFFu, !ok)) {
          aborted = true;
          break;
        }
        tc_fence_after();
        // scales of head h for this warp's token slice, into its buffer [K | V]
        float *ts = reinterpret_cast<float *>(smem + kOffTs) + warp * 2 * kRwTok;
        {
          const float *sc = reinterpret_cast<const float *>(smem + kOffSc + b * 2 * kScBytes);
#pragma unroll
          for (int i = 0; i < RC / 32; ++i) {
            const int tk = copy * RC + lane + 32 * i;
            ts[lane + 32 * i] = sc[4 * tk + (h & 3)];
            ts[RC + lane + 32 * i] = sc[kRwTok * 4 + 4 * tk + (h & 3)];
          }
        }
        __syncwarp();
        const int lim = vis - j0;               // tokens jj < lim of the slice are seen
        const uint32_t scol = tl + RwCols<RC>::S(sb) + copy * RC;
        const uint32_t ocol = tl + kColO + 128 * gp;
        const float m0 = m_ref;                 // the references O buffer gp is under
        const int e0 = E;
        // P'' of the slice (references moved on the way where needed)
        float lchunk = 0.0f;
        uint32_t pk[RC < 128 ? RC / 2 : 1];
        const float *ks = ts, *vs = ts + RC;
        if constexpr (RC == 128) {
          rows_chunk_p_direct(scol, ks, vs, lim, rowf, m_ref, E, lchunk, lsum);
        } else {
          rows_chunk_p<RC>(scol, BAR(kBarSFree + sb), lane, ks, vs, lim, rowf, m_ref, E, lchunk,
                           lsum, pk);
          // P'' buffer gp and O buffer gp were last used by PV(s - 2)
          if (s >= 2 && __any_sync(0xFFFFFFFFu, !rw_wait_fast(BAR(kBarPvDone + sb),
                                                              ((s >> 1) - 1) & 1, abort_s))) {
            aborted = true;
            break;
          }
          tc_fence_after();
        }
        if constexpr (RC < 128) convert_v(s, k);
        // O buffer gp holds the group's earlier chunks of the unit under the
        // references of the chunk's start: brought to the present ones if they
        // moved (no MMA in flight on it: PV(s - 2) has completed)
        if (mine > 0 && __any_sync(0xFFFFFFFFu, m_ref != m0 || E != e0))
          rows_rescale_o(ocol, (m0 == -INFINITY) ? 0.0f : rw_ex2(m0 - m_ref) * pow2f_down(e0 - E));
        lsum += lchunk;
        // this slice's P'' columns of buffer gp (the others stay zero)
        if constexpr (RwCols<RC>::kSplitP) {
          const uint32_t pbase = tl + RwCols<RC>::P(sb) + copy * (RC / 2);
#pragma unroll
          for (int c = 0; c < RC / 2; c += 16) {
            uint32_t w16[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) w16[i] = pk[c + i];
            tmem_st16u(pbase + c, w16);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(BAR(kBarReady + sb));
        ++mine;
      }
      // ---- the next unit's query rows into registers: their loads overlap
      //      this unit's epilogue
      w.advance_segment(pre, p.context_lens, geo, N);
      if (w.valid)
        rows_fetch_q<RC>(qrows, qa, w.sg.r, w.sg.h, 128 * w.sg.t, min(p.M - 128 * w.sg.t, RC),
                         warp, lane);
      // ---- the unit's piece: wait for its last PV (the MMAs complete in order)
      if (!aborted && sg.n > 0) {
        const int se = s_first + sg.n - 1;
        if (!rw_wait_fast(BAR(kBarPvDone + (se & 1)), (se >> 1) & 1, abort_s)) aborted = true;
      }
      if (soft_barrier_or(aborted || *abort_s)) {
        aborted = true;
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(BAR(kBarOFree));
        break;
      }
      tc_fence_after();
      // ---- merge each row's partial results -- kRwGroups x kCopies of them
      //      (group, token slice) -- exchanging (m, l, E); group 0 then reads
      //      both groups' O buffers and sums the slices through shared memory
      //      (the query tile's space, idle until the next unit)
      constexpr int kParts = kRwGroups * kCopies;
      ml_s[gp * 128 + L32] = make_float4(m_ref, lsum, static_cast<float>(E), 0.0f);
      soft_barrier();
      float m_all = -INFINITY;
      int e_all = -126;
#pragma unroll
      for (int c = 0; c < kParts; ++c) {
        const float4 v = ml_s[(c / kCopies) * 128 + (c % kCopies) * RC + mrow];
        m_all = fmaxf(m_all, v.x);
        if (v.x != -INFINITY) e_all = max(e_all, static_cast<int>(v.z));
      }
      float l_all = 0.0f;
#pragma unroll
      for (int c = 0; c < kParts; ++c) {
        const float4 v = ml_s[(c / kCopies) * 128 + (c % kCopies) * RC + mrow];
        if (v.x != -INFINITY) l_all += rw_ex2(v.x - m_all) * v.y;
      }
      const bool writer = gp == 0 && (copy == kCopies - 1) && row_ok;
      const bool direct = (sg.c0 == 0 && sg.n == sg.C);
      const float vsc = pow2f(e_all);           // undo the 2^-E of P''
      const int ir = ma / p.G, gq = ma - ir * p.G;
      const int64_t orow = (static_cast<int64_t>(r) * p.R + ir) * p.Hq + h * p.G + gq;
      const int b_first = static_cast<int>(sg.first / B);
      const int slot = 2 * static_cast<int>(blockIdx.x) +
                       (static_cast<int>(blockIdx.x) == b_first ? 1 : 0);
      const float inv = (l_all > 0.0f) ? vsc / l_all : 0.0f;
      if (gp == 0) {
        // this lane's rows of both O buffers under the unit's references (a
        // buffer a group did not write in this unit -- one chunk -- is not read)
        const float4 v1 = ml_s[128 + L32];
        const float f0 = (m_ref == -INFINITY) ? 0.0f
                                              : rw_ex2(m_ref - m_all) * pow2f_down(E - e_all);
        const float f1 = (v1.x == -INFINITY)
                             ? 0.0f
                             : rw_ex2(v1.x - m_all) * pow2f_down(static_cast<int>(v1.z) - e_all);
        const bool has0 = mine > 0;
        const bool has1 = sg.n + (s_first & 1) >= 2;   // group 1 had a chunk of the unit
        // 32 dims of this lane's row from both buffers, under the unit's
        // references
        auto o_rows = [&](int d0, float (&o)[32]) {
          if (has0) {
            tmem_ld32(tl + kColO + d0, o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] *= f0;
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = 0.0f;
          }
          if (has1) {
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              float o2[16];
              tmem_ld16(tl + kColO + 128 + d0 + 16 * hh, o2);
#pragma unroll
              for (int i = 0; i < 16; ++i) o[16 * hh + i] = fmaf(o2[i], f1, o[16 * hh + i]);
            }
          }
        };
        if constexpr (kCopies == 1) {
          // one slice: the thread holds its whole row
#pragma unroll 1
          for (int pc = 0; pc < 4; ++pc) {
            float o[32];
            o_rows(32 * pc, o);
            if (row_ok) {
              if (direct) {
                uint4 *dst = reinterpret_cast<uint4 *>(p.out + orow * kHeadDim + 32 * pc);
#pragma unroll
                for (int c8 = 0; c8 < 4; ++c8)
                  dst[c8] = make_uint4(pack_bf16x2(o[8 * c8] * inv, o[8 * c8 + 1] * inv),
                                       pack_bf16x2(o[8 * c8 + 2] * inv, o[8 * c8 + 3] * inv),
                                       pack_bf16x2(o[8 * c8 + 4] * inv, o[8 * c8 + 5] * inv),
                                       pack_bf16x2(o[8 * c8 + 6] * inv, o[8 * c8 + 7] * inv));
              } else {
                float4 *dst = reinterpret_cast<float4 *>(
                    p.o_part + (static_cast<int64_t>(slot) * RC + mrow) * kHeadDim + 32 * pc);
#pragma unroll
                for (int c4 = 0; c4 < 8; ++c4)
                  dst[c4] = make_float4(o[4 * c4] * vsc, o[4 * c4 + 1] * vsc,
                                        o[4 * c4 + 2] * vsc, o[4 * c4 + 3] * vsc);
              }
            }
          }
        } else {
          // the slices' rows through shared memory (the query tile's space),
          // 64 dims at a time: every thread puts its row's dims there, then
          // sums the slices over kSl of them for its row and writes those
          constexpr int kSl = 64 / kCopies;
          float *xs = reinterpret_cast<float *>(smem + kOffQ);   // [copy][64 dims][RC]
#pragma unroll 1
          for (int half = 0; half < 2; ++half) {
            // (both 32-dim reads of a half unrolled: verify 904 vs 909 us)
#pragma unroll
            for (int pc = 0; pc < 2; ++pc) {
              float o[32];
              o_rows(64 * half + 32 * pc, o);
#pragma unroll
              for (int i = 0; i < 32; ++i) xs[(copy * 64 + 32 * pc + i) * RC + mrow] = o[i];
            }
            group0_barrier();
            float a[kSl];
#pragma unroll
            for (int j = 0; j < kSl; ++j) {
              float t = 0.0f;
#pragma unroll
              for (int c = 0; c < kCopies; ++c) t += xs[(c * 64 + copy * kSl + j) * RC + mrow];
              a[j] = t;
            }
            const int d0 = 64 * half + copy * kSl;
            if (row_ok) {
              if (direct) {
                uint4 *dst = reinterpret_cast<uint4 *>(p.out + orow * kHeadDim + d0);
#pragma unroll
                for (int c8 = 0; c8 < kSl / 8; ++c8)
                  dst[c8] = make_uint4(pack_bf16x2(a[8 * c8] * inv, a[8 * c8 + 1] * inv),
                                       pack_bf16x2(a[8 * c8 + 2] * inv, a[8 * c8 + 3] * inv),
                                       pack_bf16x2(a[8 * c8 + 4] * inv, a[8 * c8 + 5] * inv),
                                       pack_bf16x2(a[8 * c8 + 6] * inv, a[8 * c8 + 7] * inv));
              } else {
                float4 *dst = reinterpret_cast<float4 *>(
                    p.o_part + (static_cast<int64_t>(slot) * RC + mrow) * kHeadDim + d0);
#pragma unroll
                for (int c4 = 0; c4 < kSl / 4; ++c4)
                  dst[c4] = make_float4(a[4 * c4] * vsc, a[4 * c4 + 1] * vsc,
                                        a[4 * c4 + 2] * vsc, a[4 * c4 + 3] * vsc);
              }
            }
            group0_barrier();                   // (before the next half overwrites xs)
          }
        }
      }
      // the O rows have been read (group 1's arrival only counts): the next
      // unit's PVs may overwrite them
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR(kBarOFree));
      if (!direct) {
        // a piece: slot 1 of this CTA if the unit continues past its range
        // (its first CTA), else slot 0; the piece that lands last merges
        if (writer) {
          p.ml_part[static_cast<int64_t>(slot) * RC + mrow] = make_float2(m_all, l_all);
          __threadfence();
        }
        soft_barrier();
        const int b_last = static_cast<int>((sg.first + sg.C - 1) / B);
        const int64_t unit = (static_cast<int64_t>(r) * p.H + h) * p.T + sg.t;
        if (tid == 0) {
          const uint32_t landed = ticket_take(p.tickets + unit, p.tag);
          const bool last = landed == static_cast<uint32_t>(b_last - b_first + 1);
          *ticket_s = last ? 1 : 0;
          if (last) p.tickets[unit] = 0ull;
          if (landed == 0u && p.err_flags) atomicOr(p.err_flags, KVQ_ERRF_WAIT_TIMEOUT);
          __threadfence();
        }
        soft_barrier();
        if (*ticket_s) {
          // every piece of the unit: warp per row, lane per 4 dims, running
          // log-sum-exp over the pieces
          for (int m = warp; m < rows_here; m += kRwGroupWarps) {
            float mw = -INFINITY, ls = 0.0f;
            float4 a4 = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int bb = b_first; bb <= b_last; ++bb) {
              const int sl = 2 * bb + (bb == b_first ? 1 : 0);
              const float2 v = __ldcg(p.ml_part + static_cast<int64_t>(sl) * RC + m);
              const float4 o4 = __ldcg(reinterpret_cast<const float4 *>(
                  p.o_part + (static_cast<int64_t>(sl) * RC + m) * kHeadDim) + lane);
              if (v.x == -INFINITY) continue;
              const float mn = fmaxf(mw, v.x);
              const float fa = rw_ex2(mw - mn), fb = rw_ex2(v.x - mn);
              ls = ls * fa + v.y * fb;
              a4.x = a4.x * fa + o4.x * fb;
              a4.y = a4.y * fa + o4.y * fb;
              a4.z = a4.z * fa + o4.z * fb;
              a4.w = a4.w * fa + o4.w * fb;
              mw = mn;
            }
            const float iv = (ls > 0.0f) ? 1.0f / ls : 0.0f;
            const int mab = row0 + m, i2 = mab / p.G, g2 = mab - i2 * p.G;
            const int64_t orw = (static_cast<int64_t>(r) * p.R + i2) * p.Hq + h * p.G + g2;
            *reinterpret_cast<uint2 *>(p.out + orw * kHeadDim + 4 * lane) =
                make_uint2(pack_bf16x2(a4.x * iv, a4.y * iv), pack_bf16x2(a4.z * iv, a4.w * iv));
          }
        }
      }
      soft_barrier();                           // the merge scratch is free again
    }
    if (aborted && lane == 0 && p.err_flags) atomicOr(p.err_flags, KVQ_ERRF_WAIT_TIMEOUT);
    if (aborted) *abort_s = 1;
    // units whose rows see no token: zero rows, spread over the grid
    if (!aborted) {
      const int n_units = N * p.H * p.T;
      for (int u = blockIdx.x * kRwGroupWarps + warp; u < n_units;
           u += gridDim.x * kRwGroupWarps) {
        const int t = u % p.T, rh = u / p.T, h = rh % p.H, r = rh / p.H;
        const int L = clamp_len(p.context_lens[r], p.ctx_limit);
        if (tile_tokens(geo, L, t) > 0) continue;
        const int rows = min(p.M - 128 * t, 128);
        for (int m = 0; m < rows; ++m) {
          const int ma = 128 * t + m, ir = ma / p.G, gq = ma - ir * p.G;
          const int64_t orow = (static_cast<int64_t>(r) * p.R + ir) * p.Hq + h * p.G + gq;
          *reinterpret_cast<uint2 *>(p.out + orow * kHeadDim + 4 * lane) = make_uint2(0u, 0u);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kRwWarpTma) {
    tc_fence_after();
    tmem_dealloc(tmem, kRwTmemCols);
  }
}

}  // namespace

int32_t attn_rows_per_tile(int32_t rows) { return rows <= 32 ? 32 : (rows <= 64 ? 64 : 128); }

bool attn_rows_supported(const kvq_cache &c, const AttnShape &s) {
  const int bs = 1 << s.log2_block;
  return s.rows >= 1 && bs >= 16 && c.num_kv_heads % 4 == 0 && c.num_slots > 0 &&
         c.num_slots < (int64_t(1) << 31) && s.num_requests <= kRowsMaxRequests &&
         (reinterpret_cast<uintptr_t>(c.k_scales) & 15u) == 0 &&
         (reinterpret_cast<uintptr_t>(c.v_scales) & 15u) == 0;
}

size_t attn_rows_workspace_bytes(const AttnShape &s, int32_t num_kv_heads) {
  const int64_t T = (s.rows + 127) / 128;
  const int64_t units = static_cast<int64_t>(s.num_requests) * num_kv_heads * T;
  const int64_t rc = attn_rows_per_tile(s.rows);
  const int64_t grid = s.sms > 0 ? s.sms : 152;
  const size_t tickets = (static_cast<size_t>(units) * 8 + 255) / 256 * 256;
  const size_t o = static_cast<size_t>(grid) * 2 * rc * kHeadDim * sizeof(float);
  const size_t ml = static_cast<size_t>(grid) * 2 * rc * sizeof(float2);
  return tickets + (o + 255) / 256 * 256 + (ml + 255) / 256 * 256;
}

cudaError_t launch_attn_rows(const kvq_cache &c, const AttnShape &s, const void *q,
                             const int32_t *block_tables, const int32_t *context_lens,
                             float sm_scale, void *out, void *workspace, int32_t *err_flags,
                             cudaStream_t stream, int32_t code_format) {
  RwParams p;
  p.num_blocks = static_cast<uint32_t>(c.num_slots >> s.log2_block);
  p.H = c.num_kv_heads;
  p.log2_bs = s.log2_block;
  p.box = (1 << s.log2_block) < kRwTok ? (1 << s.log2_block) : kRwTok;
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
  p.T = (s.rows + 127) / 128;
  p.qk_scale = sm_scale * 1.4426950408889634f;
  const int64_t units = static_cast<int64_t>(s.num_requests) * c.num_kv_heads * p.T;
  const int rc = attn_rows_per_tile(s.rows);
  const int grid = s.sms > 0 ? s.sms : 152;
  char *ws = static_cast<char *>(workspace);
  p.tickets = reinterpret_cast<unsigned long long *>(ws);
  p.tag = next_call_tag();
  ws += (static_cast<size_t>(units) * 8 + 255) / 256 * 256;
  p.o_part = reinterpret_cast<float *>(ws);
  ws += (static_cast<size_t>(grid) * 2 * rc * kHeadDim * sizeof(float) + 255) / 256 * 256;
  p.ml_part = reinterpret_cast<float2 *>(ws);
  p.err_flags = err_flags;
  CUtensorMap mkc, mvc, mks, mvs;
  if (!encode_code_tensor_map(&mkc, c.k_codes, c.num_slots, c.num_kv_heads, p.box) ||
      !encode_code_tensor_map(&mvc, c.v_codes, c.num_slots, c.num_kv_heads, p.box) ||
      !encode_scale_tensor_map(&mks, c.k_scales, c.num_slots, c.num_kv_heads, p.box) ||
      !encode_scale_tensor_map(&mvs, c.v_scales, c.num_slots, c.num_kv_heads, p.box))
    return cudaErrorInvalidValue;
  using Kernel = void (*)(RwParams, CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap);
  const bool e5 = code_format == KVQ_CODES_E5M2;
  const Kernel kernel =
      rc == 32 ? (e5 ? attn_rows_kernel<32, KVQ_CODES_E5M2> : attn_rows_kernel<32, KVQ_CODES_E4M3>)
      : rc == 64 ? (e5 ? attn_rows_kernel<64, KVQ_CODES_E5M2> : attn_rows_kernel<64, KVQ_CODES_E4M3>)
                 : (e5 ? attn_rows_kernel<128, KVQ_CODES_E5M2>
                       : attn_rows_kernel<128, KVQ_CODES_E4M3>);
  static std::atomic<uint64_t> configured[6];
  const int which = (rc == 32 ? 0 : (rc == 64 ? 1 : 2)) + (e5 ? 3 : 0);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = (dev >= 0 && dev < 64) ? (uint64_t(1) << dev) : 0;
  if (bit == 0 || !(configured[which].load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kRwSmem);
    if (e != cudaSuccess) return e;
    configured[which].fetch_or(bit, std::memory_order_acq_rel);
  }
  return launch_overlapped(kernel, dim3(grid), dim3(kRwThreads), kRwSmem, stream, p, mkc, mvc,
                           mks, mvs);
}

}  // namespace kvq
