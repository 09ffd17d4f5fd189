// kvq_attention.cu -- paged GQA decode / multi-row verify attention over the
// FP8 E4M3 cache: split-K partials on the tensor cores, then a combine pass.
//
// ROCm/ATOM PR #2655 "fix(qwen4-exp): register the QSA FP8 scale planes for KV
// offload", PR description:
//  * K/V bullet: attention runs on the E4M3 tiles themselves; a token's key
//    scale is applied to its score after the code dot product, and its value
//    scale to its probability ahead of the PV product;
//  * stacked decode scorer: all query rows of a verify step (4 of them) and
//    all heads reading the same keys go into one MMA operand, so each key tile
//    is loaded once per step for every one of those rows.
// sgl-project/sglang-jax #1776 "feat(dsa): implement fp8 KV cache (e4m3) with
// a bf16 indexer cache", Modifications: the cached block is upcast to the query
// dtype before the score dot, and P is never rounded to fp8.
//
// Work decomposition.  One CTA = (KV head h, row group, context partition p,
// request r).  The CTA's M rows are the (query row i, head g) pairs of request r
// that read KV head h, stacked as m = i*G + g (at most 32 per row group: one or
// two m16 tiles).  Four warps stream the partition's tokens through a 3-stage
// cp.async pipeline of 64-token stages (16 tokens per warp per stage); each
// token's 128-byte code rows are found through the block table.  Per 16-token
// chunk a warp:
//   1. runs S = Q K^T on the FP8 tensor cores (m16n8k32 e4m3, fp32
//      accumulate) with the K code bytes themselves as B fragments -- no
//      decode -- against Q split into two e4m3 pieces per element, q =
//      2^e (p1 + p2), exact for elements >= 2^-9 of the row's largest and off
//      by at most 2^-17 of it below that;
//   2. multiplies each score column by its key scale and sm_scale*log2(e),
//      masks causally (row i sees tokens j < L - R + 1 + i), and updates a
//      running max per row, rescaling the accumulators only when the max grows
//      by more than 2^8 (so p <= 256);
//   3. folds the value scale into p (P' = p * v_scale * 2^-E, rounded once to
//      f16, where 2^E is a running power-of-two bound on the v_scales the warp
//      has seen, so P' <= 256 always fits f16), accumulates the denominator
//      with the unscaled p, and runs O += P' V with f16 MMAs on V codes decoded
//      exactly to f16 (value * 2^-8; the 2^(E+8) is applied once at the end).
//      f16 keeps 11 mantissa bits of P' where bf16 keeps 8: with the outputs'
//      cancellation between large terms, bf16 P' alone costs up to ~1.6%
//      elementwise, f16 about the output's own bf16 rounding.
// The warps' (max, denominator, O) are merged through shared memory; a request
// with a single partition writes its bf16 output directly, otherwise the
// partial is stored and the combine kernel merges the partitions (log-sum-exp
// weights).
//
// The contraction index of Q K^T is permuted so that each lane's B fragments
// are two words of its token's code row: in k32-step s2, the lane with
// c = lane % 4 feeds dims 32c + 8 s2 + 0..3 as k = 4c..4c+3 and dims
// 32c + 8 s2 + 4..7 as k = 4c+16..4c+19; Q's A fragments use the same map.  For P V the output columns are
// permuted instead: n-tile i, column u stands for dim 16u + i, so each lane
// reads 16 consecutive code bytes per token.  Shared-memory code rows are
// stored with their 16-byte chunks XOR-swizzled by (token & 7), which keeps
// both read patterns free of bank conflicts.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstring>

#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {

namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kStageTok = 64;
constexpr int kStages = 3;
constexpr int kGroupRows = 32;
constexpr float kLazyRescale = 8.0f;   // rescale only when the max grows by > 2^8
constexpr float kLog2e = 1.4426950408889634f;

// Shared memory, from a 1024-byte aligned base (the TMA 128-byte swizzle
// pattern repeats every 1024 bytes):
//   K code stages  kStages x 64 rows x 128 B   (row = one token of one head)
//   V code stages  kStages x 64 rows x 128 B
//   K, V scales    kStages x 64 fp32 each
//   Q fragments    MT x 8 x 32 uint4
//   block ids      kMaxPages int32          (TMA staging only)
//   mbarriers      kStages x 8 B            (TMA staging only)
//   row exponents  32 fp32                  (2^e_m of each query row)
// Within a code row the 16-byte chunk c of token row t sits at chunk c ^ (t & 7).
constexpr int kCodeStage = kStageTok * kHeadDim;                 // 8 KiB
constexpr int kOffK = 0;
constexpr int kOffV = kStages * kCodeStage;
constexpr int kOffKs = 2 * kStages * kCodeStage;
constexpr int kOffVs = kOffKs + kStages * kStageTok * 4;
constexpr int kOffQ = kOffVs + kStages * kStageTok * 4;
constexpr int kMaxPages = 1024;
constexpr int kMinTmaBlock = 8;    // a page box of >= 8 rows keeps 1024-byte alignment

__host__ __device__ constexpr int off_bt(int mt) { return kOffQ + mt * 8 * 32 * 16; }
__host__ __device__ constexpr int off_mbar(int mt) { return off_bt(mt) + kMaxPages * 4; }
__host__ __device__ constexpr int off_rowexp(int mt) { return off_mbar(mt) + kStages * 8; }
__host__ __device__ constexpr int smem_bytes(int mt) { return off_rowexp(mt) + 32 * 4 + 1024; }

struct AttnParams {
  const uint8_t *k_codes;
  const uint8_t *v_codes;
  const float *k_scales;
  const float *v_scales;
  int64_t num_blocks;
  int32_t H;
  int32_t log2_bs;
  const uint16_t *q;
  uint16_t *out;
  const int32_t *block_tables;
  int32_t max_blocks;
  const int32_t *context_lens;
  int32_t ctx_limit;        // min(max_context_len, max_blocks << log2_bs)
  int32_t R, Hq, G, M;
  int32_t row_groups;
  float qk_scale;           // sm_scale * log2(e)
  int32_t part_tokens;
  int32_t n_parts_max;
  float *o_part;
  float2 *ml_part;
  int32_t *err_flags;
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint4 lds128(const void *p) {
  return *reinterpret_cast<const uint4 *>(p);
}

__device__ __forceinline__ int clamp_context(const AttnParams &p, int r, bool report) {
  int L = p.context_lens[r];
  if (L < 0 || L > p.ctx_limit) {
    if (report && p.err_flags) atomicOr(p.err_flags, KVQ_ERRF_CONTEXT_RANGE);
    L = L < 0 ? 0 : p.ctx_limit;
  }
  return L;
}

// Issue the cp.async copies of one 64-token stage (tokens [tok0, tok0+64) of
// the request; those at or past t_end are zero-filled).  Used when the block
// size is below kMinTmaBlock.
__device__ __forceinline__ void issue_stage_cp(const AttnParams &p, uint8_t *kdst,
                                               uint8_t *vdst, float *ksd, float *vsd, int r,
                                               int h, int tok0, int t_end, int tid) {
  const int32_t *bt = p.block_tables + static_cast<int64_t>(r) * p.max_blocks;
  const int bs_mask = (1 << p.log2_bs) - 1;
  // code rows: 128 rows (64 K then 64 V) x 8 chunks of 16 bytes; thread tid
  // copies chunk tid%8 of rows tid/8 + 16*it, so 8 consecutive lanes move one
  // full 128-byte row.
  const int chunk = tid & 7;
#pragma unroll
  for (int it = 0; it < 8; ++it) {
    const int row = (tid >> 3) + 16 * it;
    const int tl = row & (kStageTok - 1);
    const bool is_v = row >= kStageTok;
    const int j = tok0 + tl;
    const uint8_t *base = is_v ? p.v_codes : p.k_codes;
    const uint8_t *src = base;
    uint32_t nbytes = 0;
    if (j < t_end) {
      const int64_t blk = bt[j >> p.log2_bs];
      if (blk >= 0 && blk < p.num_blocks) {
        const int64_t slot = (blk << p.log2_bs) + (j & bs_mask);
        src = base + (slot * p.H + h) * kHeadDim + chunk * 16;
        nbytes = 16;
      } else if (p.err_flags) {
        atomicOr(p.err_flags, KVQ_ERRF_BLOCK_RANGE);
      }
    }
    uint8_t *dst = (is_v ? vdst : kdst) + tl * kHeadDim + ((chunk ^ (tl & 7)) << 4);
    cp_async_16(dst, src, nbytes);
  }
  // scales: thread tid copies token tid%64's K (tid < 64) or V scale
  {
    const int tl = tid & (kStageTok - 1);
    const bool is_v = tid >= kStageTok;
    const int j = tok0 + tl;
    const float *base = is_v ? p.v_scales : p.k_scales;
    const float *src = base;
    uint32_t nbytes = 0;
    if (j < t_end) {
      const int64_t blk = bt[j >> p.log2_bs];
      if (blk >= 0 && blk < p.num_blocks) {
        const int64_t slot = (blk << p.log2_bs) + (j & bs_mask);
        src = base + slot * p.H + h;
        nbytes = 4;
      }
    }
    cp_async_4((is_v ? vsd : ksd) + tl, src, nbytes);
  }
}

// Issue one 64-token stage with TMA: thread 0 copies each page's 128-byte code
// rows of KV head h (a box of min(bs, 64) rows) for K and for V, completing on
// the stage's mbarrier; every thread copies one scale with cp.async.  Block
// ids come from the partition's copy in shared memory (bt_s, first page
// page0).  Pages at or past t_end, or with an out-of-range block id, are not
// copied; their scales are zero-filled so the compute stays finite.
__device__ __forceinline__ void issue_stage_tma(const AttnParams &p, const void *tmap_k,
                                                const void *tmap_v, uint32_t kdst,
                                                uint32_t vdst, float *ksd, float *vsd,
                                                uint32_t bar, const int32_t *bt_s, int page0,
                                                int h, int tok0, int t_end, int tid) {
  const int bs_mask = (1 << p.log2_bs) - 1;
  if (tid == 0) {
    const int rows = p.log2_bs >= 6 ? kStageTok : (1 << p.log2_bs);
    uint32_t bytes = 0;
    bool bad = false;
    fence_proxy_async_smem();   // earlier generic reads of this buffer come first
    for (int i = 0; i < kStageTok / rows; ++i) {
      const int j = tok0 + i * rows;
      if (j >= t_end) break;
      const int64_t blk = bt_s[(j >> p.log2_bs) - page0];
      if (blk < 0 || blk >= p.num_blocks) {
        bad = true;
        continue;
      }
      const int z = static_cast<int>((blk << p.log2_bs) + (j & bs_mask));
      tma_load_3d(kdst + i * rows * kHeadDim, tmap_k, 0, h, z, bar);
      tma_load_3d(vdst + i * rows * kHeadDim, tmap_v, 0, h, z, bar);
      bytes += 2u * rows * kHeadDim;
    }
    if (bad && p.err_flags) atomicOr(p.err_flags, KVQ_ERRF_BLOCK_RANGE);
    mbar_arrive_expect_tx(bar, bytes);
  }
  {
    const int tl = tid & (kStageTok - 1);
    const bool is_v = tid >= kStageTok;
    const int j = tok0 + tl;
    const float *base = is_v ? p.v_scales : p.k_scales;
    const float *src = base;
    uint32_t nbytes = 0;
    if (j < t_end) {
      const int64_t blk = bt_s[(j >> p.log2_bs) - page0];
      if (blk >= 0 && blk < p.num_blocks) {
        src = base + ((blk << p.log2_bs) + (j & bs_mask)) * p.H + h;
        nbytes = 4;
      }
    }
    cp_async_4((is_v ? vsd : ksd) + tl, src, nbytes);
  }
}

template <int MT, bool kTma>
__global__ void __launch_bounds__(kThreads, (MT == 1) ? 3 : 2)
attn_partials_kernel(const AttnParams p, const __grid_constant__ CUtensorMap tmap_k,
                     const __grid_constant__ CUtensorMap tmap_v) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint4 *qfrag = reinterpret_cast<uint4 *>(smem + kOffQ);
  int32_t *bt_s = reinterpret_cast<int32_t *>(smem + off_bt(MT));
  uint64_t *mbar = reinterpret_cast<uint64_t *>(smem + off_mbar(MT));
  __shared__ int timed_out;

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int g4 = lane >> 2;
  const int c4 = lane & 3;
  const int h = blockIdx.x / p.row_groups;
  const int row_base = (blockIdx.x - h * p.row_groups) * kGroupRows;
  const int part = blockIdx.y;
  const int r = blockIdx.z;

  grid_dependency_wait();
  allow_dependents_launch();
  const int L = clamp_context(p, r, part == 0 && tid == 0 && blockIdx.x == 0);
  const int n_parts = (L + p.part_tokens - 1) / p.part_tokens;
  if (part >= (n_parts > 0 ? n_parts : 1)) return;
  const int t0 = part * p.part_tokens;
  const int t_end = min(L, t0 + p.part_tokens);
  const int n_stages = (t_end > t0) ? (t_end - t0 + kStageTok - 1) / kStageTok : 0;
  const int page0 = t0 >> p.log2_bs;

  auto kst = [&](int b) { return smem + kOffK + b * kCodeStage; };
  auto vst = [&](int b) { return smem + kOffV + b * kCodeStage; };
  auto kss = [&](int b) { return reinterpret_cast<float *>(smem + kOffKs) + b * kStageTok; };
  auto vss = [&](int b) { return reinterpret_cast<float *>(smem + kOffVs) + b * kStageTok; };
  auto issue = [&](int s) {
    const int b = s % kStages;
    if constexpr (kTma) {
      issue_stage_tma(p, &tmap_k, &tmap_v, smem_addr(kst(b)), smem_addr(vst(b)), kss(b), vss(b),
                      smem_addr(&mbar[b]), bt_s, page0, h, t0 + s * kStageTok, t_end, tid);
    } else {
      issue_stage_cp(p, kst(b), vst(b), kss(b), vss(b), r, h, t0 + s * kStageTok, t_end, tid);
    }
  };

  if constexpr (kTma) {
    // the partition's block ids, once; then the barriers
    const int n_pages = (t_end > t0) ? ((t_end - 1) >> p.log2_bs) - page0 + 1 : 0;
    const int32_t *bt = p.block_tables + static_cast<int64_t>(r) * p.max_blocks + page0;
    for (int i = tid; i < n_pages; i += kThreads) bt_s[i] = bt[i];
    if (tid == 0) {
      timed_out = 0;
      for (int b = 0; b < kStages; ++b) mbar_init(smem_addr(&mbar[b]), 1);
      fence_mbarrier_init();
      fence_proxy_async_smem();
    }
    __syncthreads();
  }

  // Start the pipeline before anything else.
#pragma unroll
  for (int s = 0; s < kStages - 1; ++s) {
    if (s < n_stages) issue(s);
    cp_async_commit();
  }

  // Q as two e4m3 pieces per element, stored per lane in fragment order.
  // Row m is scaled by 2^-e_m (e_m from the row's largest |q|, so the largest
  // scaled element lies in [128, 256)); p1 = e4m3_rne(x) and p2 = e4m3_rne(x -
  // p1).  x has 8 significant bits and p1 keeps the top 4, so the residual is a
  // multiple of x's ulp no larger than 8 ulps, and p2 holds it exactly when
  // that ulp is at least e4m3's smallest step 2^-9, i.e. for |x| >= 2^-2 (every
  // element >= 2^-9 of the row's largest).  For smaller elements p2 rounds to
  // the 2^-9 grid: q = 2^e_m (p1 + p2) is then off by at most 2^-10 2^e_m,
  // which is at most 2^-17 of the row's largest.  2^e_m multiplies the row's
  // scores later.
  float *row_exp = reinterpret_cast<float *>(smem + off_rowexp(MT));   // [MT * 16]
  const int rows_here = min(MT * 16, p.M - row_base);
  auto q_row = [&](int m) {   // m < rows_here
    const int mg = row_base + m;
    const int i = mg / p.G, gq = mg - i * p.G;
    return p.q + ((static_cast<int64_t>(r) * p.R + i) * p.Hq + h * p.G + gq) * kHeadDim;
  };
  // (a) row exponents
  for (int m = warp; m < MT * 16; m += kWarps) {
    float amax = 0.0f;
    if (m < rows_here) {
      const uint2 v = *reinterpret_cast<const uint2 *>(q_row(m) + 4 * lane);
      amax = fmaxf(fmaxf(fabsf(bf16_lo(v.x)), fabsf(bf16_hi(v.x))),
                   fmaxf(fabsf(bf16_lo(v.y)), fabsf(bf16_hi(v.y))));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
      amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, off));
    if (lane == 0) {
      // exponent e with 2^(e+7) <= amax < 2^(e+8), clamped so 2^-e is normal
      const int ex = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFFu);
      int e = (ex == 0) ? -126 : ex - 127 - 7;
      e = e < -126 ? -126 : (e > 126 ? 126 : e);
      row_exp[m] = (amax == 0.0f) ? 0.0f : __int_as_float((127 + e) << 23);   // 2^e
    }
  }
  __syncthreads();
  // (b) the two pieces of every element of the real rows, in row order, into
  // the last stage's code buffers (not written by any copy before the main
  // loop starts): plane 1 in the K buffer, plane 2 in the V buffer
  uint8_t *plane1 = kst(kStages - 1);
  uint8_t *plane2 = vst(kStages - 1);
  for (int idx = tid; idx < MT * 16 * 32; idx += kThreads) {
    const int m = idx >> 5, qd = idx & 31;
    uint32_t c1w = 0u, c2w = 0u;
    if (m < rows_here && row_exp[m] != 0.0f) {
      const uint2 v = *reinterpret_cast<const uint2 *>(q_row(m) + 4 * qd);
      const float inv = __int_as_float((254u << 23) - __float_as_uint(row_exp[m]));   // 2^-e
      const float xs[4] = {bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y)};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float x = xs[e] * inv;
        const uint32_t c1 = e4m3_round(x, x);
        const float res = x - e4m3_to_f32(c1);
        c1w |= c1 << (8 * e);
        c2w |= e4m3_round(res, res) << (8 * e);
      }
    }
    *reinterpret_cast<uint32_t *>(plane1 + m * kHeadDim + 4 * qd) = c1w;
    *reinterpret_cast<uint32_t *>(plane2 + m * kHeadDim + 4 * qd) = c2w;
  }
  __syncthreads();
  // (c) fragments: dims 32c + 8 s2 + 0..3 are k = 4c..4c+3, dims + 4..7 are
  // k = 4c+16..4c+19
  for (int idx = warp; idx < MT * 4; idx += kWarps) {
    const int mt = idx >> 2, s2 = idx & 3;
    const int off = 32 * c4 + 8 * s2;
#pragma unroll
    for (int pc = 0; pc < 2; ++pc) {
      const uint8_t *pl = pc ? plane2 : plane1;
      const uint2 a = *reinterpret_cast<const uint2 *>(pl + (mt * 16 + g4) * kHeadDim + off);
      const uint2 b = *reinterpret_cast<const uint2 *>(pl + (mt * 16 + g4 + 8) * kHeadDim + off);
      qfrag[((mt * 4 + s2) * 2 + pc) * 32 + lane] = make_uint4(a.x, b.x, a.y, b.y);
    }
  }
  float rowf[MT][2];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) rowf[mt][hf] = row_exp[mt * 16 + g4 + 8 * hf];

  // Per-thread rows: (mt, half) -> M row row_base + mt*16 + g4 + 8*half.
  int vis[MT][2];
  float m_run[MT][2], l_run[MT][2];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      const int m = row_base + mt * 16 + g4 + 8 * hf;
      vis[mt][hf] = (m < p.M) ? (L - p.R + 1 + m / p.G) : 0;
      m_run[mt][hf] = -INFINITY;
      l_run[mt][hf] = 0.0f;
    }
  float o[MT][16][4];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int i = 0; i < 16; ++i)
#pragma unroll
      for (int e = 0; e < 4; ++e) o[mt][i][e] = 0.0f;
  // running exponent E: every v_scale this warp has folded so far is <= 2^E
  // (warp-uniform; -1000 = none yet; otherwise clamped to [-126, 126])
  int ev = -1000;

  for (int st = 0; st < n_stages; ++st) {
    cp_async_wait<kStages - 2>();
    if constexpr (kTma) {
      if (!mbar_wait_bounded(smem_addr(&mbar[st % kStages]), (st / kStages) & 1))
        timed_out = 1;
    }
    __syncthreads();
    if constexpr (kTma) {
      if (timed_out) {
        // give up on this CTA: report, let the copies in flight land (bounded),
        // and leave without writing outputs
        if (tid == 0) {
          if (p.err_flags) atomicOr(p.err_flags, KVQ_ERRF_WAIT_TIMEOUT);
          for (int s2 = st; s2 < min(n_stages, st + kStages - 1); ++s2)
            mbar_wait_bounded(smem_addr(&mbar[s2 % kStages]), (s2 / kStages) & 1);
        }
        cp_async_wait<0>();
        return;
      }
    }
    {
      const int nxt = st + kStages - 1;
      if (nxt < n_stages) issue(nxt);
      cp_async_commit();
    }
    const int sbuf = st % kStages;
    const uint8_t *sb_k = kst(sbuf);
    const uint8_t *sb_v = vst(sbuf);
    const float *sb_ks = kss(sbuf);
    const float *sb_vs = vss(sbuf);
    const int tb = warp * 16;                         // this warp's 16 tokens
    const int jbase = t0 + st * kStageTok + tb;       // request position of token tb

    // ---- S = Q K^T over this warp's 16 tokens (two n-tiles of 8)
    float sacc[MT][2][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) sacc[mt][nt][e] = 0.0f;
    uint32_t kw[2][8];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const int tl = tb + nt * 8 + g4;
      const uint8_t *row = sb_k + tl * kHeadDim;
      const uint4 k0 = lds128(row + (((2 * c4) ^ (tl & 7)) << 4));
      const uint4 k1 = lds128(row + (((2 * c4 + 1) ^ (tl & 7)) << 4));
      kw[nt][0] = k0.x; kw[nt][1] = k0.y; kw[nt][2] = k0.z; kw[nt][3] = k0.w;
      kw[nt][4] = k1.x; kw[nt][5] = k1.y; kw[nt][6] = k1.z; kw[nt][7] = k1.w;
    }
#pragma unroll
    for (int s2 = 0; s2 < 4; ++s2) {
#pragma unroll
      for (int pc = 0; pc < 2; ++pc) {
        uint32_t a[MT][4];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          const uint4 f = qfrag[((mt * 4 + s2) * 2 + pc) * 32 + lane];
          a[mt][0] = f.x; a[mt][1] = f.y; a[mt][2] = f.z; a[mt][3] = f.w;
        }
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int mt = 0; mt < MT; ++mt)
            mma_e4m3_16832(sacc[mt][nt], a[mt], kw[nt][2 * s2], kw[nt][2 * s2 + 1]);
      }
    }

    // ---- scale, mask, online softmax (lazy rescale)
    float ksc[2][2], vsc[2][2];
    float vmax = 0.0f;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const float2 kk = *reinterpret_cast<const float2 *>(sb_ks + tb + nt * 8 + 2 * c4);
      const float2 vv = *reinterpret_cast<const float2 *>(sb_vs + tb + nt * 8 + 2 * c4);
      ksc[nt][0] = kk.x * p.qk_scale;
      ksc[nt][1] = kk.y * p.qk_scale;
      vsc[nt][0] = vv.x;
      vsc[nt][1] = vv.y;
      vmax = fmaxf(vmax, fmaxf(vv.x, vv.y));
    }
    // the 4 lanes of a quad hold all 16 tokens' scales: the quad max is the
    // chunk max, the same in every quad
    vmax = fmaxf(vmax, __shfl_xor_sync(0xFFFFFFFFu, vmax, 1));
    vmax = fmaxf(vmax, __shfl_xor_sync(0xFFFFFFFFu, vmax, 2));
    float vfac = 1.0f;
    bool vgrow = false;
    {
      const uint32_t bits = __float_as_uint(vmax);
      const int ex = static_cast<int>((bits >> 23) & 0xFFu);
      int ec = (ex == 0) ? -126 : ex - 127 + ((bits & 0x7FFFFFu) != 0u ? 1 : 0);
      ec = ec > 126 ? 126 : ec;   // finite scales are below 2^120
      if (ec > ev) {
        const int d = ev - ec;   // < 0
        vfac = (d >= -126) ? __int_as_float((127 + d) << 23) : 0.0f;
        ev = ec;
        vgrow = true;
      }
    }
    const float vnorm = __int_as_float((127 - ev) << 23);   // 2^-E, E in [-126, 126]
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      vsc[nt][0] *= vnorm;
      vsc[nt][1] *= vnorm;
    }
    float fac[MT][2];
    bool grow = false;
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        float mx = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int j = jbase + nt * 8 + 2 * c4 + e;
            float x = sacc[mt][nt][2 * hf + e] * ksc[nt][e] * rowf[mt][hf];
            x = (j < vis[mt][hf]) ? x : -INFINITY;
            sacc[mt][nt][2 * hf + e] = x;
            mx = fmaxf(mx, x);
          }
        mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 2));
        const float mold = m_run[mt][hf];
        if (mx > mold + kLazyRescale) {
          fac[mt][hf] = ex2(mold - mx);
          m_run[mt][hf] = mx;
          grow = true;
        } else {
          fac[mt][hf] = 1.0f;
        }
      }
    if (__any_sync(0xFFFFFFFFu, grow) || vgrow) {
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          l_run[mt][hf] *= fac[mt][hf];
          const float f = fac[mt][hf] * vfac;
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            o[mt][i][2 * hf] *= f;
            o[mt][i][2 * hf + 1] *= f;
          }
        }
    }
    uint32_t pa[MT][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      float pv[2][4];
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const float msub = (m_run[mt][hf] == -INFINITY) ? 0.0f : m_run[mt][hf];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const float pr = ex2(sacc[mt][nt][2 * hf + e] - msub);
            l_run[mt][hf] += pr;
            pv[nt][2 * hf + e] = pr * vsc[nt][e];
          }
      }
      pa[mt][0] = pack_f16x2(pv[0][0], pv[0][1]);   // row g4,   tokens 2c, 2c+1
      pa[mt][1] = pack_f16x2(pv[0][2], pv[0][3]);   // row g4+8, tokens 2c, 2c+1
      pa[mt][2] = pack_f16x2(pv[1][0], pv[1][1]);   // row g4,   tokens 2c+8, 2c+9
      pa[mt][3] = pack_f16x2(pv[1][2], pv[1][3]);   // row g4+8, tokens 2c+8, 2c+9
    }

    // ---- O += P' V.  Lane reads dims [16*g4, 16*g4+16) of tokens 2c, 2c+1, 2c+8, 2c+9.
    uint4 va, vb, vc, vd;
    {
      const int t_a = tb + 2 * c4, t_b = t_a + 1, t_c = t_a + 8, t_d = t_a + 9;
      va = lds128(sb_v + t_a * kHeadDim + ((g4 ^ (t_a & 7)) << 4));
      vb = lds128(sb_v + t_b * kHeadDim + ((g4 ^ (t_b & 7)) << 4));
      vc = lds128(sb_v + t_c * kHeadDim + ((g4 ^ (t_c & 7)) << 4));
      vd = lds128(sb_v + t_d * kHeadDim + ((g4 ^ (t_d & 7)) << 4));
    }
    const uint32_t wa[4] = {va.x, va.y, va.z, va.w};
    const uint32_t wb[4] = {vb.x, vb.y, vb.z, vb.w};
    const uint32_t wc[4] = {vc.x, vc.y, vc.z, vc.w};
    const uint32_t wd[4] = {vd.x, vd.y, vd.z, vd.w};
#pragma unroll
    for (int wi = 0; wi < 4; ++wi) {
      const uint32_t ab01 = prmt(wa[wi], wb[wi], 0x5410u);   // [a0 a1 b0 b1]
      const uint32_t ab23 = prmt(wa[wi], wb[wi], 0x7632u);   // [a2 a3 b2 b3]
      const uint32_t cd01 = prmt(wc[wi], wd[wi], 0x5410u);
      const uint32_t cd23 = prmt(wc[wi], wd[wi], 0x7632u);
      uint32_t b0[4], b1[4];
      b0[0] = e4m3x2_b02_to_f16x2_lo8(ab01); b1[0] = e4m3x2_b02_to_f16x2_lo8(cd01);
      b0[1] = e4m3x2_b13_to_f16x2_lo8(ab01); b1[1] = e4m3x2_b13_to_f16x2_lo8(cd01);
      b0[2] = e4m3x2_b02_to_f16x2_lo8(ab23); b1[2] = e4m3x2_b02_to_f16x2_lo8(cd23);
      b0[3] = e4m3x2_b13_to_f16x2_lo8(ab23); b1[3] = e4m3x2_b13_to_f16x2_lo8(cd23);
#pragma unroll
      for (int e = 0; e < 4; ++e)
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) mma_f16_16816(o[mt][4 * wi + e], pa[mt], b0[e], b1[e]);
    }
  }

  // ---- merge the four warps' partial results.  Warps 1..3 park their
  // (rescaled) accumulators in shared memory in fragment order (conflict-free
  // 16-byte stores), warp 0 adds them to its registers and writes the rows.
  cp_async_wait<0>();
  __syncthreads();
  constexpr int kRows = MT * 16;
  float *m_w = reinterpret_cast<float *>(smem);                   // [kWarps][kRows]
  float *l_w = m_w + kWarps * kRows;                              // [kWarps][kRows]
  float4 *parked = reinterpret_cast<float4 *>(l_w + kWarps * kRows);  // [3][MT][16][32]
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      float l = l_run[mt][hf];
      l += __shfl_xor_sync(0xFFFFFFFFu, l, 1);
      l += __shfl_xor_sync(0xFFFFFFFFu, l, 2);
      l_run[mt][hf] = l;
      if (c4 == 0) {
        const int rl = mt * 16 + g4 + 8 * hf;
        m_w[warp * kRows + rl] = m_run[mt][hf];
        l_w[warp * kRows + rl] = l;
      }
    }
  __syncthreads();
  float mrow[MT][2], lrow[MT][2], frow[MT][2];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      const int rl = mt * 16 + g4 + 8 * hf;
      float mx = -INFINITY;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) mx = fmaxf(mx, m_w[w * kRows + rl]);
      float lt = 0.0f;
      if (mx != -INFINITY) {
#pragma unroll
        for (int w = 0; w < kWarps; ++w) lt += l_w[w * kRows + rl] * ex2(m_w[w * kRows + rl] - mx);
      }
      mrow[mt][hf] = mx;
      lrow[mt][hf] = lt;
      // softmax merge weight times 2^E (the accumulators hold O * 2^-(E+8);
      // the remaining 2^8 is applied with a second multiply below)
      frow[mt][hf] = (mx == -INFINITY || ev == -1000)
                         ? 0.0f : ldexpf(ex2(m_run[mt][hf] - mx), ev);
    }
  if (warp > 0) {
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int i = 0; i < 16; ++i)
        parked[(((warp - 1) * MT + mt) * 16 + i) * 32 + lane] =
            make_float4(o[mt][i][0] * 256.0f * frow[mt][0], o[mt][i][1] * 256.0f * frow[mt][0],
                        o[mt][i][2] * 256.0f * frow[mt][1], o[mt][i][3] * 256.0f * frow[mt][1]);
  }
  __syncthreads();
  if (warp != 0) return;
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      float4 acc = make_float4(o[mt][i][0] * 256.0f * frow[mt][0],
                               o[mt][i][1] * 256.0f * frow[mt][0],
                               o[mt][i][2] * 256.0f * frow[mt][1],
                               o[mt][i][3] * 256.0f * frow[mt][1]);
#pragma unroll
      for (int w = 0; w < kWarps - 1; ++w) {
        const float4 x = parked[((w * MT + mt) * 16 + i) * 32 + lane];
        acc.x += x.x; acc.y += x.y; acc.z += x.z; acc.w += x.w;
      }
      o[mt][i][0] = acc.x; o[mt][i][1] = acc.y; o[mt][i][2] = acc.z; o[mt][i][3] = acc.w;
    }

  // ---- write.  Lane (g4, c4) holds, for row g4 (+8), dims 32*c4 + i (element
  // 0/2 of n-tile i) and 32*c4 + 16 + i (element 1/3): 32 consecutive dims.
  const bool direct = n_parts <= 1;
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      const int m = row_base + mt * 16 + g4 + 8 * hf;
      if (m >= p.M) continue;
      const int i = m / p.G, gq = m - i * p.G;
      const int64_t orow = (static_cast<int64_t>(r) * p.R + i) * p.Hq + h * p.G + gq;
      const int d0 = 32 * c4;
      if (direct) {
        const float inv = (lrow[mt][hf] > 0.0f) ? 1.0f / lrow[mt][hf] : 0.0f;
        uint32_t pk[16];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          pk[j] = pack_bf16x2(o[mt][2 * j][2 * hf] * inv, o[mt][2 * j + 1][2 * hf] * inv);
          pk[8 + j] = pack_bf16x2(o[mt][2 * j][2 * hf + 1] * inv, o[mt][2 * j + 1][2 * hf + 1] * inv);
        }
        uint4 *dst = reinterpret_cast<uint4 *>(p.out + orow * kHeadDim + d0);
#pragma unroll
        for (int j = 0; j < 4; ++j) dst[j] = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
      } else {
        const int64_t slot = orow * p.n_parts_max + part;
        float4 *dst = reinterpret_cast<float4 *>(p.o_part + slot * kHeadDim + d0);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          dst[j] = make_float4(o[mt][4 * j][2 * hf], o[mt][4 * j + 1][2 * hf],
                               o[mt][4 * j + 2][2 * hf], o[mt][4 * j + 3][2 * hf]);
          dst[4 + j] = make_float4(o[mt][4 * j][2 * hf + 1], o[mt][4 * j + 1][2 * hf + 1],
                                   o[mt][4 * j + 2][2 * hf + 1], o[mt][4 * j + 3][2 * hf + 1]);
        }
        if (c4 == 0) p.ml_part[slot] = make_float2(mrow[mt][hf], lrow[mt][hf]);
      }
    }
}

// ---------------------------------------------------------------------------
struct CombineParams {
  const int32_t *context_lens;
  int32_t ctx_limit;
  int32_t R, Hq;
  int64_t rows_total;
  int32_t part_tokens;
  int32_t n_parts_max;
  const float *o_part;
  const float2 *ml_part;
  uint16_t *out;
};


// One CTA of kCombineWarps warps per output row (4, or 16 when a row can span
// 64 or more partitions).  Warp w folds partitions w, w+kCombineWarps, ... (4
// dims per lane) with a running log-sum-exp, loading four partitions' (max,
// sum) and outputs before using any, so the merge costs one memory round trip
// per four partitions of a warp; the warps' (max, sum, output) meet in shared
// memory.
template <int kCombineWarps, int kPre>
__global__ void __launch_bounds__(kCombineWarps * 32)
attn_combine_kernel(const CombineParams p) {
  __shared__ float red[kCombineWarps];
  __shared__ float4 part_o[kCombineWarps - 1][32];
  __shared__ float part_l[kCombineWarps];
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int64_t row = blockIdx.x;
  const int r = static_cast<int>(row / (static_cast<int64_t>(p.R) * p.Hq));
  allow_dependents_launch();
  grid_dependency_wait();                         // before any global read
  int L = p.context_lens[r];
  L = L < 0 ? 0 : (L > p.ctx_limit ? p.ctx_limit : L);
  const int n_parts = (L + p.part_tokens - 1) / p.part_tokens;
  if (n_parts <= 1) return;                       // written by the partials kernel
  const float2 *ml = p.ml_part + row * p.n_parts_max;
  const float4 *op = reinterpret_cast<const float4 *>(p.o_part + row * p.n_parts_max * kHeadDim) +
                     lane;
  // warp w folds partitions w, w+W, ... with a running log-sum-exp; kPre of
  // its partitions' (max, sum) and outputs are loaded before any is used
  float m_w = -INFINITY, lsum = 0.0f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int q0 = warp; q0 < n_parts; q0 += kPre * kCombineWarps) {
    float2 v[kPre];
    float4 o[kPre];
#pragma unroll
    for (int k = 0; k < kPre; ++k) {
      const int q = q0 + k * kCombineWarps;
      v[k] = make_float2(-INFINITY, 0.0f);
      o[k] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (q < n_parts) {
        v[k] = ml[q];
        o[k] = op[static_cast<int64_t>(q) * (kHeadDim / 4)];
      }
    }
#pragma unroll
    for (int k = 0; k < kPre; ++k) {
      if (v[k].x == -INFINITY) continue;          // a partition that saw no token
      const float mn = fmaxf(m_w, v[k].x);
      const float a = ex2(m_w - mn), b = ex2(v[k].x - mn);
      lsum = lsum * a + v[k].y * b;
      acc.x = acc.x * a + o[k].x * b;
      acc.y = acc.y * a + o[k].y * b;
      acc.z = acc.z * a + o[k].z * b;
      acc.w = acc.w * a + o[k].w * b;
      m_w = mn;
    }
  }
  if (lane == 0) red[warp] = m_w;
  __syncthreads();
  float mx = red[0];
#pragma unroll
  for (int w = 1; w < kCombineWarps; ++w) mx = fmaxf(mx, red[w]);
  {
    const float a = (m_w == -INFINITY) ? 0.0f : ex2(m_w - mx);
    lsum *= a;
    acc.x *= a;
    acc.y *= a;
    acc.z *= a;
    acc.w *= a;
  }
  if (warp > 0) part_o[warp - 1][lane] = acc;
  if (lane == 0) part_l[warp] = lsum;
  __syncthreads();
  if (warp != 0) return;
#pragma unroll
  for (int w = 0; w < kCombineWarps - 1; ++w) {
    const float4 v = part_o[w][lane];
    acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
  }
#pragma unroll
  for (int w = 1; w < kCombineWarps; ++w) lsum += part_l[w];
  const float inv = (lsum > 0.0f) ? 1.0f / lsum : 0.0f;
  uint2 packed;
  packed.x = pack_bf16x2(acc.x * inv, acc.y * inv);
  packed.y = pack_bf16x2(acc.z * inv, acc.w * inv);
  *reinterpret_cast<uint2 *>(p.out + row * kHeadDim + 4 * lane) = packed;
}

// Rows of few partitions (<= 16): one warp per row, eight rows per CTA.  Lane
// l folds dims 4l..4l+3 over the row's partitions with a running log-sum-exp,
// four partitions' (max, sum) and outputs loaded before any is used, and
// writes the row: no shared memory, no CTA barrier.
constexpr int kCombineRowsPerCta = 8;

__global__ void __launch_bounds__(kCombineRowsPerCta * 32)
attn_combine_rows_kernel(const CombineParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kCombineRowsPerCta + (threadIdx.x >> 5);
  allow_dependents_launch();
  if (row >= p.rows_total) return;
  const int r = static_cast<int>(row / (static_cast<int64_t>(p.R) * p.Hq));
  grid_dependency_wait();                         // before any global read
  int L = p.context_lens[r];
  L = L < 0 ? 0 : (L > p.ctx_limit ? p.ctx_limit : L);
  const int n_parts = (L + p.part_tokens - 1) / p.part_tokens;
  if (n_parts <= 1) return;                       // written by the partials kernel
  const float2 *ml = p.ml_part + row * p.n_parts_max;
  const float4 *op = reinterpret_cast<const float4 *>(p.o_part + row * p.n_parts_max * kHeadDim) +
                     lane;
  float m_w = -INFINITY, lsum = 0.0f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int q0 = 0; q0 < n_parts; q0 += 4) {
    float2 v[4];
    float4 o[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      v[k] = make_float2(-INFINITY, 0.0f);
      o[k] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (q0 + k < n_parts) {
        v[k] = ml[q0 + k];
        o[k] = op[static_cast<int64_t>(q0 + k) * (kHeadDim / 4)];
      }
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      if (v[k].x == -INFINITY) continue;          // a partition that saw no token
      const float mn = fmaxf(m_w, v[k].x);
      const float a = ex2(m_w - mn), b = ex2(v[k].x - mn);
      lsum = lsum * a + v[k].y * b;
      acc.x = acc.x * a + o[k].x * b;
      acc.y = acc.y * a + o[k].y * b;
      acc.z = acc.z * a + o[k].z * b;
      acc.w = acc.w * a + o[k].w * b;
      m_w = mn;
    }
  }
  const float inv = (lsum > 0.0f) ? 1.0f / lsum : 0.0f;
  uint2 packed;
  packed.x = pack_bf16x2(acc.x * inv, acc.y * inv);
  packed.y = pack_bf16x2(acc.z * inv, acc.w * inv);
  *reinterpret_cast<uint2 *>(p.out + row * kHeadDim + 4 * lane) = packed;
}

template <int MT, bool kTma>
cudaError_t launch_partials_mt(const AttnParams &p, const CUtensorMap &mk, const CUtensorMap &mv,
                               dim3 grid, cudaStream_t stream) {
  constexpr int smem = smem_bytes(MT);
  static_assert(kOffQ >= 2 * kWarps * MT * 16 * 4 + (kWarps - 1) * MT * 16 * 32 * 16,
                "epilogue buffers must fit in the stage buffers");
  // the shared-memory opt-in is a per-device function attribute: set it once
  // per device (a host-side call, no stream work)
  static std::atomic<uint64_t> configured{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = (dev >= 0 && dev < 64) ? (uint64_t(1) << dev) : 0;
  if (bit == 0 || !(configured.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(attn_partials_kernel<MT, kTma>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit, std::memory_order_acq_rel);
  }
  return launch_overlapped(attn_partials_kernel<MT, kTma>, grid, dim3(kThreads), smem, stream, p, mk, mv);
}

void carve_workspace(void *ws, int64_t rows_total, int32_t n_parts, float **o_part,
                     float2 **ml_part) {
  const size_t o = static_cast<size_t>(rows_total) * n_parts * kHeadDim * sizeof(float);
  *o_part = static_cast<float *>(ws);
  *ml_part = reinterpret_cast<float2 *>(static_cast<char *>(ws) + ((o + 255) / 256) * 256);
}

int32_t context_cap(const AttnShape &s) {
  const int64_t cap = static_cast<int64_t>(s.max_blocks_per_req) << s.log2_block;
  return static_cast<int32_t>(cap < s.max_context_len ? cap : s.max_context_len);
}

}  // namespace

namespace {
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// against libcuda); looked up once.
EncodeTiledFn encode_tiled_fn() {
  static std::atomic<EncodeTiledFn> fn{nullptr};
  EncodeTiledFn f = fn.load(std::memory_order_acquire);
  if (f == nullptr) {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || ptr == nullptr) {
      cudaGetLastError();
      return nullptr;
    }
    f = reinterpret_cast<EncodeTiledFn>(ptr);
    fn.store(f, std::memory_order_release);
  }
  return f;
}

}  // namespace

// A map over one code plane [num_slots, H, 128] uint8: boxes of `rows` slots of
// one head, 128-byte swizzled in shared memory.  A box row is one 128-byte
// line and the next slot's row of the same head is H lines further, so L2
// promotion stays at 128 bytes: wider promotion would fetch the neighbouring
// head's line from DRAM, wasted unless that head's reader comes by while it
// is still in L2.
bool encode_code_tensor_map(CUtensorMap *map, const uint8_t *codes, int64_t num_slots, int H,
                            int rows) {
  EncodeTiledFn f = encode_tiled_fn();
  if (f == nullptr) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(H),
                              static_cast<cuuint64_t>(num_slots)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(kHeadDim),
                                 static_cast<cuuint64_t>(H) * kHeadDim};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(kHeadDim), 1u, static_cast<cuuint32_t>(rows)};
  const cuuint32_t estride[3] = {1u, 1u, 1u};
  return f(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t *>(codes), dims, strides,
           box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
           CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_code_tensor_map_strided(CUtensorMap *map, const uint8_t *codes, int64_t num_slots,
                                    int H) {
  EncodeTiledFn f = encode_tiled_fn();
  if (f == nullptr || H < 4) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(num_slots),
                              static_cast<cuuint64_t>(H)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(H) * kHeadDim,
                                 static_cast<cuuint64_t>(kHeadDim)};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(kHeadDim), 16u, 4u};
  const cuuint32_t estride[3] = {1u, 1u, 1u};
  return f(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t *>(codes), dims, strides,
           box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A map over one scale plane [num_slots, H] fp32: boxes of 4 consecutive heads
// x `rows` slots, unswizzled (16 bytes per slot row in shared memory).
bool encode_scale_tensor_map(CUtensorMap *map, const float *scales, int64_t num_slots, int H,
                             int rows) {
  EncodeTiledFn f = encode_tiled_fn();
  if (f == nullptr || H % 4 != 0) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(num_slots)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(H) * sizeof(float)};
  const cuuint32_t box[2] = {4u, static_cast<cuuint32_t>(rows)};
  const cuuint32_t estride[2] = {1u, 1u};
  return f(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(scales), dims, strides,
           box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
           CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t attn_workspace_bytes(int64_t rows_total, int32_t num_partitions) {
  if (num_partitions <= 1) return 0;
  const size_t o = static_cast<size_t>(rows_total) * num_partitions * kHeadDim * sizeof(float);
  const size_t ml = static_cast<size_t>(rows_total) * num_partitions * 2 * sizeof(float);
  const size_t total = ((o + 255) / 256) * 256 + ml;
  return ((total + 255) / 256) * 256;
}

cudaError_t launch_attn_partials(const kvq_cache &c, const AttnShape &s, const void *q,
                                 const int32_t *block_tables, const int32_t *context_lens,
                                 float sm_scale, void *out, void *workspace,
                                 int32_t *err_flags, cudaStream_t stream,
                                 const AppendRows *append) {
  // a decode step's new rows: stored inside the load-balanced kernel, else by
  // the store's own launch ahead of the attention
  if (append != nullptr && !(s.stream && !s.rows_kernel && s.rows_per_request <= kStreamNewRows)) {
    const cudaError_t e = launch_quantize_positions(
        c, append->k, append->k_stride, append->v, append->v_stride, s.num_requests,
        s.rows_per_request, block_tables, s.max_blocks_per_req, context_lens, context_cap(s),
        s.log2_block, err_flags, stream);
    if (e != cudaSuccess) return e;
    append = nullptr;
  }
  AttnParams p;
  p.k_codes = c.k_codes;
  p.v_codes = c.v_codes;
  p.k_scales = c.k_scales;
  p.v_scales = c.v_scales;
  p.num_blocks = c.num_slots >> s.log2_block;
  p.H = c.num_kv_heads;
  p.log2_bs = s.log2_block;
  p.q = static_cast<const uint16_t *>(q);
  p.out = static_cast<uint16_t *>(out);
  p.block_tables = block_tables;
  p.max_blocks = s.max_blocks_per_req;
  p.context_lens = context_lens;
  p.ctx_limit = context_cap(s);
  p.R = s.rows_per_request;
  p.Hq = s.num_q_heads;
  p.G = s.group;
  p.M = s.rows;
  p.row_groups = s.row_groups;
  p.qk_scale = sm_scale * kLog2e;
  p.part_tokens = s.partition_tokens;
  p.n_parts_max = s.num_partitions;
  p.err_flags = err_flags;
  const int64_t rows_total =
      static_cast<int64_t>(s.num_requests) * s.rows_per_request * s.num_q_heads;
  p.o_part = nullptr;
  p.ml_part = nullptr;
  if (s.num_partitions > 1)
    carve_workspace(workspace, rows_total, s.num_partitions, &p.o_part, &p.ml_part);
  if (s.rows_kernel)
    return launch_attn_rows(c, s, q, block_tables, context_lens, sm_scale, out, workspace,
                            err_flags, stream);
  if (s.stream)
    return launch_attn_partials_stream(c, s, q, block_tables, context_lens, sm_scale, out,
                                       workspace, err_flags, stream, append);
  // the page-major kernel reads 4 heads per CTA: worth it once its grid is at
  // least ~3 waves (3 CTAs per SM); smaller grids go to one CTA per head
  const int64_t page_ctas =
      static_cast<int64_t>(c.num_kv_heads / 4) * s.num_partitions * s.num_requests;
  if (attn_page_supported(c, s) && page_ctas >= 9LL * (s.sms > 0 ? s.sms : 152))
    return launch_attn_partials_page(c, s, q, block_tables, context_lens, sm_scale, out,
                                     p.o_part, p.ml_part, err_flags, stream);
  if (attn_skinny_supported(c, s))
    return launch_attn_partials_skinny(c, s, q, block_tables, context_lens, sm_scale, out,
                                       p.o_part, p.ml_part, err_flags, stream);
  if (attn_tc_supported(c, s))
    return launch_attn_partials_tc(c, s, q, block_tables, context_lens, sm_scale, out,
                                   p.o_part, p.ml_part, err_flags, stream);
  dim3 grid(c.num_kv_heads * s.row_groups, s.num_partitions, s.num_requests);
  // TMA staging needs page boxes of >= 8 rows (1024-byte aligned swizzle
  // atoms), a partition's block ids in shared memory and 32-bit slot
  // coordinates; other shapes stage with cp.async
  CUtensorMap mk, mv;
  const int rows = s.log2_block >= 6 ? kStageTok : (1 << s.log2_block);
  const int64_t pages = static_cast<int64_t>(s.partition_tokens) / rows + 1;
  const bool tma = (1 << s.log2_block) >= kMinTmaBlock && pages <= kMaxPages &&
                   c.num_slots > 0 && c.num_slots < (int64_t(1) << 31) &&
                   encode_code_tensor_map(&mk, c.k_codes, c.num_slots, c.num_kv_heads, rows) &&
                   encode_code_tensor_map(&mv, c.v_codes, c.num_slots, c.num_kv_heads, rows);
  if (!tma) {
    memset(&mk, 0, sizeof(mk));
    memset(&mv, 0, sizeof(mv));
  }
  if (s.rows <= 16)
    return tma ? launch_partials_mt<1, true>(p, mk, mv, grid, stream)
               : launch_partials_mt<1, false>(p, mk, mv, grid, stream);
  return tma ? launch_partials_mt<2, true>(p, mk, mv, grid, stream)
             : launch_partials_mt<2, false>(p, mk, mv, grid, stream);
}

cudaError_t launch_attn_combine(const AttnShape &s, const int32_t *context_lens, void *out,
                                void *workspace, cudaStream_t stream) {
  if (s.rows_kernel) return cudaSuccess;       // pieces merged by the partials kernel
  if (s.stream) return launch_attn_combine_stream(s, out, workspace, stream);
  if (s.num_partitions <= 1) return cudaSuccess;
  CombineParams p;
  p.context_lens = context_lens;
  p.ctx_limit = context_cap(s);
  p.R = s.rows_per_request;
  p.Hq = s.num_q_heads;
  p.rows_total = static_cast<int64_t>(s.num_requests) * s.rows_per_request * s.num_q_heads;
  p.part_tokens = s.partition_tokens;
  p.n_parts_max = s.num_partitions;
  float *o_part;
  float2 *ml_part;
  carve_workspace(workspace, p.rows_total, s.num_partitions, &o_part, &ml_part);
  p.o_part = o_part;
  p.ml_part = ml_part;
  p.out = static_cast<uint16_t *>(out);
  if (s.num_partitions <= 16) {
    const int64_t ctas = (p.rows_total + kCombineRowsPerCta - 1) / kCombineRowsPerCta;
    return launch_overlapped(attn_combine_rows_kernel, dim3(static_cast<unsigned>(ctas)),
                             dim3(kCombineRowsPerCta * 32), 0, stream, p);
  }
  // few, long rows (long contexts): more warps per row and more partitions
  // per memory round trip
  if (s.num_partitions >= 256)
    return launch_overlapped(attn_combine_kernel<32, 8>, dim3(static_cast<unsigned>(p.rows_total)),
                             dim3(32 * 32), 0, stream, p);
  if (s.num_partitions >= 64)
    return launch_overlapped(attn_combine_kernel<16, 4>, dim3(static_cast<unsigned>(p.rows_total)),
                             dim3(16 * 32), 0, stream, p);
  return launch_overlapped(attn_combine_kernel<4, 4>, dim3(static_cast<unsigned>(p.rows_total)),
                           dim3(4 * 32), 0, stream, p);
}

}  // namespace kvq
