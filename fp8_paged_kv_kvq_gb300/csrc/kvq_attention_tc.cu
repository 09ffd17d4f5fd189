// kvq_attention_tc.cu -- paged verify attention for 9..32 stacked query rows
// per KV head on the 5th-generation tensor cores (tcgen05), FP8 cache.
//
// The method is the one of kvq_attention.cu (ROCm/ATOM PR #2655 "fix(qwen4-exp):
// register the QSA FP8 scale planes for KV offload", PR description, K/V
// bullet: each token's key scale is applied to its score after the code dot
// product and its value scale to its probability ahead of PV; the R verify rows
// of a request that share a KV head are stacked into one tile).  Laid out for sm_103a:
//
//  * CTA = (KV head, partition, request), one per SM, 14 warps with fixed
//    roles.  Warp 12 (one lane) streams 128-token stages through a 4-deep ring
//    with TMA: per page one box of K codes, one of V codes (128-byte swizzled
//    rows) and one of each scale plane.
//  * Warp 13 (one lane) issues the MMAs.  S^T = K Q^T is one M=128 (tokens) x
//    N=64 x K=128 product on e4m3 operands (kind::f8f6f4): the K code tile
//    straight from shared memory as A (K-major), and as B the two e4m3 pieces
//    of Q (exact for elements >= 2^-9 of the row's largest, off by at most
//    2^-17 of it below) stacked as 64 rows (piece 1 of the 32 rows, then piece 2), so
//    each K step is one instruction; the softmax adds the two column halves.
//    (A tcgen05 MMA costs about the same for N = 32 as for N = 128.)  O^T += V^T P^T is M=128 (dims) x N=32 x K=128
//    (tokens) on f16 operands (kind::f16), both MN-major from shared memory,
//    accumulating in TMEM for the whole partition.
//  * Warps 0-7 run the softmax, two per TMEM lane quarter: a thread owns one
//    token (one TMEM lane) and 16 of the 32 rows.  It reads those scores,
//    folds key scale and sm_scale, applies the causal mask, and runs the
//    online softmax with a lazy per-row reference: a row's reference moves
//    only when one of its scores exceeds it by more than 2^14 (or a value scale
//    exceeds the running power-of-two bound 2^E).  The rows that moved are
//    agreed CTA-wide behind one named barrier, and only they are reduced.  A change rescales the running
//    denominators in registers and moves the PV accumulation on to a fresh
//    TMEM buffer (12 of them; the epilogue merges the buffers with the ratios
//    of their references), so it never waits for the tensor cores; only
//    after the 12th change does a change rescale the live buffer in place.
//    They write P''^T =
//    p * v_scale * 2^-E (f16, <= 2^14) in the MMA's canonical swizzled layout,
//    and at the end each thread reads one dim of O^T back from TMEM.
//  * Warps 8-11 own one token each and convert its V codes exactly to f16 (the
//    V^T operand, also in its canonical layout) while the softmax runs.
//  * Every wait is bounded; a role that gives up raises a shared abort flag,
//    the others leave their loops, copies and MMAs in flight complete, the
//    CTA frees its tensor memory and writes nothing (KVQ_ERRF_WAIT_TIMEOUT).
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <climits>

#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {

namespace {

constexpr int kTcTok = 128;                  // tokens per stage (the QK MMA's M)
constexpr int kTcStages = 4;                 // code ring depth
constexpr int kTcRows = 32;                  // stacked query rows (the MMAs' N), padded
constexpr int kTcSoftWarps = 8;             // softmax: two per TMEM lane quarter
constexpr int kTcHalf = 16;                 // rows per softmax thread
constexpr int kTcConvertWarps = 4;          // V code -> f16 operand warps
constexpr int kTcWarpTma = kTcSoftWarps + kTcConvertWarps;
constexpr int kTcWarpMma = kTcWarpTma + 1;
constexpr int kTcThreads = (kTcWarpMma + 1) * 32;
constexpr int kTcMaxPages = 512;             // block ids of one partition kept in smem
constexpr int kTcTmemCols = 512;             // S buffers 0, 1 | O buffers 0..11
constexpr int kColS = 0;                     // S^T buffer b: columns 64 b .. 64 b + 63
constexpr int kColO = 128;
constexpr int kTcOBufs = (kTcTmemCols - kColO) / kTcRows;
constexpr float kTcLazy = 14.0f;             // log2 of the largest unnormalised p
constexpr float kTcOvershoot = 4.0f;         // a moved reference sits this far above the max

// shared memory, offsets from a 1024-byte aligned base
constexpr int kCodeStage = 2 * kTcTok * kHeadDim;          // K codes | V codes
constexpr int kVfBytes = kTcTok * kHeadDim * 2;            // f16 V^T operand
constexpr int kPBytes = kTcTok * kTcRows * 2;              // f16 P^T operand
constexpr int kQBytes = kTcRows * kHeadDim;                // one e4m3 piece of Q
constexpr int kScBytes = kTcTok * 16;                      // [token][4 heads] f32
constexpr int kOffVf = kTcStages * kCodeStage;
constexpr int kOffP = kOffVf + kVfBytes;
constexpr int kOffQ = kOffP + 2 * kPBytes;
constexpr int kOffSc = kOffQ + 2 * kQBytes;
constexpr int kOffBt = kOffSc + kTcStages * 2 * kScBytes;
constexpr int kOffBar = kOffBt + kTcMaxPages * 4;
constexpr int kBarKvFull = 0;
constexpr int kBarKvEmpty = kTcStages;
constexpr int kBarSFull = 2 * kTcStages;
constexpr int kBarSEmpty = kBarSFull + 2;
constexpr int kBarPReady = kBarSEmpty + 2;
constexpr int kBarPvDone = kBarPReady + 2;
constexpr int kNumBars = kBarPvDone + 2;
constexpr int kOffMisc = kOffBar + kNumBars * 8;           // tmem base, abort, flags
constexpr int kOffRed = kOffMisc + 256;                    // [4 quarters][32 rows] scratch
constexpr int kOffRow = kOffRed + 4 * kTcRows * 4;         // 4 x [32] f32
constexpr int kOffOb = kOffRow + 4 * kTcRows * 4;          // per O buffer: [32] refs, E
constexpr int kTcSmem = kOffOb + kTcOBufs * (kTcRows + 1) * 4 + 1024;

static_assert(kOffVf % 1024 == 0 && kOffP % 1024 == 0 && kOffQ % 1024 == 0 &&
              kOffSc % 1024 == 0, "operand buffers need 1024-byte alignment");
static_assert(kTcSmem <= 227 * 1024, "shared memory budget");

constexpr uint32_t kIdescQK = mma_idesc(kTcTok, 2 * kTcRows, false, false);
constexpr uint32_t kIdescPV = mma_idesc(kHeadDim, kTcRows, true, true);

struct TcParams {
  int64_t num_blocks;
  int32_t log2_bs;
  int32_t bs;
  const uint16_t *q;
  uint16_t *out;
  const int32_t *block_tables;
  int32_t max_blocks;
  const int32_t *context_lens;
  int32_t ctx_limit;
  int32_t R, Hq, G, M;
  float qk_scale;            // sm_scale * log2(e)
  int32_t part_tokens;
  int32_t n_parts_max;
  float *o_part;
  float2 *ml_part;
  int32_t *err_flags;
};

__device__ __forceinline__ float tc_ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Order-preserving integer image of a float (for max reductions on integers).
__device__ __forceinline__ int float_key(float x) {
  const int b = __float_as_int(x);
  return b >= 0 ? b : b ^ 0x7FFFFFFF;
}

__device__ __forceinline__ float key_float(int k) {
  return __int_as_float(k >= 0 ? k : k ^ 0x7FFFFFFF);
}

// Bounded wait that also gives up once another role raised the abort flag.
__device__ __forceinline__ bool tc_wait(uint32_t bar, uint32_t parity, volatile int *abort) {
  for (int i = 0; i < (1 << 19); ++i) {
    if (mbar_try_wait_sleep(bar, parity, 2000u)) return true;
    if ((i & 15) == 15 && *abort) return false;
  }
  *abort = 1;
  return false;
}

// Smallest e in [-126, 126] with 2^e >= v (v >= 0 given as its bits).
__device__ __forceinline__ int pow2_ceil_exp(uint32_t bits) {
  const int ex = static_cast<int>((bits >> 23) & 0xFFu);
  int e = (ex == 0) ? -126 : ex - 127 + ((bits & 0x7FFFFFu) != 0u ? 1 : 0);
  return e > 126 ? 126 : e;
}

__global__ void __launch_bounds__(kTcThreads, 1)
attn_tc_kernel(const TcParams p, const __grid_constant__ CUtensorMap tm_kc,
               const __grid_constant__ CUtensorMap tm_vc, const __grid_constant__ CUtensorMap tm_ks,
               const __grid_constant__ CUtensorMap tm_vs) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int h = blockIdx.x;
  const int part = blockIdx.y;
  const int r = blockIdx.z;

  grid_dependency_wait();
  allow_dependents_launch();
  int L = p.context_lens[r];
  if (L < 0 || L > p.ctx_limit) {
    if (part == 0 && tid == 0 && h == 0 && p.err_flags) atomicOr(p.err_flags, KVQ_ERRF_CONTEXT_RANGE);
    L = L < 0 ? 0 : p.ctx_limit;
  }
  const int n_parts = (L + p.part_tokens - 1) / p.part_tokens;
  if (part >= (n_parts > 0 ? n_parts : 1)) return;
  const int t0 = part * p.part_tokens;
  const int t_end = min(L, t0 + p.part_tokens);
  const int n_st = (t_end > t0) ? (t_end - t0 + kTcTok - 1) / kTcTok : 0;
  const int page0 = t0 >> p.log2_bs;

  int32_t *bt_s = reinterpret_cast<int32_t *>(smem + kOffBt);
  const uint32_t bar0 = smem_addr(smem + kOffBar);
  auto BAR = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kOffMisc);
  volatile int *abort_s = reinterpret_cast<volatile int *>(smem + kOffMisc + 4);
  volatile int *ob_s = reinterpret_cast<volatile int *>(smem + kOffMisc + 8);     // [2]
  uint32_t *trig_s = reinterpret_cast<uint32_t *>(smem + kOffMisc + 32);  // [2][8] row masks
  uint32_t *vmax_s = reinterpret_cast<uint32_t *>(smem + kOffMisc + 96);  // [2][8]
  int *flag_s = reinterpret_cast<int *>(smem + kOffMisc + 160);           // [2][8] give-up
  int *red_i = reinterpret_cast<int *>(smem + kOffRed);
  float *rowf_s = reinterpret_cast<float *>(smem + kOffRow);   // 2^e_m * sm_scale * log2e
  float *mcur_s = rowf_s + kTcRows;                            // row references
  float *lsum_s = rowf_s + 3 * kTcRows;                        // denominators
  float *obm_s = reinterpret_cast<float *>(smem + kOffOb);     // [buffer][32] references
  int *obe_s = reinterpret_cast<int *>(obm_s + kTcOBufs * kTcRows);   // [buffer] E

  // ---- set-up: block ids, barriers, tensor memory, query pieces
  {
    const int n_pages = (t_end > t0) ? ((t_end - 1) >> p.log2_bs) - page0 + 1 : 0;
    const int32_t *bt = p.block_tables + static_cast<int64_t>(r) * p.max_blocks + page0;
    for (int i = tid; i < n_pages; i += kTcThreads) bt_s[i] = bt[i];
  }
  if (tid == 0) {
    for (int s = 0; s < kTcStages; ++s) {
      mbar_init(BAR(kBarKvFull + s), 1);
      mbar_init(BAR(kBarKvEmpty + s), kTcSoftWarps + kTcConvertWarps);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(BAR(kBarSFull + b), 1);
      mbar_init(BAR(kBarSEmpty + b), kTcSoftWarps);
      mbar_init(BAR(kBarPReady + b), kTcSoftWarps + kTcConvertWarps);
      mbar_init(BAR(kBarPvDone + b), 1);
    }
    *abort_s = 0;
    fence_mbarrier_init();
  }
  if (warp == kTcWarpTma) {
    tmem_alloc(smem_addr(tmem_slot), kTcTmemCols);
    tmem_relinquish();
  }
  if (warp < kTcSoftWarps) {
    // rows 4w .. 4w+3; lane holds dims 4*lane .. 4*lane+3.  q = 2^e (p1 + p2),
    // p1 = e4m3(q 2^-e), p2 = e4m3(q 2^-e - p1): 8 significant bits, all of bf16's
#pragma unroll 1
    for (int i = 0; i < 4; ++i) {
      const int m = 4 * warp + i;
      uint2 v = make_uint2(0u, 0u);
      if (m < p.M) {
        const int ir = m / p.G, gq = m - ir * p.G;
        v = *reinterpret_cast<const uint2 *>(
            p.q + ((static_cast<int64_t>(r) * p.R + ir) * p.Hq + h * p.G + gq) * kHeadDim +
            4 * lane);
      }
      const float xs[4] = {bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y)};
      float amax = fmaxf(fmaxf(fabsf(xs[0]), fabsf(xs[1])), fmaxf(fabsf(xs[2]), fabsf(xs[3])));
#pragma unroll
      for (int off = 16; off > 0; off >>= 1)
        amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, off));
      const int ex = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFFu);
      int e = (ex == 0) ? -126 : ex - 127 - 7;
      e = e < -126 ? -126 : (e > 126 ? 126 : e);
      const float rexp = __int_as_float((127 + e) << 23);
      const float inv = __int_as_float((127 - e) << 23);
      uint32_t c1w = 0u, c2w = 0u;
      if (amax != 0.0f) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float x = xs[k] * inv;
          const uint32_t c1 = e4m3_round(x, x);
          const float res = x - e4m3_to_f32(c1);
          c1w |= c1 << (8 * k);
          c2w |= e4m3_round(res, res) << (8 * k);
        }
      }
      if (lane == 0) {
        rowf_s[m] = (amax != 0.0f) ? rexp * p.qk_scale : 0.0f;
        mcur_s[m] = -INFINITY;
      }
      // K-major, 128-byte swizzle: row m at m * 128, 16-byte chunk c at (c ^ (m & 7))
      const int off = m * kHeadDim + (((lane >> 2) ^ (m & 7)) << 4) + 4 * (lane & 3);
      *reinterpret_cast<uint32_t *>(smem + kOffQ + off) = c1w;
      *reinterpret_cast<uint32_t *>(smem + kOffQ + kQBytes + off) = c2w;
    }
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  bool aborted = false;

  if (warp == kTcWarpTma) {
    // ---------------------------------------------------------------- TMA
    if (lane == 0) {
      const int box = p.bs;                      // pages are 16..128 tokens
      const int nbox = kTcTok / box;
      int issued = 0;
      bool bad = false;
      for (int s = 0; s < n_st; ++s) {
        const int b = s % kTcStages;
        if (s >= kTcStages &&
            !tc_wait(BAR(kBarKvEmpty + b), ((s / kTcStages) - 1) & 1, abort_s))
          break;
        const uint32_t kdst = smem_addr(smem + b * kCodeStage);
        const uint32_t vdst = kdst + kTcTok * kHeadDim;
        const uint32_t ksd = smem_addr(smem + kOffSc + 2 * b * kScBytes);
        const uint32_t vsd = ksd + kScBytes;
        const uint32_t fb = BAR(kBarKvFull + b);
        fence_proxy_async_smem();
        uint32_t bytes = 0;
        const int j0 = t0 + s * kTcTok;
        for (int i = 0; i < nbox; ++i) {
          const int j = j0 + i * box;
          if (j >= t_end) break;
          const int64_t blk = bt_s[(j >> p.log2_bs) - page0];
          if (blk < 0 || blk >= p.num_blocks) {
            bad = true;
            continue;
          }
          const int z = static_cast<int>(blk << p.log2_bs);
          tma_load_3d(kdst + i * box * kHeadDim, &tm_kc, 0, h, z, fb);
          tma_load_3d(vdst + i * box * kHeadDim, &tm_vc, 0, h, z, fb);
          tma_load_2d(ksd + i * box * 16, &tm_ks, h & ~3, z, fb);
          tma_load_2d(vsd + i * box * 16, &tm_vs, h & ~3, z, fb);
          bytes += 2u * box * kHeadDim + 2u * box * 16u;
        }
        mbar_arrive_expect_tx(fb, bytes);
        ++issued;
      }
      if (bad && p.err_flags) atomicOr(p.err_flags, KVQ_ERRF_BLOCK_RANGE);
      // copies still in flight (after an abort) land before the CTA leaves
      for (int s = (issued > kTcStages ? issued - kTcStages : 0); s < issued; ++s)
        mbar_wait_sleep_bounded(BAR(kBarKvFull + s % kTcStages), (s / kTcStages) & 1);
    }
  } else if (warp == kTcWarpMma) {
    // ---------------------------------------------------------------- MMA
    if (lane == 0) {
      const uint32_t kc0 = smem_addr(smem);
      const uint32_t vf0 = smem_addr(smem + kOffVf);
      const uint32_t p0 = smem_addr(smem + kOffP);
      const uint32_t q0 = smem_addr(smem + kOffQ);
      uint32_t last_bar = 0, last_par = 0;
      bool any = false;
      int prev_ob = -1;
      for (int s = 0; s <= n_st; ++s) {
        if (s < n_st) {
          const int b = s % kTcStages, sb = s & 1;
          if (!tc_wait(BAR(kBarKvFull + b), (s / kTcStages) & 1, abort_s)) break;
          if (s >= 2 && !tc_wait(BAR(kBarSEmpty + sb), ((s >> 1) - 1) & 1, abort_s)) break;
          tc_fence_after();
          const uint64_t ad = smem_desc(kc0 + b * kCodeStage, 16, 1024, kSmemSwizzle128);
          const uint64_t bd = smem_desc(q0, 16, 1024, kSmemSwizzle128);   // both pieces, 64 rows
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)      // K steps of 32 bytes inside the row
            tc_mma_e4m3(tmem + kColS + 2 * kTcRows * sb, ad + 2 * kk, bd + 2 * kk, kIdescQK,
                        kk != 0);
          tc_commit(BAR(kBarSFull + sb));
          last_bar = BAR(kBarSFull + sb);
          last_par = (s >> 1) & 1;
          any = true;
        }
        if (s >= 1) {
          const int u = s - 1, ub = u & 1;
          if (!tc_wait(BAR(kBarPReady + ub), (u >> 1) & 1, abort_s)) break;
          tc_fence_after();
          const int obu = ob_s[ub];                // the O buffer this stage accumulates into
          const uint64_t ad = smem_desc(vf0, kVfBytes / 2, 1024, kSmemSwizzle128);
          const uint64_t bd = smem_desc(p0 + ub * kPBytes, kPBytes, 512, kSmemSwizzle64);
#pragma unroll
          for (int kk = 0; kk < kTcTok / 16; ++kk)   // 16 tokens: 2 groups of 8 rows
            tc_mma_f16(tmem + kColO + kTcRows * obu, ad + (2048 >> 4) * kk,
                       bd + (1024 >> 4) * kk, kIdescPV, (obu == prev_ob || kk > 0) ? 1u : 0u);
          prev_ob = obu;
          tc_commit(BAR(kBarPvDone + ub));
          last_bar = BAR(kBarPvDone + ub);
          last_par = (u >> 1) & 1;
          any = true;
        }
      }
      // every MMA issued has completed before the tensor memory is freed
      if (any) mbar_wait_sleep_bounded(last_bar, last_par);
    }
  } else if (warp >= kTcSoftWarps) {
    // ------------------------------------------------ V codes -> f16 V^T
    // Token t's codes -> f16, MN-major, 128-byte swizzle: dims 64j.. in block j
    // (16 KiB apart), token t at (t/8)*1024 + (t%8)*128, the chunk of dims
    // 8c'.. at (c' ^ (t % 8)).  Tokens outside the partition get zeros: their
    // stage rows hold stale codes, and a NaN code would poison the product
    // even at p = 0.
    const int t = 32 * (warp - kTcSoftWarps) + lane;
    for (int s = 0; s < n_st; ++s) {
      const int b = s % kTcStages, sb = s & 1;
      const bool valid = t < t_end - (t0 + s * kTcTok);
      bool ok = tc_wait(BAR(kBarKvFull + b), (s / kTcStages) & 1, abort_s);
      // the f16 buffer is free once the PV of the previous stage has completed
      if (s >= 1) ok = tc_wait(BAR(kBarPvDone + (sb ^ 1)), ((s - 1) >> 1) & 1, abort_s) && ok;
      if (__any_sync(0xFFFFFFFFu, !ok)) break;
      const uint8_t *vrow = smem + b * kCodeStage + kTcTok * kHeadDim + t * kHeadDim;
      uint8_t *vf = smem + kOffVf + (t >> 3) * 1024 + (t & 7) * 128;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        uint4 w4 = make_uint4(0u, 0u, 0u, 0u);
        if (valid) w4 = *reinterpret_cast<const uint4 *>(vrow + ((c ^ (t & 7)) << 4));
        const uint4 lo = make_uint4(e4m3x2_to_f16x2(w4.x), e4m3x2_to_f16x2(w4.x >> 16),
                                    e4m3x2_to_f16x2(w4.y), e4m3x2_to_f16x2(w4.y >> 16));
        const uint4 hi = make_uint4(e4m3x2_to_f16x2(w4.z), e4m3x2_to_f16x2(w4.z >> 16),
                                    e4m3x2_to_f16x2(w4.w), e4m3x2_to_f16x2(w4.w >> 16));
        uint8_t *blk = vf + (c >> 2) * (kVfBytes / 2);
        const int c0 = (2 * c) & 7;
        *reinterpret_cast<uint4 *>(blk + ((c0 ^ (t & 7)) << 4)) = lo;
        *reinterpret_cast<uint4 *>(blk + (((c0 + 1) ^ (t & 7)) << 4)) = hi;
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(BAR(kBarPReady + sb));
        mbar_arrive(BAR(kBarKvEmpty + b));
      }
    }
  } else {
    // ----------------------------------------------------------- softmax
    const int qt = warp & 3;                    // TMEM lane quarter: tokens 32 qt ..
    const int hf = warp >> 2;                   // rows 16 hf .. 16 hf + 15
    const int t = 32 * qt + lane;               // the token (TMEM lane) this thread owns
    const uint32_t tl = tmem + (static_cast<uint32_t>(32 * qt) << 16);
    constexpr uint32_t kSoftThreads = kTcSoftWarps * 32;
    float mr[kTcHalf], lr[kTcHalf], rowf[kTcHalf];
#pragma unroll
    for (int i = 0; i < kTcHalf; ++i) {
      mr[i] = -INFINITY;
      lr[i] = 0.0f;
      rowf[i] = rowf_s[kTcHalf * hf + i];
    }
    int E = -126;                               // running bound 2^E >= every v_scale seen
    int ob = 0;                                 // O buffer the PVs accumulate into
    bool ob_used = false;                       // ... and whether one has been submitted
    const int vis0 = L - p.R + 1;               // row m sees tokens j < vis0 + m / G
    const uint32_t row_mask = (p.M >= 32) ? 0xFFFFFFFFu : ((1u << p.M) - 1u);
    for (int s = 0; s < n_st; ++s) {
      const int b = s % kTcStages, sb = s & 1;
      const int j0 = t0 + s * kTcTok;
      const int lim = t_end - j0;               // tokens t < lim belong to the partition
      bool ok = tc_wait(BAR(kBarKvFull + b), (s / kTcStages) & 1, abort_s);
      ok = tc_wait(BAR(kBarSFull + sb), (s >> 1) & 1, abort_s) && ok;
      tc_fence_after();
      float x[kTcHalf], x2[kTcHalf];
      tmem_ld16(tl + kColS + 2 * kTcRows * sb + kTcHalf * hf, x);             // piece 1
      tmem_ld16(tl + kColS + 2 * kTcRows * sb + kTcRows + kTcHalf * hf, x2);  // piece 2
#pragma unroll
      for (int i = 0; i < kTcHalf; ++i) x[i] += x2[i];
      tc_fence_before();
      const bool valid = t < lim;
      const float *sc = reinterpret_cast<const float *>(smem + kOffSc + 2 * b * kScBytes);
      const float ks = valid ? sc[4 * t + (h & 3)] : 0.0f;
      const float vs = valid ? sc[kTcTok * 4 + 4 * t + (h & 3)] : 0.0f;
      __syncwarp();                             // scores and scales are read
      if (lane == 0) {
        mbar_arrive(BAR(kBarSEmpty + sb));
        mbar_arrive(BAR(kBarKvEmpty + b));
      }
      // rows that see token j0 + t: m >= G * (j0 + t - vis0 + 1), m < M
      uint32_t vis_mask = row_mask;
      if (j0 + kTcTok > vis0 || lim < kTcTok) {
        const int lo = valid ? p.G * (j0 + t - vis0 + 1) : 32;
        vis_mask = (lo <= 0) ? row_mask : (lo >= 32 ? 0u : (row_mask & (0xFFFFFFFFu << lo)));
      }
      vis_mask >>= kTcHalf * hf;
      uint32_t trig = 0u;
#pragma unroll
      for (int i = 0; i < kTcHalf; ++i) {
        const float xm = ((vis_mask >> i) & 1u) ? x[i] * (ks * rowf[i]) : -INFINITY;
        x[i] = xm;
        trig |= (xm - mr[i] > kTcLazy) ? (1u << i) : 0u;
      }
      const uint32_t wtrig = __reduce_or_sync(0xFFFFFFFFu, trig);
      const uint32_t wv = __reduce_max_sync(0xFFFFFFFFu, __float_as_uint(vs));
      const unsigned wok = __all_sync(0xFFFFFFFFu, ok);
      if (lane == 0) {
        trig_s[(s & 1) * kTcSoftWarps + warp] = wtrig << (kTcHalf * hf);
        vmax_s[(s & 1) * kTcSoftWarps + warp] = wv;
        flag_s[(s & 1) * kTcSoftWarps + warp] = (wok && !*abort_s) ? 0 : 1;
      }
      named_barrier(1, kSoftThreads);
      uint32_t T32, vmax;
      int give_up;
      {
        const uint4 *tv = reinterpret_cast<const uint4 *>(trig_s + (s & 1) * kTcSoftWarps);
        const uint4 *vv = reinterpret_cast<const uint4 *>(vmax_s + (s & 1) * kTcSoftWarps);
        const int4 *fv = reinterpret_cast<const int4 *>(flag_s + (s & 1) * kTcSoftWarps);
        const uint4 t0v = tv[0], t1v = tv[1], v0 = vv[0], v1 = vv[1];
        const int4 f0 = fv[0], f1 = fv[1];
        T32 = (t0v.x | t0v.y | t0v.z | t0v.w) | (t1v.x | t1v.y | t1v.z | t1v.w);
        vmax = max(max(max(v0.x, v0.y), max(v0.z, v0.w)), max(max(v1.x, v1.y), max(v1.z, v1.w)));
        give_up = (f0.x | f0.y | f0.z | f0.w) | (f1.x | f1.y | f1.z | f1.w);
      }
      if (give_up) {
        aborted = true;
        break;
      }
      const int ereq = pow2_ceil_exp(vmax);
      if (T32 != 0u || ereq > E) {
        // ---- new references for the rows that moved and / or a larger value
        // bound.  The PVs so far go on under the old ones in their own buffer
        // (or, with none left, the live buffer is rescaled in place).
        const int e_new = max(E, ereq);
        const uint32_t mine = (T32 >> (kTcHalf * hf)) & 0xFFFFu;
        // the warp's max of every row of the half (independent reductions),
        // lane i keeps row i's
        int kmine = INT_MIN;
#pragma unroll
        for (int i = 0; i < kTcHalf; ++i) {
          const int k = __reduce_max_sync(0xFFFFFFFFu, float_key(x[i]));
          kmine = (lane == i) ? k : kmine;
        }
        if (lane < kTcHalf) red_i[qt * kTcRows + kTcHalf * hf + lane] = kmine;
        const bool next_buf = ob_used && ob + 1 < kTcOBufs;
        named_barrier(1, kSoftThreads);
        // lane i (< 16) settles row i of the half, then the lanes share
        float mo_l = -INFINITY;
#pragma unroll
        for (int i = 0; i < kTcHalf; ++i) mo_l = (lane == i) ? mr[i] : mo_l;
        float mn_l = mo_l, f_l = 1.0f;
        if (lane < kTcHalf) {
          const int m = kTcHalf * hf + lane;
          const int key = max(max(red_i[m], red_i[kTcRows + m]),
                              max(red_i[2 * kTcRows + m], red_i[3 * kTcRows + m]));
          if ((mine >> lane) & 1u) mn_l = fmaxf(key_float(key) + kTcOvershoot, mo_l);
          f_l = (mn_l == mo_l) ? 1.0f : tc_ex2(mo_l - mn_l);
          if (next_buf && qt == 0)              // row m's reference before the move
            obm_s[ob * kTcRows + m] = mo_l;
        }
        float f[kTcHalf];
#pragma unroll
        for (int i = 0; i < kTcHalf; ++i) {
          f[i] = __shfl_sync(0xFFFFFFFFu, f_l, i);
          mr[i] = __shfl_sync(0xFFFFFFFFu, mn_l, i);
          lr[i] *= f[i];
        }
        if (next_buf) {
          if (tid == 0) obe_s[ob] = E;
          ++ob;
          ob_used = false;
        } else if (ob_used) {
          // no buffer left: rescale the live one once the PV of the previous
          // stage is done
          const float efac =
              (e_new - E >= 127) ? 0.0f : __int_as_float((127 - (e_new - E)) << 23);
          tc_wait(BAR(kBarPvDone + ((s - 1) & 1)), ((s - 1) >> 1) & 1, abort_s);
          tc_fence_after();
          float o[kTcHalf];
          tmem_ld16(tl + kColO + kTcRows * ob + kTcHalf * hf, o);
#pragma unroll
          for (int i = 0; i < kTcHalf; ++i) o[i] *= f[i] * efac;
          tmem_st16(tl + kColO + kTcRows * ob + kTcHalf * hf, o);
          tmem_wait_st();
          tc_fence_before();
        }
        E = e_new;
      }

      // ---- P''^T of this token for the half's rows (f16) and denominators
      const float w = vs * __int_as_float((127 - E) << 23);
      uint32_t pk[kTcHalf / 2];
#pragma unroll
      for (int i = 0; i < kTcHalf / 2; ++i) {
        const float pa = tc_ex2(fmaxf(x[2 * i] - mr[2 * i], -200.0f));
        const float pb = tc_ex2(fmaxf(x[2 * i + 1] - mr[2 * i + 1], -200.0f));
        lr[2 * i] += pa;
        lr[2 * i + 1] += pb;
        pk[i] = pack_f16x2(pa * w, pb * w);
      }
      // the P buffer of stage s - 2 is free once its PV has completed
      if (s >= 2) tc_wait(BAR(kBarPvDone + sb), ((s - 2) >> 1) & 1, abort_s);
      {
        // MN-major, 64-byte swizzle: token t at (t/8)*512 + (t%8)*64, the
        // 16-byte chunk of rows 8c..8c+7 at (c ^ ((t % 8) / 2))
        uint8_t *pt = smem + kOffP + sb * kPBytes + (t >> 3) * 512 + (t & 7) * 64;
        const int sw = (t & 7) >> 1;
#pragma unroll
        for (int c = 0; c < 2; ++c)
          *reinterpret_cast<uint4 *>(pt + (((2 * hf + c) ^ sw) << 4)) =
              make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
      }
      if (tid == 0) ob_s[sb] = ob;
      ob_used = true;
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR(kBarPReady + sb));
    }

    // ---- epilogue: denominators over the 128 tokens, O^T back from TMEM
#pragma unroll
    for (int i = 0; i < kTcHalf; ++i) lr[i] += __shfl_xor_sync(0xFFFFFFFFu, lr[i], 16);
    // reduce-scatter over 16 lanes: lane i (mod 16) ends with row 16 hf + i
#pragma unroll
    for (int off = 8; off >= 1; off >>= 1) {
      const bool up = (lane & off) != 0;
#pragma unroll
      for (int i = 0; i < off; ++i) {
        const float send = up ? lr[i] : lr[i + off];
        const float keep = up ? lr[i + off] : lr[i];
        lr[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, off);
      }
    }
    float *red_f = reinterpret_cast<float *>(red_i);
    named_barrier(1, kSoftThreads);             // red_i of the last slow path is read
    if (lane < kTcHalf) red_f[qt * kTcRows + kTcHalf * hf + lane] = lr[0];
    if (qt == 0 && lane == 0) {
#pragma unroll
      for (int i = 0; i < kTcHalf; ++i) mcur_s[kTcHalf * hf + i] = mr[i];
    }
    named_barrier(1, kSoftThreads);
    if (qt == 0 && lane < kTcHalf) {
      const int m = kTcHalf * hf + lane;
      lsum_s[m] = red_f[m] + red_f[kTcRows + m] + red_f[2 * kTcRows + m] + red_f[3 * kTcRows + m];
    }
    float o[kTcHalf];
#pragma unroll
    for (int i = 0; i < kTcHalf; ++i) o[i] = 0.0f;
    if (n_st > 0 && !aborted) {
      aborted = !tc_wait(BAR(kBarPvDone + ((n_st - 1) & 1)), ((n_st - 1) >> 1) & 1, abort_s);
      tc_fence_after();
      // merge the O buffers: buffer k ran under references obm_s[k] and bound
      // 2^obe_s[k]; the live one under the final ones
      for (int k = 0; k <= ob; ++k) {
        float ok[kTcHalf];
        tmem_ld16(tl + kColO + kTcRows * k + kTcHalf * hf, ok);
        if (k == ob) {
#pragma unroll
          for (int i = 0; i < kTcHalf; ++i) o[i] += ok[i];
        } else {
          const int de = obe_s[k] - E;
          const float ef = (de <= -127) ? 0.0f : __int_as_float((127 + de) << 23);
#pragma unroll
          for (int i = 0; i < kTcHalf; ++i) {
            const float mk = obm_s[k * kTcRows + kTcHalf * hf + i];
            const float fk = (mk == -INFINITY) ? 0.0f : tc_ex2(mk - mr[i]) * ef;
            o[i] += fk * ok[i];
          }
        }
      }
    }
    aborted = __any_sync(0xFFFFFFFFu, aborted);
    if (aborted) {
      if (lane == 0 && p.err_flags) atomicOr(p.err_flags, KVQ_ERRF_WAIT_TIMEOUT);
      *abort_s = 1;
    }
    named_barrier(1, kSoftThreads);
    if (!*abort_s) {
      const float vsc = __int_as_float((127 + E) << 23);     // undo the 2^-E of P''
      const int d = t;                                        // O^T lane = head dim
      const bool direct = n_parts <= 1;
#pragma unroll
      for (int i = 0; i < kTcHalf; ++i) {
        const int m = kTcHalf * hf + i;
        if (m >= p.M) break;
        const int ir = m / p.G, gq = m - ir * p.G;
        const int64_t orow = (static_cast<int64_t>(r) * p.R + ir) * p.Hq + h * p.G + gq;
        const float l = lsum_s[m];
        if (direct) {
          const float inv = (l > 0.0f) ? vsc / l : 0.0f;
          p.out[orow * kHeadDim + d] = __bfloat16_as_ushort(__float2bfloat16_rn(o[i] * inv));
        } else {
          const int64_t slot = orow * p.n_parts_max + part;
          p.o_part[slot * kHeadDim + d] = o[i] * vsc;
          if (t == i) p.ml_part[slot] = make_float2(mcur_s[m], l);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kTcWarpTma) {
    tc_fence_after();
    tmem_dealloc(tmem, kTcTmemCols);
  }
}

}  // namespace

bool attn_tc_supported(const kvq_cache &c, const AttnShape &s) {
  const int bs = 1 << s.log2_block;
  return s.rows > 8 && s.rows <= kTcRows && bs >= 16 && bs <= kTcTok &&
         c.num_kv_heads % 4 == 0 && s.partition_tokens % kTcTok == 0 &&
         s.partition_tokens / bs <= kTcMaxPages && c.num_slots > 0 &&
         c.num_slots < (int64_t(1) << 31) &&
         (reinterpret_cast<uintptr_t>(c.k_scales) & 15u) == 0 &&
         (reinterpret_cast<uintptr_t>(c.v_scales) & 15u) == 0;
}

cudaError_t launch_attn_partials_tc(const kvq_cache &c, const AttnShape &s, const void *q,
                                    const int32_t *block_tables, const int32_t *context_lens,
                                    float sm_scale, void *out, float *o_part, float2 *ml_part,
                                    int32_t *err_flags, cudaStream_t stream) {
  TcParams p;
  p.num_blocks = c.num_slots >> s.log2_block;
  p.log2_bs = s.log2_block;
  p.bs = 1 << s.log2_block;
  p.q = static_cast<const uint16_t *>(q);
  p.out = static_cast<uint16_t *>(out);
  p.block_tables = block_tables;
  p.max_blocks = s.max_blocks_per_req;
  p.context_lens = context_lens;
  const int64_t cap = static_cast<int64_t>(s.max_blocks_per_req) << s.log2_block;
  p.ctx_limit = static_cast<int32_t>(cap < s.max_context_len ? cap : s.max_context_len);
  p.R = s.rows_per_request;
  p.Hq = s.num_q_heads;
  p.G = s.group;
  p.M = s.rows;
  p.qk_scale = sm_scale * 1.4426950408889634f;
  p.part_tokens = s.partition_tokens;
  p.n_parts_max = s.num_partitions;
  p.o_part = o_part;
  p.ml_part = ml_part;
  p.err_flags = err_flags;
  CUtensorMap mkc, mvc, mks, mvs;
  if (!encode_code_tensor_map(&mkc, c.k_codes, c.num_slots, c.num_kv_heads, p.bs) ||
      !encode_code_tensor_map(&mvc, c.v_codes, c.num_slots, c.num_kv_heads, p.bs) ||
      !encode_scale_tensor_map(&mks, c.k_scales, c.num_slots, c.num_kv_heads, p.bs) ||
      !encode_scale_tensor_map(&mvs, c.v_scales, c.num_slots, c.num_kv_heads, p.bs))
    return cudaErrorInvalidValue;
  static std::atomic<uint64_t> configured{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = (dev >= 0 && dev < 64) ? (uint64_t(1) << dev) : 0;
  if (bit == 0 || !(configured.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kTcSmem);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit, std::memory_order_acq_rel);
  }
  dim3 grid(c.num_kv_heads, s.num_partitions, s.num_requests);
  return launch_overlapped(attn_tc_kernel, grid, dim3(kTcThreads), kTcSmem, stream, p, mkc, mvc,
                           mks, mvs);
}

}  // namespace kvq
