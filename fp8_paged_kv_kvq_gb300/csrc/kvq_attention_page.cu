// kvq_attention_page.cu -- paged decode attention for up to 8 stacked query
// rows per KV head, the pages of four KV heads at a time, FP8 cache.
//
// Same method and per-chunk arithmetic as kvq_attention_skinny.cu (ROCm/ATOM
// PR #2655 "fix(qwen4-exp): register the QSA FP8 scale planes for KV offload",
// PR description, K/V bullet: per-token key scale on the score after the code
// dot, per-token value scale on the probability ahead of PV; transposed tiles S^T = K Q^T on FP8
// tensor cores with Q as two e4m3 pieces (exact for elements >= 2^-9 of the row's
// largest, off by <= 2^-17 of it below), O^T = V^T P^T on f16 tensor
// cores), with the loads laid out page-major:
//
//  * CTA = (group of 4 KV heads, partition, request).  Warps 0-3 each own one
//    KV head for the whole partition (no merge between warps); warp 4, one
//    lane, is the producer.
//  * The code planes are addressed through tensor maps ordered (128 bytes,
//    slots, heads): one 3-D box of 16 slots x 4 heads brings the 16-token
//    chunk of all four heads (8 KB, each head's rows 128-byte swizzled exactly
//    as one head's box would be) for K, one for V, and a 2-D box each scale
//    plane's 16 x 4 entries, into a 3-deep ring completing on the stage's
//    mbarrier.  Per byte this is a quarter of the TMA boxes of per-head loads,
//    the four heads of a page arrive together, and the compute warps never
//    issue a copy: they wait on the stage, compute, and release it.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>

#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {

namespace {

constexpr int kPgHeads = 4;                          // KV heads per CTA = compute warps
constexpr int kPgThreads = (kPgHeads + 1) * 32;      // + the producer warp
constexpr int kChunk = 16;                           // tokens per stage
constexpr int kPgStages = 3;
constexpr int kPgRows = 8;                           // stacked query rows per KV head
constexpr int kPgMaxPages = 512;
constexpr float kPgLazyRescale = 8.0f;

// shared memory from a 1024-byte aligned base; a stage is
// [K: head][row][128 B] | [V: head][row][128 B] | K scales [row][head] | V scales
constexpr int kPgCodeBytes = kPgHeads * kChunk * kHeadDim;            // 8 KiB
constexpr int kPgScBytes = kChunk * kPgHeads * 4;                     // 256 B
constexpr int kPgStageBytes = ((2 * kPgCodeBytes + 2 * kPgScBytes) + 1023) / 1024 * 1024;
constexpr int kOffPgQ = kPgStages * kPgStageBytes;                    // [head][2][8][128]
constexpr int kOffPgRowExp = kOffPgQ + kPgHeads * 2 * kPgRows * kHeadDim;
constexpr int kOffPgBt = kOffPgRowExp + kPgHeads * kPgRows * 4;
constexpr int kOffPgBar = kOffPgBt + kPgMaxPages * 4;
constexpr int kOffPgAbort = kOffPgBar + 2 * kPgStages * 8;
constexpr int kPgSmem = kOffPgAbort + 16 + 1024;

struct PgParams {
  int64_t num_blocks;
  int32_t H;
  int32_t log2_bs;
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

__device__ __forceinline__ float sk_ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Bounded wait that also gives up once another warp raised the abort flag.
__device__ __forceinline__ bool pg_wait(uint32_t bar, uint32_t parity, volatile int *abort) {
  for (int i = 0; i < (1 << 19); ++i) {
    if (mbar_try_wait_sleep(bar, parity, 2000u)) return true;
    if ((i & 15) == 15 && *abort) return false;
  }
  *abort = 1;
  return false;
}

__global__ void __launch_bounds__(kPgThreads, 3)
attn_page_kernel(const PgParams p, const __grid_constant__ CUtensorMap tmap_k,
                 const __grid_constant__ CUtensorMap tmap_v,
                 const __grid_constant__ CUtensorMap tmap_ks,
                 const __grid_constant__ CUtensorMap tmap_vs) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int g = lane >> 2;
  const int c = lane & 3;
  const int h0 = blockIdx.x * kPgHeads;
  const int part = blockIdx.y;
  const int r = blockIdx.z;

  // The launch overlaps the previous kernel's drain; every global access
  // (context lengths, block tables, queries, the cache, the outputs) comes
  // after the wait, so whatever a previous kernel wrote is visible.
  allow_dependents_launch();
  grid_dependency_wait();
  int L = p.context_lens[r];
  if (L < 0 || L > p.ctx_limit) {
    if (part == 0 && tid == 0 && h0 == 0 && p.err_flags) atomicOr(p.err_flags, KVQ_ERRF_CONTEXT_RANGE);
    L = L < 0 ? 0 : p.ctx_limit;
  }
  const int n_parts = (L + p.part_tokens - 1) / p.part_tokens;
  if (part >= (n_parts > 0 ? n_parts : 1)) return;
  const int t0 = part * p.part_tokens;
  const int t_end = min(L, t0 + p.part_tokens);
  const int n_chunks = (t_end > t0) ? (t_end - t0 + kChunk - 1) / kChunk : 0;
  const int page0 = t0 >> p.log2_bs;
  const int bs_mask = (1 << p.log2_bs) - 1;

  int32_t *bt_s = reinterpret_cast<int32_t *>(smem + kOffPgBt);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + kOffPgBar);
  uint64_t *empty = full + kPgStages;
  volatile int *abort_s = reinterpret_cast<volatile int *>(smem + kOffPgAbort);
  float *row_exp = reinterpret_cast<float *>(smem + kOffPgRowExp);

  // ---- partition block ids, barriers
  {
    const int n_pages = (t_end > t0) ? ((t_end - 1) >> p.log2_bs) - page0 + 1 : 0;
    const int32_t *bt = p.block_tables + static_cast<int64_t>(r) * p.max_blocks + page0;
    for (int i = tid; i < n_pages; i += kPgThreads) bt_s[i] = bt[i];
  }
  if (tid == 0) {
    for (int s = 0; s < kPgStages; ++s) {
      mbar_init(smem_addr(&full[s]), 1);
      mbar_init(smem_addr(&empty[s]), kPgHeads);
    }
    *abort_s = 0;
    fence_mbarrier_init();
  }
  __syncthreads();

  if (warp == kPgHeads) {
    // ---------------------------------------------------------- producer
    if (lane == 0) {
      int issued = 0;
      bool bad = false;
      for (int u = 0; u < n_chunks; ++u) {
        const int st = u % kPgStages;
        if (u >= kPgStages && !pg_wait(smem_addr(&empty[st]), ((u / kPgStages) - 1) & 1, abort_s))
          break;
        uint8_t *sb = smem + st * kPgStageBytes;
        const uint32_t fb = smem_addr(&full[st]);
        const int j = t0 + kChunk * u;                   // chunks lie within a page (bs >= 16)
        const int64_t blk = bt_s[(j >> p.log2_bs) - page0];
        uint32_t bytes = 0;
        if (blk < 0 || blk >= p.num_blocks) {
          bad = true;
        } else {
          const int z = static_cast<int>((blk << p.log2_bs) + (j & bs_mask));
          tma_load_3d(smem_addr(sb), &tmap_k, 0, z, h0, fb);
          tma_load_3d(smem_addr(sb + kPgCodeBytes), &tmap_v, 0, z, h0, fb);
          tma_load_2d(smem_addr(sb + 2 * kPgCodeBytes), &tmap_ks, h0, z, fb);
          tma_load_2d(smem_addr(sb + 2 * kPgCodeBytes + kPgScBytes), &tmap_vs, h0, z, fb);
          bytes = 2u * kPgCodeBytes + 2u * kPgScBytes;
        }
        mbar_arrive_expect_tx(fb, bytes);
        ++issued;
      }
      if (bad && p.err_flags) atomicOr(p.err_flags, KVQ_ERRF_BLOCK_RANGE);
      // copies still in flight (after an abort) land before the CTA leaves
      for (int u = (issued > kPgStages ? issued - kPgStages : 0); u < issued; ++u)
        mbar_wait_sleep_bounded(smem_addr(&full[u % kPgStages]), (u / kPgStages) & 1);
    }
    return;
  }

  // ------------------------------------------------------------ head warp
  const int w = warp;
  const int h = h0 + w;
  uint8_t *plane = smem + kOffPgQ + w * 2 * kPgRows * kHeadDim;   // [2][8][128]
  float *rexp = row_exp + w * kPgRows;
  auto q_row = [&](int m) {   // m < M
    const int i = m / p.G, gq = m - i * p.G;
    return p.q + ((static_cast<int64_t>(r) * p.R + i) * p.Hq + h * p.G + gq) * kHeadDim;
  };
  // query row exponents, then the two e4m3 pieces of each element:
  // q = 2^e (p1 + p2), 8 significant bits, all of bf16's
  // (all rows' loads first: one memory round trip for the warp's rows)
  uint2 vq[kPgRows];
#pragma unroll
  for (int m = 0; m < kPgRows; ++m)
    vq[m] = (m < p.M) ? *reinterpret_cast<const uint2 *>(q_row(m) + 4 * lane) : make_uint2(0u, 0u);
#pragma unroll
  for (int m = 0; m < kPgRows; ++m) {
    const uint2 v = vq[m];
    float amax = fmaxf(fmaxf(fabsf(bf16_lo(v.x)), fabsf(bf16_hi(v.x))),
                       fmaxf(fabsf(bf16_lo(v.y)), fabsf(bf16_hi(v.y))));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
      amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, off));
    const int ex = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFFu);
    int e = (ex == 0) ? -126 : ex - 127 - 7;
    e = e < -126 ? -126 : (e > 126 ? 126 : e);
    const float rx = (amax == 0.0f) ? 0.0f : __int_as_float((127 + e) << 23);   // 2^e
    if (lane == 0) rexp[m] = rx;
    uint32_t c1w = 0u, c2w = 0u;
    if (rx != 0.0f) {
      const float inv = __int_as_float((254u << 23) - __float_as_uint(rx));
      const float xs[4] = {bf16_lo(v.x) * inv, bf16_hi(v.x) * inv, bf16_lo(v.y) * inv,
                           bf16_hi(v.y) * inv};
      e4m3_pieces4(xs, c1w, c2w);
    }
    *reinterpret_cast<uint32_t *>(plane + m * kHeadDim + 4 * lane) = c1w;
    *reinterpret_cast<uint32_t *>(plane + kPgRows * kHeadDim + m * kHeadDim + 4 * lane) = c2w;
  }
  __syncwarp();
  uint32_t qb[4][2][2];
#pragma unroll
  for (int s2 = 0; s2 < 4; ++s2)
#pragma unroll
    for (int pc = 0; pc < 2; ++pc) {
      const uint2 wv = *reinterpret_cast<const uint2 *>(plane + pc * kPgRows * kHeadDim +
                                                        g * kHeadDim + 32 * c + 8 * s2);
      qb[s2][pc][0] = wv.x;
      qb[s2][pc][1] = wv.y;
    }

  // this thread's rows: n = 2c + e
  int vis[2];
  float rowf[2], m_run[2], l_run[2];
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    const int n = 2 * c + e;
    vis[e] = (n < p.M) ? (L - p.R + 1 + n / p.G) : 0;
    rowf[e] = (n < p.M) ? rexp[n] * p.qk_scale : 0.0f;
    m_run[e] = -INFINITY;
    l_run[e] = 0.0f;
  }
  float o[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int e = 0; e < 4; ++e) o[i][e] = 0.0f;
  int ev = -1000;
  bool timed_out = false;

  for (int u = 0; u < n_chunks; ++u) {
    const int st = u % kPgStages;
    if (!pg_wait(smem_addr(&full[st]), (u / kPgStages) & 1, abort_s)) {
      timed_out = true;
      break;
    }
    const uint8_t *sbase = smem + st * kPgStageBytes;
    const uint8_t *kb = sbase + w * kChunk * kHeadDim;
    const uint8_t *vb = sbase + kPgCodeBytes + w * kChunk * kHeadDim;
    const float *ksv = reinterpret_cast<const float *>(sbase + 2 * kPgCodeBytes) + w;
    const float *vsv = reinterpret_cast<const float *>(sbase + 2 * kPgCodeBytes + kPgScBytes) + w;
    const int j0 = t0 + kChunk * u;

    // ---- S^T = K Q^T: A = code rows of tokens g and g+8, dims 32c..32c+31
    uint32_t kl[8], kh[8];
    {
      const uint8_t *rl = kb + g * kHeadDim;
      const uint8_t *rh = kb + (g + 8) * kHeadDim;
      const uint4 a0 = *reinterpret_cast<const uint4 *>(rl + (((2 * c) ^ (g & 7)) << 4));
      const uint4 a1 = *reinterpret_cast<const uint4 *>(rl + (((2 * c + 1) ^ (g & 7)) << 4));
      const uint4 b0 = *reinterpret_cast<const uint4 *>(rh + (((2 * c) ^ (g & 7)) << 4));
      const uint4 b1 = *reinterpret_cast<const uint4 *>(rh + (((2 * c + 1) ^ (g & 7)) << 4));
      kl[0] = a0.x; kl[1] = a0.y; kl[2] = a0.z; kl[3] = a0.w;
      kl[4] = a1.x; kl[5] = a1.y; kl[6] = a1.z; kl[7] = a1.w;
      kh[0] = b0.x; kh[1] = b0.y; kh[2] = b0.z; kh[3] = b0.w;
      kh[4] = b1.x; kh[5] = b1.y; kh[6] = b1.z; kh[7] = b1.w;
    }
    // two independent accumulation chains (one per Q piece), added at the end
    float sacc[4] = {0.f, 0.f, 0.f, 0.f}, sacc2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int s2 = 0; s2 < 4; ++s2) {
      const uint32_t a[4] = {kl[2 * s2], kh[2 * s2], kl[2 * s2 + 1], kh[2 * s2 + 1]};
      mma_e4m3_16832(sacc, a, qb[s2][0][0], qb[s2][0][1]);
      mma_e4m3_16832(sacc2, a, qb[s2][1][0], qb[s2][1][1]);
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) sacc[e] += sacc2[e];

    // ---- scale, mask, online softmax.  sacc: [tok g][row 2c], [g][2c+1],
    // [g+8][2c], [g+8][2c+1]
    const float ks_lo = ksv[4 * g], ks_hi = ksv[4 * (g + 8)];
    float vs_lo = vsv[4 * g], vs_hi = vsv[4 * (g + 8)];
    float x[4];
    x[0] = sacc[0] * ks_lo * rowf[0];
    x[1] = sacc[1] * ks_lo * rowf[1];
    x[2] = sacc[2] * ks_hi * rowf[0];
    x[3] = sacc[3] * ks_hi * rowf[1];
    if (j0 + kChunk > min(vis[0], vis[1])) {      // some token of the chunk is masked
      x[0] = (j0 + g < vis[0]) ? x[0] : -INFINITY;
      x[1] = (j0 + g < vis[1]) ? x[1] : -INFINITY;
      x[2] = (j0 + g + 8 < vis[0]) ? x[2] : -INFINITY;
      x[3] = (j0 + g + 8 < vis[1]) ? x[3] : -INFINITY;
      // slots past the context end hold whatever they held: keep their value
      // scales out of the running bound
      vs_lo = (j0 + g < L) ? vs_lo : 0.0f;
      vs_hi = (j0 + g + 8 < L) ? vs_hi : 0.0f;
    }
    float mx0 = fmaxf(x[0], x[2]), mx1 = fmaxf(x[1], x[3]);
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
        if (mxs[e] > m_run[e] + kPgLazyRescale) {
          fac[e] = sk_ex2(m_run[e] - mxs[e]);
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
    const float vnorm = __int_as_float((127 - ev) << 23);
    const float ms0 = (m_run[0] == -INFINITY) ? 0.0f : m_run[0];
    const float ms1 = (m_run[1] == -INFINITY) ? 0.0f : m_run[1];
    const float p0 = sk_ex2(x[0] - ms0), p1 = sk_ex2(x[1] - ms1);
    const float p2 = sk_ex2(x[2] - ms0), p3 = sk_ex2(x[3] - ms1);
    l_run[0] += p0 + p2;
    l_run[1] += p1 + p3;
    const float wl = vs_lo * vnorm, wh = vs_hi * vnorm;
    // row 2c: (tok g, tok g+8); row 2c+1: (tok g, tok g+8)
    const uint32_t X = pack_f16x2(p0 * wl, p2 * wh);
    const uint32_t Y = pack_f16x2(p1 * wl, p3 * wh);
    // B = P^T: this lane (column = row g) needs tokens 2c, 2c+1 (b0) and 2c+8,
    // 2c+9 (b1) of row g, held by lanes 4*(2c) + g/2 and 4*(2c+1) + g/2
    const int la = 8 * c + (g >> 1), lb = la + 4;
    const uint32_t xa = __shfl_sync(0xFFFFFFFFu, X, la), ya = __shfl_sync(0xFFFFFFFFu, Y, la);
    const uint32_t xb = __shfl_sync(0xFFFFFFFFu, X, lb), yb = __shfl_sync(0xFFFFFFFFu, Y, lb);
    const uint32_t va = (g & 1) ? ya : xa;      // (tok 2c,   tok 2c+8)
    const uint32_t vc = (g & 1) ? yb : xb;      // (tok 2c+1, tok 2c+9)
    const uint32_t pb0 = prmt(va, vc, 0x5410u);
    const uint32_t pb1 = prmt(va, vc, 0x7632u);

    // ---- O^T += V^T P^T.  m-tile i, row g -> dim 16g + 2i, row g+8 -> 16g + 2i + 1;
    // this lane reads dims 16g..16g+15 of tokens 2c, 2c+1, 2c+8, 2c+9
    uint32_t wa[4], wb[4], wc[4], wd[4];
    {
      const int ta = 2 * c, tb = ta + 1, tc = ta + 8, td = ta + 9;
      const uint4 A = *reinterpret_cast<const uint4 *>(vb + ta * kHeadDim + ((g ^ (ta & 7)) << 4));
      const uint4 Bv = *reinterpret_cast<const uint4 *>(vb + tb * kHeadDim + ((g ^ (tb & 7)) << 4));
      const uint4 C = *reinterpret_cast<const uint4 *>(vb + tc * kHeadDim + ((g ^ (tc & 7)) << 4));
      const uint4 Dv = *reinterpret_cast<const uint4 *>(vb + td * kHeadDim + ((g ^ (td & 7)) << 4));
      wa[0] = A.x; wa[1] = A.y; wa[2] = A.z; wa[3] = A.w;
      wb[0] = Bv.x; wb[1] = Bv.y; wb[2] = Bv.z; wb[3] = Bv.w;
      wc[0] = C.x; wc[1] = C.y; wc[2] = C.z; wc[3] = C.w;
      wd[0] = Dv.x; wd[1] = Dv.y; wd[2] = Dv.z; wd[3] = Dv.w;
      // tokens at or past the context end hold whatever the slot or the stage
      // buffer held (a NaN code would poison the PV product even times p = 0)
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
    // m-tile i: dims 16g + 2i (a0, a2) and 16g + 2i + 1 (a1, a3) -- byte pairs
    // (token 2c, 2c+1) and (2c+8, 2c+9) of code bytes 2i, 2i+1
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
    if (lane == 0 && p.err_flags) atomicOr(p.err_flags, KVQ_ERRF_WAIT_TIMEOUT);
    return;
  }

  // ---- the warp's (max, denominator, O) are the partition's for its head
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    float l = l_run[e];
    l += __shfl_xor_sync(0xFFFFFFFFu, l, 4);
    l += __shfl_xor_sync(0xFFFFFFFFu, l, 8);
    l += __shfl_xor_sync(0xFFFFFFFFu, l, 16);
    l_run[e] = l;
  }
  // undo the 2^-ev of P''
  const float vsc = (ev == -1000) ? 0.0f : __int_as_float((127 + ev) << 23);
  // lane (g, c) holds rows 2c, 2c+1 at dims 16g + 2i (elements 0/1) and
  // 16g + 2i + 1 (elements 2/3): 16 consecutive dims per row
  const bool direct = n_parts <= 1;
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    const int n = 2 * c + e;
    if (n >= p.M) continue;
    const int i = n / p.G, gq = n - i * p.G;
    const int64_t orow = (static_cast<int64_t>(r) * p.R + i) * p.Hq + h * p.G + gq;
    if (direct) {
      const float inv = (l_run[e] > 0.0f) ? vsc / l_run[e] : 0.0f;
      uint32_t pk[8];
#pragma unroll
      for (int t = 0; t < 8; ++t) pk[t] = pack_bf16x2(o[t][e] * inv, o[t][2 + e] * inv);
      uint4 *dst = reinterpret_cast<uint4 *>(p.out + orow * kHeadDim + 16 * g);
      dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
      dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
    } else {
      const int64_t slot = orow * p.n_parts_max + part;
      float4 *dst = reinterpret_cast<float4 *>(p.o_part + slot * kHeadDim + 16 * g);
#pragma unroll
      for (int t = 0; t < 4; ++t)
        dst[t] = make_float4(o[2 * t][e] * vsc, o[2 * t][2 + e] * vsc, o[2 * t + 1][e] * vsc,
                             o[2 * t + 1][2 + e] * vsc);
      if (g == 0) p.ml_part[slot] = make_float2(m_run[e], l_run[e]);
    }
  }
}

// A map over one code plane [num_slots, H, 128] uint8 ordered (128 bytes,
// slots, heads): boxes of 16 slots x 4 heads, 128-byte swizzled per head.
bool encode_code_page_map(CUtensorMap *map, const uint8_t *codes, int64_t num_slots, int H) {
  return encode_code_tensor_map_strided(map, codes, num_slots, H);
}

}  // namespace

bool attn_page_supported(const kvq_cache &c, const AttnShape &s) {
  const int bs = 1 << s.log2_block;
  return s.rows <= kPgRows && bs >= kChunk && c.num_kv_heads % kPgHeads == 0 &&
         c.num_slots > 0 && c.num_slots < (int64_t(1) << 31) &&
         static_cast<int64_t>(s.partition_tokens) / bs + 1 <= kPgMaxPages &&
         (reinterpret_cast<uintptr_t>(c.k_scales) & 15u) == 0 &&
         (reinterpret_cast<uintptr_t>(c.v_scales) & 15u) == 0;
}

cudaError_t launch_attn_partials_page(const kvq_cache &c, const AttnShape &s, const void *q,
                                      const int32_t *block_tables, const int32_t *context_lens,
                                      float sm_scale, void *out, float *o_part, float2 *ml_part,
                                      int32_t *err_flags, cudaStream_t stream) {
  PgParams p;
  p.num_blocks = c.num_slots >> s.log2_block;
  p.H = c.num_kv_heads;
  p.log2_bs = s.log2_block;
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
  CUtensorMap mk, mv, mks, mvs;
  if (!encode_code_page_map(&mk, c.k_codes, c.num_slots, c.num_kv_heads) ||
      !encode_code_page_map(&mv, c.v_codes, c.num_slots, c.num_kv_heads) ||
      !encode_scale_tensor_map(&mks, c.k_scales, c.num_slots, c.num_kv_heads, kChunk) ||
      !encode_scale_tensor_map(&mvs, c.v_scales, c.num_slots, c.num_kv_heads, kChunk))
    return cudaErrorInvalidValue;
  static std::atomic<uint64_t> configured{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = (dev >= 0 && dev < 64) ? (uint64_t(1) << dev) : 0;
  if (bit == 0 || !(configured.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(attn_page_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kPgSmem);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit, std::memory_order_acq_rel);
  }
  dim3 grid(c.num_kv_heads / kPgHeads, s.num_partitions, s.num_requests);
  return launch_overlapped(attn_page_kernel, grid, dim3(kPgThreads), kPgSmem, stream, p, mk, mv,
                           mks, mvs);
}

}  // namespace kvq
