// kvq_attention_skinny.cu -- paged decode attention for up to 8 stacked query
// rows per KV head (decode with GQA <= 8, or short verify), FP8 cache.
//
// Same method as kvq_attention.cu (ROCm/ATOM PR #2655 "fix(qwen4-exp): register
// the QSA FP8 scale planes for KV offload", PR description, K/V bullet:
// per-token key scale on the score after the code dot, per-token value scale on
// the probability ahead of PV), laid out for few rows:
//
//  * The tiles are transposed: S^T = K Q^T and O^T = V^T P^T, so the tokens (and
//    the head dims) fill the MMA's 16-row M side and the <= 8 query rows the
//    8-wide N side.  QK^T runs on FP8 tensor cores (m16n8k32 e4m3) with the K
//    code bytes as the A operand as they sit in shared memory -- no decode --
//    and Q as two e4m3 pieces per element (B operand, registers; q = 2^e (p1 +
//    p2) exactly for elements >= 2^-9 of the row's largest, off by at most
//    2^-17 of it below that).  PV runs
//    on f16 tensor cores (m16n8k16) with V codes converted exactly to f16 by
//    the hardware e4m3x2 conversion and P'' = p * v_scale * 2^-E <= 1 (E a
//    running power-of-two bound on the value scales) moved from the S^T
//    fragment layout to the B layout with four shuffles per 16 tokens.
//  * Every warp streams its own 16-token chunks (chunks w, w+4, ... of the
//    partition) through its own 2-deep TMA pipeline: one box of min(bs, 16) code
//    rows per page for K and for V, completing on the warp's own mbarrier, and
//    the chunk's 32 scales by cp.async.  The main loop has no CTA-wide barrier.
//  * The four warps' (max, denominator, O) merge in shared memory at the end.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstring>

#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {

namespace {

constexpr int kSkWarps = 4;
constexpr int kSkThreads = kSkWarps * 32;
constexpr int kChunk = 16;                           // tokens per warp step
constexpr int kSkStages = 2;                         // chunks in flight per warp
constexpr int kChunkBytes = kChunk * kHeadDim;       // 2 KiB of codes per K or V
constexpr int kSkMaxPages = 1024;
constexpr int kSkRows = 8;                           // query rows per KV head handled
constexpr float kSkLazyRescale = 8.0f;
constexpr float kSkLog2e = 1.4426950408889634f;

// shared memory from a 1024-byte aligned base
constexpr int kWarpCode = kSkStages * 2 * kChunkBytes;                    // 8 KiB
constexpr int kOffSkScales = kSkWarps * kWarpCode;                         // [w][stage][32] f32
constexpr int kOffSkBar = kOffSkScales + kSkWarps * kSkStages * 2 * kChunk * 4;
constexpr int kOffSkQ = kOffSkBar + kSkWarps * kSkStages * 8;             // 2 planes x 8 x 128 B
constexpr int kOffSkRowExp = kOffSkQ + 2 * kSkRows * kHeadDim;
constexpr int kOffSkBt = kOffSkRowExp + kSkRows * 4;
constexpr int kSkSmem = kOffSkBt + kSkMaxPages * 4 + 1024;

struct SkParams {
  const uint8_t *k_codes;
  const uint8_t *v_codes;
  const float *k_scales;
  const float *v_scales;
  uint32_t num_blocks;        // < 2^31 (slots < 2^31)
  int32_t H;
  int32_t log2_bs;
  int32_t box_rows;          // min(bs, 16)
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

__global__ void __launch_bounds__(kSkThreads, 4)
attn_skinny_kernel(const SkParams p, const __grid_constant__ CUtensorMap tmap_k,
                   const __grid_constant__ CUtensorMap tmap_v) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int g = lane >> 2;
  const int c = lane & 3;
  const int h = blockIdx.x;
  const int part = blockIdx.y;
  const int r = blockIdx.z;

  // The launch overlaps the previous kernel's drain; every global access
  // (context lengths, block tables, queries, the cache, the outputs) comes
  // after the wait, so whatever a previous kernel wrote is visible.
  allow_dependents_launch();
  grid_dependency_wait();
  int L = p.context_lens[r];
  if (L < 0 || L > p.ctx_limit) {
    if (part == 0 && tid == 0 && h == 0 && p.err_flags) atomicOr(p.err_flags, KVQ_ERRF_CONTEXT_RANGE);
    L = L < 0 ? 0 : p.ctx_limit;
  }
  const int n_parts = (L + p.part_tokens - 1) / p.part_tokens;
  if (part >= (n_parts > 0 ? n_parts : 1)) return;
  const int t0 = part * p.part_tokens;
  const int t_end = min(L, t0 + p.part_tokens);
  const int n_chunks = (t_end > t0) ? (t_end - t0 + kChunk - 1) / kChunk : 0;
  const int page0 = t0 >> p.log2_bs;
  const int bs_mask = (1 << p.log2_bs) - 1;

  int32_t *bt_s = reinterpret_cast<int32_t *>(smem + kOffSkBt);
  uint64_t *bar = reinterpret_cast<uint64_t *>(smem + kOffSkBar) + warp * kSkStages;
  uint8_t *wcode = smem + warp * kWarpCode;           // [stage][K 2K | V 2K]
  float *wscale = reinterpret_cast<float *>(smem + kOffSkScales) + warp * kSkStages * 2 * kChunk;
  uint8_t *plane = smem + kOffSkQ;                    // [2][8][128]
  float *row_exp = reinterpret_cast<float *>(smem + kOffSkRowExp);

  // ---- partition block ids, barriers, query row exponents
  {
    const int n_pages = (t_end > t0) ? ((t_end - 1) >> p.log2_bs) - page0 + 1 : 0;
    const int32_t *bt = p.block_tables + static_cast<int64_t>(r) * p.max_blocks + page0;
    for (int i = tid; i < n_pages; i += kSkThreads) bt_s[i] = bt[i];
  }
  if (tid == 0) {
    uint64_t *all = reinterpret_cast<uint64_t *>(smem + kOffSkBar);
    for (int b = 0; b < kSkWarps * kSkStages; ++b) mbar_init(smem_addr(&all[b]), 1);
    fence_mbarrier_init();
    fence_proxy_async_smem();
  }
  auto q_row = [&](int m) {   // m < M
    const int i = m / p.G, gq = m - i * p.G;
    return p.q + ((static_cast<int64_t>(r) * p.R + i) * p.Hq + h * p.G + gq) * kHeadDim;
  };
  // ---- query rows m = warp, warp + 4: both loaded at once, then per row its
  // exponent and the two e4m3 pieces of each element, q = 2^e (p1 + p2), into
  // the B planes
  {
    constexpr int kRowsPerWarp = kSkRows / kSkWarps;
    uint2 v[kRowsPerWarp];
#pragma unroll
    for (int k = 0; k < kRowsPerWarp; ++k) {
      const int m = warp + kSkWarps * k;
      v[k] = (m < p.M) ? *reinterpret_cast<const uint2 *>(q_row(m) + 4 * lane) : make_uint2(0u, 0u);
    }
#pragma unroll
    for (int k = 0; k < kRowsPerWarp; ++k) {
      const int m = warp + kSkWarps * k;
      float amax = fmaxf(fmaxf(fabsf(bf16_lo(v[k].x)), fabsf(bf16_hi(v[k].x))),
                         fmaxf(fabsf(bf16_lo(v[k].y)), fabsf(bf16_hi(v[k].y))));
#pragma unroll
      for (int off = 16; off > 0; off >>= 1)
        amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, off));
      const int ex = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFFu);
      int e = (ex == 0) ? -126 : ex - 127 - 7;
      e = e < -126 ? -126 : (e > 126 ? 126 : e);
      const float rx = (amax == 0.0f) ? 0.0f : __int_as_float((127 + e) << 23);   // 2^e
      if (lane == 0) row_exp[m] = rx;
      uint32_t c1w = 0u, c2w = 0u;
      if (rx != 0.0f) {
        const float inv = __int_as_float((254u << 23) - __float_as_uint(rx));
        const float xs[4] = {bf16_lo(v[k].x) * inv, bf16_hi(v[k].x) * inv, bf16_lo(v[k].y) * inv,
                             bf16_hi(v[k].y) * inv};
        e4m3_pieces4(xs, c1w, c2w);
      }
      *reinterpret_cast<uint32_t *>(plane + m * kHeadDim + 4 * lane) = c1w;
      *reinterpret_cast<uint32_t *>(plane + kSkRows * kHeadDim + m * kHeadDim + 4 * lane) = c2w;
    }
  }
  __syncthreads();

  // ---- the warp's pipeline: chunk u of this warp covers tokens
  // t0 + 16 * (warp + 4u) .. +16
  const int n_my = (n_chunks > warp) ? (n_chunks - warp + kSkWarps - 1) / kSkWarps : 0;
  const float *scale_base = ((lane < 16) ? p.k_scales : p.v_scales) + h;
  auto issue = [&](int u) {
    if (u < n_my) {
      const int sb = u % kSkStages;
      const int j0 = t0 + kChunk * (warp + kSkWarps * u);
      if (lane == 0) {
        const uint32_t kdst = smem_addr(wcode + sb * 2 * kChunkBytes);
        const uint32_t vdst = kdst + kChunkBytes;
        const uint32_t b = smem_addr(&bar[sb]);
        uint32_t bytes = 0;
        bool bad = false;
        fence_proxy_async_smem();
        for (int i = 0; i < kChunk / p.box_rows; ++i) {
          const int j = j0 + i * p.box_rows;
          if (j >= t_end) break;
          const uint32_t blk = static_cast<uint32_t>(bt_s[(j >> p.log2_bs) - page0]);
          if (blk >= p.num_blocks) {             // also every negative id
            bad = true;
            continue;
          }
          const int z = static_cast<int>((blk << p.log2_bs) | (j & bs_mask));
          tma_load_3d(kdst + i * p.box_rows * kHeadDim, &tmap_k, 0, h, z, b);
          tma_load_3d(vdst + i * p.box_rows * kHeadDim, &tmap_v, 0, h, z, b);
          bytes += 2u * p.box_rows * kHeadDim;
        }
        if (bad && p.err_flags) atomicOr(p.err_flags, KVQ_ERRF_BLOCK_RANGE);
        mbar_arrive_expect_tx(b, bytes);
      }
      // lanes 0..15: K scales, 16..31: V scales of the chunk's tokens (32-bit
      // slot arithmetic: slots < 2^31)
      const int j = j0 + (lane & 15);
      const float *src = scale_base;
      uint32_t nbytes = 0;
      if (j < t_end) {
        const uint32_t blk = static_cast<uint32_t>(bt_s[(j >> p.log2_bs) - page0]);
        if (blk < p.num_blocks) {
          src = scale_base + static_cast<uint64_t>((blk << p.log2_bs) | (j & bs_mask)) * p.H;
          nbytes = 4;
        }
      }
      cp_async_4(wscale + sb * 2 * kChunk + lane, src, nbytes);
    }
    cp_async_commit();
  };
#pragma unroll
  for (int u = 0; u < kSkStages; ++u) issue(u);

  // B fragments of the query pieces for k-step s2 (dims 32 s2 .. +31), row g:
  // b0 = dims 32 s2 + 4c + 0..3, b1 = dims 32 s2 + 16 + 4c + 0..3
  uint32_t qb[4][2][2];
#pragma unroll
  for (int s2 = 0; s2 < 4; ++s2)
#pragma unroll
    for (int pc = 0; pc < 2; ++pc) {
      const uint8_t *qr = plane + pc * kSkRows * kHeadDim + g * kHeadDim + 32 * s2 + 4 * c;
      qb[s2][pc][0] = *reinterpret_cast<const uint32_t *>(qr);
      qb[s2][pc][1] = *reinterpret_cast<const uint32_t *>(qr + 16);
    }
  // this lane's ldmatrix row address within a K tile, per k-step: token row
  // (lane & 7) + 8 ((lane >> 3) & 1), 16-byte chunk 2 s2 + (lane >> 4), 128-byte
  // swizzled (chunk ^ row & 7)
  const int ld_row = (lane & 7) + 8 * ((lane >> 3) & 1);
  uint32_t ld_off[4];
#pragma unroll
  for (int s2 = 0; s2 < 4; ++s2)
    ld_off[s2] = ld_row * kHeadDim + (((2 * s2 + (lane >> 4)) ^ (lane & 7)) << 4);

  // this thread's rows: n = 2c + e
  int vis[2];
  float rowf[2], m_run[2], l_run[2];
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    const int n = 2 * c + e;
    vis[e] = (n < p.M) ? (L - p.R + 1 + n / p.G) : 0;
    rowf[e] = (n < p.M) ? row_exp[n] * p.qk_scale : 0.0f;
    m_run[e] = -INFINITY;
    l_run[e] = 0.0f;
  }
  float o[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int e = 0; e < 4; ++e) o[i][e] = 0.0f;
  int ev = -1000;
  // cached forms of the running state: the rescale thresholds m_run + lazy
  // margin, the exponent base (0 while no score was seen), the value bound
  // 2^ev (below every scale before the first chunk) and 2^-ev
  float thr[2] = {-INFINITY, -INFINITY}, ms[2] = {0.0f, 0.0f};
  float vbound = -1.0f, vnorm = 1.0f;
  bool timed_out = false;

#pragma unroll 2
  for (int u = 0; u < n_my; ++u) {
    const int sb = u % kSkStages;
    cp_async_wait<kSkStages - 1>();
    const bool ok = mbar_wait_sleep_bounded(smem_addr(&bar[sb]), (u / kSkStages) & 1);
    if (__any_sync(0xFFFFFFFFu, !ok)) {
      // give up on this warp's chunks: let its copies in flight land (bounded)
      timed_out = true;
      for (int v = u; v < min(n_my, u + kSkStages); ++v)
        mbar_wait_sleep_bounded(smem_addr(&bar[v % kSkStages]), (v / kSkStages) & 1);
      break;
    }
    __syncwarp();
    const uint8_t *kb = wcode + sb * 2 * kChunkBytes;
    const uint8_t *vb = kb + kChunkBytes;
    const float *ksv = wscale + sb * 2 * kChunk;
    const float *vsv = ksv + kChunk;
    const int j0 = t0 + kChunk * (warp + kSkWarps * u);

    // ---- S^T = K Q^T: A = the K tile's code rows (tokens) by ldmatrix, in
    // fragment order; two independent accumulation chains (one per Q piece)
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

    // ---- scale, mask, online softmax.  sacc: [tok g][row 2c], [g][2c+1],
    // [g+8][2c], [g+8][2c+1]
    const float ks_lo = ksv[g], ks_hi = ksv[g + 8];
    const float vs_lo = vsv[g], vs_hi = vsv[g + 8];
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
    }
    // The running max moves only when a score passes it by more than the lazy
    // margin and the value bound only when a scale passes it; after the first
    // chunks both are rare, so the warp reductions and the rescale run only
    // when some lane sees one (the same updates as reducing every chunk).
    const bool need = x[0] > thr[0] || x[2] > thr[0] || x[1] > thr[1] || x[3] > thr[1] ||
                      vs_lo > vbound || vs_hi > vbound;
    if (__any_sync(0xFFFFFFFFu, need)) {
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
          if (mxs[e] > m_run[e] + kSkLazyRescale) {
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
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        thr[e] = m_run[e] + kSkLazyRescale;
        ms[e] = (m_run[e] == -INFINITY) ? 0.0f : m_run[e];
      }
      vbound = __int_as_float((127 + ev) << 23);      // 2^ev, ev in [-126, 126]
      vnorm = __int_as_float((127 - ev) << 23);
    }
    const float ms0 = ms[0], ms1 = ms[1];
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
    issue(u + kSkStages);
  }

  // ---- merge the warps (a CTA with a warp that gave up writes nothing)
  cp_async_wait<0>();
  if (timed_out && lane == 0 && p.err_flags) atomicOr(p.err_flags, KVQ_ERRF_WAIT_TIMEOUT);
  if (__syncthreads_or(timed_out ? 1 : 0)) return;
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    float l = l_run[e];
    l += __shfl_xor_sync(0xFFFFFFFFu, l, 4);
    l += __shfl_xor_sync(0xFFFFFFFFu, l, 8);
    l += __shfl_xor_sync(0xFFFFFFFFu, l, 16);
    l_run[e] = l;
  }
  float *m_w = reinterpret_cast<float *>(smem);               // [4][8]
  float *l_w = m_w + kSkWarps * kSkRows;                       // [4][8]
  float4 *parked = reinterpret_cast<float4 *>(l_w + kSkWarps * kSkRows);   // [3][8][32]
  if (g == 0) {
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      m_w[warp * kSkRows + 2 * c + e] = m_run[e];
      l_w[warp * kSkRows + 2 * c + e] = l_run[e];
    }
  }
  __syncthreads();
  float mrow[2], lrow[2], frow[2];
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    const int n = 2 * c + e;
    float mx = -INFINITY;
#pragma unroll
    for (int w = 0; w < kSkWarps; ++w) mx = fmaxf(mx, m_w[w * kSkRows + n]);
    float lt = 0.0f;
    if (mx != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kSkWarps; ++w) lt += l_w[w * kSkRows + n] * sk_ex2(m_w[w * kSkRows + n] - mx);
    }
    mrow[e] = mx;
    lrow[e] = lt;
    frow[e] = (mx == -INFINITY || ev == -1000) ? 0.0f : ldexpf(sk_ex2(m_run[e] - mx), ev);
  }
  if (warp > 0) {
#pragma unroll
    for (int i = 0; i < 8; ++i)
      parked[((warp - 1) * 8 + i) * 32 + lane] =
          make_float4(o[i][0] * frow[0], o[i][1] * frow[1], o[i][2] * frow[0], o[i][3] * frow[1]);
  }
  __syncthreads();
  if (warp != 0) return;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    float4 acc = make_float4(o[i][0] * frow[0], o[i][1] * frow[1], o[i][2] * frow[0], o[i][3] * frow[1]);
#pragma unroll
    for (int w = 0; w < kSkWarps - 1; ++w) {
      const float4 v = parked[(w * 8 + i) * 32 + lane];
      acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
    }
    o[i][0] = acc.x; o[i][1] = acc.y; o[i][2] = acc.z; o[i][3] = acc.w;
  }
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
      const float inv = (lrow[e] > 0.0f) ? 1.0f / lrow[e] : 0.0f;
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
        dst[t] = make_float4(o[2 * t][e], o[2 * t][2 + e], o[2 * t + 1][e], o[2 * t + 1][2 + e]);
      if (g == 0) p.ml_part[slot] = make_float2(mrow[e], lrow[e]);
    }
  }
}

}  // namespace

bool attn_skinny_supported(const kvq_cache &c, const AttnShape &s) {
  const int bs = 1 << s.log2_block;
  return s.rows <= kSkRows && bs >= 8 && c.num_slots > 0 && c.num_slots < (int64_t(1) << 31) &&
         static_cast<int64_t>(s.partition_tokens) / (bs < 16 ? bs : 16) + 1 <= kSkMaxPages;
}

cudaError_t launch_attn_partials_skinny(const kvq_cache &c, const AttnShape &s, const void *q,
                                        const int32_t *block_tables, const int32_t *context_lens,
                                        float sm_scale, void *out, float *o_part,
                                        float2 *ml_part, int32_t *err_flags,
                                        cudaStream_t stream) {
  SkParams p;
  p.k_codes = c.k_codes;
  p.v_codes = c.v_codes;
  p.k_scales = c.k_scales;
  p.v_scales = c.v_scales;
  p.num_blocks = static_cast<uint32_t>(c.num_slots >> s.log2_block);
  p.H = c.num_kv_heads;
  p.log2_bs = s.log2_block;
  const int bs = 1 << s.log2_block;
  p.box_rows = bs < kChunk ? bs : kChunk;
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
  p.qk_scale = sm_scale * kSkLog2e;
  p.part_tokens = s.partition_tokens;
  p.n_parts_max = s.num_partitions;
  p.o_part = o_part;
  p.ml_part = ml_part;
  p.err_flags = err_flags;
  CUtensorMap mk, mv;
  if (!encode_code_tensor_map(&mk, c.k_codes, c.num_slots, c.num_kv_heads, p.box_rows) ||
      !encode_code_tensor_map(&mv, c.v_codes, c.num_slots, c.num_kv_heads, p.box_rows))
    return cudaErrorInvalidValue;
  static std::atomic<uint64_t> configured{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = (dev >= 0 && dev < 64) ? (uint64_t(1) << dev) : 0;
  if (bit == 0 || !(configured.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(attn_skinny_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSkSmem);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit, std::memory_order_acq_rel);
  }
  dim3 grid(c.num_kv_heads, s.num_partitions, s.num_requests);
  return launch_overlapped(attn_skinny_kernel, grid, dim3(kSkThreads), kSkSmem, stream, p, mk, mv);
}

}  // namespace kvq
