// kvq_index_scores.cu -- stacked index scoring over the compressed index keys.
//
// ROCm/ATOM PR #2655 "fix(qwen4-exp): register the QSA FP8 scale planes for KV
// offload", PR description: the decode-time scorer there multiplies all R query
// rows x H index heads of a request against each cached index key in a single
// matrix product, so every key is loaded once per step; each head's dot product
// is clipped at zero (ReLU) and the clipped values are added into the row's
// score.  Keys are FP8 plus an FP32 scale for each row, or MXFP4 (two E2M1
// codes per byte and an E8M0 exponent for every 32 dims):
//     score(r, i, t) = sum_h max(0, <q(r, i, h), khat_t>),
// -inf where row i does not see token t (t >= L - R + 1 + i).
//
// Layout of the work: a persistent grid (CTAs resident at once) over the
// flattened sequence of (request, 128-token chunk) units, each CTA a
// contiguous run of it.  One producer warp streams the chunks' index keys --
// codes and the per-token scale / exponent bytes, one bulk copy per page
// segment -- into a ring of shared-memory stages; four consumer warps take two
// 16-token tiles of each chunk.  The tokens fill the MMA's M side and the
// R * H <= 16 query vectors its N side (two n8 tiles): S^T = K Q^T on f16
// tensor cores (m16n8k16), fp32 accumulate.  Both key formats convert exactly
// to f16 (every e4m3 and E2M1 value is an f16).  The k order of the
// contraction is permuted so that lane c of a quad holds the contiguous dims
// 32c .. 32c + 31 of its two token rows -- for MXFP4 exactly one exponent
// group -- and the query's B fragments follow the same permutation.  MXFP4
// groups are brought to the token's largest exponent before the MMA (powers of
// two, exact down to f16's smallest subnormal) and the token scale is applied
// after it; each query vector is held in f16 scaled by a power of two, set up
// by every consumer warp from global memory when its run enters a request.
#include <cuda_runtime.h>

#include <atomic>

#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {

namespace {

constexpr int kScWarps = 4;                          // consumer warps
constexpr int kScThreads = (kScWarps + 1) * 32;      // + the producer warp
constexpr int kScTile = 16;                          // tokens per MMA tile
constexpr int kScChunk = 128;                        // tokens per stage
constexpr int kScStages = 4;
constexpr int kScIdAhead = 8;                        // chunks whose block ids are in flight
constexpr int kScCols = 16;                          // stacked query vectors

template <int kFormat>
struct ScFmt {
  static constexpr int kRowBytes = kFormat == KVQ_INDEX_MXFP4 ? kHeadDim / 2 : kHeadDim;
  static constexpr int kCodeBytes = kScChunk * kRowBytes;
  static constexpr int kStageBytes = kCodeBytes + kScChunk * 4;   // + scale / exponent words
  static constexpr int kOffBars = kScStages * kStageBytes;
  static constexpr int kOffIds = kOffBars + 2 * kScStages * 8 + 16;   // [kScIdAhead + 1][32]
  static constexpr int kSmem = kOffIds + (kScIdAhead + 1) * 32 * 4;
};

struct ScParams {
  const uint8_t *codes;
  const float *scales;
  const uint8_t *exps;
  uint32_t num_blocks;
  int32_t log2_bs;                                   // >= 4
  const uint16_t *q;
  int32_t R;
  const int32_t *block_tables;
  int32_t max_blocks;
  const int32_t *context_lens;
  int32_t ctx_limit;
  int32_t max_len;
  int32_t nch;                                       // chunks per request
  int64_t total;                                     // num_requests * nch
  float *out;
  int32_t *err_flags;
};

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Two bytes of E2M1 pairs (low byte first) to two f16x2 words, low nibble in
// the low half.
__device__ __forceinline__ void e2m1x4_to_f16x2x2(uint32_t w16, uint32_t &lo, uint32_t &hi) {
  asm("{\n .reg .b8 c0, c1;\n mov.b16 {c0, c1}, %2;\n cvt.rn.f16x2.e2m1x2 %0, c0;\n"
      " cvt.rn.f16x2.e2m1x2 %1, c1;\n}\n"
      : "=r"(lo), "=r"(hi) : "h"(static_cast<uint16_t>(w16)));
}

// 2^x as binary32 for x in [-149, 127].
__device__ __forceinline__ float exp2i(int x) {
  return x >= -126 ? __uint_as_float(static_cast<uint32_t>(127 + x) << 23)
                   : __uint_as_float(1u << (x + 149));
}

// 1-D bulk copy global -> shared, completing on `bar` (16-byte aligned
// addresses, size a multiple of 16).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n"
      :: "r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}

// Bounded wait that also gives up once another warp raised the abort flag.
__device__ __forceinline__ bool sc_wait(uint32_t bar, uint32_t parity, volatile int *abort) {
  for (int i = 0; i < (1 << 19); ++i) {
    if (mbar_try_wait_sleep(bar, parity, 2000u)) return true;
    if ((i & 15) == 15 && *abort) return false;
  }
  *abort = 1;
  return false;
}

__device__ __forceinline__ int sc_context(const ScParams &p, int r) {
  const int L = p.context_lens[r];
  return L < 0 ? 0 : (L > p.ctx_limit ? p.ctx_limit : L);
}

template <int kFormat, int kH>
__global__ void __launch_bounds__(kScThreads, 4)
index_scores_kernel(const ScParams p) {
  using F = ScFmt<kFormat>;
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + F::kOffBars);
  uint64_t *empty = full + kScStages;
  volatile int *abort_s = reinterpret_cast<volatile int *>(empty + kScStages);
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int64_t x_begin = blockIdx.x * p.total / gridDim.x;
  const int64_t x_end = (blockIdx.x + 1) * p.total / gridDim.x;
  const int n_units = static_cast<int>(x_end - x_begin);

  // The launch overlaps the previous kernel's drain; every global access comes
  // after the wait, so whatever a previous kernel wrote is visible.
  allow_dependents_launch();
  grid_dependency_wait();
  if (tid == 0) {
    for (int s = 0; s < kScStages; ++s) {
      mbar_init(smem_addr(&full[s]), 1);
      mbar_init(smem_addr(&empty[s]), kScWarps);
    }
    *abort_s = 0;
    fence_mbarrier_init();
  }
  __syncthreads();
  if (n_units <= 0) return;
  const int r_begin = static_cast<int>(x_begin / p.nch);
  const int k_begin = static_cast<int>(x_begin - static_cast<int64_t>(r_begin) * p.nch);

  if (warp == kScWarps) {
    // ------------------------------------------------------------ producer
    // lane i copies page segment i of a chunk: tokens [128k + i*seg, +seg)
    const int seg = p.log2_bs >= 7 ? kScChunk : (1 << p.log2_bs);
    const int nseg = kScChunk / seg;
    bool bad = false, stop = false;
    // Block ids go to shared memory by cp.async kScIdAhead chunks ahead of
    // their stage (one commit group per chunk; lane i: page segment i), so no
    // chunk waits for a block-table read.
    int32_t *ids = reinterpret_cast<int32_t *>(smem + F::kOffIds);
    const int nreq = static_cast<int>(p.total / p.nch);
    int fr = r_begin, fk = k_begin, fu = 0;
    int fL = sc_context(p, fr);
    auto fetch_next = [&]() {
      if (fu < n_units) {
        const int j = fk * kScChunk + lane * seg;
        const bool need = lane < nseg && j < fL;
        const int32_t *src = p.block_tables + static_cast<int64_t>(fr) * p.max_blocks +
                             (need ? (j >> p.log2_bs) : 0);
        cp_async_4(ids + (fu % (kScIdAhead + 1)) * 32 + lane, src, need ? 4u : 0u);
        if (++fk == p.nch) {
          fk = 0;
          if (++fr < nreq) fL = sc_context(p, fr);
        }
      }
      cp_async_commit();
      ++fu;
    };
    for (int a = 0; a < kScIdAhead; ++a) fetch_next();
    int r = r_begin, k = k_begin;
    int L = sc_context(p, r);
    int u = 0;
    for (; u < n_units; ++u) {
      fetch_next();                             // chunk u + kScIdAhead
      cp_async_wait<kScIdAhead>();              // chunk u's ids have landed
      __syncwarp();
      const int j = k * kScChunk + lane * seg;
      const bool has = lane < nseg && j < L;
      const uint32_t blk = has ? static_cast<uint32_t>(ids[(u % (kScIdAhead + 1)) * 32 + lane])
                               : 0u;
      const int st = u % kScStages;
      if (u >= kScStages) {
        if (lane == 0)
          stop = !sc_wait(smem_addr(&empty[st]), ((u / kScStages) - 1) & 1, abort_s);
        stop = __shfl_sync(0xFFFFFFFFu, stop ? 1 : 0, 0) != 0;
        if (stop) break;
      }
      const bool ok = has && blk < p.num_blocks;     // also every negative id
      bad |= has && !ok;
      const uint32_t bytes = ok ? static_cast<uint32_t>(seg * (F::kRowBytes + 4)) : 0u;
      const uint32_t tx = __reduce_add_sync(0xFFFFFFFFu, bytes);
      const uint32_t fb = smem_addr(&full[st]);
      if (lane == 0) mbar_arrive_expect_tx(fb, tx);
      __syncwarp();
      if (ok) {
        const int64_t slot = (static_cast<int64_t>(blk) << p.log2_bs) |
                             (j & ((1 << p.log2_bs) - 1));
        uint8_t *sb = smem + st * F::kStageBytes;
        bulk_load(smem_addr(sb + lane * seg * F::kRowBytes), p.codes + slot * F::kRowBytes,
                  static_cast<uint32_t>(seg * F::kRowBytes), fb);
        const void *side = kFormat == KVQ_INDEX_FP8
                               ? static_cast<const void *>(p.scales + slot)
                               : static_cast<const void *>(p.exps + slot * 4);
        bulk_load(smem_addr(sb + F::kCodeBytes + lane * seg * 4), side,
                  static_cast<uint32_t>(seg * 4), fb);
      }
      if (++k == p.nch) {
        k = 0;
        if (++r < nreq) L = sc_context(p, r);
      }
    }
    cp_async_wait<0>();
    bad = __any_sync(0xFFFFFFFFu, bad);
    if (lane == 0) {
      if (bad && p.err_flags) atomicOr(p.err_flags, KVQ_ERRF_BLOCK_RANGE);
      // copies still in flight (after an abort) land before the CTA leaves
      for (int v = (u > kScStages ? u - kScStages : 0); v < u; ++v)
        mbar_wait_sleep_bounded(smem_addr(&full[v % kScStages]), (v / kScStages) & 1);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int g = lane >> 2;
  const int c = lane & 3;
  const int nq = p.R * kH;
  constexpr int kU = kH == 1 ? 2 : 1;
  uint32_t qb[2][8][2];
  float hcs[2][2];                                   // column scales / 2
  float *orow[2][kU];
  int vis[2][kU];
  int L = 0, vis_min = 0;
  // the request's query vectors as B fragments -- tile t (vector 8t + g),
  // k-step s: b0 = dims 32c + 4s + 0, 1; b1 = dims 32c + 4s + 2, 3 -- each
  // vector scaled by 2^-e so that its largest magnitude lies in [2^7, 2^8)
  auto setup = [&](int r) {
    const int Lraw = p.context_lens[r];
    if ((Lraw < 0 || Lraw > p.ctx_limit) && tid == 0 && p.err_flags)
      atomicOr(p.err_flags, KVQ_ERRF_CONTEXT_RANGE);
    L = sc_context(p, r);
    vis_min = L - p.R + 1;                           // row 0 sees the fewest tokens
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const int n = 8 * t + g;
      uint4 v[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) v[i] = make_uint4(0u, 0u, 0u, 0u);
      if (n < nq) {
        const uint4 *src = reinterpret_cast<const uint4 *>(
            p.q + (static_cast<int64_t>(r) * nq + n) * kHeadDim + 32 * c);
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = __ldg(src + i);
      }
      // largest magnitude from the bf16 bits (|x| orders as the bits do)
      uint32_t m2 = 0;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        m2 = __vmaxu2(m2, v[i].x & 0x7FFF7FFFu);
        m2 = __vmaxu2(m2, v[i].y & 0x7FFF7FFFu);
        m2 = __vmaxu2(m2, v[i].z & 0x7FFF7FFFu);
        m2 = __vmaxu2(m2, v[i].w & 0x7FFF7FFFu);
      }
      uint32_t mb = max(m2 & 0xFFFFu, m2 >> 16);
      mb = max(mb, __shfl_xor_sync(0xFFFFFFFFu, mb, 1));
      mb = max(mb, __shfl_xor_sync(0xFFFFFFFFu, mb, 2));
      const float amax = __uint_as_float(mb << 16);
      int e = 0;
      if (amax != 0.0f) {
        int kx;
        frexpf(amax, &kx);                           // amax in [2^(kx-1), 2^kx)
        e = kx - 8;
      }
      const int ne = -e;                             // in [-120, 141]
      const float s1 = exp2i(ne < 127 ? ne : 127), s2 = exp2i(ne < 127 ? 0 : ne - 127);
      const uint32_t w[16] = {v[0].x, v[0].y, v[0].z, v[0].w, v[1].x, v[1].y, v[1].z, v[1].w,
                              v[2].x, v[2].y, v[2].z, v[2].w, v[3].x, v[3].y, v[3].z, v[3].w};
#pragma unroll
      for (int m = 0; m < 16; ++m) {
        const uint32_t h2 = pack_f16x2(bf16_lo(w[m]) * s1 * s2, bf16_hi(w[m]) * s1 * s2);
        qb[t][m >> 1][m & 1] = h2;
      }
      const float qsc = amax == 0.0f ? 0.0f : exp2i(e);
      hcs[t][0] = 0.5f * __shfl_sync(0xFFFFFFFFu, qsc, 4 * (2 * c));
      hcs[t][1] = 0.5f * __shfl_sync(0xFFFFFFFFu, qsc, 4 * (2 * c + 1));
      // accumulator column 2c + u is vector 8t + 2c + u = row n / H, head
      // n % H.  With H = 1 a lane owns two rows per tile; otherwise a row's
      // heads sit on 1, 2 or 4 lanes and the lowest of them writes.
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int nn = 8 * t + 2 * c + u;
        const int i = nn / kH;
        const bool writer = kH <= 2 || (kH == 4 ? (c & 1) == 0 : c == 0);
        orow[t][u] = (writer && i < p.R)
                         ? p.out + (static_cast<int64_t>(r) * p.R + i) * p.max_len : nullptr;
        vis[t][u] = L - p.R + 1 + i;
      }
    }
  };

  int r = r_begin, k = k_begin, cur_r = r_begin;
  setup(r_begin);
  for (int u = 0; u < n_units; ++u) {
    if (r != cur_r) {
      setup(r);
      cur_r = r;
    }
    const int st = u % kScStages;
    if (!sc_wait(smem_addr(&full[st]), (u / kScStages) & 1, abort_s)) {
      if (lane == 0 && p.err_flags) atomicOr(p.err_flags, KVQ_ERRF_WAIT_TIMEOUT);
      break;
    }
    const uint8_t *sb = smem + st * F::kStageBytes;
    const uint32_t *sx = reinterpret_cast<const uint32_t *>(sb + F::kCodeBytes);
    // the warp's two tiles of the chunk unrolled, so that their conversions
    // and MMA chains interleave (59.6 vs 61.8 us on 64 requests of MXFP4 keys,
    // 55.9 vs 57.4 with FP8 keys; 96 registers either way)
#pragma unroll
    for (int tile = warp; tile < kScChunk / kScTile; tile += kScWarps) {
      const int j0 = k * kScChunk + kScTile * tile;
      if (j0 >= p.max_len) break;
      float acc[2][4];
      float tok_scale[2];
#pragma unroll
      for (int t = 0; t < 2; ++t)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[t][e] = 0.0f;
      if (j0 < L) {
        // this lane's two token rows (g, g + 8), dims 32c .. 32c + 31 of
        // each: raw code words, converted to f16 pairs one k-step at a time
        // (pair m holds dims 32c + 2m, 32c + 2m + 1)
        constexpr int kW = F::kRowBytes / 16;        // words of a row per lane
        uint32_t rw[2][kW];
        uint32_t f2[2] = {0u, 0u};                   // MXFP4 group factor, f16x2
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int tt = kScTile * tile + g + 8 * h;
          const uint32_t side = sx[tt];
          if (kFormat == KVQ_INDEX_FP8) {
            const uint4 w0 = *reinterpret_cast<const uint4 *>(sb + tt * F::kRowBytes + 32 * c);
            const uint4 w1 =
                *reinterpret_cast<const uint4 *>(sb + tt * F::kRowBytes + 32 * c + 16);
            rw[h][0] = w0.x; rw[h][1] = w0.y; rw[h][2] = w0.z; rw[h][3] = w0.w;
            rw[h][kW > 4 ? 4 : 0] = w1.x; rw[h][kW > 5 ? 5 : 0] = w1.y;
            rw[h][kW > 6 ? 6 : 0] = w1.z; rw[h][kW > 7 ? 7 : 0] = w1.w;
            tok_scale[h] = __uint_as_float(side);
          } else {
            const uint4 w0 = *reinterpret_cast<const uint4 *>(sb + tt * F::kRowBytes + 16 * c);
            rw[h][0] = w0.x; rw[h][1] = w0.y; rw[h][2] = w0.z; rw[h][3] = w0.w;
            // the token's groups brought to its largest exponent: lane c
            // holds group c, the quad the token.  2^(X_c - Xmax) as binary32
            // (0 below 2^-126), then rounded to f16 -- exact down to f16's
            // smallest subnormal 2^-24, 0 below it
            const int xb = static_cast<int>((side >> (8 * c)) & 0xFFu);
            int mb = max(xb, __shfl_xor_sync(0xFFFFFFFFu, xb, 1));
            mb = max(mb, __shfl_xor_sync(0xFFFFFFFFu, mb, 2));
            const float fx = __uint_as_float(static_cast<uint32_t>(max(xb - mb + 127, 0)) << 23);
            f2[h] = pack_f16x2(fx, fx);
            // 2^Xmax: the largest exponent byte is the binary32 exponent
            // field (byte 0: 2^-127, a subnormal)
            tok_scale[h] = __uint_as_float(mb ? static_cast<uint32_t>(mb) << 23 : 1u << 22);
          }
        }
        // S^T = K Q^T over the 8 k-steps, both query tiles: a0/a2 = row g
        // pairs 2s / 2s + 1, a1/a3 = row g + 8
#pragma unroll
        for (int s = 0; s < 8; ++s) {
          uint32_t a[4];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            if (kFormat == KVQ_INDEX_FP8) {
              // pairs 2s, 2s + 1 = bytes 4s .. 4s + 3 = word s
              a[h] = e4m3x2_to_f16x2(rw[h][s]);
              a[2 + h] = e4m3x2_to_f16x2(rw[h][s] >> 16);
            } else {
              // pairs 2s, 2s + 1 = bytes 2s, 2s + 1 = half s & 1 of word s / 2
              uint32_t lo, hi;
              e2m1x4_to_f16x2x2(rw[h][s >> 1] >> (16 * (s & 1)), lo, hi);
              a[h] = hmul2(lo, f2[h]);
              a[2 + h] = hmul2(hi, f2[h]);
            }
          }
          mma_f16_16816(acc[0], a, qb[0][s][0], qb[0][s][1]);
          mma_f16_16816(acc[1], a, qb[1][s][0], qb[1][s][1]);
        }
      } else {
        tok_scale[0] = tok_scale[1] = 0.0f;          // past the context: every entry -inf
      }
      // acc[t] = (token g, col 2c), (g, 2c + 1), (g + 8, 2c), (g + 8, 2c + 1).
      // The token and column scales are >= 0, so the ReLU goes first, as
      // (x + |x|) / 2: score = tok * sum_h cs_h * max(0, acc_h).  A tile that
      // every row sees in full needs no mask.
      const bool plain = j0 + kScTile <= vis_min && j0 + kScTile <= p.max_len;
#pragma unroll
      for (int t = 0; t < 2; ++t)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int j = j0 + g + 8 * h;
          const float r0 = (acc[t][2 * h] + fabsf(acc[t][2 * h])) * hcs[t][0];
          const float r1 = (acc[t][2 * h + 1] + fabsf(acc[t][2 * h + 1])) * hcs[t][1];
          if (kH == 1) {
#pragma unroll
            for (int u2 = 0; u2 < kU; ++u2) {
              if (orow[t][u2] == nullptr) continue;
              float v = (u2 ? r1 : r0) * tok_scale[h];
              if (!plain) {
                if (j >= p.max_len) continue;
                v = j < vis[t][u2] ? v : -INFINITY;
              }
              orow[t][u2][j] = v;
            }
          } else {
            float sum = r0 + r1;
            if (kH >= 4) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 1);
            if (kH >= 8) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 2);
            if (orow[t][0] != nullptr) {
              float v = sum * tok_scale[h];
              if (plain) {
                orow[t][0][j] = v;
              } else if (j < p.max_len) {
                orow[t][0][j] = j < vis[t][0] ? v : -INFINITY;
              }
            }
          }
        }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_addr(&empty[st]));
    if (++k == p.nch) {
      k = 0;
      ++r;
    }
  }
}

template <int kFormat>
cudaError_t launch_scores_fmt(const ScParams &p, int32_t H, int32_t sms, cudaStream_t stream) {
  using F = ScFmt<kFormat>;
  void (*kernels[4])(const ScParams) = {
      index_scores_kernel<kFormat, 1>, index_scores_kernel<kFormat, 2>,
      index_scores_kernel<kFormat, 4>, index_scores_kernel<kFormat, 8>};
  const int ki = H == 1 ? 0 : (H == 2 ? 1 : (H == 4 ? 2 : 3));
  // per kernel and device: shared memory opted in once; resident CTAs per SM
  // (the same on every device of this architecture)
  static std::atomic<uint64_t> configured[4];
  static std::atomic<int> resident[4];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = (dev >= 0 && dev < 64) ? (uint64_t(1) << dev) : 0;
  if (bit == 0 || !(configured[ki].load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(kernels[ki], cudaFuncAttributeMaxDynamicSharedMemorySize, F::kSmem);
    if (e != cudaSuccess) return e;
    configured[ki].fetch_or(bit, std::memory_order_acq_rel);
  }
  int occ = resident[ki].load(std::memory_order_acquire);
  if (occ == 0) {
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kernels[ki], kScThreads, F::kSmem);
    if (e != cudaSuccess) return e;
    if (occ < 1) occ = 1;
    resident[ki].store(occ, std::memory_order_release);
  }
  const int64_t want = static_cast<int64_t>(occ) * (sms > 0 ? sms : 152);
  const int grid = static_cast<int>(p.total < want ? p.total : want);
  return launch_overlapped(kernels[ki], dim3(grid), dim3(kScThreads), F::kSmem, stream, p);
}

}  // namespace

bool index_scores_supported(int32_t rows_per_request, int32_t num_index_heads) {
  const int H = num_index_heads;
  return (H == 1 || H == 2 || H == 4 || H == 8) && rows_per_request >= 1 &&
         rows_per_request * H <= kScCols;
}

cudaError_t launch_index_scores(const kvq_index_cache &c, int32_t log2_block, const void *q,
                                int32_t num_requests, int32_t rows_per_request,
                                int32_t num_index_heads, const int32_t *block_tables,
                                int32_t max_blocks_per_req, const int32_t *context_lens,
                                int32_t max_context_len, float *out, int32_t *err_flags,
                                int32_t sms, cudaStream_t stream) {
  ScParams p;
  p.codes = c.codes;
  p.scales = c.scales;
  p.exps = c.exponents;
  p.num_blocks = static_cast<uint32_t>(c.num_slots >> log2_block);
  p.log2_bs = log2_block;
  p.q = static_cast<const uint16_t *>(q);
  p.R = rows_per_request;
  p.block_tables = block_tables;
  p.max_blocks = max_blocks_per_req;
  p.context_lens = context_lens;
  const int64_t cap = static_cast<int64_t>(max_blocks_per_req) << log2_block;
  p.ctx_limit = static_cast<int32_t>(cap < max_context_len ? cap : max_context_len);
  p.max_len = max_context_len;
  p.nch = (max_context_len + kScChunk - 1) / kScChunk;
  p.total = static_cast<int64_t>(num_requests) * p.nch;
  p.out = out;
  p.err_flags = err_flags;
  if (p.total <= 0) return cudaSuccess;
  if (c.format == KVQ_INDEX_FP8)
    return launch_scores_fmt<KVQ_INDEX_FP8>(p, num_index_heads, sms, stream);
  return launch_scores_fmt<KVQ_INDEX_MXFP4>(p, num_index_heads, sms, stream);
}

}  // namespace kvq
