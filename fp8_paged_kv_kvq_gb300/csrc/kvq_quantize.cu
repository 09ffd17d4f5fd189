// kvq_quantize.cu -- fused quantize + scatter of bf16 K/V rows into the FP8
// E4M3 paged cache, and the row dequantiser.
//
// FreeToken PR #354 "feat(kvcache): store the KV cache as fp8 e4m3 codes", PR
// description: every cached (token, KV head) row, of K as of V, is held as
// head_dim e4m3 bytes and a single symmetric fp32 scale (ROCm/ATOM PR #2655, PR
// description, K/V bullet: the scale is the row's largest magnitude over the
// FP8 maximum); one launch handles K and V and takes its slot ids from device
// memory, so it can be captured in a CUDA graph.  The fix commit "give the V tensor its own row pitch in the fp8 KV
// store": K and V each carry their own token pitch.
//
// Layout of the work: each 4-lane group owns one 128-element row (32 elements,
// 64 bytes, per lane: four 16-byte loads) of the grid-wide list of rows
// ordered (token, K heads then V heads), so a token's K rows are one
// contiguous read and every row costs one memory round trip.  The row amax is
// an integer max over the bf16 magnitude bits (order-preserving for finite
// values) reduced across the 4 lanes with shuffles; a lane's 32 codes leave as
// two 16-byte stores, so a row's 128 codes are one contiguous 128-byte line.
// Four lanes per row (rather than 8, 2 or 1) measured fastest: the per-row
// work (token index, scale, reciprocal) is shared by fewer threads while each
// thread still holds few registers.  The quotients run two at a time on the
// packed f32x2 FMA path.
#include <cuda_runtime.h>

#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {

namespace {

constexpr int kQuantWarps = 4;   // 128-thread CTAs, at least 12 resident per SM

struct QuantParams {
  const uint16_t *k;
  const uint16_t *v;
  int64_t k_stride;
  int64_t v_stride;
  int64_t num_tokens;
  const int64_t *slot_ids;
  uint8_t *k_codes;
  uint8_t *v_codes;
  float *k_scales;
  float *v_scales;
  int64_t num_slots;
  int32_t num_kv_heads;
  int32_t *err_flags;
  uint64_t rows_per_token_magic;   // ceil(2^shift / (2H)): row id / (2H) by a multiply
  int32_t rows_per_token_shift;    // 32 + ceil(log2(2H))
  // slot_ids == nullptr: token t = r R + i goes to position L_r - R + i of
  // request r's block table (a decode step's new rows)
  const int32_t *block_tables;
  int32_t max_blocks;
  const int32_t *context_lens;
  int32_t R;
  int32_t log2_bs;
  int32_t ctx_limit;
};

// The slot of token t under the block-table positions (-1: skip; a page id out
// of range is flagged).
__device__ __forceinline__ int64_t position_slot(const QuantParams &p, int64_t t) {
  const uint32_t r = static_cast<uint32_t>(t) / static_cast<uint32_t>(p.R);   // t < 2^31
  const int i = static_cast<int>(static_cast<uint32_t>(t) - r * static_cast<uint32_t>(p.R));
  int L = __ldg(p.context_lens + r);
  L = L < 0 ? 0 : (L > p.ctx_limit ? p.ctx_limit : L);
  const int pos = L - p.R + i;
  if (pos < 0) return -1;
  const uint32_t blk = static_cast<uint32_t>(__ldg(p.block_tables + static_cast<int64_t>(r) * p.max_blocks + (pos >> p.log2_bs)));
  if (static_cast<int64_t>(blk) >= (p.num_slots >> p.log2_bs)) {
    if (i == 0 && p.err_flags) atomicOr(p.err_flags, KVQ_ERRF_BLOCK_RANGE);
    return -1;
  }
  return (static_cast<int64_t>(blk) << p.log2_bs) | (pos & ((1 << p.log2_bs) - 1));
}

__device__ __forceinline__ uint32_t max_mag_bf16x2(uint4 a, uint4 b) {
  const uint32_t m = 0x7FFF7FFFu;
  uint32_t r = __vmaxu2(a.x & m, a.y & m);
  r = __vmaxu2(r, a.z & m);
  r = __vmaxu2(r, a.w & m);
  r = __vmaxu2(r, b.x & m);
  r = __vmaxu2(r, b.y & m);
  r = __vmaxu2(r, b.z & m);
  r = __vmaxu2(r, b.w & m);
  return r;
}

template <bool kFast>
__device__ __forceinline__ uint4 encode16(uint4 a, uint4 b, float s, float y) {
  uint4 out;
  out.x = encode4<kFast>(a.x, a.y, s, y);
  out.y = encode4<kFast>(a.z, a.w, s, y);
  out.z = encode4<kFast>(b.x, b.y, s, y);
  out.w = encode4<kFast>(b.z, b.w, s, y);
  return out;
}

constexpr int kLanesPerRow = 4;
constexpr int kRowsPerWarp = 32 / kLanesPerRow;
constexpr int kPerLane = kHeadDim / kLanesPerRow;      // elements
constexpr int kVec = kPerLane / 16;                     // 16-element pieces per lane

__global__ void __launch_bounds__(kQuantWarps * 32, 12)
quantize_scatter_kernel(const QuantParams p) {
  const int lane = threadIdx.x & 31;
  const int sub = lane & (kLanesPerRow - 1);
  const unsigned gmask = ((1u << kLanesPerRow) - 1u) << (lane & ~(kLanesPerRow - 1));
  const uint32_t rid = blockIdx.x * (kQuantWarps * kRowsPerWarp) + (threadIdx.x / kLanesPerRow);
  const int H = p.num_kv_heads;
  const uint32_t t32 =
      static_cast<uint32_t>((static_cast<uint64_t>(rid) * p.rows_per_token_magic) >> p.rows_per_token_shift);
  grid_dependency_wait();
  allow_dependents_launch();
  if (t32 >= p.num_tokens) return;
  const int64_t t = t32;
  const int rem = static_cast<int>(rid - t32 * static_cast<uint32_t>(2 * H));
  const bool is_v = rem >= H;
  const int h = is_v ? rem - H : rem;
  const uint16_t *src = (is_v ? p.v + t * p.v_stride : p.k + t * p.k_stride) + h * kHeadDim + sub * kPerLane;
  uint4 a[kVec], b[kVec];
#pragma unroll
  for (int k = 0; k < kVec; ++k) {
    a[k] = __ldg(reinterpret_cast<const uint4 *>(src + 16 * k));
    b[k] = __ldg(reinterpret_cast<const uint4 *>(src + 16 * k + 8));
  }
  const int64_t slot = p.slot_ids ? __ldg(p.slot_ids + t) : position_slot(p, t);
  if (slot < 0) return;
  if (slot >= p.num_slots) {
    if (sub == 0 && rem == 0 && p.err_flags) atomicOr(p.err_flags, KVQ_ERRF_SLOT_RANGE);
    return;
  }
  uint32_t m = max_mag_bf16x2(a[0], b[0]);
#pragma unroll
  for (int k = 1; k < kVec; ++k) m = __vmaxu2(m, max_mag_bf16x2(a[k], b[k]));
#pragma unroll
  for (int off = 1; off < kLanesPerRow; off <<= 1) m = __vmaxu2(m, __shfl_xor_sync(gmask, m, off));
  const float amax = __uint_as_float(max(m & 0xFFFFu, m >> 16) << 16);
  uint4 out[kVec];
#pragma unroll
  for (int k = 0; k < kVec; ++k) out[k] = make_uint4(0u, 0u, 0u, 0u);
  float s = 0.0f;
  if (amax != 0.0f) {
    s = row_scale(amax);
    if (s >= kMarksteinMinScale) {
      const float y = __frcp_rn(s);
#pragma unroll
      for (int k = 0; k < kVec; ++k) out[k] = encode16<true>(a[k], b[k], s, y);
    } else {
#pragma unroll
      for (int k = 0; k < kVec; ++k) out[k] = encode16<false>(a[k], b[k], s, 0.0f);
    }
  }
  const int64_t row = slot * H + h;
  uint4 *dst = reinterpret_cast<uint4 *>((is_v ? p.v_codes : p.k_codes) + row * kHeadDim + sub * kPerLane);
#pragma unroll
  for (int k = 0; k < kVec; ++k) dst[k] = out[k];
  if (sub == 0) (is_v ? p.v_scales : p.k_scales)[row] = s;
}

// ---------------------------------------------------------------------------
// The unscaled store of the codec ablation (sgl-project/sglang-jax #1776, design
// points: an O(1) cache cast to fp8 with no scale): each bf16 value is cast
// to e4m3 (saturating at 448) or e5m2 (saturating at 57344) with round-to-
// nearest-even by the hardware conversion, the sign of a zero code taken from
// its input, and both scale planes are set to 1 so the attention kernels read
// the codes' own values.  Same row layout and lanes as the scaled store.
__device__ __forceinline__ uint32_t e5m2x2_rn(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

template <int kFormat>   // KVQ_CODES_E4M3 or KVQ_CODES_E5M2
__device__ __forceinline__ uint32_t cast4(uint32_t w0, uint32_t w1) {
  const float q0 = bf16_lo(w0), q1 = bf16_hi(w0), q2 = bf16_lo(w1), q3 = bf16_hi(w1);
  const uint32_t signs = prmt(w0, w1, 0x7531u) & 0x80808080u;
  if (kFormat == KVQ_CODES_E5M2) return e5m2x2_rn(q0, q1) | (e5m2x2_rn(q2, q3) << 16) | signs;
  return e4m3x2_rn(q0, q1) | (e4m3x2_rn(q2, q3) << 16) | signs;
}

template <int kFormat>
__global__ void __launch_bounds__(kQuantWarps * 32, 12)
quantize_unscaled_kernel(const QuantParams p) {
  const int lane = threadIdx.x & 31;
  const int sub = lane & (kLanesPerRow - 1);
  const uint32_t rid = blockIdx.x * (kQuantWarps * kRowsPerWarp) + (threadIdx.x / kLanesPerRow);
  const int H = p.num_kv_heads;
  const uint32_t t32 =
      static_cast<uint32_t>((static_cast<uint64_t>(rid) * p.rows_per_token_magic) >> p.rows_per_token_shift);
  grid_dependency_wait();
  allow_dependents_launch();
  if (t32 >= p.num_tokens) return;
  const int64_t t = t32;
  const int rem = static_cast<int>(rid - t32 * static_cast<uint32_t>(2 * H));
  const bool is_v = rem >= H;
  const int h = is_v ? rem - H : rem;
  const uint16_t *src = (is_v ? p.v + t * p.v_stride : p.k + t * p.k_stride) + h * kHeadDim + sub * kPerLane;
  uint4 a[kVec], b[kVec];
#pragma unroll
  for (int k = 0; k < kVec; ++k) {
    a[k] = __ldg(reinterpret_cast<const uint4 *>(src + 16 * k));
    b[k] = __ldg(reinterpret_cast<const uint4 *>(src + 16 * k + 8));
  }
  const int64_t slot = __ldg(p.slot_ids + t);
  if (slot < 0) return;
  if (slot >= p.num_slots) {
    if (sub == 0 && rem == 0 && p.err_flags) atomicOr(p.err_flags, KVQ_ERRF_SLOT_RANGE);
    return;
  }
  const int64_t row = slot * H + h;
  uint4 *dst = reinterpret_cast<uint4 *>((is_v ? p.v_codes : p.k_codes) + row * kHeadDim + sub * kPerLane);
#pragma unroll
  for (int k = 0; k < kVec; ++k)
    dst[k] = make_uint4(cast4<kFormat>(a[k].x, a[k].y), cast4<kFormat>(a[k].z, a[k].w),
                        cast4<kFormat>(b[k].x, b[k].y), cast4<kFormat>(b[k].z, b[k].w));
  if (sub == 0) (is_v ? p.v_scales : p.k_scales)[row] = 1.0f;
}

// ---------------------------------------------------------------------------
struct DequantParams {
  const uint8_t *k_codes;
  const uint8_t *v_codes;
  const float *k_scales;
  const float *v_scales;
  int64_t num_slots;
  int32_t num_kv_heads;
  const int64_t *slot_ids;
  int64_t n;
  int32_t out_bf16;
  void *out_k;
  void *out_v;
  int32_t *err_flags;
};

__global__ void __launch_bounds__(kQuantWarps * 32)
dequant_rows_kernel(const DequantParams p) {
  const int lane = threadIdx.x & 31;
  const int sub = lane & 7;
  const int grp = lane >> 3;
  const int64_t i = static_cast<int64_t>(blockIdx.x) * kQuantWarps + (threadIdx.x >> 5);
  grid_dependency_wait();
  allow_dependents_launch();
  if (i >= p.n) return;
  const int64_t slot = p.slot_ids[i];
  const bool valid = slot >= 0 && slot < p.num_slots;
  if (slot >= p.num_slots && lane == 0 && p.err_flags)
    atomicOr(p.err_flags, KVQ_ERRF_SLOT_RANGE);
  const int H = p.num_kv_heads;
  for (int r = grp; r < 2 * H; r += 4) {
    const bool is_v = r >= H;
    const int h = is_v ? r - H : r;
    void *outp = is_v ? p.out_v : p.out_k;
    if (outp == nullptr) continue;
    uint4 codes = make_uint4(0u, 0u, 0u, 0u);
    float s = 0.0f;
    if (valid) {
      const int64_t row = slot * H + h;
      codes = __ldg(reinterpret_cast<const uint4 *>(
          (is_v ? p.v_codes : p.k_codes) + row * kHeadDim + sub * 16));
      s = __ldg((is_v ? p.v_scales : p.k_scales) + row);
    }
    float v[16];
    const uint32_t w[4] = {codes.x, codes.y, codes.z, codes.w};
#pragma unroll
    for (int j = 0; j < 16; ++j)
      v[j] = __fmul_rn(e4m3_to_f32((w[j >> 2] >> (8 * (j & 3))) & 0xFFu), s);
    const int64_t o = (i * H + h) * kHeadDim + sub * 16;
    if (p.out_bf16) {
      uint4 lo, hi;
      lo.x = pack_bf16x2(v[0], v[1]);   lo.y = pack_bf16x2(v[2], v[3]);
      lo.z = pack_bf16x2(v[4], v[5]);   lo.w = pack_bf16x2(v[6], v[7]);
      hi.x = pack_bf16x2(v[8], v[9]);   hi.y = pack_bf16x2(v[10], v[11]);
      hi.z = pack_bf16x2(v[12], v[13]); hi.w = pack_bf16x2(v[14], v[15]);
      uint4 *dst = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(outp) + o);
      dst[0] = lo;
      dst[1] = hi;
    } else {
      float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(outp) + o);
      dst[0] = make_float4(v[0], v[1], v[2], v[3]);
      dst[1] = make_float4(v[4], v[5], v[6], v[7]);
      dst[2] = make_float4(v[8], v[9], v[10], v[11]);
      dst[3] = make_float4(v[12], v[13], v[14], v[15]);
    }
  }
}


// ---------------------------------------------------------------------------
// Compressed index keys (ATOM PR #2655, PR description, index-key bullet):
// FP8 with one FP32 scale per row (the K/V row format), or MXFP4 -- two E2M1
// codes per byte and one E8M0 exponent per 32 dims, the exponent taken large
// enough that no element of its group exceeds the E2M1 range.  Rows of 128 values, one per token; each 4-lane group owns a row and
// each lane 32 values, which for MXFP4 is exactly one exponent group.
struct IndexParams {
  const uint16_t *x;
  int64_t x_stride;
  int64_t num_tokens;
  const int64_t *slot_ids;
  uint8_t *codes;
  float *scales;
  uint8_t *exps;
  int64_t num_slots;
  int32_t *err_flags;
};

constexpr int kIdxWarps = 4;

// Two E2M1 codes (round to nearest even, saturating; low nibble = lo).
__device__ __forceinline__ uint32_t e2m1x2_rn(float lo, float hi) {
  uint16_t r;
  asm("{\n .reg .b8 t;\n cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n mov.b16 %0, {t, 0};\n}\n"
      : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// The group exponent X from the bf16 bits of the group's largest magnitude:
// the smallest integer with amax <= 6 * 2^X, clamped to [-127, 127].  With
// amax = (1 + m/128) 2^(E-127): X = E - 129 when 1 + m/128 <= 1.5 (m <= 64),
// else E - 128; zero and subnormal amax (below 2^-126) clamp to -127.
__device__ __forceinline__ int mxfp4_group_exponent(uint32_t amax_bits) {
  const int E = static_cast<int>((amax_bits >> 7) & 0xFFu);
  if (E == 0) return -127;
  int X = E - 129 + ((amax_bits & 0x7Fu) > 0x40u ? 1 : 0);
  return X < -127 ? -127 : X;
}

// Four codes of elements (w0 lo, w0 hi, w1 lo, w1 hi) scaled by y = 2^-X:
// two bytes, even element in the low nibble, each code with its element's
// sign (bf16 bits 15 of the halves).
__device__ __forceinline__ uint32_t mxfp4_encode4(uint32_t w0, uint32_t w1, float y) {
  const uint32_t c = e2m1x2_rn(bf16_lo(w0) * y, bf16_hi(w0) * y) |
                     (e2m1x2_rn(bf16_lo(w1) * y, bf16_hi(w1) * y) << 8);
  const uint32_t signs = ((w0 >> 12) & 0x8u) | ((w0 >> 24) & 0x80u) | ((w1 >> 4) & 0x800u) |
                         ((w1 >> 16) & 0x8000u);
  return c | signs;
}

template <int kFormat>
__global__ void __launch_bounds__(kIdxWarps * 32, 12)
index_quantize_kernel(const IndexParams p) {
  const int lane = threadIdx.x & 31;
  const int sub = lane & 3;
  const unsigned gmask = 0xFu << (lane & 28);
  const int64_t t = static_cast<int64_t>(blockIdx.x) * (kIdxWarps * 8) + (threadIdx.x >> 2);
  grid_dependency_wait();
  allow_dependents_launch();
  if (t >= p.num_tokens) return;
  const uint16_t *src = p.x + t * p.x_stride + sub * 32;
  uint4 a[2], b[2];
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    a[k] = __ldg(reinterpret_cast<const uint4 *>(src + 16 * k));
    b[k] = __ldg(reinterpret_cast<const uint4 *>(src + 16 * k + 8));
  }
  const int64_t slot = __ldg(p.slot_ids + t);
  if (slot < 0) return;
  if (slot >= p.num_slots) {
    if (sub == 0 && p.err_flags) atomicOr(p.err_flags, KVQ_ERRF_SLOT_RANGE);
    return;
  }
  uint32_t m = __vmaxu2(max_mag_bf16x2(a[0], b[0]), max_mag_bf16x2(a[1], b[1]));
  if (kFormat == KVQ_INDEX_FP8) {
    m = __vmaxu2(m, __shfl_xor_sync(gmask, m, 1));
    m = __vmaxu2(m, __shfl_xor_sync(gmask, m, 2));
    const float amax = __uint_as_float(max(m & 0xFFFFu, m >> 16) << 16);
    uint4 out0 = make_uint4(0u, 0u, 0u, 0u), out1 = out0;
    float s = 0.0f;
    if (amax != 0.0f) {
      s = row_scale(amax);
      if (s >= kMarksteinMinScale) {
        const float y = __frcp_rn(s);
        out0 = encode16<true>(a[0], b[0], s, y);
        out1 = encode16<true>(a[1], b[1], s, y);
      } else {
        out0 = encode16<false>(a[0], b[0], s, 0.0f);
        out1 = encode16<false>(a[1], b[1], s, 0.0f);
      }
    }
    uint4 *dst = reinterpret_cast<uint4 *>(p.codes + slot * kHeadDim + sub * 32);
    dst[0] = out0;
    dst[1] = out1;
    if (sub == 0) p.scales[slot] = s;
  } else {
    // this lane's 32 values are one group
    const int X = mxfp4_group_exponent(max(m & 0xFFFFu, m >> 16));
    const float y = (X == 127) ? __uint_as_float(0x00400000u)              // 2^-127
                               : __uint_as_float(static_cast<uint32_t>(127 - X) << 23);
    uint4 out;
    out.x = mxfp4_encode4(a[0].x, a[0].y, y) | (mxfp4_encode4(a[0].z, a[0].w, y) << 16);
    out.y = mxfp4_encode4(b[0].x, b[0].y, y) | (mxfp4_encode4(b[0].z, b[0].w, y) << 16);
    out.z = mxfp4_encode4(a[1].x, a[1].y, y) | (mxfp4_encode4(a[1].z, a[1].w, y) << 16);
    out.w = mxfp4_encode4(b[1].x, b[1].y, y) | (mxfp4_encode4(b[1].z, b[1].w, y) << 16);
    *reinterpret_cast<uint4 *>(p.codes + slot * (kHeadDim / 2) + sub * 16) = out;
    p.exps[slot * (kHeadDim / 32) + sub] = static_cast<uint8_t>(X + 127);
  }
}

// Rows back to real values, one warp per row: FP8 fl32(e4m3(c) * scale); MXFP4
// fl32(e2m1(c) * 2^X) (exact products but for overflow), optionally rounded
// again to bf16.
struct IndexDequantParams {
  const uint8_t *codes;
  const float *scales;
  const uint8_t *exps;
  int64_t num_slots;
  const int64_t *slot_ids;
  int64_t n;
  int32_t out_bf16;
  void *out;
  int32_t *err_flags;
};

__device__ __forceinline__ void f16x2_to_f32x2(uint32_t h2, float &lo, float &hi) {
  asm("{\n .reg .b16 l, h;\n mov.b32 {l, h}, %2;\n cvt.f32.f16 %0, l;\n cvt.f32.f16 %1, h;\n}\n"
      : "=f"(lo), "=f"(hi) : "r"(h2));
}

template <int kFormat>
__global__ void __launch_bounds__(kIdxWarps * 32)
index_dequant_kernel(const IndexDequantParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t i = static_cast<int64_t>(blockIdx.x) * kIdxWarps + (threadIdx.x >> 5);
  grid_dependency_wait();
  allow_dependents_launch();
  if (i >= p.n) return;
  const int64_t slot = p.slot_ids[i];
  const bool valid = slot >= 0 && slot < p.num_slots;
  if (slot >= p.num_slots && lane == 0 && p.err_flags) atomicOr(p.err_flags, KVQ_ERRF_SLOT_RANGE);
  float v[4] = {0.f, 0.f, 0.f, 0.f};                 // dims 4 lane .. 4 lane + 3
  if (valid) {
    if (kFormat == KVQ_INDEX_FP8) {
      const uint32_t w = __ldg(reinterpret_cast<const uint32_t *>(p.codes + slot * kHeadDim) + lane);
      const float s = __ldg(p.scales + slot);
#pragma unroll
      for (int j = 0; j < 4; ++j) v[j] = __fmul_rn(e4m3_to_f32((w >> (8 * j)) & 0xFFu), s);
    } else {
      const uint16_t w = __ldg(reinterpret_cast<const uint16_t *>(p.codes + slot * (kHeadDim / 2)) + lane);
      const int X = static_cast<int>(__ldg(p.exps + slot * (kHeadDim / 32) + lane / 8)) - 127;
      const float sc = (X == -127) ? __uint_as_float(0x00400000u)
                                   : __uint_as_float(static_cast<uint32_t>(127 + X) << 23);
      uint32_t h01, h23;
      asm("{\n .reg .b8 c0, c1;\n mov.b16 {c0, c1}, %2;\n cvt.rn.f16x2.e2m1x2 %0, c0;\n"
          " cvt.rn.f16x2.e2m1x2 %1, c1;\n}\n" : "=r"(h01), "=r"(h23) : "h"(w));
      f16x2_to_f32x2(h01, v[0], v[1]);
      f16x2_to_f32x2(h23, v[2], v[3]);
#pragma unroll
      for (int j = 0; j < 4; ++j) v[j] = __fmul_rn(v[j], sc);
    }
  }
  const int64_t o = i * kHeadDim + 4 * lane;
  if (p.out_bf16) {
    uint2 pk;
    pk.x = pack_bf16x2(v[0], v[1]);
    pk.y = pack_bf16x2(v[2], v[3]);
    *reinterpret_cast<uint2 *>(static_cast<uint16_t *>(p.out) + o) = pk;
  } else {
    *reinterpret_cast<float4 *>(static_cast<float *>(p.out) + o) = make_float4(v[0], v[1], v[2], v[3]);
  }
}

}  // namespace

namespace {

QuantParams quant_params(const kvq_cache &c, const void *k, int64_t k_stride, const void *v,
                         int64_t v_stride, int64_t num_tokens, const int64_t *slot_ids,
                         int32_t *err_flags) {
  QuantParams p;
  p.k = static_cast<const uint16_t *>(k);
  p.v = static_cast<const uint16_t *>(v);
  p.k_stride = k_stride;
  p.v_stride = v_stride;
  p.num_tokens = num_tokens;
  p.slot_ids = slot_ids;
  p.k_codes = c.k_codes;
  p.v_codes = c.v_codes;
  p.k_scales = c.k_scales;
  p.v_scales = c.v_scales;
  p.num_slots = c.num_slots;
  p.num_kv_heads = c.num_kv_heads;
  p.err_flags = err_flags;
  p.block_tables = nullptr;
  p.max_blocks = 0;
  p.context_lens = nullptr;
  p.R = 1;
  p.log2_bs = 0;
  p.ctx_limit = 0;
  {
    // n / d == (n * ceil(2^S / d)) >> S for every n < 2^31 when S = 32 + ceil(log2 d):
    // the multiplier's excess e = M d - 2^S is below d <= 2^(S-32), so n e < 2^S
    const uint64_t d = 2u * static_cast<uint64_t>(c.num_kv_heads);
    int l = 0;
    while ((uint64_t(1) << l) < d) ++l;
    p.rows_per_token_shift = 32 + l;
    p.rows_per_token_magic = ((uint64_t(1) << (32 + l)) + d - 1) / d;
  }
  return p;
}

}  // namespace

cudaError_t launch_quantize_scatter(const kvq_cache &c, const void *k, int64_t k_stride,
                                    const void *v, int64_t v_stride, int64_t num_tokens,
                                    const int64_t *slot_ids, int32_t *err_flags,
                                    cudaStream_t stream) {
  const QuantParams p = quant_params(c, k, k_stride, v, v_stride, num_tokens, slot_ids, err_flags);
  const int64_t rows = num_tokens * 2 * c.num_kv_heads;
  const int64_t blocks = (rows + kQuantWarps * kRowsPerWarp - 1) / (kQuantWarps * kRowsPerWarp);
  return launch_overlapped(quantize_scatter_kernel, dim3(static_cast<unsigned>(blocks)),
                           dim3(kQuantWarps * 32), 0, stream, p);
}

cudaError_t launch_quantize_positions(const kvq_cache &c, const void *k, int64_t k_stride,
                                     const void *v, int64_t v_stride, int32_t num_requests,
                                     int32_t rows_per_request, const int32_t *block_tables,
                                     int32_t max_blocks_per_req, const int32_t *context_lens,
                                     int32_t ctx_limit, int32_t log2_block, int32_t *err_flags,
                                     cudaStream_t stream) {
  const int64_t num_tokens = static_cast<int64_t>(num_requests) * rows_per_request;
  QuantParams p = quant_params(c, k, k_stride, v, v_stride, num_tokens, nullptr, err_flags);
  p.block_tables = block_tables;
  p.max_blocks = max_blocks_per_req;
  p.context_lens = context_lens;
  p.R = rows_per_request;
  p.log2_bs = log2_block;
  p.ctx_limit = ctx_limit;
  const int64_t rows = num_tokens * 2 * c.num_kv_heads;
  const int64_t blocks = (rows + kQuantWarps * kRowsPerWarp - 1) / (kQuantWarps * kRowsPerWarp);
  return launch_overlapped(quantize_scatter_kernel, dim3(static_cast<unsigned>(blocks)),
                           dim3(kQuantWarps * 32), 0, stream, p);
}

cudaError_t launch_quantize_unscaled(const kvq_cache &c, int32_t code_format, const void *k,
                                     int64_t k_stride, const void *v, int64_t v_stride,
                                     int64_t num_tokens, const int64_t *slot_ids,
                                     int32_t *err_flags, cudaStream_t stream) {
  const QuantParams p = quant_params(c, k, k_stride, v, v_stride, num_tokens, slot_ids, err_flags);
  const int64_t rows = num_tokens * 2 * c.num_kv_heads;
  const int64_t blocks = (rows + kQuantWarps * kRowsPerWarp - 1) / (kQuantWarps * kRowsPerWarp);
  if (code_format == KVQ_CODES_E5M2)
    return launch_overlapped(quantize_unscaled_kernel<KVQ_CODES_E5M2>,
                             dim3(static_cast<unsigned>(blocks)), dim3(kQuantWarps * 32), 0,
                             stream, p);
  return launch_overlapped(quantize_unscaled_kernel<KVQ_CODES_E4M3>,
                           dim3(static_cast<unsigned>(blocks)), dim3(kQuantWarps * 32), 0,
                           stream, p);
}

cudaError_t launch_dequant_rows(const kvq_cache &c, const int64_t *slot_ids, int64_t n,
                                int32_t out_dtype, void *out_k, void *out_v,
                                int32_t *err_flags, cudaStream_t stream) {
  DequantParams p;
  p.k_codes = c.k_codes;
  p.v_codes = c.v_codes;
  p.k_scales = c.k_scales;
  p.v_scales = c.v_scales;
  p.num_slots = c.num_slots;
  p.num_kv_heads = c.num_kv_heads;
  p.slot_ids = slot_ids;
  p.n = n;
  p.out_bf16 = out_dtype == 1;
  p.out_k = out_k;
  p.out_v = out_v;
  p.err_flags = err_flags;
  const int64_t blocks = (n + kQuantWarps - 1) / kQuantWarps;
  return launch_overlapped(dequant_rows_kernel, dim3(static_cast<unsigned>(blocks)),
                           dim3(kQuantWarps * 32), 0, stream, p);
}

}  // namespace kvq

namespace kvq {

cudaError_t launch_index_quantize_scatter(const kvq_index_cache &c, const void *x,
                                          int64_t x_stride, int64_t num_tokens,
                                          const int64_t *slot_ids, int32_t *err_flags,
                                          cudaStream_t stream) {
  IndexParams p;
  p.x = static_cast<const uint16_t *>(x);
  p.x_stride = x_stride;
  p.num_tokens = num_tokens;
  p.slot_ids = slot_ids;
  p.codes = c.codes;
  p.scales = c.scales;
  p.exps = c.exponents;
  p.num_slots = c.num_slots;
  p.err_flags = err_flags;
  const int64_t blocks = (num_tokens + kIdxWarps * 8 - 1) / (kIdxWarps * 8);
  if (c.format == KVQ_INDEX_FP8)
    return launch_overlapped(index_quantize_kernel<KVQ_INDEX_FP8>,
                             dim3(static_cast<unsigned>(blocks)), dim3(kIdxWarps * 32), 0,
                             stream, p);
  return launch_overlapped(index_quantize_kernel<KVQ_INDEX_MXFP4>,
                           dim3(static_cast<unsigned>(blocks)), dim3(kIdxWarps * 32), 0, stream,
                           p);
}

cudaError_t launch_index_dequant_rows(const kvq_index_cache &c, const int64_t *slot_ids,
                                      int64_t n, int32_t out_dtype, void *out,
                                      int32_t *err_flags, cudaStream_t stream) {
  IndexDequantParams p;
  p.codes = c.codes;
  p.scales = c.scales;
  p.exps = c.exponents;
  p.num_slots = c.num_slots;
  p.slot_ids = slot_ids;
  p.n = n;
  p.out_bf16 = out_dtype == 1;
  p.out = out;
  p.err_flags = err_flags;
  const int64_t blocks = (n + kIdxWarps - 1) / kIdxWarps;
  if (c.format == KVQ_INDEX_FP8)
    return launch_overlapped(index_dequant_kernel<KVQ_INDEX_FP8>,
                             dim3(static_cast<unsigned>(blocks)), dim3(kIdxWarps * 32), 0,
                             stream, p);
  return launch_overlapped(index_dequant_kernel<KVQ_INDEX_MXFP4>,
                           dim3(static_cast<unsigned>(blocks)), dim3(kIdxWarps * 32), 0, stream,
                           p);
}

}  // namespace kvq
