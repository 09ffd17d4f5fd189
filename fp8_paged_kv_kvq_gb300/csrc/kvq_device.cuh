// kvq_device.cuh -- device-side building blocks shared by the libkvq kernels:
// the software E4M3 codec, packed bf16 helpers, cp.async and mma.sync wrappers.
//
// The E4M3 ("fn") format: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa
// bits; E = 0 is subnormal (M * 2^-9); S.1111.111 is NaN; the largest finite
// magnitude is 448.  FreeToken PR #354 "feat(kvcache): store the KV cache as
// fp8 e4m3 codes", PR description: codes live in a plain uint8 buffer, so
// every card holds the same bytes.  Decoding is done here with bit placement;
// the store encodes with the hardware e4m3x2 conversion, whose rounding
// (nearest-even, saturating) is the one defined below, bit for bit.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>

namespace kvq {

constexpr int kHeadDim = 128;

// ---------------------------------------------------------------------------
// Encode.  q = fl32(x / s) (IEEE division, round-to-nearest-even), then the
// nearest e4m3 magnitude, ties to the even mantissa, |q| >= 448 saturating to
// 448.  The sign is taken from x, which equals the sign of q for s > 0 and
// keeps the sign of zero.  Works on the binary32 bit pattern:
//  * |q| >= 2^-6 (e4m3 normal range): drop the 20 low mantissa bits with
//    round-half-even; the rounded exponent/mantissa field, rebased from bias
//    127 to bias 7 (subtract 120 << 3), is the code, carries included;
//  * |q| < 2^-6 (subnormal range): adding 2^14 rounds |q| to a multiple of
//    2^-9 (the ulp of 2^14) with the hardware's nearest-even addition, and the
//    bit-pattern difference to 2^14 is the subnormal mantissa 0..8 (8 lands
//    exactly on the smallest normal code).
// The rounding step alone: code of the finite value q (sign from `sgn`).
__device__ __forceinline__ uint32_t e4m3_round(float q, float sgn) {
  const uint32_t a = __float_as_uint(q) & 0x7FFFFFFFu;
  const uint32_t sign = (__float_as_uint(sgn) >> 24) & 0x80u;
  uint32_t mag;
  if (a >= 0x43E00000u) {                       // >= 448
    mag = 0x7Eu;
  } else if (a >= 0x3C800000u) {                // >= 2^-6
    mag = ((a + 0x7FFFFu + ((a >> 20) & 1u)) >> 20) - 0x3C0u;
  } else {
    mag = __float_as_uint(__fadd_rn(__uint_as_float(a), 16384.0f)) - 0x46800000u;
  }
  return mag | sign;
}

// Two codes at once through the hardware conversion (round-to-nearest-even,
// saturating to +-448, the sign of zero kept): the low byte is lo's code.  It
// rounds a binary32 value exactly as e4m3_round does.
__device__ __forceinline__ uint32_t e4m3x2_rn(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Correctly rounded x / s given y = fl32(1 / s), by Markstein's correction
// (P. Markstein, "Computation of elementary functions on the IBM RISC
// System/6000 processor", IBM J. Res. Dev. 34(1), 1990): q0 = x*y is within
// 1.5 ulp of x / s; one step q1 = q0 + (x - s*q0)*y brings it within 1 ulp,
// and with the remainder exact (an FMA) a second step rounds correctly.  Valid
// while no step underflows: for s >= 2^-90 every quotient >= 2^-11 (the only
// ones whose e4m3 code is not 0) has an exact remainder; smaller quotients
// stay below 2^-10 and encode to zero either way.  For x != 0 the result has
// the sign of x; x = -0 gives +0 (the caller restores the sign of zero).
constexpr float kMarksteinMinScale = 0x1p-90f;

__device__ __forceinline__ float div_markstein(float x, float s, float y) {
  const float q0 = __fmul_rn(x, y);
  const float r0 = __fmaf_rn(-q0, s, x);
  const float q1 = __fmaf_rn(r0, y, q0);
  const float r1 = __fmaf_rn(-q1, s, x);
  return __fmaf_rn(r1, y, q1);
}

// Packed pairs of fp32 (low half = first element) for the f32x2 arithmetic.
__device__ __forceinline__ uint64_t pack_f32x2(float lo, float hi) {
  uint64_t d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
  return d;
}
__device__ __forceinline__ void unpack_f32x2(uint64_t d, float &lo, float &hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(d));
}
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t mul_f32x2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// div_markstein on a packed pair: x holds two dividends, ns and y hold -s and
// fl32(1 / s) in both halves; the same five roundings per element as the
// scalar form, on the f32x2 FMA path.
__device__ __forceinline__ uint64_t div_markstein_x2(uint64_t x, uint64_t ns, uint64_t y) {
  const uint64_t q0 = mul_f32x2(x, y);
  const uint64_t r0 = fma_f32x2(q0, ns, x);
  const uint64_t q1 = fma_f32x2(r0, y, q0);
  const uint64_t r1 = fma_f32x2(q1, ns, x);
  return fma_f32x2(r1, y, q1);
}



// ---------------------------------------------------------------------------
// Decode to bf16, exactly.  Placing the 7 magnitude bits of a code at bf16 bits
// 10..4 (exponent low bits + top mantissa bits) and its sign at bit 15 gives a
// bf16 whose value is e4m3(c) * 2^-120 exactly -- subnormal codes land on bf16
// subnormals with the same mantissa -- and one bf16 multiply by 2^120 (exact:
// a power of two, result in the normal range) restores e4m3(c).
//
// Pair helpers take two codes held in the same byte of the two 16-bit halves of
// a word and return the bf16x2 of their values (low half from the low code).
__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

constexpr uint32_t kBf16x2Pow2_120 = 0x7B807B80u;   // bf16 2^120 in both halves

// codes in bytes 0 and 2 of w (bytes 1 and 3 ignored)
__device__ __forceinline__ uint32_t e4m3x2_b02_to_bf16x2(uint32_t w) {
  const uint32_t mag = (w << 4) & 0x07F007F0u;
  const uint32_t sgn = (w << 8) & 0x80008000u;
  return bf16x2_mul(mag | sgn, kBf16x2Pow2_120);
}

// codes in bytes 1 and 3 of w (bytes 0 and 2 ignored)
__device__ __forceinline__ uint32_t e4m3x2_b13_to_bf16x2(uint32_t w) {
  const uint32_t mag = (w >> 4) & 0x07F007F0u;
  const uint32_t sgn = w & 0x80008000u;
  return bf16x2_mul(mag | sgn, kBf16x2Pow2_120);
}

// Two codes (low byte -> low half) to their exact f16 values through the
// hardware conversion; every e4m3 value, subnormals included, is an f16.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t w16) {
  uint32_t d;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(d) : "h"(static_cast<uint16_t>(w16)));
  return d;
}

// Decode to f16 times 2^-8, exactly: the 7 magnitude bits at f16 bits 13..7
// and the sign at bit 15 give a half whose value is e4m3(c) * 2^-8 (f16 has a
// 5-bit exponent with bias 15 against e4m3's 4 bits with bias 7); subnormal
// codes land on f16 subnormals (M * 2^-17) with the same mantissa.  No
// multiply is needed: the 2^8 is folded into the operand on the other side.
// codes in bytes 0 and 2 of w (bytes 1 and 3 ignored)
__device__ __forceinline__ uint32_t e4m3x2_b02_to_f16x2_lo8(uint32_t w) {
  return ((w << 7) & 0x3F803F80u) | ((w << 8) & 0x80008000u);
}

// codes in bytes 1 and 3 of w (bytes 0 and 2 ignored)
__device__ __forceinline__ uint32_t e4m3x2_b13_to_f16x2_lo8(uint32_t w) {
  return ((w >> 1) & 0x3F803F80u) | (w & 0x80008000u);
}

// Decode one code to fp32 exactly: bits at binary32 positions give
// e4m3(c) * 2^-120 (subnormal codes become binary32 subnormals), times 2^120.
__device__ __forceinline__ float e4m3_to_f32(uint32_t c) {
  const uint32_t bits = ((c & 0x7Fu) << 20) | ((c & 0x80u) << 24);
  return __fmul_rn(__uint_as_float(bits), 0x1p120f);
}

// The two e4m3 pieces of four query elements: p1 = e4m3(x), p2 = e4m3(x - p1)
// (the difference is exact in binary32), four codes per word, element t in
// byte t.  Through the hardware conversions: e4m3x2_rn rounds as e4m3_round,
// and every e4m3 value is an f16.  For x of at most 8 significant bits inside
// e4m3's range, x = p1 + p2 exactly.
__device__ __forceinline__ void e4m3_pieces4(const float (&x)[4], uint32_t &c1w, uint32_t &c2w) {
  const uint32_t a = e4m3x2_rn(x[0], x[1]), b = e4m3x2_rn(x[2], x[3]);
  float d[4];
  asm("{\n .reg .b16 l0, h0, l1, h1;\n mov.b32 {l0, h0}, %4;\n mov.b32 {l1, h1}, %5;\n"
      " cvt.f32.f16 %0, l0;\n cvt.f32.f16 %1, h0;\n cvt.f32.f16 %2, l1;\n cvt.f32.f16 %3, h1;\n}\n"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(e4m3x2_to_f16x2(a)), "r"(e4m3x2_to_f16x2(b)));
  c1w = a | (b << 16);
  c2w = e4m3x2_rn(x[0] - d[0], x[1] - d[1]) | (e4m3x2_rn(x[2] - d[2], x[3] - d[3]) << 16);
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// ---------------------------------------------------------------------------
// The row codec of the store (FreeToken PR #354 "feat(kvcache): store the KV
// cache as fp8 e4m3 codes"; ROCm/ATOM PR #2655, K/V bullet): one fp32 scale
// per (token, KV head) row, the row's largest magnitude over 448, and e4m3
// codes of x / scale rounded to nearest even.

constexpr float kInv448 = 1.0f / 448.0f;               // fl32(1 / 448): rounded by the compiler

// fl32(amax / 448): Markstein's correction through the correctly rounded
// constant reciprocal while no step underflows, else IEEE division.
__device__ __forceinline__ float row_scale(float amax) {
  return (amax >= kMarksteinMinScale) ? div_markstein(amax, 448.0f, kInv448)
                                      : __fdiv_rn(amax, 448.0f);
}

// Four codes from the two bf16 pairs (w0: elements 0,1; w1: elements 2,3):
// fl32(x / s) then e4m3 round-to-nearest-even.  kFast divides through the
// row's reciprocal y with Markstein's correction (exact for s >= 2^-90), two
// elements per packed f32x2 operation; otherwise plain IEEE division.  The four sign bits of x (bytes 1 and 3 of
// each bf16 pair) are ORed into the code bytes: a nonzero code already has
// its sign, and a zero code takes the sign of its input (-0 stays 0x80).
template <bool kFast>
__device__ __forceinline__ uint32_t encode4(uint32_t w0, uint32_t w1, float s, float y) {
  float q[4] = {bf16_lo(w0), bf16_hi(w0), bf16_lo(w1), bf16_hi(w1)};
  if (kFast) {
    const uint64_t ns = pack_f32x2(-s, -s), yy = pack_f32x2(y, y);
    unpack_f32x2(div_markstein_x2(pack_f32x2(q[0], q[1]), ns, yy), q[0], q[1]);
    unpack_f32x2(div_markstein_x2(pack_f32x2(q[2], q[3]), ns, yy), q[2], q[3]);
  } else {
#pragma unroll
    for (int e = 0; e < 4; ++e) q[e] = __fdiv_rn(q[e], s);
  }
  const uint32_t signs = prmt(w0, w1, 0x7531u) & 0x80808080u;
  return e4m3x2_rn(q[0], q[1]) | (e4m3x2_rn(q[2], q[3]) << 16) | signs;
}

// ---------------------------------------------------------------------------
// Asynchronous global -> shared copies (Ampere-style cp.async, available on
// sm_103a).  src_bytes = 0 zero-fills the destination without reading.
__device__ __forceinline__ void cp_async_16(void *smem, const void *gmem, uint32_t src_bytes) {
  const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n"
               :: "r"(s), "l"(gmem), "r"(src_bytes));
}

__device__ __forceinline__ void cp_async_4(void *smem, const void *gmem, uint32_t src_bytes) {
  const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n"
               :: "r"(s), "l"(gmem), "r"(src_bytes));
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n"); }

template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" :: "n"(N));
}

// ---------------------------------------------------------------------------
// mbarrier + TMA (cp.async.bulk.tensor).  The copy engine signals completion
// on an mbarrier as transaction bytes; waits are bounded so that a copy that
// never lands cannot hang the GPU: the caller gets `false` and reports it.
__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" :: "r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n"
               :: "r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
  return ok != 0;
}

// Bounded wait for phase `parity` of the barrier (about a second at most).
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity) {
  for (int i = 0; i < (1 << 20); ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

// As mbar_try_wait, but a thread whose phase is not complete may sleep until it
// completes or about `ns` nanoseconds pass, instead of spinning.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity, uint32_t ns) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok) : "r"(bar), "r"(parity), "r"(ns) : "memory");
  return ok != 0;
}

// Bounded sleeping wait: at most 2^19 tries of at most 2 us each (about a
// second); returns false if the phase never completed.
__device__ __forceinline__ bool mbar_wait_sleep_bounded(uint32_t bar, uint32_t parity) {
  for (int i = 0; i < (1 << 19); ++i)
    if (mbar_try_wait_sleep(bar, parity, 2000u)) return true;
  return false;
}

// Programmatic dependent launch.  A kernel launched with programmatic stream
// serialization may start while the previous kernel of the stream drains:
// grid_dependency_wait() returns once that kernel has completed and its writes
// are visible, so it comes before the first read of anything a previous kernel
// may have written; allow_dependents_launch() lets the next kernel start early.
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
}

__device__ __forceinline__ void allow_dependents_launch() {
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}

// Piece counter of a unit of work cut into pieces by CTA range boundaries.
// The 64-bit word holds (call tag << 32) | pieces landed; a piece that finds
// another call's tag -- or whatever the workspace held before -- starts the
// count for this call, so the word needs no initialisation.  Returns the
// pieces landed including this one (0 if the word could not be claimed).  The
// piece that completes the count resets the word to 0, so a graph replay that
// reuses the tag starts from zero too.
__device__ __forceinline__ uint32_t ticket_take(unsigned long long *t, uint32_t tag) {
  unsigned long long cur = *reinterpret_cast<volatile unsigned long long *>(t);
  for (int i = 0; i < 4096; ++i) {
    const unsigned long long want = (static_cast<uint32_t>(cur >> 32) == tag)
                                        ? cur + 1ull
                                        : ((static_cast<unsigned long long>(tag) << 32) | 1ull);
    const unsigned long long prev = atomicCAS(t, cur, want);
    if (prev == cur) return static_cast<uint32_t>(want & 0xFFFFFFFFull);
    cur = prev;
  }
  return 0u;
}

// Makes barrier initialisation visible to the copy engine.
__device__ __forceinline__ void fence_mbarrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}

// 3-D tiled TMA load of one box into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void *tmap, int x, int y, int z,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];\n"
      :: "r"(dst), "l"(tmap), "r"(x), "r"(y), "r"(z), "r"(bar) : "memory");
}

// ---------------------------------------------------------------------------
// Plain arrive (count 1) on an mbarrier.
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" :: "r"(bar) : "memory");
}

// 2-D tiled TMA load of one box into shared memory, completing on `bar`.
// An L2 policy that marks lines first in line for eviction (data read once).
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;\n" : "=l"(p));
  return p;
}
// An L2 policy with the default eviction priority.
__device__ __forceinline__ uint64_t l2_policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;\n" : "=l"(p));
  return p;
}
// tma_load_3d under an L2 cache policy.
__device__ __forceinline__ void tma_load_3d_hint(uint32_t dst, const void *tmap, int x, int y,
                                                 int z, uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;\n"
      :: "r"(dst), "l"(tmap), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(policy) : "memory");
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void *tmap, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];\n"
      :: "r"(dst), "l"(tmap), "r"(x), "r"(y), "r"(bar) : "memory");
}

// Barrier `id` (1..15) over the first `count` threads that reach it.
__device__ __forceinline__ void named_barrier(uint32_t id, uint32_t count) {
  asm volatile("bar.sync %0, %1;\n" :: "r"(id), "r"(count) : "memory");
}

// ---------------------------------------------------------------------------
// 5th-generation tensor cores (tcgen05).  Accumulators live in tensor memory
// (TMEM: 128 lanes x 512 columns of 32 bits per SM; an address is lane << 16 |
// column); a warp reads and writes only the 32 lanes of its quarter (warp id
// mod 4).  MMA operands come from shared memory through 64-bit descriptors:
//   bits  0-13  start address >> 4
//   bits 16-29  leading byte offset >> 4
//   bits 32-45  stride byte offset >> 4
//   bits 46-47  descriptor version (1)
//   bits 61-63  swizzle: 0 none, 2 128-byte, 4 64-byte, 6 32-byte
// For a K-major operand with the 128-byte swizzle (rows of 128 bytes, 8-row
// atoms) the stride offset is the distance between 8-row groups and the
// leading offset is unused; a K step inside the 128-byte row advances the
// start address.  For an MN-major operand the leading offset is the distance
// between blocks of one swizzle width along M or N and the stride offset the
// distance between groups of 8 rows along K.
constexpr uint32_t kSmemSwizzle128 = 2;
constexpr uint32_t kSmemSwizzle64 = 4;

__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo,
                                              uint32_t swizzle) {
  return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) |
         (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (uint64_t(1) << 46) |
         (static_cast<uint64_t>(swizzle) << 61);
}

// Instruction descriptor of a dense MMA with fp32 accumulation:
//   bits 4-5 D format (1 = f32), 7-9 A format, 10-12 B format (kind::f16:
//   0 = f16, 1 = bf16; kind::f8f6f4: 0 = e4m3), bit 15 A MN-major, bit 16 B
//   MN-major, bits 17-22 N >> 3, bits 24-28 M >> 4.
__host__ __device__ constexpr uint32_t mma_idesc(int m, int n, bool a_mn_major, bool b_mn_major) {
  return (1u << 4) | (a_mn_major ? (1u << 15) : 0u) | (b_mn_major ? (1u << 16) : 0u) |
         (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(m >> 4) << 24);
}

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n"
               :: "r"(dst_smem), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n"
               :: "r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
}

// D (TMEM) = A * B^T (+ D if accumulate), e4m3 operands.
__device__ __forceinline__ void tc_mma_e4m3(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}\n"
      :: "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate) : "memory");
}

// D (TMEM) = A * B^T (+ D if accumulate), f16 operands.
__device__ __forceinline__ void tc_mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n"
      :: "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate) : "memory");
}

// D (TMEM) = A * B (+ D if accumulate), f16 operands, A read from tensor
// memory: row i of A in TMEM lane i, its K elements two to a 32-bit column
// (element 2c in the low half of column c), so a K step of 16 advances the A
// address by 8 columns; B from shared memory through its descriptor.
__device__ __forceinline__ void tc_mma_f16_tmem_a(uint32_t d_tmem, uint32_t a_tmem,
                                                  uint64_t b_desc, uint32_t idesc,
                                                  uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n"
      :: "r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate) : "memory");
}

// One arrive on `bar` once every MMA this thread issued so far has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n"
               :: "r"(bar) : "memory");
}

// 32 consecutive columns of this thread's TMEM lane (32x32b shape, x32).  The
// wait for the load sits in the same asm statement, so no use of the
// registers can be scheduled before the data has arrived.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n"
               "tcgen05.wait::ld.sync.aligned;\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
               : "r"(taddr) : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
  uint32_t r[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(v[i]);
  asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};\n"
               :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31]) : "memory");
}

// 16 consecutive columns of this thread's TMEM lane (32x32b shape, x16), the
// wait for the load in the same statement.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];\n"
               "tcgen05.wait::ld.sync.aligned;\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
               : "r"(taddr) : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float (&v)[16]) {
  uint32_t r[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) r[i] = __float_as_uint(v[i]);
  asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};\n"
               :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]) : "memory");
}

// 16 consecutive 32-bit columns of this thread's TMEM lane from raw words.
__device__ __forceinline__ void tmem_st16u(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};\n"
               :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]) : "memory");
}

// 8 consecutive 32-bit columns of this thread's TMEM lane from raw words.
__device__ __forceinline__ void tmem_st8u(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};\n"
               :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]),
                  "r"(r[6]), "r"(r[7]) : "memory");
}

// 8 consecutive 32-bit columns of this thread's TMEM lane as raw words, the
// wait for the load in the same statement.
__device__ __forceinline__ void tmem_ld8u(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];\n"
               "tcgen05.wait::ld.sync.aligned;\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                 "=r"(r[6]), "=r"(r[7])
               : "r"(taddr) : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
}

__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
}

// ---------------------------------------------------------------------------
// D = A * B + D on the tensor cores, 16x8x16, bf16 operands, fp32 accumulate.
// Fragment ownership (lane = 4*g + c):
//   A (16x16, row-major): a0 = A[g][2c..2c+1], a1 = A[g+8][2c..2c+1],
//                         a2 = A[g][2c+8..2c+9], a3 = A[g+8][2c+8..2c+9]
//   B (16x8, col-major):  b0 = B[2c..2c+1][g],  b1 = B[2c+8..2c+9][g]
//   C (16x8):             c0,c1 = C[g][2c..2c+1], c2,c3 = C[g+8][2c..2c+1]
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4],
                                               uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// The same with f16 operands.
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4],
                                              uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Four 8x8 matrices of 16-bit elements from shared memory in mma fragment
// order: lanes 8m..8m+7 give the row addresses of matrix m; register m of
// lane t holds row t/4, elements 2(t%4), 2(t%4)+1 of matrix m.  On byte
// tiles (two bytes per element) this is the 8-bit m16n8k32 A fragment: rows
// 0-7 / 8-15 in matrices 0/1 (k 0-15) and 2/3 (k 16-31).
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}

// D = A * B + D, 16x8x32, e4m3 operands (the cache's own code bytes), fp32
// accumulate.  Each register holds four consecutive k of one row (A) or one
// column (B):
//   a0 = A[g][4c..4c+3], a1 = A[g+8][4c..4c+3], a2 = A[g][4c+16..4c+19],
//   a3 = A[g+8][4c+16..4c+19];  b0 = B[4c..4c+3][g], b1 = B[4c+16..4c+19][g]
__device__ __forceinline__ void mma_e4m3_16832(float (&d)[4], const uint32_t (&a)[4],
                                               uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

}  // namespace kvq
