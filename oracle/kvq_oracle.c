/*
 * kvq_oracle.c -- the CPU oracle for the FP8 E4M3 paged KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product (the fp8_paged_kv_kvq_gb300
 * package, its CUDA library or its C ABI) includes, links or calls this file.
 * Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline / reference
 * leg load it.  It shares no code, header, table or constant generator with the
 * CUDA path: everything here is written from the format definition and from the
 * pages' description of the method, in the plainest form, single-threaded.
 *
 * Build: plain C11, -O2 -ffp-contract=off, no -ffast-math, so that every float
 * operation below is one IEEE-754 binary32 operation rounded to nearest-even.
 *
 * Sources (web pages; cited by title and section):
 *  [ATOM]   ROCm/ATOM PR #2655, "fix(qwen4-exp): register the QSA FP8 scale
 *           planes for KV offload" -- PR description, K/V bullet: E4M3 codes
 *           and, per (token, KV head), an FP32 scale equal to the row's largest
 *           magnitude over the FP8 maximum; the
 *           attention applies a token's key scale to its score after the code
 *           dot product and its value scale to its probability ahead of PV.
 *  [FT]     FlashML-org/FreeToken PR #354, "feat(kvcache): store the KV cache as
 *           fp8 e4m3 codes (--kv-cache-dtype fp8)" -- PR description: a row is
 *           head_dim code bytes and a single symmetric fp32 scale, the bytes in
 *           a uint8 buffer shaped like the 16-bit cache, written by a fused
 *           quantize-and-scatter to slot ids held on the device; review thread and fix commit "give the V tensor its
 *           own row pitch in the fp8 KV store": K and V each have their own row
 *           pitch; codes are checked against a round-to-nearest-even reference.
 *  [SGJ]    sgl-project/sglang-jax #1776, "feat(dsa): implement fp8 KV cache
 *           (e4m3) with a bf16 indexer cache" -- design points: e4m3 range 448,
 *           0.0156 floor of the normal range, ~6% worst-case relative error.
 *
 * Readings of points the pages leave open:
 *  - the encode divides by the stored fp32 scale: q = fl32(x / s);
 *  - rounding is round-to-nearest-even onto the e4m3 grid, |q| >= 448 saturates
 *    to the largest finite code (0x7E magnitude); NaN codes are never produced;
 *  - an all-zero row stores s = 0 and all codes 0x00 (even for -0.0 inputs);
 *  - in a nonzero row the sign of zero is kept (-0.0 or a negative value that
 *    rounds to zero gives 0x80);
 *  - GQA maps query head hq to KV head hq / (Hq / H);
 *  - a request with R query rows (multi-token verify) is causal: row i sees the
 *    first L - R + 1 + i cached tokens; a row that sees nothing outputs zeros;
 *  - slot ids < 0 are padding and are skipped; ids >= num_slots are skipped and
 *    reported in the error word (bit 0).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define KVQO_ERR_SLOT_RANGE 1
#define KVQO_ERR_BLOCK_RANGE 2
#define KVQO_ERR_CONTEXT_RANGE 4

/* ------------------------------------------------------------------------ */
/* bfloat16 <-> float, by definition of the format (upper half of binary32). */

float kvqo_bf16_to_float(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round a finite float to bfloat16, nearest-even: the 16 dropped bits decide. */
uint16_t kvqo_float_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    uint32_t upper = u >> 16;
    uint32_t lower = u & 0xFFFFu;
    if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u)))
        upper += 1u;
    return (uint16_t)upper;
}

/* ------------------------------------------------------------------------ */
/* E4M3 ("fn" variant: no infinities, S.1111.111 is NaN, max finite 448).
 * A code is 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits.
 *   E in 1..15: value = 2^(E-7) * (1 + M/8)
 *   E == 0:     value = 2^(-6) * (M/8)          (subnormal)
 * [SGJ] design points give the 448 top and the 0.0156 bottom of the normal
 * range; the format itself is the OCP 8-bit floating point "E4M3" encoding. */

double kvqo_e4m3_decode(uint8_t c)
{
    int sign = (c >> 7) & 1;
    int e = (c >> 3) & 0xF;
    int m = c & 0x7;
    double mag;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        mag = ldexp((double)m / 8.0, -6);
    else
        mag = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -mag : mag;
}

/* The 127 finite nonnegative magnitudes, grid[c] = decode(c) for c = 0..0x7E,
 * filled once when the library loads. */
static double grid[0x7F];

/* decode(c) for all 256 codes, for the attention loops below. */
static double dec[256];

__attribute__((constructor)) static void fill_tables(void)
{
    for (int c = 0; c < 0x7F; ++c)
        grid[c] = kvqo_e4m3_decode((uint8_t)c);
    for (int c = 0; c < 256; ++c)
        dec[c] = kvqo_e4m3_decode((uint8_t)c);
}

/* Encode a finite binary32 value: round to the nearest representable e4m3
 * magnitude, ties to the code whose mantissa is even, saturating at 448.
 * The magnitudes increase with the code, so a bisection over the grid finds
 * the two neighbours of |q|. */
uint8_t kvqo_e4m3_encode(float q)
{
    uint8_t sign = signbit(q) ? 0x80 : 0x00;
    double a = fabs((double)q);
    if (a >= 448.0)
        return (uint8_t)(sign | 0x7E);
    /* invariant: grid[lo] <= a < grid[hi] */
    int lo = 0, hi = 0x7E;
    while (hi - lo > 1) {
        int mid = (lo + hi) / 2;
        if (grid[mid] <= a)
            lo = mid;
        else
            hi = mid;
    }
    double vlo = grid[lo];
    double vhi = grid[hi];
    double half = 0.5 * (vlo + vhi); /* exact: both have few significant bits */
    int pick;
    if (a < half)
        pick = lo;
    else if (a > half)
        pick = hi;
    else
        pick = (lo & 1) ? hi : lo; /* the mantissa LSB is the code LSB */
    return (uint8_t)(sign | pick);
}

/* Element-wise forms of the two functions above, for arrays. */
void kvqo_e4m3_encode_array(const float *q, int64_t n, uint8_t *codes)
{
    for (int64_t i = 0; i < n; ++i)
        codes[i] = kvqo_e4m3_encode(q[i]);
}

void kvqo_float_to_bf16_array(const float *x, int64_t n, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = kvqo_float_to_bf16(x[i]);
}

/* ------------------------------------------------------------------------ */
/* One (token, KV head) row: [ATOM] PR description (K/V bullet) and [FT] PR
 * description: the scale is the row's largest magnitude over 448, and each
 * code is e4m3(x / scale). */

void kvqo_quantize_row(const uint16_t *x, int D, uint8_t *codes, float *scale)
{
    float amax = 0.0f;
    for (int d = 0; d < D; ++d) {
        float a = fabsf(kvqo_bf16_to_float(x[d]));
        if (a > amax)
            amax = a;
    }
    if (amax == 0.0f) {
        *scale = 0.0f;
        memset(codes, 0, (size_t)D);
        return;
    }
    float s = amax / 448.0f;
    *scale = s;
    for (int d = 0; d < D; ++d) {
        float q = kvqo_bf16_to_float(x[d]) / s;
        codes[d] = kvqo_e4m3_encode(q);
    }
}

/* Many rows at once: x [n_rows, D] -> codes [n_rows, D], scales [n_rows]. */
void kvqo_quantize_rows(const uint16_t *x, int64_t n_rows, int D, uint8_t *codes, float *scales)
{
    for (int64_t i = 0; i < n_rows; ++i)
        kvqo_quantize_row(x + i * D, D, codes + i * D, &scales[i]);
}

/* Fused quantize + scatter, [FT] PR description and fix commit: token t's K
 * row for head h starts at k + t*k_token_stride + h*D (elements), V's at
 * v + t*v_token_stride + h*D, each with its own pitch; the codes land in the
 * cache at slot slot_ids[t], laid out [num_slots, H, D] (the 16-bit buffer's
 * geometry), the scales at [num_slots, H]. Returns the error word. */
int32_t kvqo_quantize_scatter(const uint16_t *k, int64_t k_token_stride,
                              const uint16_t *v, int64_t v_token_stride,
                              int64_t num_tokens, int H, int D,
                              const int64_t *slot_ids, int64_t num_slots,
                              uint8_t *k_codes, uint8_t *v_codes,
                              float *k_scales, float *v_scales)
{
    int32_t err = 0;
    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_ids[t];
        if (slot < 0)
            continue;
        if (slot >= num_slots) {
            err |= KVQO_ERR_SLOT_RANGE;
            continue;
        }
        for (int h = 0; h < H; ++h) {
            int64_t row = slot * H + h;
            kvqo_quantize_row(k + t * k_token_stride + (int64_t)h * D, D,
                              k_codes + row * D, &k_scales[row]);
            kvqo_quantize_row(v + t * v_token_stride + (int64_t)h * D, D,
                              v_codes + row * D, &v_scales[row]);
        }
    }
    return err;
}

/* ------------------------------------------------------------------------ */
/* Dequantize rows at the given slots: value = fl32(decode(c) * s), one IEEE
 * multiply (decode(c) is exact in binary32); out_dtype 1 rounds that float
 * once more to bfloat16 (nearest-even). Layout of out: [n, H, D]. */

void kvqo_dequant_rows(const uint8_t *codes, const float *scales, int64_t num_slots,
                       int H, int D, const int64_t *slot_ids, int64_t n,
                       int out_dtype, void *out)
{
    for (int64_t i = 0; i < n; ++i) {
        int64_t slot = slot_ids[i];
        for (int h = 0; h < H; ++h) {
            for (int d = 0; d < D; ++d) {
                int64_t o = (i * H + h) * D + d;
                float val = 0.0f;
                if (slot >= 0 && slot < num_slots) {
                    int64_t row = slot * H + h;
                    val = (float)kvqo_e4m3_decode(codes[row * D + d]) * scales[row];
                }
                if (out_dtype == 0)
                    ((float *)out)[o] = val;
                else
                    ((uint16_t *)out)[o] = kvqo_float_to_bf16(val);
            }
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Paged GQA attention in fp64 over the dequantised cache.
 *
 * Requests r = 0..N-1 each have R query rows (R = 1: decode; R > 1: the rows
 * of a multi-token verify, the last R tokens already in the cache) and Hq
 * query heads sharing H KV heads (G = Hq / H, head hq reads KV head hq / G).
 * Cached token j of request r lives at slot
 *     block_tables[r * max_blocks + j / bs] * bs + j % bs.
 * Row i of request r sees the first  L_r - R + 1 + i  tokens.
 *
 * For each visible token: k_hat = decode(code) * k_scale, v_hat likewise
 * (exact in double); score = sm_scale * <q, k_hat>; p = softmax(score);
 * out = sum_j p_j * v_hat_j.  Scaling the score by the key scale after the
 * code dot and p by the value scale ahead of PV ([ATOM] PR description) gives
 * the same quantity in exact arithmetic; the oracle takes the plain definition.
 *
 * q: bf16 [N*R, Hq, D]; out: double [N*R, Hq, D]. Returns the error word
 * (bit 1: a block id outside [0, num_slots/bs); bit 2: a context length
 * outside [0, max_blocks*bs]); offending tokens / rows are left out.
 * `scores` is caller scratch of at least max_blocks*bs doubles. */
static int32_t attention_row(const uint8_t *k_codes, const uint8_t *v_codes,
                             const float *k_scales, const float *v_scales,
                             int64_t num_slots, int H, int D, int bs,
                             const uint16_t *qrow, int kvh,
                             const int32_t *bt_row, int visible, double sm_scale,
                             double *scores, double *out)
{
    int32_t err = 0;
    int64_t num_blocks = num_slots / bs;
    double mx = -INFINITY;
    for (int j = 0; j < visible; ++j) {
        int64_t blk = bt_row[j / bs];
        if (blk < 0 || blk >= num_blocks) {
            err |= KVQO_ERR_BLOCK_RANGE;
            scores[j] = -INFINITY;
            continue;
        }
        int64_t row = (blk * bs + j % bs) * H + kvh;
        double ks = (double)k_scales[row];
        double dot = 0.0;
        for (int d = 0; d < D; ++d) {
            double kh = dec[k_codes[row * D + d]] * ks;
            dot += (double)kvqo_bf16_to_float(qrow[d]) * kh;
        }
        scores[j] = sm_scale * dot;
        if (scores[j] > mx)
            mx = scores[j];
    }
    for (int d = 0; d < D; ++d)
        out[d] = 0.0;
    if (mx == -INFINITY)
        return err; /* nothing visible: zeros */
    double l = 0.0;
    for (int j = 0; j < visible; ++j) {
        if (scores[j] == -INFINITY)
            continue;
        double p = exp(scores[j] - mx);
        l += p;
        int64_t row = ((int64_t)bt_row[j / bs] * bs + j % bs) * H + kvh;
        double vs = (double)v_scales[row];
        for (int d = 0; d < D; ++d)
            out[d] += p * (dec[v_codes[row * D + d]] * vs);
    }
    for (int d = 0; d < D; ++d)
        out[d] /= l;
    return err;
}

int32_t kvqo_paged_attention(const uint8_t *k_codes, const uint8_t *v_codes,
                             const float *k_scales, const float *v_scales,
                             int64_t num_slots, int H, int D, int bs,
                             const uint16_t *q, int N, int R, int Hq,
                             const int32_t *block_tables, int max_blocks,
                             const int32_t *context_lens, double sm_scale,
                             double *out)
{
    int32_t err = 0;
    int G = Hq / H;
    double *scores = (double *)malloc(sizeof(double) * ((size_t)max_blocks * bs + 1));
    if (!scores)
        return -1;
    for (int r = 0; r < N; ++r) {
        int L = context_lens[r];
        if (L < 0 || (int64_t)L > (int64_t)max_blocks * bs) {
            err |= KVQO_ERR_CONTEXT_RANGE;
            L = L < 0 ? 0 : max_blocks * bs;
        }
        for (int i = 0; i < R; ++i) {
            int visible = L - R + 1 + i;
            if (visible < 0)
                visible = 0;
            for (int hq = 0; hq < Hq; ++hq) {
                int64_t orow = ((int64_t)(r * R + i) * Hq + hq);
                err |= attention_row(k_codes, v_codes, k_scales, v_scales, num_slots,
                                     H, D, bs, q + orow * D, hq / G,
                                     block_tables + (int64_t)r * max_blocks, visible,
                                     sm_scale, scores, out + orow * D);
            }
        }
    }
    free(scores);
    return err;
}

/* The same attention for a chosen list of (request, row, query head) units,
 * written to out[u * D ..]: lets a test or a timing sample cover part of a
 * large batch. units: int32 triples (r, i, hq). */
int32_t kvqo_paged_attention_units(const uint8_t *k_codes, const uint8_t *v_codes,
                                   const float *k_scales, const float *v_scales,
                                   int64_t num_slots, int H, int D, int bs,
                                   const uint16_t *q, int N, int R, int Hq,
                                   const int32_t *block_tables, int max_blocks,
                                   const int32_t *context_lens, double sm_scale,
                                   const int32_t *units, int64_t num_units,
                                   double *out)
{
    int32_t err = 0;
    int G = Hq / H;
    double *scores = (double *)malloc(sizeof(double) * ((size_t)max_blocks * bs + 1));
    if (!scores)
        return -1;
    for (int64_t u = 0; u < num_units; ++u) {
        int r = units[3 * u], i = units[3 * u + 1], hq = units[3 * u + 2];
        if (r < 0 || r >= N || i < 0 || i >= R || hq < 0 || hq >= Hq) {
            free(scores);
            return -1;
        }
        int L = context_lens[r];
        if (L < 0 || (int64_t)L > (int64_t)max_blocks * bs) {
            err |= KVQO_ERR_CONTEXT_RANGE;
            L = L < 0 ? 0 : max_blocks * bs;
        }
        int visible = L - R + 1 + i;
        if (visible < 0)
            visible = 0;
        int64_t orow = ((int64_t)(r * R + i) * Hq + hq);
        err |= attention_row(k_codes, v_codes, k_scales, v_scales, num_slots, H, D, bs,
                             q + orow * D, hq / G, block_tables + (int64_t)r * max_blocks,
                             visible, sm_scale, scores, out + u * D);
    }
    free(scores);
    return err;
}

/* ------------------------------------------------------------------------ */
/* Compressed index keys, [ATOM] PR description, index-key bullet: FP8 with a
 * per-row FP32 scale (the rows above, one index head per token: H = 1), or
 * MXFP4 -- two E2M1 codes per byte and one E8M0 exponent per 32 dims, the
 * exponent rounded up until no element of the group overflows; the FP4 codes
 * are decoded by bit manipulation.
 *
 * Readings of what the bullet leaves open:
 *  - E2M1 is the OCP microscaling element format: 1 sign bit, 2 exponent bits
 *    (bias 1), 1 mantissa bit; magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6.
 *  - E8M0 is a biased exponent: byte X + 127 stands for the group scale 2^X.
 *  - the exponent rounded up so no element overflows: X is the smallest integer with
 *    group amax <= 6 * 2^X (the largest E2M1 magnitude), clamped to
 *    [-127, 127]; an all-zero group gets X = -127.
 *  - Each element becomes the E2M1 value nearest to x / 2^X (exact: a power
 *    of two), ties to the code with an even mantissa bit, with x's sign (so
 *    -0.0 and negative values that round to zero keep the sign bit).
 *  - Element 2i goes to the low nibble of byte i, element 2i + 1 to the high.
 *  - Dequantisation is decode(code) * 2^X rounded once to binary32. */

double kvqo_e2m1_decode(uint8_t c)
{
    int sign = (c >> 3) & 1;
    int e = (c >> 1) & 3;
    int m = c & 1;
    double mag = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return sign ? -mag : mag;
}

/* Nearest E2M1 magnitude code (0..7) to a >= 0, ties to the even code. */
static uint8_t e2m1_round_mag(double a)
{
    if (a >= 6.0)
        return 7;
    int lo = 0;
    while (lo < 7 && kvqo_e2m1_decode((uint8_t)(lo + 1)) <= a)
        ++lo;
    /* decode(lo) <= a < decode(lo + 1) */
    double vlo = kvqo_e2m1_decode((uint8_t)lo);
    double vhi = kvqo_e2m1_decode((uint8_t)(lo + 1));
    double half = 0.5 * (vlo + vhi);
    if (a < half)
        return (uint8_t)lo;
    if (a > half)
        return (uint8_t)(lo + 1);
    return (uint8_t)((lo & 1) ? lo + 1 : lo); /* the mantissa bit is the code LSB */
}

uint8_t kvqo_e2m1_encode(double q)
{
    uint8_t sign = signbit(q) ? 0x8 : 0x0;
    return (uint8_t)(sign | e2m1_round_mag(fabs(q)));
}

/* The group exponent X: the smallest integer with amax <= 6 * 2^X, clamped to
 * [-127, 127] (-127 for an all-zero group). */
int kvqo_mxfp4_group_exponent(double amax)
{
    if (amax == 0.0)
        return -127;
    int k;
    frexp(amax, &k);                        /* amax in [2^(k-1), 2^k) */
    int X = k - 4;                          /* 6 * 2^(k-4) < 2^(k-1) <= amax */
    while (6.0 * ldexp(1.0, X) < amax)
        ++X;
    if (X < -127)
        X = -127;
    if (X > 127)
        X = 127;
    return X;
}

/* One row of D bf16 values (D a multiple of 32): codes [D/2] bytes, exps
 * [D/32] E8M0 bytes. */
void kvqo_mxfp4_quantize_row(const uint16_t *x, int D, uint8_t *codes, uint8_t *exps)
{
    for (int g = 0; g < D / 32; ++g) {
        double amax = 0.0;
        for (int d = 32 * g; d < 32 * g + 32; ++d) {
            double a = fabs((double)kvqo_bf16_to_float(x[d]));
            if (a > amax)
                amax = a;
        }
        int X = kvqo_mxfp4_group_exponent(amax);
        exps[g] = (uint8_t)(X + 127);
        for (int d = 32 * g; d < 32 * g + 32; d += 2) {
            uint8_t c0 = kvqo_e2m1_encode(ldexp((double)kvqo_bf16_to_float(x[d]), -X));
            uint8_t c1 = kvqo_e2m1_encode(ldexp((double)kvqo_bf16_to_float(x[d + 1]), -X));
            codes[d / 2] = (uint8_t)(c0 | (c1 << 4));
        }
    }
}

void kvqo_mxfp4_quantize_rows(const uint16_t *x, int64_t n_rows, int D, uint8_t *codes,
                              uint8_t *exps)
{
    for (int64_t i = 0; i < n_rows; ++i)
        kvqo_mxfp4_quantize_row(x + i * D, D, codes + i * (D / 2), exps + i * (D / 32));
}

/* Rows [n, D] back to binary32: decode(code) * 2^X, one rounding. */
void kvqo_mxfp4_dequant_rows(const uint8_t *codes, const uint8_t *exps, int64_t n_rows, int D,
                             float *out)
{
    for (int64_t i = 0; i < n_rows; ++i) {
        for (int d = 0; d < D; ++d) {
            uint8_t byte = codes[i * (D / 2) + d / 2];
            uint8_t c = (d & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 0xF);
            int X = (int)exps[i * (D / 32) + d / 32] - 127;
            out[i * D + d] = (float)ldexp(kvqo_e2m1_decode(c), X);
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Index scoring over the compressed index keys, [ATOM] PR description: the
 * stacked decode scorer lets R query rows x H index heads of a request meet
 * each cached key once, applies the per-head ReLU and sums the heads.  For
 * request r, query row i and cached token t (slot from the block table):
 *     score(r, i, t) = sum_h max(0, <q(r, i, h), khat_t>)
 * with khat_t the dequantised key, computed in double.  Readings:
 * no per-head weight (a caller folds one into q); row i sees the tokens
 * t < L_r - R + 1 + i, as the attention rows do; every other position up to
 * max_len gets -inf.
 *   format 0: codes [S, D] e4m3, scales [S]; format 1: codes [S, D/2] E2M1
 *   pairs, exps [S, D/32] E8M0.  q: bf16 [N*R, H, D]; out: double [N*R, max_len].
 * Returns the error word (block or context range). */
static double index_key_value(int format, const uint8_t *codes, const float *scales,
                              const uint8_t *exps, int64_t slot, int D, int d)
{
    if (format == 0)
        return kvqo_e4m3_decode(codes[slot * D + d]) * (double)scales[slot];
    uint8_t byte = codes[slot * (D / 2) + d / 2];
    uint8_t c = (d & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 0xF);
    return ldexp(kvqo_e2m1_decode(c), (int)exps[slot * (D / 32) + d / 32] - 127);
}

int32_t kvqo_index_scores(int format, const uint8_t *codes, const float *scales,
                          const uint8_t *exps, int64_t num_slots, int D, int bs,
                          const int32_t *block_tables, int max_blocks,
                          const int32_t *context_lens, int N, int R, int H,
                          const uint16_t *q, int max_len, double *out)
{
    int32_t err = 0;
    for (int r = 0; r < N; ++r) {
        int L = context_lens[r];
        if (L < 0 || L > max_len || (int64_t)L > (int64_t)max_blocks * bs) {
            err |= KVQO_ERR_CONTEXT_RANGE;
            L = L < 0 ? 0 : L;
            if (L > max_len) L = max_len;
            if ((int64_t)L > (int64_t)max_blocks * bs) L = max_blocks * bs;
        }
        for (int i = 0; i < R; ++i) {
            double *o = out + (int64_t)(r * R + i) * max_len;
            int visible = L - R + 1 + i;
            for (int t = 0; t < max_len; ++t)
                o[t] = -INFINITY;
            for (int t = 0; t < visible; ++t) {
                int64_t blk = block_tables[(int64_t)r * max_blocks + t / bs];
                if (blk < 0 || (blk + 1) * bs > num_slots) {
                    err |= KVQO_ERR_BLOCK_RANGE;
                    continue;
                }
                int64_t slot = blk * bs + t % bs;
                double score = 0.0;
                for (int h = 0; h < H; ++h) {
                    const uint16_t *qv = q + ((int64_t)(r * R + i) * H + h) * D;
                    double dot = 0.0;
                    for (int d = 0; d < D; ++d)
                        dot += (double)kvqo_bf16_to_float(qv[d]) *
                               index_key_value(format, codes, scales, exps, slot, D, d);
                    if (dot > 0.0)
                        score += dot;
                }
                o[t] = score;
            }
        }
    }
    return err;
}

/* ------------------------------------------------------------------------ */
/* E5M2, for the unscaled-cache ablation.  [SGJ] design points: the fp8 cache
 * of that page casts O(1) values to e4m3 or e5m2 with no scale at all, and
 * prefers e4m3 for its extra mantissa bit.  E5M2: 1 sign, 5 exponent bits with
 * bias 15, 2 mantissa bits; exponent field 0 is subnormal (m/4 * 2^-14),
 * exponent field 31 holds infinity (m = 0) and NaN (m != 0).
 * Reading: the cast rounds to nearest, ties to the even mantissa, and
 * saturates at the largest finite magnitude 57344 (as the e4m3 encode does at
 * 448), so no infinity or NaN code is produced from a finite input. */

double kvqo_e5m2_decode(uint8_t c)
{
    int sign = (c >> 7) & 1;
    int e = (c >> 2) & 0x1F;
    int m = c & 0x3;
    double mag;
    if (e == 31)
        mag = (m == 0) ? INFINITY : NAN;
    else if (e == 0)
        mag = ldexp((double)m / 4.0, -14);
    else
        mag = ldexp(1.0 + (double)m / 4.0, e - 15);
    return sign ? -mag : mag;
}

/* The 124 finite nonnegative magnitudes, code 0 .. 0x7B, ascending. */
static double grid52[0x7C];

__attribute__((constructor)) static void fill_e5m2_table(void)
{
    for (int c = 0; c < 0x7C; ++c)
        grid52[c] = kvqo_e5m2_decode((uint8_t)c);
}

/* Nearest e5m2 magnitude by bisection over the ascending grid, ties to the
 * code with the even mantissa (the code's least significant bit). */
uint8_t kvqo_e5m2_encode(float q)
{
    uint8_t sign = signbit(q) ? 0x80 : 0x00;
    double a = fabs((double)q);
    if (a >= 57344.0)
        return (uint8_t)(sign | 0x7B);
    int lo = 0, hi = 0x7B;                 /* grid52[lo] <= a < grid52[hi] */
    while (hi - lo > 1) {
        int mid = (lo + hi) / 2;
        if (grid52[mid] <= a)
            lo = mid;
        else
            hi = mid;
    }
    double half = 0.5 * (grid52[lo] + grid52[hi]);
    int pick;
    if (a < half)
        pick = lo;
    else if (a > half)
        pick = hi;
    else
        pick = (lo & 1) ? hi : lo;
    return (uint8_t)(sign | pick);
}

void kvqo_e5m2_encode_array(const float *q, int64_t n, uint8_t *codes)
{
    for (int64_t i = 0; i < n; ++i)
        codes[i] = kvqo_e5m2_encode(q[i]);
}
