/*
 * qoracle.c - the plain, slow, scalar CPU oracle for the ggml/GGUF
 * block-quantized matrix-vector product.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file: it is used by tests/, by the smoke check and by the CPU
 * baseline leg of bench.py.  It shares no code, header, table or helper with
 * the CUDA library.
 *
 * Build: gcc -std=c11 -O2 -ffp-contract=off -fPIC -shared (see build.py).
 * -ffp-contract=off forbids fused multiply-adds, so every float expression
 * below rounds exactly as written.
 *
 * Sources (page titles and sections of the reference pages):
 *   [rml]      "Quantization" (rayaq.ca/rml): The type table; Block layouts;
 *              Unpacking the packed fields (Q4_K element-200 trace);
 *              A worked example: Q4_0; Quantized dot products;
 *              Kernels and references.
 *   [sipllm]   "Quantization" (sipllm docs): On-disk block geometry;
 *              Per-format dequant; The fused matmul.
 *   [lesson21] "Building Q8_0 and Q4_0 Like ggml": Examples 1-2 (Q8_0 layout
 *              and quantizer), 5-6 (Q4_0 scale, code rule, nibble order),
 *              7 (Q4_1 min/max rule and layout), 8 (Q5_0 rule, qh packing
 *              and decode), 10 (Q8_0 x Q8_0 dot), 11 (Q4_0 x Q8_0 dot),
 *              14 (byte-exact blocks of all four formats).
 *   [candle]   "量化格式" (quantized formats, candle): GgmlDType table;
 *              block structure table; "一些边界值" (special values);
 *              VecDotType pairing table; vec_dot_unopt.
 *
 * Readings where the pages leave a step open (each is also listed in the
 * design notes):
 *   - Q8_K activation rule: the Q8_0 rule over 256 elements with d kept as
 *     f32 (not rounded to f16), codes clamped to [-127, 127], and
 *     bsums[k] = sum of codes 16k..16k+15.
 *   - Q6_K element mapping: for e = 128h + 32k + l (h in 0..1, k in 0..3,
 *     l in 0..31) the low 4 bits come from ql[64h + 32(k&1) + l] (low nibble
 *     for k < 2, high nibble for k >= 2), the high 2 bits from
 *     (qh[32h + l] >> 2k) & 3, and the sub-block scale is scales[e / 16].
 *   - Q4_K sub-blocks 0..3: scale = scales[j] & 63, min = scales[j+4] & 63.
 *   - Q2_K, Q3_K and Q5_K (the pages give their sizes and, for Q5_K, that
 *     it carries dmin and Q4_K's packed 6-bit scales and mins): the ggml
 *     file layouts, written out at q2_k_code, q3_k_code and q5_k_code below.
 *     Element e = 128n + 32j + 16h + l of Q2_K/Q3_K takes bits 2j..2j+1 of
 *     qs[32n + 16h + l] and lies in the 16-element sub-block e / 16; Q3_K's
 *     third bit is bit 4n + j of hmask[16h + l] (set means the 2-bit value
 *     as is, clear means 4 less) and its sixteen 6-bit scales, stored
 *     biased by 32, keep their low 4 bits in the nibbles of bytes 0..7 and
 *     their high 2 bits in bytes 8..11; Q5_K is Q4_K plus a fifth bit, bit j
 *     of qh[e % 32] for sub-block j = e / 32.
 *   - NaN inputs to a quantizer are ignored by the amax and give code 0
 *     (candle's special-value table).
 *   - Q8_1 activations (paired with Q4_1 by [candle]'s VecDotType table;
 *     the byte layout is not printed): f16 d, f16 s, 32 int8 codes
 *     (36 bytes), where d and the codes follow the Q8_0 rule and
 *     s = f16(d * sum of the codes) in f32 with the unrounded d (a NaN s,
 *     which only a block holding inf produces, is stored as 0x7E00). The
 *     Q4_1 x Q8_1 block term is d_w * d_x * S + m_w * s_x (S = sum of
 *     code * q_x), so it carries s's f16 rounding.
 *
 * Parity pins: every function here is pinned by tests under tests/ against
 * values the pages print, closed forms or brute force; the Q6_K element
 * mapping, the Q8_K rule, Q8_1's s field and the Q2_K/Q3_K/Q5_K layouts
 * are pinned only by structural invariants (and Q5_K also by its reduction
 * to the pinned Q4_K): the pages do not define them, so they are "parity
 * unpinned" against ggml itself.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* Type table ([rml] The type table; [candle] GgmlDType table).             */
/* Numbers are the ggml element-type ids stored in GGUF tensor records.     */
/* ------------------------------------------------------------------------ */
enum {
    OR_F32 = 0, OR_F16 = 1, OR_Q4_0 = 2, OR_Q4_1 = 3, OR_Q5_0 = 6, OR_Q8_0 = 8, OR_Q8_1 = 9,
    OR_Q2_K = 10, OR_Q3_K = 11, OR_Q4_K = 12, OR_Q5_K = 13, OR_Q6_K = 14, OR_Q8_K = 15
};

/* Returns 0 and fills (elems, bytes) for a known id, -1 otherwise. */
int or_type_info(int type, int *elems, int *bytes) {
    switch (type) {
    case OR_F32:  *elems = 1;   *bytes = 4;   return 0;
    case OR_F16:  *elems = 1;   *bytes = 2;   return 0;
    case OR_Q4_0: *elems = 32;  *bytes = 18;  return 0;
    case OR_Q4_1: *elems = 32;  *bytes = 20;  return 0;
    case OR_Q5_0: *elems = 32;  *bytes = 22;  return 0;
    case OR_Q8_1: *elems = 32;  *bytes = 36;  return 0;
    case OR_Q8_0: *elems = 32;  *bytes = 34;  return 0;
    case OR_Q2_K: *elems = 256; *bytes = 84;  return 0;
    case OR_Q3_K: *elems = 256; *bytes = 110; return 0;
    case OR_Q4_K: *elems = 256; *bytes = 144; return 0;
    case OR_Q5_K: *elems = 256; *bytes = 176; return 0;
    case OR_Q6_K: *elems = 256; *bytes = 210; return 0;
    case OR_Q8_K: *elems = 256; *bytes = 292; return 0;
    default: return -1;
    }
}

/* n elements take n / elems * bytes bytes; -1 if n is not whole blocks
 * ([rml] The type table; [sipllm] type_nbytes). */
int64_t or_type_nbytes(int type, int64_t n) {
    int elems, bytes;
    if (or_type_info(type, &elems, &bytes) != 0) return -1;
    if (n < 0 || n % elems != 0) return -1;
    return n / elems * bytes;
}

/* ------------------------------------------------------------------------ */
/* Block layouts ([rml] Block layouts; [candle] block structure table).     */
/* Plain structs whose bytes match the file format; sizes pinned below.     */
/* ------------------------------------------------------------------------ */
typedef struct { uint16_t d; int8_t qs[32]; } or_block_q8_0;
typedef struct { uint16_t d; uint8_t qs[16]; } or_block_q4_0;
typedef struct { uint16_t d, m; uint8_t qs[16]; } or_block_q4_1;
typedef struct { uint16_t d; uint8_t qh[4]; uint8_t qs[16]; } or_block_q5_0;
typedef struct { uint16_t d, s; int8_t qs[32]; } or_block_q8_1;
typedef struct {
    uint16_t d;
    uint16_t dmin;
    uint8_t scales[12];
    uint8_t qs[128];
} or_block_q4_k;
typedef struct {
    uint8_t ql[128];
    uint8_t qh[64];
    int8_t scales[16];
    uint16_t d;
} or_block_q6_k;
typedef struct {
    uint8_t scales[16];  /* low nibble: scale, high nibble: min */
    uint8_t qs[64];
    uint16_t d;
    uint16_t dmin;
} or_block_q2_k;
typedef struct {
    uint8_t hmask[32];
    uint8_t qs[64];
    uint8_t scales[12];
    uint16_t d;
} or_block_q3_k;
typedef struct {
    uint16_t d;
    uint16_t dmin;
    uint8_t scales[12];
    uint8_t qh[32];
    uint8_t qs[128];
} or_block_q5_k;
typedef struct { float d; int8_t qs[256]; int16_t bsums[16]; } or_block_q8_k;

_Static_assert(sizeof(or_block_q8_0) == 34, "Q8_0 block is 34 bytes");
_Static_assert(sizeof(or_block_q4_0) == 18, "Q4_0 block is 18 bytes");
_Static_assert(sizeof(or_block_q4_1) == 20, "Q4_1 block is 20 bytes");
_Static_assert(sizeof(or_block_q5_0) == 22, "Q5_0 block is 22 bytes");
_Static_assert(sizeof(or_block_q8_1) == 36, "Q8_1 block is 36 bytes");
_Static_assert(sizeof(or_block_q4_k) == 144, "Q4_K block is 144 bytes");
_Static_assert(sizeof(or_block_q6_k) == 210, "Q6_K block is 210 bytes");
_Static_assert(sizeof(or_block_q2_k) == 84, "Q2_K block is 84 bytes");
_Static_assert(sizeof(or_block_q3_k) == 110, "Q3_K block is 110 bytes");
_Static_assert(sizeof(or_block_q5_k) == 176, "Q5_K block is 176 bytes");
_Static_assert(sizeof(or_block_q8_k) == 292, "Q8_K block is 292 bytes");

/* ------------------------------------------------------------------------ */
/* IEEE 754 binary16 codec, written from the format's definition:           */
/* 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits; exponent 0 is   */
/* zero/subnormal (value = m * 2^-24), exponent 31 is inf/NaN.  Encoding    */
/* rounds to nearest, ties to even; overflow gives inf.                     */
/* ------------------------------------------------------------------------ */
float or_f16_to_f32(uint16_t h) {
    int sign = h >> 15;
    int e = (h >> 10) & 31;
    int m = h & 1023;
    double v;
    if (e == 0) {
        v = ldexp((double)m, -24);
    } else if (e == 31) {
        v = (m == 0) ? INFINITY : NAN;
    } else {
        v = ldexp((double)(1024 + m), e - 25);
    }
    return (float)(sign ? -v : v);
}

/* Round a non-negative double to the nearest integer, ties to even. */
static double or_round_half_even(double s) {
    double fl = floor(s);
    double diff = s - fl;
    if (diff > 0.5) return fl + 1.0;
    if (diff < 0.5) return fl;
    return (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
}

uint16_t or_f32_to_f16(float f) {
    uint16_t sign = signbit(f) ? 0x8000 : 0;
    if (isnan(f)) return (uint16_t)(sign | 0x7E00);
    double a = fabs((double)f);
    if (a >= 65520.0) return (uint16_t)(sign | 0x7C00); /* 65504 + half ulp, tie goes up to 2^16 */
    if (a < ldexp(1.0, -14)) {
        /* subnormal range: value = m * 2^-24, m rounded half to even */
        double m = or_round_half_even(a * ldexp(1.0, 24));
        return (uint16_t)(sign | (uint16_t)m); /* m == 1024 encodes the smallest normal */
    }
    int ex;
    frexp(a, &ex);            /* a in [2^(ex-1), 2^ex) */
    int E = ex - 1;           /* unbiased exponent, -14..15 */
    double r = or_round_half_even(a * ldexp(1.0, 10 - E)); /* significand in [1024, 2048] */
    if (r == 2048.0) { r = 1024.0; E += 1; }
    if (E > 15) return (uint16_t)(sign | 0x7C00);
    return (uint16_t)(sign | (uint16_t)((E + 15) << 10) | (uint16_t)(r - 1024.0));
}

/* ------------------------------------------------------------------------ */
/* Code conversions shared by the quantizers.                               */
/* ------------------------------------------------------------------------ */

/* roundf result -> int8 code.  NaN gives 0 and out-of-range values
 * saturate, as the special-value table of [candle] shows; for finite
 * inputs the quantizers never leave [-127, 127]. */
static int or_code_from_rounded(float r, int lo, int hi) {
    if (isnan(r)) return 0;
    if (r < (float)lo) return lo;
    if (r > (float)hi) return hi;
    return (int)r;
}

/* ------------------------------------------------------------------------ */
/* Quantizers                                                               */
/* ------------------------------------------------------------------------ */

/* Q8_0 ([lesson21] Example 2, [candle] BlockQ8_0::from_float): per block of
 * 32, amax = largest |x| (NaN ignored), d = amax / 127 in f32, id = 1/d
 * (0 when d == 0), store f16(d), code = roundf(x * id) with halves away
 * from zero; codes use the unrounded id. Used for weights and activations. */
void or_quantize_q8_0(const float *x, uint8_t *out, int64_t n) {
    for (int64_t b = 0; b < n / 32; ++b) {
        const float *xb = x + b * 32;
        float amax = 0.0f;
        for (int j = 0; j < 32; ++j) {
            float a = fabsf(xb[j]);
            if (a > amax) amax = a;
        }
        float d = amax / 127.0f;
        float id = (d != 0.0f) ? 1.0f / d : 0.0f;
        or_block_q8_0 blk;
        blk.d = or_f32_to_f16(d);
        for (int j = 0; j < 32; ++j) {
            float scaled = xb[j] * id;
            blk.qs[j] = (int8_t)or_code_from_rounded(roundf(scaled), -128, 127);
        }
        memcpy(out + b * 34, &blk, 34);
    }
}

/* The float-to-int cast of the lesson's Java code ([lesson21] Examples 5, 7
 * and 8 are Java): truncation toward zero, 0 for NaN, and the int range's end
 * for values beyond it. C leaves (int) undefined for NaN and out-of-range
 * values, so the cast is written out. A NaN element, or a block whose scale
 * is so small that 1/d overflows to infinity, reaches these cases. */
static int or_java_f2i(float f) {
    if (isnan(f)) return 0;
    if (f >= 2147483648.0f) return INT32_MAX;
    if (f <= -2147483648.0f) return INT32_MIN;
    return (int)f;
}

/* Q4_0 ([lesson21] Example 5, [rml] A worked example: Q4_0): per block the
 * FIRST element of strictly largest magnitude gives max (a later tie does
 * not replace it), d = max / -8, id = 1/d (0 when d == 0), code =
 * min(15, (int)(x*id + 8.5f)) with the multiply and the add rounded
 * separately; byte j holds element j (low nibble) and j+16 (high nibble). */
void or_quantize_q4_0(const float *x, uint8_t *out, int64_t n) {
    for (int64_t b = 0; b < n / 32; ++b) {
        const float *xb = x + b * 32;
        float amax = 0.0f, max = 0.0f;
        for (int j = 0; j < 32; ++j) {
            if (amax < fabsf(xb[j])) {
                amax = fabsf(xb[j]);
                max = xb[j];
            }
        }
        float d = max / -8.0f;
        float id = (d != 0.0f) ? 1.0f / d : 0.0f;
        int code[32];
        for (int j = 0; j < 32; ++j) {
            float scaled = xb[j] * id;
            float shifted = scaled + 8.5f;
            int c = or_java_f2i(shifted);
            code[j] = c < 15 ? c : 15;
        }
        or_block_q4_0 blk;
        blk.d = or_f32_to_f16(d);
        /* low 4 bits of each code (a code below 0 comes only from -inf) */
        for (int j = 0; j < 16; ++j)
            blk.qs[j] = (uint8_t)((code[j] & 0x0F) | ((code[j + 16] & 0x0F) << 4));
        memcpy(out + b * 18, &blk, 18);
    }
}

/* Q4_1 ([lesson21] Example 7): per block of 32, min and max of the values,
 * d = (max - min) / 15, id = 1/d (0 when d == 0), store f16(d) and
 * f16(min), code = min(15, (int)((x - min) * id + 0.5f)) with the
 * subtraction, the multiply and the add each rounded in f32, using the
 * unrounded min; nibbles in Q4_0's order (byte j: element j low, j+16 high). */
void or_quantize_q4_1(const float *x, uint8_t *out, int64_t n) {
    for (int64_t b = 0; b < n / 32; ++b) {
        const float *xb = x + b * 32;
        float mn = 3.4028234663852886e38f, mx = -3.4028234663852886e38f;
        for (int j = 0; j < 32; ++j) {
            if (xb[j] < mn) mn = xb[j];
            if (xb[j] > mx) mx = xb[j];
        }
        float d = (mx - mn) / 15.0f;
        float id = (d != 0.0f) ? 1.0f / d : 0.0f;
        int code[32];
        for (int j = 0; j < 32; ++j) {
            float diff = xb[j] - mn;
            float scaled = diff * id;
            float shifted = scaled + 0.5f;
            int c = or_java_f2i(shifted);
            code[j] = c < 15 ? c : 15;
        }
        or_block_q4_1 blk;
        blk.d = or_f32_to_f16(d);
        blk.m = or_f32_to_f16(mn);
        for (int j = 0; j < 16; ++j)
            blk.qs[j] = (uint8_t)((code[j] & 0x0F) | ((code[j + 16] & 0x0F) << 4));
        memcpy(out + b * 20, &blk, 20);
    }
}

/* Q5_0 ([lesson21] Example 8): the Q4_0 rule with 5-bit codes -- the first
 * element of strictly largest magnitude gives max, d = max / -16, id = 1/d
 * (0 when d == 0), code = min(31, (int)(x * id + 16.5f)) with the multiply
 * and the add rounded separately. The low 4 bits go into nibbles as in
 * Q4_0; bit j of the 32-bit little-endian word qh is bit 4 of code j. */
void or_quantize_q5_0(const float *x, uint8_t *out, int64_t n) {
    for (int64_t b = 0; b < n / 32; ++b) {
        const float *xb = x + b * 32;
        float amax = 0.0f, max = 0.0f;
        for (int j = 0; j < 32; ++j) {
            if (amax < fabsf(xb[j])) {
                amax = fabsf(xb[j]);
                max = xb[j];
            }
        }
        float d = max / -16.0f;
        float id = (d != 0.0f) ? 1.0f / d : 0.0f;
        int code[32];
        for (int j = 0; j < 32; ++j) {
            float scaled = xb[j] * id;
            float shifted = scaled + 16.5f;
            int c = or_java_f2i(shifted);
            code[j] = c < 31 ? c : 31;
        }
        or_block_q5_0 blk;
        blk.d = or_f32_to_f16(d);
        uint32_t qh = 0;
        for (int j = 0; j < 32; ++j) qh |= (((uint32_t)code[j] >> 4) & 1u) << j;
        for (int i = 0; i < 4; ++i) blk.qh[i] = (uint8_t)(qh >> (8 * i));
        for (int j = 0; j < 16; ++j)
            blk.qs[j] = (uint8_t)((code[j] & 0x0F) | ((code[j + 16] & 0x0F) << 4));
        memcpy(out + b * 22, &blk, 22);
    }
}

/* Q8_1 activations (the reading stated at the top of this file): the Q8_0
 * rule, plus s = f16(d * sum of codes) with the f32 d; a NaN s (only from a
 * block holding inf) is stored as 0x7E00. */
void or_quantize_q8_1(const float *x, uint8_t *out, int64_t n) {
    for (int64_t b = 0; b < n / 32; ++b) {
        const float *xb = x + b * 32;
        float amax = 0.0f;
        for (int j = 0; j < 32; ++j) {
            float a = fabsf(xb[j]);
            if (a > amax) amax = a;
        }
        float d = amax / 127.0f;
        float id = (d != 0.0f) ? 1.0f / d : 0.0f;
        or_block_q8_1 blk;
        int sum = 0;
        for (int j = 0; j < 32; ++j) {
            float scaled = xb[j] * id;
            blk.qs[j] = (int8_t)or_code_from_rounded(roundf(scaled), -128, 127);
            sum += blk.qs[j];
        }
        blk.d = or_f32_to_f16(d);
        float sv = (float)sum * d;
        /* a block holding inf has d = inf, codes 0 and s = 0 * inf: store
         * the one quiet NaN 0x7E00 whatever sign the host's NaN carries */
        blk.s = isnan(sv) ? (uint16_t)0x7E00 : or_f32_to_f16(sv);
        memcpy(out + b * 36, &blk, 36);
    }
}

/* Q8_K activations ([candle] block table: f32 d, 256 codes, 16 bsums, each
 * the sum of 16 codes; [rml] Quantized dot products: bsums serve the K-quant
 * min term).  The rule itself is not printed; the reading used here is the
 * Q8_0 rule over 256 elements with d kept in f32 and codes clamped to
 * [-127, 127]. */
void or_quantize_q8_k(const float *x, uint8_t *out, int64_t n) {
    for (int64_t b = 0; b < n / 256; ++b) {
        const float *xb = x + b * 256;
        float amax = 0.0f;
        for (int j = 0; j < 256; ++j) {
            float a = fabsf(xb[j]);
            if (a > amax) amax = a;
        }
        float d = amax / 127.0f;
        float id = (d != 0.0f) ? 1.0f / d : 0.0f;
        or_block_q8_k blk;
        blk.d = d;
        for (int j = 0; j < 256; ++j) {
            float scaled = xb[j] * id;
            blk.qs[j] = (int8_t)or_code_from_rounded(roundf(scaled), -127, 127);
        }
        for (int k = 0; k < 16; ++k) {
            int s = 0;
            for (int i = 0; i < 16; ++i) s += blk.qs[16 * k + i];
            blk.bsums[k] = (int16_t)s;
        }
        memcpy(out + b * 292, &blk, 292);
    }
}

/* ------------------------------------------------------------------------ */
/* Readable unpacking helpers (one per packed field).                       */
/* ------------------------------------------------------------------------ */

/* Q4_0 element e of a block: byte e mod 16, low nibble for e < 16, high
 * nibble otherwise; the stored code c means c - 8 ([lesson21] Example 5). */
static int q4_0_code(const or_block_q4_0 *b, int e) {
    uint8_t byte = b->qs[e % 16];
    return (e < 16) ? (byte & 0x0F) : (byte >> 4);
}

/* Q5_0 element e: low 4 bits as in Q4_0, bit 4 = bit e of qh (the
 * decoder of [lesson21] Example 8 rebuilds it from bit j and bit j + 16);
 * the stored code c means c - 16. */
static int q5_0_code(const or_block_q5_0 *b, int e) {
    uint32_t qh = (uint32_t)b->qh[0] | ((uint32_t)b->qh[1] << 8) | ((uint32_t)b->qh[2] << 16) |
                  ((uint32_t)b->qh[3] << 24);
    uint8_t byte = b->qs[e % 16];
    int lo4 = (e < 16) ? (byte & 0x0F) : (byte >> 4);
    return lo4 | (int)(((qh >> e) & 1u) << 4);
}

/* Q4_1 element e: the nibble in Q4_0's order; its value is code * d + m. */
static int q4_1_code(const or_block_q4_1 *b, int e) {
    uint8_t byte = b->qs[e % 16];
    return (e < 16) ? (byte & 0x0F) : (byte >> 4);
}

/* Q4_K sub-block j scale and min from the 12 packed bytes
 * ([rml] Unpacking the packed fields; [candle] get_scale_min_k4 text):
 * sub-blocks 0..3 keep both in the low 6 bits of bytes j (scale) and j+4
 * (min); sub-blocks 4..7 keep their low 4 bits in byte j+4 (scale in the
 * low nibble, min in the high nibble) and borrow the top 2 bits of byte
 * j-4 (scale) and byte j (min). */
static void q4_k_scale_min(const uint8_t s[12], int j, int *scale, int *min) {
    if (j < 4) {
        *scale = s[j] & 63;
        *min = s[j + 4] & 63;
    } else {
        *scale = (s[j + 4] & 0x0F) | ((s[j - 4] >> 6) << 4);
        *min = (s[j + 4] >> 4) | ((s[j] >> 6) << 4);
    }
}

/* Q4_K element e: chunk e/64 of 32 bytes, low nibble for position < 32
 * in the chunk, high nibble otherwise ([rml] element-200 trace). */
static int q4_k_code(const or_block_q4_k *b, int e) {
    int chunk = e / 64, p = e % 64;
    if (p < 32) return b->qs[32 * chunk + p] & 0x0F;
    return b->qs[32 * chunk + p - 32] >> 4;
}

/* Q6_K element e (reading stated in the file header): low 4 bits from ql,
 * high 2 bits from qh; the stored q in 0..63 means q - 32 ([candle] block
 * table: d * sc[j] * (q - 32)). */
static int q6_k_code(const or_block_q6_k *b, int e) {
    int h = e / 128, k = (e % 128) / 32, l = e % 32;
    uint8_t lbyte = b->ql[64 * h + 32 * (k & 1) + l];
    int lo4 = (k < 2) ? (lbyte & 0x0F) : (lbyte >> 4);
    int hi2 = (b->qh[32 * h + l] >> (2 * k)) & 3;
    return lo4 | (hi2 << 4);
}

/* Q5_K element e: Q4_K's nibble plus a fifth bit, bit j of qh[e % 32] for
 * the 32-element sub-block j = e / 32 (reading in the file header). */
static int q5_k_code(const or_block_q5_k *b, int e) {
    int chunk = e / 64, p = e % 64, j = e / 32;
    int lo4 = (p < 32) ? (b->qs[32 * chunk + p] & 0x0F) : (b->qs[32 * chunk + p - 32] >> 4);
    int bit = (b->qh[e % 32] >> j) & 1;
    return lo4 | (bit << 4);
}

/* Q2_K element e = 128n + 32j + 16h + l: bits 2j..2j+1 of qs[32n + 16h + l]
 * (reading in the file header); its sub-block e / 16 has scale
 * scales[e/16] & 15 and min scales[e/16] >> 4. */
static int q2_k_code(const or_block_q2_k *b, int e) {
    int n = e / 128, j = (e % 128) / 32, h = (e % 32) / 16, l = e % 16;
    return (b->qs[32 * n + 16 * h + l] >> (2 * j)) & 3;
}

/* Q3_K element e = 128n + 32j + 16h + l: the 2-bit value as in Q2_K, less 4
 * when bit 4n + j of hmask[16h + l] is clear; the result is in -4..3. */
static int q3_k_code(const or_block_q3_k *b, int e) {
    int n = e / 128, j = (e % 128) / 32, h = (e % 32) / 16, l = e % 16;
    int q2 = (b->qs[32 * n + 16 * h + l] >> (2 * j)) & 3;
    int high = (b->hmask[16 * h + l] >> (4 * n + j)) & 1;
    return q2 - (high ? 0 : 4);
}

/* Q3_K sub-block scale j (0..15), unbiased to -32..31: low 4 bits in the
 * low nibble of byte j (j < 8) or the high nibble of byte j - 8, high 2
 * bits at bits 2(j/4)..2(j/4)+1 of byte 8 + j % 4. */
static int q3_k_scale(const uint8_t s[12], int j) {
    int lo4 = (j < 8) ? (s[j] & 0x0F) : (s[j - 8] >> 4);
    int hi2 = (s[8 + j % 4] >> (2 * (j / 4))) & 3;
    return (lo4 | (hi2 << 4)) - 32;
}

/* ------------------------------------------------------------------------ */
/* Dequantization ([sipllm] Per-format dequant; [candle] block table;      */
/* [rml] Dequantization: memcpy each block into a local struct first).      */
/* ------------------------------------------------------------------------ */
static void dequant_block(int type, const uint8_t *src, float *dst) {
    switch (type) {
    case OR_Q8_0: {
        or_block_q8_0 b; memcpy(&b, src, sizeof b);
        float d = or_f16_to_f32(b.d);
        for (int e = 0; e < 32; ++e) dst[e] = (float)b.qs[e] * d;
        break;
    }
    case OR_Q4_0: {
        or_block_q4_0 b; memcpy(&b, src, sizeof b);
        float d = or_f16_to_f32(b.d);
        for (int e = 0; e < 32; ++e) dst[e] = (float)(q4_0_code(&b, e) - 8) * d;
        break;
    }
    case OR_Q4_1: {
        or_block_q4_1 b; memcpy(&b, src, sizeof b);
        float d = or_f16_to_f32(b.d), m = or_f16_to_f32(b.m);
        for (int e = 0; e < 32; ++e) {
            float value = (float)q4_1_code(&b, e) * d; /* exact: 11 + 4 bits */
            dst[e] = value + m;                         /* the only rounding */
        }
        break;
    }
    case OR_Q5_0: {
        or_block_q5_0 b; memcpy(&b, src, sizeof b);
        float d = or_f16_to_f32(b.d);
        for (int e = 0; e < 32; ++e) dst[e] = (float)(q5_0_code(&b, e) - 16) * d;
        break;
    }
    case OR_Q8_1: {
        or_block_q8_1 b; memcpy(&b, src, sizeof b);
        float d = or_f16_to_f32(b.d);
        for (int e = 0; e < 32; ++e) dst[e] = (float)b.qs[e] * d;
        break;
    }
    case OR_Q4_K: {
        or_block_q4_k b; memcpy(&b, src, sizeof b);
        float d = or_f16_to_f32(b.d), dmin = or_f16_to_f32(b.dmin);
        for (int e = 0; e < 256; ++e) {
            int sc, m;
            q4_k_scale_min(b.scales, e / 32, &sc, &m);
            float scaled = d * (float)sc;      /* exact: 11 + 6 bits */
            float value = scaled * (float)q4_k_code(&b, e); /* exact: 21 bits */
            float offset = dmin * (float)m;    /* exact: 17 bits */
            dst[e] = value - offset;           /* the only rounding */
        }
        break;
    }
    case OR_Q5_K: {
        or_block_q5_k b; memcpy(&b, src, sizeof b);
        float d = or_f16_to_f32(b.d), dmin = or_f16_to_f32(b.dmin);
        for (int e = 0; e < 256; ++e) {
            int sc, m;
            q4_k_scale_min(b.scales, e / 32, &sc, &m);
            float scaled = d * (float)sc;      /* exact: 11 + 6 bits */
            float value = scaled * (float)q5_k_code(&b, e); /* exact: 22 bits */
            float offset = dmin * (float)m;    /* exact: 17 bits */
            dst[e] = value - offset;           /* the only rounding */
        }
        break;
    }
    case OR_Q2_K: {
        or_block_q2_k b; memcpy(&b, src, sizeof b);
        float d = or_f16_to_f32(b.d), dmin = or_f16_to_f32(b.dmin);
        for (int e = 0; e < 256; ++e) {
            int sc = b.scales[e / 16] & 0x0F, m = b.scales[e / 16] >> 4;
            float value = (d * (float)sc) * (float)q2_k_code(&b, e); /* exact: 17 bits */
            float offset = dmin * (float)m;                          /* exact: 15 bits */
            dst[e] = value - offset;                                 /* the only rounding */
        }
        break;
    }
    case OR_Q3_K: {
        or_block_q3_k b; memcpy(&b, src, sizeof b);
        float d = or_f16_to_f32(b.d);
        for (int e = 0; e < 256; ++e) {
            float scaled = d * (float)q3_k_scale(b.scales, e / 16); /* exact: 11 + 6 bits */
            dst[e] = scaled * (float)q3_k_code(&b, e);               /* exact: 20 bits */
        }
        break;
    }
    case OR_Q6_K: {
        or_block_q6_k b; memcpy(&b, src, sizeof b);
        float d = or_f16_to_f32(b.d);
        for (int e = 0; e < 256; ++e) {
            float scaled = d * (float)b.scales[e / 16];          /* exact: 11 + 7 bits */
            dst[e] = scaled * (float)(q6_k_code(&b, e) - 32);    /* exact: 24 bits */
        }
        break;
    }
    case OR_Q8_K: {
        or_block_q8_k b; memcpy(&b, src, sizeof b);
        for (int e = 0; e < 256; ++e) dst[e] = (float)b.qs[e] * b.d;
        break;
    }
    default:
        break;
    }
}

/* Dequantize n elements (whole blocks) of `type`. Returns 0, or -1 for an
 * unsupported type or a length that is not whole blocks. */
int or_dequantize(int type, const uint8_t *src, float *dst, int64_t n) {
    int elems, bytes;
    if (or_type_info(type, &elems, &bytes) != 0) return -1;
    if (type == OR_F32 || type == OR_F16) return -1;
    if (n % elems != 0) return -1;
    for (int64_t b = 0; b < n / elems; ++b)
        dequant_block(type, src + b * bytes, dst + b * elems);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Weight -> activation pairing ([rml] DotActivationType; [candle]          */
/* VecDotType table): Q4_0, Q5_0 and Q8_0 pair with Q8_0, Q4_1 with Q8_1,   */
/* the K-quants with Q8_K.                                                  */
/* ------------------------------------------------------------------------ */
int or_act_type(int wtype) {
    switch (wtype) {
    case OR_Q4_0: case OR_Q5_0: case OR_Q8_0: return OR_Q8_0;
    case OR_Q4_1: return OR_Q8_1;
    case OR_Q2_K: case OR_Q3_K: case OR_Q4_K: case OR_Q5_K: case OR_Q6_K: return OR_Q8_K;
    default: return -1;
    }
}

/* Number of int32 sums per (vector, row, block): the types with a dmin
 * (Q2_K, Q4_K, Q5_K) keep the scale sum S_q and the min sum S_m apart,
 * every other type has one sum S. */
int or_isums_per_block(int wtype) {
    return (wtype == OR_Q2_K || wtype == OR_Q4_K || wtype == OR_Q5_K) ? 2 : 1;
}

/* ------------------------------------------------------------------------ */
/* Per-block exact integer sums, element by element (the reference form of  */
/* [rml] Kernels and references: each q decoded on its own, the K-quant min */
/* term summed per element rather than through bsums).                      */
/*                                                                          */
/*   Q8_0: S = sum_i qw_i * qx_i                 ([lesson21] Example 10)    */
/*   Q4_0: S = sum_i (code_i - 8) * qx_i         ([lesson21] Example 11)    */
/*   Q5_0: S = sum_i (code_i - 16) * qx_i        ([lesson21] Example 8)     */
/*   Q4_1: S = sum_i code_i * qx_i (the min m enters with s_x, below)       */
/*   Q4_K: S_q = sum_j sc_j * sum_{i in j} q_i * a_i,                       */
/*         S_m = sum_j m_j * sum_{i in j} a_i    ([rml] Quantized dot)      */
/*   Q6_K: S = sum_j sc_j * sum_{i in j} (q_i - 32) * a_i                   */
/*   Q5_K: as Q4_K with the 5-bit q; Q2_K: as Q4_K over 16-element          */
/*         sub-blocks; Q3_K: S = sum_j sc_j * sum_{i in j} q_i * a_i with   */
/*         q in -4..3 and sc in -32..31                                     */
/* ------------------------------------------------------------------------ */
static void block_sums(int wtype, const uint8_t *wblk, const uint8_t *xblk, int32_t *out) {
    switch (wtype) {
    case OR_Q8_0: {
        or_block_q8_0 w, x; memcpy(&w, wblk, 34); memcpy(&x, xblk, 34);
        int32_t s = 0;
        for (int i = 0; i < 32; ++i) s += (int32_t)w.qs[i] * (int32_t)x.qs[i];
        out[0] = s;
        break;
    }
    case OR_Q4_0: {
        or_block_q4_0 w; or_block_q8_0 x; memcpy(&w, wblk, 18); memcpy(&x, xblk, 34);
        int32_t s = 0;
        for (int i = 0; i < 32; ++i) s += (int32_t)(q4_0_code(&w, i) - 8) * (int32_t)x.qs[i];
        out[0] = s;
        break;
    }
    case OR_Q5_0: {
        or_block_q5_0 w; or_block_q8_0 x; memcpy(&w, wblk, 22); memcpy(&x, xblk, 34);
        int32_t s = 0;
        for (int i = 0; i < 32; ++i) s += (int32_t)(q5_0_code(&w, i) - 16) * (int32_t)x.qs[i];
        out[0] = s;
        break;
    }
    case OR_Q4_1: {
        or_block_q4_1 w; or_block_q8_1 x; memcpy(&w, wblk, 20); memcpy(&x, xblk, 36);
        int32_t s = 0;
        for (int i = 0; i < 32; ++i) s += (int32_t)q4_1_code(&w, i) * (int32_t)x.qs[i];
        out[0] = s;
        break;
    }
    case OR_Q4_K: {
        or_block_q4_k w; or_block_q8_k x; memcpy(&w, wblk, 144); memcpy(&x, xblk, 292);
        int32_t sq = 0, sm = 0;
        for (int j = 0; j < 8; ++j) {
            int sc, m;
            q4_k_scale_min(w.scales, j, &sc, &m);
            int32_t dot = 0, asum = 0;
            for (int i = 32 * j; i < 32 * j + 32; ++i) {
                dot += (int32_t)q4_k_code(&w, i) * (int32_t)x.qs[i];
                asum += (int32_t)x.qs[i];
            }
            sq += sc * dot;
            sm += m * asum;
        }
        out[0] = sq;
        out[1] = sm;
        break;
    }
    case OR_Q5_K: {
        or_block_q5_k w; or_block_q8_k x; memcpy(&w, wblk, 176); memcpy(&x, xblk, 292);
        int32_t sq = 0, sm = 0;
        for (int j = 0; j < 8; ++j) {
            int sc, m;
            q4_k_scale_min(w.scales, j, &sc, &m);
            int32_t dot = 0, asum = 0;
            for (int i = 32 * j; i < 32 * j + 32; ++i) {
                dot += (int32_t)q5_k_code(&w, i) * (int32_t)x.qs[i];
                asum += (int32_t)x.qs[i];
            }
            sq += sc * dot;
            sm += m * asum;
        }
        out[0] = sq;
        out[1] = sm;
        break;
    }
    case OR_Q2_K: {
        or_block_q2_k w; or_block_q8_k x; memcpy(&w, wblk, 84); memcpy(&x, xblk, 292);
        int32_t sq = 0, sm = 0;
        for (int j = 0; j < 16; ++j) {
            int32_t dot = 0, asum = 0;
            for (int i = 16 * j; i < 16 * j + 16; ++i) {
                dot += (int32_t)q2_k_code(&w, i) * (int32_t)x.qs[i];
                asum += (int32_t)x.qs[i];
            }
            sq += (w.scales[j] & 0x0F) * dot;
            sm += (w.scales[j] >> 4) * asum;
        }
        out[0] = sq;
        out[1] = sm;
        break;
    }
    case OR_Q3_K: {
        or_block_q3_k w; or_block_q8_k x; memcpy(&w, wblk, 110); memcpy(&x, xblk, 292);
        int32_t s = 0;
        for (int j = 0; j < 16; ++j) {
            int32_t dot = 0;
            for (int i = 16 * j; i < 16 * j + 16; ++i)
                dot += (int32_t)q3_k_code(&w, i) * (int32_t)x.qs[i];
            s += q3_k_scale(w.scales, j) * dot;
        }
        out[0] = s;
        break;
    }
    case OR_Q6_K: {
        or_block_q6_k w; or_block_q8_k x; memcpy(&w, wblk, 210); memcpy(&x, xblk, 292);
        int32_t s = 0;
        for (int j = 0; j < 16; ++j) {
            int32_t dot = 0;
            for (int i = 16 * j; i < 16 * j + 16; ++i)
                dot += (int32_t)(q6_k_code(&w, i) - 32) * (int32_t)x.qs[i];
            s += (int32_t)w.scales[j] * dot;
        }
        out[0] = s;
        break;
    }
    default:
        break;
    }
}

/* Block scales as doubles: (d_w, dmin_w, d_x) and the additive term off
 * (Q4_1: m_w * s_x, else 0). dmin_w is 0 except Q2_K, Q4_K and Q5_K. */
static void block_scales(int wtype, const uint8_t *wblk, const uint8_t *xblk,
                         double *dw, double *dmin, double *dx, double *off) {
    *dmin = 0.0;
    *off = 0.0;
    switch (wtype) {
    case OR_Q5_0: { or_block_q5_0 w; or_block_q8_0 x; memcpy(&w, wblk, 22); memcpy(&x, xblk, 34);
        *dw = or_f16_to_f32(w.d); *dx = or_f16_to_f32(x.d); break; }
    case OR_Q4_1: { or_block_q4_1 w; or_block_q8_1 x; memcpy(&w, wblk, 20); memcpy(&x, xblk, 36);
        *dw = or_f16_to_f32(w.d); *dx = or_f16_to_f32(x.d);
        *off = (double)or_f16_to_f32(w.m) * (double)or_f16_to_f32(x.s); break; }
    case OR_Q8_0: { or_block_q8_0 w, x; memcpy(&w, wblk, 34); memcpy(&x, xblk, 34);
        *dw = or_f16_to_f32(w.d); *dx = or_f16_to_f32(x.d); break; }
    case OR_Q4_0: { or_block_q4_0 w; or_block_q8_0 x; memcpy(&w, wblk, 18); memcpy(&x, xblk, 34);
        *dw = or_f16_to_f32(w.d); *dx = or_f16_to_f32(x.d); break; }
    case OR_Q4_K: { or_block_q4_k w; or_block_q8_k x; memcpy(&w, wblk, 144); memcpy(&x, xblk, 292);
        *dw = or_f16_to_f32(w.d); *dmin = or_f16_to_f32(w.dmin); *dx = x.d; break; }
    case OR_Q6_K: { or_block_q6_k w; or_block_q8_k x; memcpy(&w, wblk, 210); memcpy(&x, xblk, 292);
        *dw = or_f16_to_f32(w.d); *dx = x.d; break; }
    case OR_Q5_K: { or_block_q5_k w; or_block_q8_k x; memcpy(&w, wblk, 176); memcpy(&x, xblk, 292);
        *dw = or_f16_to_f32(w.d); *dmin = or_f16_to_f32(w.dmin); *dx = x.d; break; }
    case OR_Q2_K: { or_block_q2_k w; or_block_q8_k x; memcpy(&w, wblk, 84); memcpy(&x, xblk, 292);
        *dw = or_f16_to_f32(w.d); *dmin = or_f16_to_f32(w.dmin); *dx = x.d; break; }
    case OR_Q3_K: { or_block_q3_k w; or_block_q8_k x; memcpy(&w, wblk, 110); memcpy(&x, xblk, 292);
        *dw = or_f16_to_f32(w.d); *dx = x.d; break; }
    default: *dw = 0.0; *dx = 0.0; break;
    }
}

static int geometry(int wtype, int64_t n_in, int *wel, int *wby, int *xby) {
    int at = or_act_type(wtype), xel;
    if (at < 0) return -1;
    if (or_type_info(wtype, wel, wby) != 0) return -1;
    if (or_type_info(at, &xel, xby) != 0) return -1;
    if (xel != *wel || n_in % *wel != 0) return -1;
    return 0;
}

/* Per-(vector, row, block) sums, written to
 * isums[((v * n_out + o) * nb + b) * k + t], k = or_isums_per_block(wtype).
 * W is [n_out][n_in] in blocks of wtype; xq is [n_vec][n_in] in blocks of
 * the paired activation type. Returns 0 or -1 on a bad type/shape. */
int or_block_isums(int wtype, const uint8_t *W, const uint8_t *xq, int32_t *isums,
                   int64_t n_out, int64_t n_in, int64_t n_vec) {
    int wel, wby, xby;
    if (geometry(wtype, n_in, &wel, &wby, &xby) != 0) return -1;
    int64_t nb = n_in / wel;
    int k = or_isums_per_block(wtype);
    for (int64_t v = 0; v < n_vec; ++v)
        for (int64_t o = 0; o < n_out; ++o)
            for (int64_t b = 0; b < nb; ++b)
                block_sums(wtype, W + (o * nb + b) * wby, xq + (v * nb + b) * xby,
                           isums + ((v * n_out + o) * nb + b) * k);
    return 0;
}

/* y[v * n_out + o] for rows o in [row0, row1), accumulated in f64 over the
 * row's blocks ([lesson21] Example 10: integer sum per block times both
 * scales):  Q8_0/Q4_0/Q5_0/Q3_K/Q6_K: T_b = d_w * d_x * S;
 *           Q4_1:                     T_b = d_w * d_x * S + m_w * s_x;
 *           Q2_K/Q4_K/Q5_K:           T_b = d_x * (d_w * S_q - dmin_w * S_m). */
int or_gemv(int wtype, const uint8_t *W, const uint8_t *xq, double *y,
            int64_t n_out, int64_t n_in, int64_t n_vec, int64_t row0, int64_t row1) {
    int wel, wby, xby;
    if (geometry(wtype, n_in, &wel, &wby, &xby) != 0) return -1;
    if (row0 < 0 || row1 > n_out || row0 > row1) return -1;
    int64_t nb = n_in / wel;
    for (int64_t v = 0; v < n_vec; ++v)
        for (int64_t o = row0; o < row1; ++o) {
            double acc = 0.0;
            for (int64_t b = 0; b < nb; ++b) {
                const uint8_t *wb = W + (o * nb + b) * wby;
                const uint8_t *xb = xq + (v * nb + b) * xby;
                int32_t s[2] = {0, 0};
                double dw, dmin, dx, off;
                block_sums(wtype, wb, xb, s);
                block_scales(wtype, wb, xb, &dw, &dmin, &dx, &off);
                if (or_isums_per_block(wtype) == 2)
                    acc += dx * (dw * (double)s[0] - dmin * (double)s[1]);
                else
                    acc += dw * dx * (double)s[0] + off;
            }
            y[v * n_out + o] = acc;
        }
    return 0;
}

/* Exact value of one element as a double (no rounding at all), for the
 * brute-force form below. */
static double exact_weight(int wtype, const uint8_t *blk, int e) {
    switch (wtype) {
    case OR_Q8_0: { or_block_q8_0 b; memcpy(&b, blk, 34);
        return (double)b.qs[e] * (double)or_f16_to_f32(b.d); }
    case OR_Q4_0: { or_block_q4_0 b; memcpy(&b, blk, 18);
        return (double)(q4_0_code(&b, e) - 8) * (double)or_f16_to_f32(b.d); }
    case OR_Q5_0: { or_block_q5_0 b; memcpy(&b, blk, 22);
        return (double)(q5_0_code(&b, e) - 16) * (double)or_f16_to_f32(b.d); }
    case OR_Q4_1: { or_block_q4_1 b; memcpy(&b, blk, 20);
        return (double)q4_1_code(&b, e) * (double)or_f16_to_f32(b.d) + (double)or_f16_to_f32(b.m); }
    case OR_Q4_K: { or_block_q4_k b; memcpy(&b, blk, 144);
        int sc, m; q4_k_scale_min(b.scales, e / 32, &sc, &m);
        return (double)or_f16_to_f32(b.d) * sc * q4_k_code(&b, e)
             - (double)or_f16_to_f32(b.dmin) * m; }
    case OR_Q6_K: { or_block_q6_k b; memcpy(&b, blk, 210);
        return (double)or_f16_to_f32(b.d) * b.scales[e / 16] * (q6_k_code(&b, e) - 32); }
    case OR_Q5_K: { or_block_q5_k b; memcpy(&b, blk, 176);
        int sc, m; q4_k_scale_min(b.scales, e / 32, &sc, &m);
        return (double)or_f16_to_f32(b.d) * sc * q5_k_code(&b, e)
             - (double)or_f16_to_f32(b.dmin) * m; }
    case OR_Q2_K: { or_block_q2_k b; memcpy(&b, blk, 84);
        int sc = b.scales[e / 16] & 0x0F, m = b.scales[e / 16] >> 4;
        return (double)or_f16_to_f32(b.d) * sc * q2_k_code(&b, e)
             - (double)or_f16_to_f32(b.dmin) * m; }
    case OR_Q3_K: { or_block_q3_k b; memcpy(&b, blk, 110);
        return (double)or_f16_to_f32(b.d) * q3_k_scale(b.scales, e / 16) * q3_k_code(&b, e); }
    default: return 0.0;
    }
}

static double exact_act(int atype, const uint8_t *blk, int e) {
    if (atype == OR_Q8_0) { or_block_q8_0 b; memcpy(&b, blk, 34);
        return (double)b.qs[e] * (double)or_f16_to_f32(b.d); }
    if (atype == OR_Q8_1) { or_block_q8_1 b; memcpy(&b, blk, 36);
        return (double)b.qs[e] * (double)or_f16_to_f32(b.d); }
    or_block_q8_k b; memcpy(&b, blk, 292);
    return (double)b.qs[e] * (double)b.d;
}

/* Second form ([sipllm] The fused matmul: dequantize one row, then dot):
 * dequantize W and the quantized activations to exact doubles and take a
 * plain f64 dot. Equal to or_gemv up to f64 rounding, except for Q4_1,
 * whose block form takes the min term through the f16-rounded s_x: there
 * the two differ by sum_b m_w * (s_x - d_x * sum of codes). */
int or_gemv_dequant(int wtype, const uint8_t *W, const uint8_t *xq, double *y,
                    int64_t n_out, int64_t n_in, int64_t n_vec) {
    int wel, wby, xby;
    if (geometry(wtype, n_in, &wel, &wby, &xby) != 0) return -1;
    int at = or_act_type(wtype);
    int64_t nb = n_in / wel;
    for (int64_t v = 0; v < n_vec; ++v)
        for (int64_t o = 0; o < n_out; ++o) {
            double acc = 0.0;
            for (int64_t i = 0; i < n_in; ++i) {
                int64_t b = i / wel;
                int e = (int)(i % wel);
                acc += exact_weight(wtype, W + (o * nb + b) * wby, e)
                     * exact_act(at, xq + (v * nb + b) * xby, e);
            }
            y[v * n_out + o] = acc;
        }
    return 0;
}

/* Returns 1 when the host stores integers little-endian, as the file
 * format does (the struct decode above relies on it). */
int or_host_is_little_endian(void) {
    uint16_t probe = 1;
    uint8_t first;
    memcpy(&first, &probe, 1);
    return first == 1;
}
