/*
 * fp8_oracle.c -- plain, slow CPU oracle for FP8 scaled quantization.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this code.  It shares nothing with
 * the CUDA path (no headers, tables, helpers or constants) and is compiled
 * with gcc, -O2 -ffp-contract=off, no fast-math, so every float operation
 * below is one IEEE-754 binary32 operation rounded to nearest-even.
 *
 * What it follows ("FP8 quantized-training guide" = the scrxy.com page,
 * "Colossal-AI FP8" = the liutaoaihuanlian.com page):
 *   - E4M3 = 1 sign / 4 exponent / 3 mantissa bits, E5M2 = 1/5/2
 *     (FP8 quantized-training guide, section "format choice E4M3 and E5M2").
 *     Largest finite values 448 and 57344; E4M3 has no infinity (the "fn"
 *     encoding: S.1111.111 is NaN), E5M2 is IEEE-like.
 *   - Per-tensor current scaling: amax of the current tensor, scale =
 *     FMAX / amax (Colossal-AI FP8, "current scaling"; guide, "instant
 *     scaling scheme").
 *   - Delayed scaling: a buffer of past amaxes, scale from its maximum
 *     (Colossal-AI FP8, "delayed scaling"; guide, "delayed scaling scheme").
 *   - Blockwise scaling: 1x128 tiles for activations/gradients, 128x128 for
 *     weights, one scale per tile (guide, section "block-level scaling").
 *   - MXFP8: 1x32 blocks with an E8M0 (power of two) scale (guide, section
 *     "MXFP8 scaling").
 * Readings where the pages are silent are listed next to each function.
 *
 * Parity status of each function is stated in the test suite; all functions
 * here are pinned (closed forms, library cross-checks, brute force, invariants).
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_E4M3 0
#define ORC_E5M2 1

static float bits_to_float(uint32_t b) { float f; memcpy(&f, &b, 4); return f; }
static uint32_t float_to_bits(float f) { uint32_t b; memcpy(&b, &f, 4); return b; }

/* bf16 is the upper half of a binary32: widening is exact. */
static float bf16_to_float(uint16_t h) { return bits_to_float((uint32_t)h << 16); }

/* Largest finite magnitude of each format (1-4-3: 1.75 * 2^8; 1-5-2: 1.75 * 2^15). */
float orc_fmax(int fmt) { return fmt == ORC_E4M3 ? 448.0f : 57344.0f; }

/*
 * Value of a positive 7-bit magnitude code read with the plain exponent /
 * mantissa formula, ignoring the codes each format reserves for NaN/inf.
 *   E4M3 (bias 7):  e == 0 -> m/8 * 2^-6 ; else (1 + m/8) * 2^(e-7)
 *   E5M2 (bias 15): e == 0 -> m/4 * 2^-14; else (1 + m/4) * 2^(e-15)
 */
static double magnitude_value(unsigned mag, int fmt)
{
    if (fmt == ORC_E4M3) {
        unsigned e = (mag >> 3) & 0xF, m = mag & 0x7;
        if (e == 0) return ldexp((double)m, -9);
        return ldexp((double)(8 + m), (int)e - 10);
    } else {
        unsigned e = (mag >> 2) & 0x1F, m = mag & 0x3;
        if (e == 0) return ldexp((double)m, -16);
        return ldexp((double)(4 + m), (int)e - 17);
    }
}

static unsigned max_finite_code(int fmt) { return fmt == ORC_E4M3 ? 0x7Eu : 0x7Bu; }

/* Decode one FP8 code to binary32 (exact: every FP8 value is a binary32). */
float orc_decode(uint8_t code, int fmt)
{
    uint32_t sign = (uint32_t)(code >> 7) << 31;
    unsigned mag = code & 0x7Fu;
    if (fmt == ORC_E4M3) {
        if (mag == 0x7F) return bits_to_float(sign | 0x7FC00000u);      /* S.1111.111: NaN */
    } else {
        if (mag == 0x7C) return bits_to_float(sign | 0x7F800000u);      /* S.11111.00: inf */
        if (mag > 0x7C)  /* S.11111.mm, mm != 0: NaN; keep mm as the top payload bits */
            return bits_to_float(sign | 0x7F800000u | ((uint32_t)(mag & 3) << 21));
    }
    float v = (float)magnitude_value(mag, fmt);
    return sign ? -v : v;
}

/*
 * Round a binary32 to FP8, round-to-nearest, ties-to-even, with gradual
 * underflow.  saturate == 0: overflow past the rounding threshold of the
 * largest finite value gives NaN (E4M3) or inf (E5M2).  saturate != 0: any
 * magnitude above the largest finite value (inf included) gives +-max; this
 * is the "saturating RNE cast" of the quantizer.  NaN stays NaN (sign kept;
 * E5M2 keeps the two top payload bits, forced to 0b10 when both are zero).
 *
 * Method: the positive codes 0..max are increasing in value, so find the
 * two codes whose values bracket |v| and compare |v| with their exact
 * midpoint (all quantities are exact in double).  A tie picks the even code,
 * which is the one whose last mantissa bit is 0.
 */
uint8_t orc_encode(float v, int fmt, int saturate)
{
    uint32_t bits = float_to_bits(v);
    uint8_t sign = (uint8_t)((bits >> 31) << 7);
    if (isnan(v)) {
        if (fmt == ORC_E4M3) return (uint8_t)(sign | 0x7F);
        unsigned payload = (bits >> 21) & 3u;
        if (payload == 0) payload = 2;
        return (uint8_t)(sign | 0x7C | payload);
    }
    double a = fabs((double)v);
    unsigned maxc = max_finite_code(fmt);
    double vmax = magnitude_value(maxc, fmt);
    if (a > vmax) {
        if (saturate) return (uint8_t)(sign | maxc);
        double next = magnitude_value(maxc + 1, fmt);   /* 480 for E4M3, 65536 for E5M2 */
        double mid = 0.5 * (vmax + next);
        if (a < mid || (a == mid && (maxc & 1u) == 0)) return (uint8_t)(sign | maxc);
        return (uint8_t)(sign | (fmt == ORC_E4M3 ? 0x7F : 0x7C));
    }
    unsigned lo = 0, hi = maxc;                 /* largest code with value <= a */
    while (lo < hi) {
        unsigned mid = (lo + hi + 1) / 2;
        if (magnitude_value(mid, fmt) <= a) lo = mid; else hi = mid - 1;
    }
    double vlo = magnitude_value(lo, fmt);
    if (vlo == a) return (uint8_t)(sign | lo);
    unsigned up = lo + 1;
    double mid = 0.5 * (vlo + magnitude_value(up, fmt));
    unsigned c;
    if (a < mid) c = lo;
    else if (a > mid) c = up;
    else c = (lo & 1u) ? up : lo;
    return (uint8_t)(sign | c);
}

void orc_decode_array(const uint8_t* q, int64_t n, int fmt, float* out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = orc_decode(q[i], fmt);
}

void orc_encode_array(const float* v, int64_t n, int fmt, int saturate, uint8_t* out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = orc_encode(v[i], fmt, saturate);
}

/*
 * amax = max |x| over the elements, NaN ignored (reading: the pages take
 * "the maximum of the current batch"; NaN has no magnitude).  -0 counts as 0.
 */
float orc_amax_bf16(const uint16_t* x, int64_t n)
{
    float amax = 0.0f;
    for (int64_t i = 0; i < n; ++i) {
        float a = fabsf(bf16_to_float(x[i]));
        if (a > amax) amax = a;
    }
    return amax;
}

/*
 * The same maximum over binary32 values: the amax of a GEMM output that the
 * delayed-scaling history records when the output stays in FP32 (Colossal-AI
 * FP8 article, "delayed scaling").
 */
float orc_amax_f32(const float* x, int64_t n)
{
    float amax = 0.0f;
    for (int64_t i = 0; i < n; ++i) {
        float a = fabsf(x[i]);
        if (a > amax) amax = a;
    }
    return amax;
}

/*
 * Per-tensor (and per-tile) scale rule: scale = FMAX / amax, one binary32
 * division; scale_inv = 1 / scale.  Readings (pages silent): amax == 0 or
 * non-finite gives scale 1; a quotient that overflows to inf becomes FLT_MAX;
 * no safety margin.
 */
void orc_tensor_scale(float amax, int fmt, float* scale, float* scale_inv)
{
    float s;
    if (!(amax > 0.0f) || isinf(amax)) {
        s = 1.0f;
    } else {
        s = orc_fmax(fmt) / amax;
        if (isinf(s)) s = FLT_MAX;
    }
    *scale = s;
    *scale_inv = 1.0f / s;
}

/*
 * One delayed-scaling update: record this step's amax in the history ring,
 * advance the write position, and derive the next step's scale from the
 * maximum over the whole window (reading of "a buffer of the maxima of past
 * training steps").  A window maximum that is zero or non-finite leaves the
 * scale unchanged.
 */
void orc_history_step(float* hist, int32_t len, int32_t* pos, float amax, int fmt,
                      float* scale, float* scale_inv)
{
    hist[*pos] = amax;
    *pos = (*pos + 1) % len;
    float m = 0.0f;
    for (int32_t i = 0; i < len; ++i)
        if (hist[i] > m) m = hist[i];
    if (m > 0.0f && !isinf(m)) {
        float s = orc_fmax(fmt) / m;
        if (isinf(s)) s = FLT_MAX;
        *scale = s;
        *scale_inv = 1.0f / s;
    }
}

/*
 * MX block exponent: the smallest integer e with amax <= FMAX * 2^e, taken
 * from [-127, 127] by direct search (each comparison is exact in double).
 * Readings: amax == 0 or non-finite gives e = 0.  The stored E8M0 byte is
 * e + 127 and the block is multiplied by 2^-e before the cast, so the largest
 * element of a block never exceeds FMAX.
 */
int orc_mx_exponent(float amax, int fmt)
{
    if (!(amax > 0.0f) || isinf(amax)) return 0;
    double fmax = (double)orc_fmax(fmt);
    for (int e = -127; e <= 127; ++e)
        if ((double)amax <= ldexp(fmax, e)) return e;
    return 127;
}

/*
 * MX block exponent, floor convention -- the documented alternate (the ceil rule above
 * is the default).  e = floor(log2 amax) - emax, with emax the exponent of the format's
 * largest power of two (8 for E4M3: 256; 15 for E5M2: 32768), so the block maximum
 * scales into [2^emax, 2^(emax + 1)) and the part of the block above FMAX saturates.
 * Taken as the largest e in [-127, 127] with 2^(e + emax) <= amax, by direct search
 * (each comparison exact in double); amax == 0 or non-finite gives e = 0.
 */
int orc_mx_exponent_floor(float amax, int fmt)
{
    if (!(amax > 0.0f) || isinf(amax)) return 0;
    int emax = fmt == ORC_E4M3 ? 8 : 15;
    for (int e = 127; e >= -127; --e)
        if (ldexp(1.0, e + emax) <= (double)amax) return e;
    return -127;
}

/* 2^-e as a binary32 (exact for e in [-127, 127]; 2^-127 is subnormal). */
static float pow2_neg(int e) { return (float)ldexp(1.0, -e); }

/* Cast one element: binary32 product x * scale, then the saturating cast. */
static uint8_t quantize_one(uint16_t x, float scale, int fmt)
{
    float p = bf16_to_float(x) * scale;
    return orc_encode(p, fmt, 1);
}

/* Per-tensor quantize of a row-major [R, C] bf16 matrix with a given scale. */
void orc_quantize_tensor(const uint16_t* x, int64_t R, int64_t C, int fmt, float scale, uint8_t* q)
{
    for (int64_t i = 0; i < R * C; ++i) q[i] = quantize_one(x[i], scale, fmt);
}

/*
 * 1 x 128 blockwise quantize along the contiguous dimension: each run of
 * 128 consecutive elements of a row gets its own amax and scale.
 * s_inv is row-major [R, C/128].  C must be a multiple of 128.
 */
void orc_quantize_1x128(const uint16_t* x, int64_t R, int64_t C, int fmt, uint8_t* q, float* s_inv)
{
    int64_t nb = C / 128;
    for (int64_t r = 0; r < R; ++r) {
        for (int64_t b = 0; b < nb; ++b) {
            const uint16_t* blk = x + r * C + b * 128;
            float scale, sinv;
            orc_tensor_scale(orc_amax_bf16(blk, 128), fmt, &scale, &sinv);
            for (int64_t j = 0; j < 128; ++j) q[r * C + b * 128 + j] = quantize_one(blk[j], scale, fmt);
            s_inv[r * nb + b] = sinv;
        }
    }
}

/*
 * 128 x 128 blockwise quantize: one amax and scale per 128x128 tile.
 * s_inv is row-major [R/128, C/128].  R and C must be multiples of 128.
 */
void orc_quantize_128x128(const uint16_t* x, int64_t R, int64_t C, int fmt, uint8_t* q, float* s_inv)
{
    int64_t nbr = R / 128, nbc = C / 128;
    for (int64_t br = 0; br < nbr; ++br) {
        for (int64_t bc = 0; bc < nbc; ++bc) {
            float amax = 0.0f;
            for (int64_t i = 0; i < 128; ++i) {
                float a = orc_amax_bf16(x + (br * 128 + i) * C + bc * 128, 128);
                if (a > amax) amax = a;
            }
            float scale, sinv;
            orc_tensor_scale(amax, fmt, &scale, &sinv);
            for (int64_t i = 0; i < 128; ++i)
                for (int64_t j = 0; j < 128; ++j) {
                    int64_t idx = (br * 128 + i) * C + bc * 128 + j;
                    q[idx] = quantize_one(x[idx], scale, fmt);
                }
            s_inv[br * nbc + bc] = sinv;
        }
    }
}

/*
 * MXFP8 quantize along the contiguous dimension: each run of 32 consecutive
 * elements of a row gets an E8M0 exponent byte.  s_e8m0 is row-major
 * [R, C/32].  C must be a multiple of 32.
 */
void orc_quantize_mx(const uint16_t* x, int64_t R, int64_t C, int fmt, uint8_t* q, uint8_t* s_e8m0)
{
    int64_t nb = C / 32;
    for (int64_t r = 0; r < R; ++r) {
        for (int64_t b = 0; b < nb; ++b) {
            const uint16_t* blk = x + r * C + b * 32;
            int e = orc_mx_exponent(orc_amax_bf16(blk, 32), fmt);
            float scale = pow2_neg(e);
            for (int64_t j = 0; j < 32; ++j) q[r * C + b * 32 + j] = quantize_one(blk[j], scale, fmt);
            s_e8m0[r * nb + b] = (uint8_t)(e + 127);
        }
    }
}

/*
 * The same four quantizers for a binary32 input matrix -- the FP32 master copy of
 * a weight quantized directly (search-result page, mixed-precision dataflow
 * paragraph: weights are held in higher precision and quantized to FP8 from
 * that copy).  Each element is one binary32 product x * scale followed by the
 * saturating cast, exactly as for bf16 inputs, whose values are a subset of the
 * binary32 ones; block amaxes are taken over the binary32 values (NaN ignored).
 */
static uint8_t quantize_one_f32(float x, float scale, int fmt)
{
    return orc_encode(x * scale, fmt, 1);
}

void orc_quantize_tensor_f32(const float* x, int64_t R, int64_t C, int fmt, float scale, uint8_t* q)
{
    for (int64_t i = 0; i < R * C; ++i) q[i] = quantize_one_f32(x[i], scale, fmt);
}

void orc_quantize_1x128_f32(const float* x, int64_t R, int64_t C, int fmt, uint8_t* q, float* s_inv)
{
    int64_t nb = C / 128;
    for (int64_t r = 0; r < R; ++r) {
        for (int64_t b = 0; b < nb; ++b) {
            const float* blk = x + r * C + b * 128;
            float scale, sinv;
            orc_tensor_scale(orc_amax_f32(blk, 128), fmt, &scale, &sinv);
            for (int64_t j = 0; j < 128; ++j) q[r * C + b * 128 + j] = quantize_one_f32(blk[j], scale, fmt);
            s_inv[r * nb + b] = sinv;
        }
    }
}

void orc_quantize_128x128_f32(const float* x, int64_t R, int64_t C, int fmt, uint8_t* q, float* s_inv)
{
    int64_t nbr = R / 128, nbc = C / 128;
    for (int64_t br = 0; br < nbr; ++br) {
        for (int64_t bc = 0; bc < nbc; ++bc) {
            float amax = 0.0f;
            for (int64_t i = 0; i < 128; ++i) {
                float a = orc_amax_f32(x + (br * 128 + i) * C + bc * 128, 128);
                if (a > amax) amax = a;
            }
            float scale, sinv;
            orc_tensor_scale(amax, fmt, &scale, &sinv);
            for (int64_t i = 0; i < 128; ++i)
                for (int64_t j = 0; j < 128; ++j) {
                    int64_t idx = (br * 128 + i) * C + bc * 128 + j;
                    q[idx] = quantize_one_f32(x[idx], scale, fmt);
                }
            s_inv[br * nbc + bc] = sinv;
        }
    }
}

void orc_quantize_mx_f32(const float* x, int64_t R, int64_t C, int fmt, uint8_t* q, uint8_t* s_e8m0)
{
    int64_t nb = C / 32;
    for (int64_t r = 0; r < R; ++r) {
        for (int64_t b = 0; b < nb; ++b) {
            const float* blk = x + r * C + b * 32;
            int e = orc_mx_exponent(orc_amax_f32(blk, 32), fmt);
            float scale = pow2_neg(e);
            for (int64_t j = 0; j < 32; ++j) q[r * C + b * 32 + j] = quantize_one_f32(blk[j], scale, fmt);
            s_e8m0[r * nb + b] = (uint8_t)(e + 127);
        }
    }
}

/* MXFP8 quantize with the floor-rule exponent (bf16 and binary32 inputs). */
void orc_quantize_mx_floor(const uint16_t* x, int64_t R, int64_t C, int fmt, uint8_t* q, uint8_t* s_e8m0)
{
    int64_t nb = C / 32;
    for (int64_t r = 0; r < R; ++r) {
        for (int64_t b = 0; b < nb; ++b) {
            const uint16_t* blk = x + r * C + b * 32;
            int e = orc_mx_exponent_floor(orc_amax_bf16(blk, 32), fmt);
            float scale = pow2_neg(e);
            for (int64_t j = 0; j < 32; ++j) q[r * C + b * 32 + j] = quantize_one(blk[j], scale, fmt);
            s_e8m0[r * nb + b] = (uint8_t)(e + 127);
        }
    }
}

void orc_quantize_mx_floor_f32(const float* x, int64_t R, int64_t C, int fmt, uint8_t* q, uint8_t* s_e8m0)
{
    int64_t nb = C / 32;
    for (int64_t r = 0; r < R; ++r) {
        for (int64_t b = 0; b < nb; ++b) {
            const float* blk = x + r * C + b * 32;
            int e = orc_mx_exponent_floor(orc_amax_f32(blk, 32), fmt);
            float scale = pow2_neg(e);
            for (int64_t j = 0; j < 32; ++j) q[r * C + b * 32 + j] = quantize_one_f32(blk[j], scale, fmt);
            s_e8m0[r * nb + b] = (uint8_t)(e + 127);
        }
    }
}

/* Plain transpose of a row-major [R, C] binary32 matrix into [C, R]. */
void orc_transpose_f32(const float* x, int64_t R, int64_t C, float* xt)
{
    for (int64_t r = 0; r < R; ++r)
        for (int64_t c = 0; c < C; ++c) xt[c * R + r] = x[r * C + c];
}

/* Plain transpose of a row-major [R, C] bf16 matrix into [C, R]. */
void orc_transpose_bf16(const uint16_t* x, int64_t R, int64_t C, uint16_t* xt)
{
    for (int64_t r = 0; r < R; ++r)
        for (int64_t c = 0; c < C; ++c) xt[c * R + r] = x[r * C + c];
}

/*
 * Dequantize to double: value = decode(q) * multiplier, where the multiplier
 * of element (r, c) is
 *   kind 0 (per tensor):  s[0]
 *   kind 1 (1 x 128):     s[r * (C/128) + c/128]
 *   kind 2 (128 x 128):   s[(r/128) * (C/128) + c/128]
 *   kind 3 (MX 1 x 32):   2^(e8m0[r * (C/32) + c/32] - 127); the byte 0xFF is
 *                         the E8M0 NaN (reading: the guide names the E8M0
 *                         format only; its all-ones code is NaN, and the
 *                         quantizer never writes it)
 * All products are exact in double (4-bit by 24-bit significands).
 */
void orc_dequantize(const uint8_t* q, int64_t R, int64_t C, int fmt, int kind,
                    const void* s, double* out)
{
    const float* sf = (const float*)s;
    const uint8_t* se = (const uint8_t*)s;
    for (int64_t r = 0; r < R; ++r) {
        for (int64_t c = 0; c < C; ++c) {
            double v = (double)orc_decode(q[r * C + c], fmt);
            double m;
            switch (kind) {
            case 0: m = (double)sf[0]; break;
            case 1: m = (double)sf[r * (C / 128) + c / 128]; break;
            case 2: m = (double)sf[(r / 128) * (C / 128) + c / 128]; break;
            default: {
                const int e = (int)se[r * (C / 32) + c / 32];
                m = e == 255 ? NAN : ldexp(1.0, e - 127);
                break;
            }
            }
            out[r * C + c] = v * m;
        }
    }
}

/*
 * Round a double to the nearest bfloat16 (8 significant bits, 8 exponent
 * bits, bias 127), ties to even, with gradual underflow (spacing 2^-133 below
 * 2^-126) and overflow to infinity at max + half an ulp; returns the bit
 * pattern.  NaN gives the quiet NaN 0x7FC0 with the input's sign.
 */
uint16_t orc_round_bf16(double v)
{
    const uint16_t sign = signbit(v) ? 0x8000u : 0u;
    if (isnan(v)) return (uint16_t)(sign | 0x7FC0u);
    double a = fabs(v);
    if (isinf(a)) return (uint16_t)(sign | 0x7F80u);
    if (a == 0.0) return sign;
    int e;
    frexp(a, &e);               /* a = f * 2^e, f in [0.5, 1): a in [2^(e-1), 2^e) */
    int ex = e - 1;
    if (ex < -126) ex = -126;   /* subnormal range: fixed spacing */
    const double quantum = ldexp(1.0, ex - 7);
    const double k = a / quantum;                 /* exact: division by a power of two */
    double n = floor(k);
    const double frac = k - n;
    if (frac > 0.5 || (frac == 0.5 && fmod(n, 2.0) != 0.0)) n += 1.0;
    const double res = n * quantum;
    if (res >= ldexp(1.0, 128)) return (uint16_t)(sign | 0x7F80u);
    const float f = (float)res;                   /* exact: every bfloat16 is a binary32 */
    uint32_t bits;
    memcpy(&bits, &f, sizeof bits);
    return (uint16_t)(sign | (bits >> 16));
}

/*
 * Dequantize to bfloat16 (the FP8 -> BF16 conversion, e.g. of weights): the
 * exact product decode(q) * multiplier of orc_dequantize, rounded once to
 * bfloat16 (reading: the pages give no rounding for this step; one rounding
 * of the exact value is the plain definition).
 */
void orc_dequantize_bf16(const uint8_t* q, int64_t R, int64_t C, int fmt, int kind,
                         const void* s, uint16_t* out)
{
    /* 128-row slabs through orc_dequantize (a slab starts on a 128-row block,
       so every kind's multiplier array is offset by whole rows of blocks) */
    double* buf = (double*)malloc((size_t)(C > 0 ? C : 1) * 128 * sizeof(double));
    if (buf == NULL) return;
    const float* sf = (const float*)s;
    const uint8_t* se = (const uint8_t*)s;
    for (int64_t r0 = 0; r0 < R; r0 += 128) {
        const int64_t rows = R - r0 < 128 ? R - r0 : 128;
        const void* sb;
        switch (kind) {
        case 0: sb = sf; break;
        case 1: sb = sf + r0 * (C / 128); break;
        case 2: sb = sf + (r0 / 128) * (C / 128); break;
        default: sb = se + r0 * (C / 32); break;
        }
        orc_dequantize(q + r0 * C, rows, C, fmt, kind, sb, buf);
        for (int64_t i = 0; i < rows * C; ++i) out[r0 * C + i] = orc_round_bf16(buf[i]);
    }
    free(buf);
}

/*
 * FP8 gradient all-reduce with a shared scale, for k data-parallel ranks whose
 * gradients are the k rows of g [k, n] (FP8-LM news article, "automatic
 * scaling": the gradient's scaling factor is adjusted so that its values stay
 * within FP8's range during the all-reduce).  Reading (the pages give no
 * formula): the ranks agree on the global amax A (an all-reduce MAX), all use
 * the per-tensor scale s = FMAX / A (orc_tensor_scale's rule), each sends
 * encode_sat(g_r * s), and the reduction sums the decoded payloads in rank
 * order in binary32, then multiplies once by scale_inv = 1 / s:
 *   out[i] = (((decode(q[0,i]) + decode(q[1,i])) + ...) + decode(q[k-1,i])) * scale_inv
 * q is [k, n]; *amax_out = A; *scale_inv_out = 1 / s.
 */
void orc_allreduce_sum(const uint16_t* g, int32_t k, int64_t n, int fmt, float* amax_out, uint8_t* q,
                       float* scale_inv_out, float* out)
{
    const float a = orc_amax_bf16(g, (int64_t)k * n);
    float s, si;
    orc_tensor_scale(a, fmt, &s, &si);
    orc_quantize_tensor(g, k, n, fmt, s, q);
    for (int64_t i = 0; i < n; ++i) {
        float acc = 0.0f;
        for (int32_t r = 0; r < k; ++r) acc = acc + (float)orc_decode(q[(int64_t)r * n + i], fmt);
        out[i] = acc * si;
    }
    *amax_out = a;
    *scale_inv_out = si;
}
