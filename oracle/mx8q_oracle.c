/*
 * CPU ORACLE for microscaling quantization (MXFP8, per-token NVFP4, MXFP4)
 * and the block-scaled GEMM those encodings feed (plus the plain BF16 GEMM of
 * the dequantized-backward mode).
 *
 * This file is TEST INFRASTRUCTURE.  Only the test suite, the smoke check and
 * the benchmark's CPU-baseline leg may load it.  It shares no code, header,
 * table or constant with the CUDA library: every rule below is restated here
 * from the source pages, in scalar loops that a reader can check by eye.
 *
 * Sources (page title -- section):
 *   [MRL]  "Miles Blackwell RL Cambia la Uniformidad BF16 por MXFP8 y NVFP4
 *          Nativos" -- sections "La Compatibilidad de Miles Blackwell Ahora
 *          Abarca Todo el Ciclo de RL" and "Un Cuantizador Compartido Es el
 *          Mecanismo Real".
 *   [NV4]  "NVIDIA presenta una metodologia de preentrenamiento de 4 bits
 *          utilizando NVFP4" -- sections "Que es realmente NVFP4" and
 *          "La metodologia de formacion de cuatro partes".
 *   [REC]  "Miles Blackwell MXFP8 / NVFP4 RL recipes" (aib.vote) -- the
 *          paragraphs on MXFP8 (row/column copies), on NVFP4 (E4M3 block
 *          scale + FP32 tensor-or-token scale) and on per-token scaling.
 *
 * Conventions that the pages leave open are fixed here and listed in the
 * design notes (scale rounding = ceiling for E8M0, round-to-nearest-even for
 * every cast, saturate-to-finite, signed zero kept, FP32 arithmetic for the
 * NVFP4 scale chain, decode scale stored per token).
 *
 * Build: gcc -O2 -fPIC -shared -ffp-contract=off  (no fast-math: every float
 * operation below must be a single IEEE round-to-nearest operation).
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>
#include <float.h>

typedef int64_t i64;

/* ------------------------------------------------------------------ */
/* bf16 <-> f32                                                        */
/* ------------------------------------------------------------------ */

/* bf16 is the upper half of an IEEE binary32; widening is exact. */
float or_bf16_to_f32(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round-to-nearest-even narrowing of a binary32 to bf16 (NaN kept quiet). */
uint16_t or_f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if (isnan(f)) return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t keep = u >> 16, rest = u & 0xFFFFu;
    if (rest > 0x8000u || (rest == 0x8000u && (keep & 1u))) keep += 1u;
    return (uint16_t)keep;
}

/* ------------------------------------------------------------------ */
/* Element and scale codecs                                            */
/* ------------------------------------------------------------------ */

/* E4M3 ([MRL] "La Compatibilidad...": 32 E4M3 values share one E8M0 scale;
 * [NV4] "Que es realmente NVFP4": the NVFP4 block scale is E4M3).
 * Layout S.EEEE.MMM, bias 7, no infinities, S.1111.111 is NaN.
 * Magnitude of code c (0..126):
 *   exponent field 0  : subnormal  m * 2^-9
 *   exponent field e>0: (8 + m) * 2^(e - 10)  == (1 + m/8) * 2^(e-7)        */
static double e4m3_magnitude(int c)
{
    int e = (c >> 3) & 0xF, m = c & 7;
    if (e == 0) return ldexp((double)m, -9);
    return ldexp((double)(8 + m), e - 10);
}

double or_e4m3_decode(uint8_t code)
{
    int c = code & 0x7F;
    if (c == 0x7F) return NAN;
    double v = e4m3_magnitude(c);
    return (code & 0x80) ? -v : v;
}

/* Round-to-nearest, ties to even, saturating finite values to +-448.
 * Codes 0..126 are in increasing order of magnitude, so "even code" is
 * "even mantissa".  Signed zero is kept (a negative value that rounds to
 * zero gives 0x80). */
uint8_t or_e4m3_encode(float v)
{
    int sign = signbit(v) ? 0x80 : 0;
    if (isnan(v)) return (uint8_t)(sign | 0x7F);
    double a = fabs((double)v);
    if (a >= 448.0) return (uint8_t)(sign | 0x7E);
    int c = 0;
    while (c < 126 && e4m3_magnitude(c + 1) <= a) c++;
    double lo = e4m3_magnitude(c), hi = e4m3_magnitude(c + 1);
    double mid = 0.5 * (lo + hi);          /* exact: few significant bits */
    if (a > mid || (a == mid && (c & 1))) c++;
    return (uint8_t)(sign | c);
}

/* E2M1 ([NV4] "Que es realmente NVFP4": 1 sign, 2 exponent, 1 mantissa bit;
 * the values are +-0, 0.5, 1, 1.5, 2, 3, 4, 6).  Bias 1:
 *   exponent field 0  : m * 0.5
 *   exponent field e>0: (1 + m/2) * 2^(e-1)                                  */
static double e2m1_magnitude(int c)
{
    int e = (c >> 1) & 3, m = c & 1;
    if (e == 0) return 0.5 * m;
    return ldexp(1.0 + 0.5 * m, e - 1);
}

double or_e2m1_decode(uint8_t code)
{
    double v = e2m1_magnitude(code & 7);
    return (code & 8) ? -v : v;
}

/* RNE to E2M1, saturating to +-6 (also for +-inf); signed zero kept.
 * NaN is outside the input contract and maps to +-6. */
uint8_t or_e2m1_encode(float v)
{
    int sign = signbit(v) ? 8 : 0;
    double a = fabs((double)v);
    if (isnan(v) || a >= 6.0) return (uint8_t)(sign | 7);
    int c = 0;
    while (c < 7 && e2m1_magnitude(c + 1) <= a) c++;
    double lo = e2m1_magnitude(c), hi = e2m1_magnitude(c + 1);
    double mid = 0.5 * (lo + hi);
    if (a > mid || (a == mid && (c & 1))) c++;
    return (uint8_t)(sign | c);
}

/* UE8M0: 8 exponent bits, no sign, no mantissa: value 2^(code-127); 255 NaN
 * ([NV4] "Que es realmente NVFP4": UE8M0 scales are powers of two). */
double or_e8m0_decode(uint8_t code)
{
    if (code == 255) return NAN;
    return ldexp(1.0, (int)code - 127);
}

/* ------------------------------------------------------------------ */
/* MXFP8                                                               */
/* ------------------------------------------------------------------ */

/* Shared exponent of one 32-element block: the smallest integer e with
 * amax <= 448 * 2^e, i.e. e = ceil(log2(amax / 448)), so the block amax maps
 * to at most the E4M3 maximum and no element saturates.  The search is
 * clamped to the E8M0 range [-127, 127]; amax == 0 gives -127. */
int or_mxfp8_block_exp(float amax)
{
    double a = (double)amax;
    int e = -127;
    while (e < 127 && a > ldexp(448.0, e)) e++;
    return e;
}

static float absf_of_bf16(uint16_t h) { return fabsf(or_bf16_to_f32(h)); }

/* Rowwise copy: 1x32 blocks along each row ([MRL] "Un Cuantizador
 * Compartido...": blocks must run along the GEMM reduction dimension).
 *   x : bf16 [R, C] with row stride ld (elements)
 *   q : E4M3 [R, C]
 *   s : E8M0 [R, C/32]   (canonical, row-major; not the tensor-core layout) */
void or_mxfp8_quantize_rowwise(const uint16_t *x, i64 R, i64 C, i64 ld,
                               uint8_t *q, uint8_t *s)
{
    i64 nb = C / 32;
    for (i64 r = 0; r < R; r++) {
        for (i64 b = 0; b < nb; b++) {
            const uint16_t *blk = x + r * ld + b * 32;
            float amax = 0.0f;
            for (int i = 0; i < 32; i++) {
                float a = absf_of_bf16(blk[i]);
                if (a > amax) amax = a;
            }
            int e = or_mxfp8_block_exp(amax);
            s[r * nb + b] = (uint8_t)(e + 127);
            for (int i = 0; i < 32; i++) {
                /* x * 2^-e is exact in double; E4M3 rounding happens once. */
                double scaled = ldexp((double)or_bf16_to_f32(blk[i]), -e);
                q[r * C + b * 32 + i] = or_e4m3_encode((float)scaled);
            }
        }
    }
}

/* Columnwise copy: 32x1 blocks down each column of the ORIGINAL bf16 input
 * (not a requantization of the rowwise copy: [MRL] "Un Cuantizador
 * Compartido..."; [REC] MXFP8 paragraph).  Stored transposed so that every
 * GEMM operand has its blocks along its contiguous dimension:
 *   qT : E4M3 [C, R]     qT[c][r] encodes x[r][c]
 *   sT : E8M0 [C, R/32]  canonical.   R must be a multiple of 32. */
void or_mxfp8_quantize_colwise(const uint16_t *x, i64 R, i64 C, i64 ld,
                               uint8_t *qT, uint8_t *sT)
{
    i64 nb = R / 32;
    for (i64 c = 0; c < C; c++) {
        for (i64 b = 0; b < nb; b++) {
            float amax = 0.0f;
            for (int i = 0; i < 32; i++) {
                float a = absf_of_bf16(x[(b * 32 + i) * ld + c]);
                if (a > amax) amax = a;
            }
            int e = or_mxfp8_block_exp(amax);
            sT[c * nb + b] = (uint8_t)(e + 127);
            for (int i = 0; i < 32; i++) {
                double scaled = ldexp((double)or_bf16_to_f32(x[(b * 32 + i) * ld + c]), -e);
                qT[c * R + b * 32 + i] = or_e4m3_encode((float)scaled);
            }
        }
    }
}

/* Dequantize an MXFP8 matrix with 1x32 blocks along its rows:
 * out = decode(q) * 2^(s - 127), computed in double and rounded once to
 * binary32 (exact unless it overflows to inf or underflows). */
void or_dequant_mxfp8(const uint8_t *q, const uint8_t *s, i64 R, i64 C, float *out)
{
    i64 nb = C / 32;
    for (i64 r = 0; r < R; r++)
        for (i64 c = 0; c < C; c++) {
            double v = or_e4m3_decode(q[r * C + c]) * or_e8m0_decode(s[r * nb + c / 32]);
            out[r * C + c] = (float)v;
        }
}

/* ------------------------------------------------------------------ */
/* MXFP4                                                               */
/* ------------------------------------------------------------------ */

/* [NV4] "Que es realmente NVFP4": MXFP4 stores 32-element blocks of E2M1
 * (values +-0, 0.5, 1, 1.5, 2, 3, 4, 6) under one UE8M0 (power-of-two)
 * scale.  The exponent rule is the MXFP8 one with the E2M1 maximum: the
 * smallest integer e with amax <= 6 * 2^e, clamped to [-127, 127]
 * (amax == 0 gives -127), so no element saturates. */
int or_mxfp4_block_exp(float amax)
{
    double a = (double)amax;
    int e = -127;
    while (e < 127 && a > ldexp(6.0, e)) e++;
    return e;
}

/* Packed E2M1 pair: element 2j in the low nibble, 2j+1 in the high one. */
static void put_nibble(uint8_t *row, i64 k, uint8_t code)
{
    if (k & 1) row[k / 2] = (uint8_t)((row[k / 2] & 0x0F) | (code << 4));
    else row[k / 2] = (uint8_t)((row[k / 2] & 0xF0) | (code & 0x0F));
}

/* Rowwise MXFP4: 1x32 blocks along each row.
 *   q : packed E2M1 [R, C/2]
 *   s : E8M0 [R, C/32]   (canonical, row-major) */
void or_mxfp4_quantize_rowwise(const uint16_t *x, i64 R, i64 C, i64 ld,
                               uint8_t *q, uint8_t *s)
{
    i64 nb = C / 32;
    for (i64 r = 0; r < R; r++) {
        for (i64 b = 0; b < nb; b++) {
            const uint16_t *blk = x + r * ld + b * 32;
            float amax = 0.0f;
            for (int i = 0; i < 32; i++) {
                float a = absf_of_bf16(blk[i]);
                if (a > amax) amax = a;
            }
            int e = or_mxfp4_block_exp(amax);
            s[r * nb + b] = (uint8_t)(e + 127);
            for (int i = 0; i < 32; i++) {
                /* x * 2^-e is exact in double; E2M1 rounding happens once. */
                double scaled = ldexp((double)or_bf16_to_f32(blk[i]), -e);
                put_nibble(q + r * (C / 2), b * 32 + i, or_e2m1_encode((float)scaled));
            }
        }
    }
}

/* Columnwise MXFP4: 32x1 blocks down each column of the bf16 input, stored
 * transposed:  qT : packed E2M1 [C, R/2] (qT row c encodes column c of x);
 * sT : E8M0 [C, R/32] canonical.  R must be a multiple of 32. */
void or_mxfp4_quantize_colwise(const uint16_t *x, i64 R, i64 C, i64 ld,
                               uint8_t *qT, uint8_t *sT)
{
    i64 nb = R / 32;
    for (i64 c = 0; c < C; c++) {
        for (i64 b = 0; b < nb; b++) {
            float amax = 0.0f;
            for (int i = 0; i < 32; i++) {
                float a = absf_of_bf16(x[(b * 32 + i) * ld + c]);
                if (a > amax) amax = a;
            }
            int e = or_mxfp4_block_exp(amax);
            sT[c * nb + b] = (uint8_t)(e + 127);
            for (int i = 0; i < 32; i++) {
                double scaled = ldexp((double)or_bf16_to_f32(x[(b * 32 + i) * ld + c]), -e);
                put_nibble(qT + c * (R / 2), b * 32 + i, or_e2m1_encode((float)scaled));
            }
        }
    }
}

/* out = decode(q) * 2^(s - 127) in double, rounded once to binary32. */
void or_dequant_mxfp4(const uint8_t *q, const uint8_t *s, i64 R, i64 C, float *out)
{
    i64 nb = C / 32;
    for (i64 r = 0; r < R; r++)
        for (i64 c = 0; c < C; c++) {
            uint8_t byte = q[r * (C / 2) + c / 2];
            uint8_t nib = (c & 1) ? (byte >> 4) : (byte & 15);
            out[r * C + c] = (float)(or_e2m1_decode(nib) * or_e8m0_decode(s[r * nb + c / 32]));
        }
}

/* ------------------------------------------------------------------ */
/* NVFP4 with an FP32 scale per token / group / tensor                  */
/* ------------------------------------------------------------------ */

/* Two-level NVFP4 ([NV4] "Que es realmente NVFP4"; [REC] NVFP4 paragraph;
 * per-token scope: [MRL] "Un Cuantizador Compartido..." and [REC]):
 *   amax_t          = max |x| over the scope (token row, group of rows, or
 *                     whole tensor)
 *   S_enc           = RN(448*6 / amax_t), clamped to FLT_MAX (amax_t = 0 or
 *                     tiny would give inf)
 *   S_dec           = RN(amax_t / (448*6))         -- the stored FP32 scale
 *   per 1x16 block  : sb = RNE_E4M3_satfinite( RN( RN(amax_b / 6) * S_enc ) )
 *                     r  = (sb == 0) ? 0 : min(RN(S_enc / sb), FLT_MAX)
 *                     code_i = RNE_E2M1_satfinite( RN(x_i * r) )
 * Every step is one binary32 operation, IEEE round-to-nearest (the fast-math
 * path is explicitly disabled for this quantizer in [MRL] "Un Cuantizador
 * Compartido...").  Element 2j goes to the low nibble, 2j+1 to the high one.
 *
 *   scope 0 (token) : s32[R], one per row
 *   scope 1 (group) : s32[G], rows [offs[g], offs[g+1]) share one scale
 *   scope 2 (tensor): s32[1]
 *   q : uint8 [R, C/2]      s : E4M3 [R, C/16] canonical                     */
static void nvfp4_scales_from_amax(float amax, float *senc, float *sdec)
{
    const float two_level_max = 2688.0f;   /* 6 (E2M1 max) * 448 (E4M3 max) */
    float e = two_level_max / amax;
    if (!(e <= FLT_MAX)) e = FLT_MAX;
    *senc = e;
    *sdec = amax / two_level_max;
}

static void nvfp4_encode_row(const uint16_t *xr, i64 C, float senc,
                             uint8_t *qr, uint8_t *sr)
{
    for (i64 b = 0; b < C / 16; b++) {
        float amax_b = 0.0f;
        for (int i = 0; i < 16; i++) {
            float a = absf_of_bf16(xr[b * 16 + i]);
            if (a > amax_b) amax_b = a;
        }
        float t = amax_b / 6.0f;
        t = t * senc;
        uint8_t sb = or_e4m3_encode(t);          /* t >= 0: sign bit clear */
        sr[b] = sb;
        float sbv = (float)or_e4m3_decode(sb);
        float r = 0.0f;
        if (sb != 0) {
            r = senc / sbv;
            if (!(r <= FLT_MAX)) r = FLT_MAX;
        }
        for (int i = 0; i < 16; i += 2) {
            float v0 = or_bf16_to_f32(xr[b * 16 + i]) * r;
            float v1 = or_bf16_to_f32(xr[b * 16 + i + 1]) * r;
            uint8_t lo = or_e2m1_encode(v0), hi = or_e2m1_encode(v1);
            qr[(b * 16 + i) / 2] = (uint8_t)(lo | (hi << 4));
        }
    }
}

static float row_amax(const uint16_t *xr, i64 C)
{
    float m = 0.0f;
    for (i64 c = 0; c < C; c++) {
        float a = absf_of_bf16(xr[c]);
        if (a > m) m = a;
    }
    return m;
}

void or_nvfp4_quantize(const uint16_t *x, i64 R, i64 C, i64 ld, int scope,
                       const i64 *offs, int G, uint8_t *q, uint8_t *s, float *s32)
{
    i64 nb = C / 16;
    if (scope == 0) {
        for (i64 r = 0; r < R; r++) {
            float senc, sdec;
            nvfp4_scales_from_amax(row_amax(x + r * ld, C), &senc, &sdec);
            s32[r] = sdec;
            nvfp4_encode_row(x + r * ld, C, senc, q + r * (C / 2), s + r * nb);
        }
        return;
    }
    i64 single[2] = {0, R};
    if (scope == 2) { offs = single; G = 1; }
    for (int g = 0; g < G; g++) {
        float amax = 0.0f;
        for (i64 r = offs[g]; r < offs[g + 1]; r++) {
            float a = row_amax(x + r * ld, C);
            if (a > amax) amax = a;
        }
        float senc, sdec;
        nvfp4_scales_from_amax(amax, &senc, &sdec);
        s32[g] = sdec;
        for (i64 r = offs[g]; r < offs[g + 1]; r++)
            nvfp4_encode_row(x + r * ld, C, senc, q + r * (C / 2), s + r * nb);
    }
}

/* NVFP4 weights with 2-D 16x16 block scaling ([NV4] "La metodologia de
 * formacion de cuatro partes": the backward pass uses the transposed weight,
 * so 1x16 blocks would quantize forward and backward weights differently;
 * 16x16 blocks give one quantized representation for both passes).  One
 * FP32 scale for the tensor, as for tensor-scope NVFP4; per 16x16 block
 * (rows 16 bi.., columns 16 bj..):
 *   amax_b = max |x| over the 256 elements
 *   sb, r  = as for a 1x16 block (E4M3 scale of RN(amax_b / 6) * S_enc)
 *   code   = RNE_E2M1_satfinite( RN(x * r) )
 * Outputs: the rowwise copy q_row [R, C/2] with s_row [R, C/16] (row n takes
 * its block's sb) and the columnwise copy q_col [C, R/2] with s_col
 * [C, R/16]: exactly the transposes of the rowwise codes and scales.
 * Requires R % 16 == 0 and C % 16 == 0. */
void or_nvfp4_quantize_2d(const uint16_t *x, i64 R, i64 C, i64 ld,
                          uint8_t *q_row, uint8_t *s_row, uint8_t *q_col, uint8_t *s_col,
                          float *s32)
{
    float amax = 0.0f;
    for (i64 r = 0; r < R; r++) {
        float a = row_amax(x + r * ld, C);
        if (a > amax) amax = a;
    }
    float senc, sdec;
    nvfp4_scales_from_amax(amax, &senc, &sdec);
    s32[0] = sdec;
    for (i64 bi = 0; bi < R / 16; bi++)
        for (i64 bj = 0; bj < C / 16; bj++) {
            float amax_b = 0.0f;
            for (int i = 0; i < 16; i++)
                for (int j = 0; j < 16; j++) {
                    float a = absf_of_bf16(x[(bi * 16 + i) * ld + bj * 16 + j]);
                    if (a > amax_b) amax_b = a;
                }
            float t = amax_b / 6.0f;
            t = t * senc;
            uint8_t sb = or_e4m3_encode(t);
            float sbv = (float)or_e4m3_decode(sb);
            float r = 0.0f;
            if (sb != 0) {
                r = senc / sbv;
                if (!(r <= FLT_MAX)) r = FLT_MAX;
            }
            for (int i = 0; i < 16; i++) {
                i64 n = bi * 16 + i;
                s_row[n * (C / 16) + bj] = sb;
                for (int j = 0; j < 16; j++) {
                    i64 k = bj * 16 + j;
                    if (i == 0) s_col[k * (R / 16) + bi] = sb;
                    uint8_t code = or_e2m1_encode(or_bf16_to_f32(x[n * ld + k]) * r);
                    put_nibble(q_row + n * (C / 2), k, code);
                    put_nibble(q_col + k * (R / 2), n, code);
                }
            }
        }
}

/* Stochastic rounding for gradients ([NV4] "La metodologia de formacion de
 * cuatro partes": round-to-nearest-even biases gradient tensors; stochastic
 * rounding picks one of the two nearest representable values with
 * probability given by the distance to each, which removes the bias; it is
 * applied to gradients only).
 *
 * Random bits: the counter-based generator Philox4x32-10 (Salmon, Moraes,
 * Dror, Shaw, "Parallel random numbers: as easy as 1, 2, 3", SC 2011): ten
 * rounds of two 32x32->64-bit multiplications with the round constants
 * M0 = 0xD2511F53, M1 = 0xCD9E8D57 and Weyl key increments
 * W0 = 0x9E3779B9, W1 = 0xBB67AE85:
 *   (hi0, lo0) = M0 * c0, (hi1, lo1) = M1 * c2,
 *   c = (hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0);  k += (W0, W1) between rounds. */
void or_philox4x32_10(const uint32_t *ctr_in, const uint32_t *key_in, uint32_t *out)
{
    const uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
    const uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
    uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
    uint32_t k0 = key_in[0], k1 = key_in[1];
    for (int round = 0; round < 10; round++) {
        if (round > 0) { k0 += W0; k1 += W1; }
        uint64_t p0 = (uint64_t)M0 * c0, p1 = (uint64_t)M1 * c2;
        uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
        uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
        uint32_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
        c0 = n0; c1 = lo1; c2 = n2; c3 = lo0;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* The 32 random bits of element e of a quantized tensor under seed: one
 * Philox block, counter (e / 4 mod 2^32, e / 4 div 2^32, 0, 0) and key
 * (seed mod 2^32, seed div 2^32), gives 4 words of 32 bits; element e takes
 * word e % 4. */
uint32_t or_sr_bits(uint64_t seed, uint64_t e)
{
    uint32_t ctr[4] = {(uint32_t)(e >> 2), (uint32_t)(e >> 34), 0, 0};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)}, out[4];
    or_philox4x32_10(ctr, key, out);
    return out[e & 3];
}

/* E2M1 code of v by stochastic rounding with 32 random bits:
 *   |v| >= 6: 6 (saturate).  Otherwise lo <= |v| < hi are the neighbouring
 *   grid values of {0, .5, 1, 1.5, 2, 3, 4, 6}, p = (|v| - lo) / (hi - lo)
 *   (exact: the spacing is a power of two), and |v| rounds up to hi when
 *   (bits >> 8) < p * 2^24, i.e. with probability p (to 2^-24).
 *   The sign is kept (a negative value rounding to 0 gives code 0x8). */
uint8_t or_e2m1_sr(float v, uint32_t bits)
{
    static const float grid[8] = {0.0f, 0.5f, 1.0f, 1.5f, 2.0f, 3.0f, 4.0f, 6.0f};
    uint8_t sign = signbit(v) ? 8 : 0;
    float a = fabsf(v);
    if (a >= 6.0f) return (uint8_t)(sign | 7);
    int i = 0;
    while (i < 6 && grid[i + 1] <= a) i++;          /* grid[i] <= a < grid[i+1] */
    float p = (a - grid[i]) / (grid[i + 1] - grid[i]);
    int up = (float)(bits >> 8) < p * 16777216.0f;
    return (uint8_t)(sign | (i + up));
}

/* 16x16 random Hadamard transform ([NV4] "La metodologia de formacion de
 * cuatro partes": the Wgrad inputs are multiplied, in 16-element tiles along
 * the reduction dimension, by a 16x16 Hadamard matrix combined with one
 * random +-1 sign vector shared by all linear layers; the transform is
 * orthogonal, so it cancels inside the Wgrad dot products):
 *   y = (1/4) * H16 * diag(s) * x,   H16[i][j] = (-1)^popcount(i & j),
 *   s_i = -1 where bit i of sign_mask is set.
 * Evaluated in binary32 as the natural-order fast Walsh-Hadamard transform:
 * v_i = s_i x_i (exact), then for h = 1, 2, 4, 8 and every pair (i, i + h)
 * with (i & h) == 0: (v_i, v_{i+h}) <- (v_i + v_{i+h}, v_i - v_{i+h}), each
 * one IEEE round-to-nearest operation; finally y_i = v_i * 0.25 (exact). */
void or_rht16(const float *x, unsigned sign_mask, float *y)
{
    float v[16];
    for (int i = 0; i < 16; i++) v[i] = ((sign_mask >> i) & 1u) ? -x[i] : x[i];
    for (int h = 1; h < 16; h <<= 1)
        for (int i = 0; i < 16; i++)
            if ((i & h) == 0) {
                float a = v[i], b = v[i + h];
                v[i] = a + b;
                v[i + h] = a - b;
            }
    for (int i = 0; i < 16; i++) y[i] = v[i] * 0.25f;
}

/* NVFP4 encode of one 16-element block of binary32 values (the steps of
 * nvfp4_encode_row, from f32 instead of bf16 inputs). */
static void nvfp4_encode_block_f32(const float *v, float senc, uint8_t *codes, uint8_t *sb_out)
{
    float amax_b = 0.0f;
    for (int i = 0; i < 16; i++) {
        float a = fabsf(v[i]);
        if (a > amax_b) amax_b = a;
    }
    float t = amax_b / 6.0f;
    t = t * senc;
    uint8_t sb = or_e4m3_encode(t);
    float sbv = (float)or_e4m3_decode(sb);
    float r = 0.0f;
    if (sb != 0) {
        r = senc / sbv;
        if (!(r <= FLT_MAX)) r = FLT_MAX;
    }
    *sb_out = sb;
    for (int i = 0; i < 16; i++) codes[i] = or_e2m1_encode(v[i] * r);
}

/* The columnwise (transposed) NVFP4 copy of a Wgrad input x [R, C] (R the
 * reduction dimension, e.g. tokens) with the 16x16 random Hadamard transform
 * applied to every 16-row chunk of every column before quantization:
 *   y[c][16 k .. 16 k + 15] = or_rht16(x[16 k .. 16 k + 15][c])
 *   one FP32 scale from the amax of y (tensor scope), then per 16-block of y
 *   the NVFP4 block scale and codes (stochastic rounding of the codes when
 *   `stochastic`, for gradient inputs).
 * qT [C, R/2], sT [C, R/16] canonical, s32[1] = S_dec.  R % 16 == 0. */
void or_nvfp4_quantize_rht_colwise(const uint16_t *x, i64 R, i64 C, i64 ld, unsigned sign_mask,
                                   int stochastic, uint64_t seed, uint8_t *qT, uint8_t *sT, float *s32)
{
    float *y = (float *)malloc(sizeof(float) * (size_t)(R * C));
    float amax = 0.0f;
    for (i64 c = 0; c < C; c++)
        for (i64 k = 0; k < R / 16; k++) {
            float in[16];
            for (int i = 0; i < 16; i++) in[i] = or_bf16_to_f32(x[(k * 16 + i) * ld + c]);
            or_rht16(in, sign_mask, y + c * R + k * 16);
            for (int i = 0; i < 16; i++) {
                float a = fabsf(y[c * R + k * 16 + i]);
                if (a > amax) amax = a;
            }
        }
    float senc, sdec;
    nvfp4_scales_from_amax(amax, &senc, &sdec);
    s32[0] = sdec;
    for (i64 c = 0; c < C; c++)
        for (i64 k = 0; k < R / 16; k++) {
            uint8_t codes[16];
            nvfp4_encode_block_f32(y + c * R + k * 16, senc, codes, sT + c * (R / 16) + k);
            if (stochastic) {
                /* same block scale; codes by stochastic rounding, element index
                 * = its position c * R + t in the transposed copy */
                uint8_t sb = sT[c * (R / 16) + k];
                float r = 0.0f;
                if (sb != 0) {
                    r = senc / (float)or_e4m3_decode(sb);
                    if (!(r <= FLT_MAX)) r = FLT_MAX;
                }
                for (int i = 0; i < 16; i++)
                    codes[i] = or_e2m1_sr(y[c * R + k * 16 + i] * r,
                                          or_sr_bits(seed, (uint64_t)(c * R + k * 16 + i)));
            }
            for (int i = 0; i < 16; i++) put_nibble(qT + c * (R / 2), k * 16 + i, codes[i]);
        }
    free(y);
}

/* Per-token NVFP4 with stochastic rounding of the element codes: the FP32
 * scale and the block scales as or_nvfp4_quantize (scope 0, round to
 * nearest even), each code from or_e2m1_sr(RN(x * r), or_sr_bits(seed,
 * r * C + c)). */
void or_nvfp4_quantize_sr(const uint16_t *x, i64 R, i64 C, i64 ld, uint64_t seed,
                          uint8_t *q, uint8_t *s, float *s32)
{
    for (i64 row = 0; row < R; row++) {
        const uint16_t *xr = x + row * ld;
        float senc, sdec;
        nvfp4_scales_from_amax(row_amax(xr, C), &senc, &sdec);
        s32[row] = sdec;
        for (i64 b = 0; b < C / 16; b++) {
            float amax_b = 0.0f;
            for (int i = 0; i < 16; i++) {
                float a = absf_of_bf16(xr[b * 16 + i]);
                if (a > amax_b) amax_b = a;
            }
            float t = amax_b / 6.0f;
            t = t * senc;
            uint8_t sb = or_e4m3_encode(t);
            s[row * (C / 16) + b] = sb;
            float r = 0.0f;
            if (sb != 0) {
                r = senc / (float)or_e4m3_decode(sb);
                if (!(r <= FLT_MAX)) r = FLT_MAX;
            }
            for (int i = 0; i < 16; i++) {
                i64 c = b * 16 + i;
                float v = or_bf16_to_f32(xr[c]) * r;
                put_nibble(q + row * (C / 2), c, or_e2m1_sr(v, or_sr_bits(seed, (uint64_t)(row * C + c))));
            }
        }
    }
}

/* FP32 decode scale of row r under s32_mode: 0 none (1), 1 per row,
 * 2 per tensor, 3 per group (offs, G). */
static double s32_of_row(const float *s32, int mode, const i64 *offs, int G, i64 r)
{
    if (mode == 0 || s32 == NULL) return 1.0;
    if (mode == 1) return (double)s32[r];
    if (mode == 2) return (double)s32[0];
    int g = 0;                           /* the group with offs[g] <= r < offs[g+1] */
    while (g < G && !(r >= offs[g] && r < offs[g + 1])) g++;
    return g < G ? (double)s32[g] : NAN;
}

/* out = RN_f32( (e2m1 * sb) * S_dec ); the inner product is exact. */
void or_dequant_nvfp4(const uint8_t *q, const uint8_t *s, const float *s32,
                      int s32_mode, const i64 *offs, int G, i64 R, i64 C, float *out)
{
    i64 nb = C / 16;
    for (i64 r = 0; r < R; r++) {
        float sd = (float)s32_of_row(s32, s32_mode, offs, G, r);
        for (i64 c = 0; c < C; c++) {
            uint8_t byte = q[r * (C / 2) + c / 2];
            uint8_t nib = (c & 1) ? (byte >> 4) : (byte & 15);
            float blockval = (float)(or_e2m1_decode(nib) * or_e4m3_decode(s[r * nb + c / 16]));
            out[r * C + c] = blockval * sd;
        }
    }
}

/* ------------------------------------------------------------------ */
/* Tensor-core scale-factor layout                                      */
/* ------------------------------------------------------------------ */

/* The block-scaled tensor-core MMA reads scale factors in 128-row x 4-column
 * tiles of 512 bytes (the pages are silent; this is the layout NVIDIA
 * documents for its block-scaled GEMMs).  Scale (r, k) of a [rows, scols]
 * canonical matrix goes to
 *     tile   = (r / 128) * ceil(scols / 4) + k / 4
 *     offset = tile*512 + (r % 32)*16 + ((r % 128) / 32)*4 + k % 4
 * in a buffer of ceil(rows/128)*128 x ceil(scols/4)*4 bytes whose padding is
 * zero.  With groups (offs != NULL), group g's rows start at the padded row
 * P_g = sum_{h<g} ceil(n_h/128)*128, so every group owns whole tiles. */
static i64 ceil_div(i64 a, i64 b) { return (a + b - 1) / b; }

i64 or_swizzled_bytes(i64 rows, i64 scols, const i64 *offs, int G)
{
    i64 ptiles = 0;
    if (offs == NULL) ptiles = ceil_div(rows, 128);
    else for (int g = 0; g < G; g++) ptiles += ceil_div(offs[g + 1] - offs[g], 128);
    return ptiles * 128 * ceil_div(scols, 4) * 4;
}

void or_swizzle_scales(const uint8_t *canon, i64 rows, i64 scols,
                       const i64 *offs, int G, uint8_t *out)
{
    i64 kt = ceil_div(scols, 4);
    memset(out, 0, (size_t)or_swizzled_bytes(rows, scols, offs, G));
    i64 single[2] = {0, rows};
    if (offs == NULL) { offs = single; G = 1; }
    i64 prow = 0;
    for (int g = 0; g < G; g++) {
        i64 n = offs[g + 1] - offs[g];
        for (i64 lr = 0; lr < n; lr++) {
            i64 r = prow + lr;
            for (i64 k = 0; k < scols; k++) {
                i64 tile = (r / 128) * kt + k / 4;
                i64 off = tile * 512 + (r % 32) * 16 + ((r % 128) / 32) * 4 + k % 4;
                out[off] = canon[(offs[g] + lr) * scols + k];
            }
        }
        prow += ceil_div(n, 128) * 128;
    }
}

/* ------------------------------------------------------------------ */
/* Block-scaled GEMM reference (FP64)                                   */
/* ------------------------------------------------------------------ */

/* Exact FP64 decode of one operand row: element * block scale * FP32 scale.
 * fmt 0 = MXFP8 (E4M3 bytes, E8M0 per 32), fmt 1 = NVFP4 (packed E2M1,
 * E4M3 per 16), fmt 2 = MXFP4 (packed E2M1, E8M0 per 32).  All products
 * have <= 30 significant bits: exact. */
static void decode_row(int fmt, const uint8_t *qrow, const uint8_t *srow, double s32,
                       i64 K, double *dst)
{
    for (i64 k = 0; k < K; k++) {
        double v;
        if (fmt == 0) {
            v = or_e4m3_decode(qrow[k]) * or_e8m0_decode(srow[k / 32]);
        } else {
            uint8_t byte = qrow[k / 2];
            uint8_t nib = (k & 1) ? (byte >> 4) : (byte & 15);
            v = or_e2m1_decode(nib) * (fmt == 1 ? or_e4m3_decode(srow[k / 16]) : or_e8m0_decode(srow[k / 32]));
        }
        dst[k] = v * s32;
    }
}

/* ref[m,n] = sum_k A^[m,k] * B^[n,k]   (Y = A * B^T, both operands stored
 * with K contiguous), accumulated in double; absref = sum_k |A^||B^| gives
 * the tolerance scale.  With pairs != NULL only the listed (m, n) outputs
 * are produced (pairs holds 2*npairs indices); otherwise all M*N, row-major.
 * a32_mode / b32_mode: 0 none, 1 per row, 2 per tensor.  The caller passes
 * a scratch buffer of 2*K doubles. */
void or_gemm_ref(int fmt, i64 M, i64 N, i64 K,
                 const uint8_t *A, const uint8_t *SA, const float *a32, int a32_mode,
                 const uint8_t *B, const uint8_t *SB, const float *b32, int b32_mode,
                 const i64 *pairs, i64 npairs, double *ref, double *absref, double *scratch)
{
    i64 bs = (fmt == 1) ? 16 : 32;
    i64 rowbytes = (fmt == 0) ? K : K / 2;
    double *ar = scratch, *br = scratch + K;
    i64 count = pairs ? npairs : M * N;
    i64 last_m = -1;
    for (i64 p = 0; p < count; p++) {
        i64 m = pairs ? pairs[2 * p] : p / N;
        i64 n = pairs ? pairs[2 * p + 1] : p % N;
        if (m != last_m) {
            decode_row(fmt, A + m * rowbytes, SA + m * (K / bs),
                       s32_of_row(a32, a32_mode, NULL, 0, m), K, ar);
            last_m = m;
        }
        decode_row(fmt, B + n * rowbytes, SB + n * (K / bs),
                   s32_of_row(b32, b32_mode, NULL, 0, n), K, br);
        double acc = 0.0, aacc = 0.0;
        for (i64 k = 0; k < K; k++) {
            acc += ar[k] * br[k];
            aacc += fabs(ar[k]) * fabs(br[k]);
        }
        ref[p] = acc;
        absref[p] = aacc;
    }
}

/* Grouped (MoE routed experts): rows [offs[g], offs[g+1]) of A belong to
 * expert g and multiply that expert's weight B[g] ([N, K]):
 *   ref[m, n] = sum_k A^[m,k] * B^_g[n,k],  g = group of row m
 * a32: per-row FP32 decode scale (per-token activations) or NULL;
 * b32: per-group FP32 decode scale [G] or NULL.
 * SA is canonical [rows, K/bs]; SB canonical [G*N, K/bs]. */
void or_grouped_gemm_ref(int fmt, int G, const i64 *offs, i64 N, i64 K,
                         const uint8_t *A, const uint8_t *SA, const float *a32,
                         const uint8_t *B, const uint8_t *SB, const float *b32,
                         const i64 *pairs, i64 npairs, double *ref, double *absref,
                         double *scratch)
{
    i64 bs = (fmt == 1) ? 16 : 32;
    i64 rowbytes = (fmt == 0) ? K : K / 2;
    double *ar = scratch, *br = scratch + K;
    i64 last_m = -1;
    for (i64 p = 0; p < npairs; p++) {
        i64 m = pairs[2 * p], n = pairs[2 * p + 1];
        int g = 0;                       /* the group with offs[g] <= m < offs[g+1] */
        while (g < G && !(m >= offs[g] && m < offs[g + 1])) g++;
        if (g == G) { ref[p] = NAN; absref[p] = NAN; continue; }
        if (m != last_m) {
            decode_row(fmt, A + m * rowbytes, SA + m * (K / bs),
                       a32 ? (double)a32[m] : 1.0, K, ar);
            last_m = m;
        }
        i64 brow = (i64)g * N + n;
        decode_row(fmt, B + brow * rowbytes, SB + brow * (K / bs),
                   b32 ? (double)b32[g] : 1.0, K, br);
        double acc = 0.0, aacc = 0.0;
        for (i64 k = 0; k < K; k++) {
            acc += ar[k] * br[k];
            aacc += fabs(ar[k]) * fabs(br[k]);
        }
        ref[p] = acc;
        absref[p] = aacc;
    }
}

/* Plain GEMM over bf16 operands, for the dequantized-backward mode ([MRL]
 * "La Compatibilidad...": Dgrad and Wgrad run in BF16 on operands rebuilt
 * from the low-precision forward copies):
 *   ref[m,n] = sum_k a[m,k] * b[n,k]   (Y = A * B^T, K contiguous in both)
 * in double; every product of two bf16 values is exact in double.  Rows of
 * A and B are lda / ldb elements apart.  pairs / npairs as in or_gemm_ref. */
void or_bf16_gemm_ref(i64 M, i64 N, i64 K, const uint16_t *A, i64 lda,
                      const uint16_t *B, i64 ldb, const i64 *pairs, i64 npairs,
                      double *ref, double *absref)
{
    i64 count = pairs ? npairs : M * N;
    for (i64 p = 0; p < count; p++) {
        i64 m = pairs ? pairs[2 * p] : p / N;
        i64 n = pairs ? pairs[2 * p + 1] : p % N;
        const uint16_t *ar = A + m * lda, *br = B + n * ldb;
        double acc = 0.0, aacc = 0.0;
        for (i64 k = 0; k < K; k++) {
            double x = (double)or_bf16_to_f32(ar[k]), y = (double)or_bf16_to_f32(br[k]);
            acc += x * y;
            aacc += fabs(x) * fabs(y);
        }
        ref[p] = acc;
        absref[p] = aacc;
    }
}

/* MoE combine: each token's expert outputs, weighted by its router weights,
 * summed back in token order (the step that closes the routed-expert layer
 * around the grouped GEMMs of [MRL] "Un Cuantizador Compartido..." and
 * [REC]'s NVFP4 MoE experts):
 *   out[t][h] = sum_{j<k} w[t][j] * y[rows[t][j]][h]
 * accumulated in binary32 in the order j = 0, 1, ..., each product and each
 * sum one round-to-nearest operation (acc = RN(acc + RN(w * y))).  y is bf16
 * [R, H]; out is f32 [T, H] (a bf16 output is RNE of it).  Rows outside
 * [0, R) contribute nothing. */
void or_moe_combine(const uint16_t *y, i64 R, i64 H, const i64 *rows, const float *w, i64 T, int k, float *out)
{
    for (i64 t = 0; t < T; t++)
        for (i64 h = 0; h < H; h++) {
            float acc = 0.0f;
            for (int j = 0; j < k; j++) {
                i64 r = rows[t * k + j];
                if (r < 0 || r >= R) continue;
                float prod = w[t * k + j] * or_bf16_to_f32(y[r * H + h]);
                acc = acc + prod;
            }
            out[t * H + h] = acc;
        }
}

/* ------------------------------------------------------------------ */
/* SwiGLU between the MoE gate|up and down GEMMs                        */
/* ------------------------------------------------------------------ */

/* Correctly rounded bf16 of a binary64 value, in one rounding step (no
 * intermediate binary32): round to nearest, ties to even, or, with
 * ties_toward_zero, a tie goes to the neighbour of smaller magnitude.
 * Overflow gives infinity; bf16 subnormals are kept (spacing 2^-133). */
static uint16_t f64_to_bf16(double v, int ties_toward_zero)
{
    if (isnan(v)) return 0x7FC0u;
    uint16_t sign = signbit(v) ? 0x8000u : 0u;
    double a = fabs(v);
    if (a == 0.0) return sign;
    if (isinf(a)) return (uint16_t)(sign | 0x7F80u);
    int e;
    frexp(a, &e);                    /* a in [2^(e-1), 2^e) */
    int k = e - 1;
    if (k < -126) k = -126;          /* below the normal range the spacing stays 2^-133 */
    double q = ldexp(a, 7 - k);      /* a in units of the bf16 spacing 2^(k-7): exact */
    double n = floor(q);
    double rest = q - n;             /* exact */
    if (rest > 0.5 || (rest == 0.5 && !ties_toward_zero && fmod(n, 2.0) != 0.0)) n += 1.0;
    double r = ldexp(n, k - 7);
    if (r >= 0x1p128) return (uint16_t)(sign | 0x7F80u);
    float f = (float)r;              /* exact: at most 9 significant bits, in binary32 range */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(sign | (u >> 16));
}

/* h[r, j] = RN_bf16( silu(g) * u ), silu(g) = g / (1 + e^-g): the exact real
 * value rounded once to bf16 ("Un Cuantizador Compartido Es el Mecanismo
 * Real": gate and up of a SwiGLU expert are one fused GEMM output).
 * Evaluated in binary64 and rounded directly to bf16.  Where 1 + e^-g == 1
 * in binary64 (g > 36.7) the quotient would return g*u itself, which can be
 * a bf16 tie; the exact value g*u*(1 - e^-g/(1 + e^-g)) lies just inside
 * g*u (less than one binary64 unit), so it rounds like g*u except that a tie
 * goes toward zero.  g*u is exact in binary64 (two 8-bit significands).
 * Elsewhere the value is never a tie (silu(g) is transcendental for g != 0)
 * and the binary64 evaluation is a few units of 2^-53 from it.
 * gu: bf16 [R, 2F] (gate columns, then up columns); h: bf16 [R, F]. */
void or_swiglu(const uint16_t *gu, i64 R, i64 F, uint16_t *h)
{
    for (i64 r = 0; r < R; r++)
        for (i64 j = 0; j < F; j++) {
            double g = (double)or_bf16_to_f32(gu[r * 2 * F + j]);
            double u = (double)or_bf16_to_f32(gu[r * 2 * F + F + j]);
            double t = exp(-g);
            if (1.0 + t == 1.0)
                h[r * F + j] = f64_to_bf16(g * u, 1);
            else
                h[r * F + j] = f64_to_bf16(g / (1.0 + t) * u, 0);
        }
}
