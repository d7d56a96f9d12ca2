/* Exhaustive check of the division method used by the CUDA NVFP4 quantizers.
 *
 * The kernels compute the two quotients of the NVFP4 block scale, amax_b / 6
 * and S_enc / sb, as Markstein's FMA-corrected quotients: with y = RN(1/b)
 * and q = RN(a * y), RN(q + (a - b q) * y) equals the IEEE quotient RN(a / b)
 * (P. Markstein, "IA-64 and Elementary Functions", 2000; J.-M. Muller et al.,
 * "Handbook of Floating-Point Arithmetic", the theorem on correcting a
 * quotient with one FMA).  The theorem excludes underflow and overflow, so
 * this program checks every input the kernels can meet instead:
 *   amax_b : every finite non-negative bf16 value (a block maximum of bf16
 *            magnitudes), divisor 6;
 *   S_enc  : min(2688 / A, FLT_MAX) for every finite positive bf16 A (the
 *            token, group or tensor amax), divided by every positive E4M3
 *            value sb, the result clamped with min(., FLT_MAX) as in the
 *            kernels (a NaN from an overflowed product maps to FLT_MAX, as
 *            fminf does on the GPU).
 * Exit status 0 when every result matches IEEE division bit for bit.
 * Build with -ffp-contract=off so that only the explicit fmaf calls fuse. */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

static float from_bits(uint32_t u) { float f; memcpy(&f, &u, sizeof f); return f; }
static uint32_t to_bits(float f) { uint32_t u; memcpy(&u, &f, sizeof u); return u; }

/* Positive E4M3 codes 1..126: S.EEEE.MMM, bias 7, subnormals for E = 0. */
static float e4m3_value(int code) {
    const int e = (code >> 3) & 15, m = code & 7;
    if (e == 0) return ldexpf((float)m, -9);
    return ldexpf(1.0f + (float)m / 8.0f, e - 7);
}

int main(void) {
    const float inv6 = 1.0f / 6.0f;
    long cases6 = 0, bad6 = 0, cases_r = 0, bad_r = 0;
    for (uint32_t h = 0; h < 0x7F80u; ++h) {
        const float x = from_bits(h << 16);
        const float want = x / 6.0f;
        const float q = x * inv6;
        const float got = fmaf(fmaf(-q, 6.0f, x), inv6, q);
        ++cases6;
        if (to_bits(got) != to_bits(want)) {
            if (bad6 < 4) printf("amax_b/6 mismatch: x=%a want=%a got=%a\n", x, want, got);
            ++bad6;
        }
        if (h == 0) continue;
        float senc = 2688.0f / x;
        if (!(senc <= FLT_MAX)) senc = FLT_MAX;
        for (int c = 1; c < 127; ++c) {
            const float b = e4m3_value(c);
            const float y = 1.0f / b;
            const float want_r = fminf(senc / b, FLT_MAX);
            const float q0 = senc * y;
            const float got_r = fminf(fmaf(fmaf(-q0, b, senc), y, q0), FLT_MAX);
            ++cases_r;
            if (to_bits(got_r) != to_bits(want_r)) {
                if (bad_r < 4) printf("S_enc/sb mismatch: senc=%a sb=%a want=%a got=%a\n", senc, b, want_r, got_r);
                ++bad_r;
            }
        }
    }
    printf("amax_b/6: %ld cases, %ld mismatches; S_enc/sb: %ld cases, %ld mismatches\n", cases6, bad6, cases_r, bad_r);
    return (bad6 == 0 && bad_r == 0) ? 0 : 1;
}
