/* Exhaustive host checks of two arithmetic shortcuts the CUDA quantisers
 * take in place of the plain definitions (test infrastructure; compiled and
 * run by tests/test_kernel_identities.py).  Each shortcut is restated here
 * from the kernel's comments and compared with the definition it replaces:
 *
 * 1. div6: for x >= 2^-125, q0 = RN(x * RN(1/6)); r = fma(-q0, 6, x);
 *    q = fma(r, RN(1/6), q0) equals the IEEE quotient RN(x / 6), for every
 *    finite float in [2^-125, FLT_MAX].
 * 2. E2M1 stochastic rounding: the rounding-up rule "(u >> 8) < p * 2^24"
 *    with p = (|v| - lo) / (hi - lo) over the grid {0, .5, 1, 1.5, 2, 3, 4,
 *    6} (saturating at 6), against the kernel's integer form on the FP32
 *    bits; checked for every finite |v| at the last word that rounds up and
 *    the first that does not (the decision is monotone in u).
 *
 * Prints "div6 <mismatches>" and "sr <mismatches>".  Build with
 * -ffp-contract=off -fopenmp. */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

static float f_of(uint32_t b) { float f; memcpy(&f, &b, 4); return f; }
static uint32_t b_of(float f) { uint32_t b; memcpy(&b, &f, 4); return b; }

static float div6_short(float x) {
    const float c = 1.0f / 6.0f;
    const float q0 = x * c;
    const float r = fmaf(-q0, 6.0f, x);
    return fmaf(r, c, q0);
}

/* the definition: magnitude code of |v| rounded up or down by word u */
static uint32_t sr_def(float v, uint32_t u) {
    static const float grid[8] = {0.0f, 0.5f, 1.0f, 1.5f, 2.0f, 3.0f, 4.0f, 6.0f};
    const float m = fabsf(v);
    if (m >= 6.0f) return 7;
    uint32_t k = 0;
    while (k < 7 && grid[k + 1] <= m) ++k;
    const float p = (m - grid[k]) / (grid[k + 1] - grid[k]);     /* exact */
    return ((float)(u >> 8) < p * 16777216.0f) ? k + 1 : k;
}

/* the kernel's integer form: m = min(|v|, 6) in code steps with 24
 * fraction bits (ceil(m * 2^25) below 1, four times the FP32 bits of m minus
 * those of 0.5 from 1 on), plus 2^24 - 1 - (u >> 8), bits 24 and up */
static uint32_t sr_short(float v, uint32_t u) {
    const float m = fminf(fabsf(v), 6.0f);
    const uint32_t mb = b_of(m);
    const uint32_t x = mb >= 0x3F800000u ? mb * 4u + 0x04000000u
                                         : (uint32_t)ceilf(m * 33554432.0f);   /* exact product, ceil */
    return (x + 0x00FFFFFFu - (u >> 8)) >> 24;
}

/* first word that does not round up: 256 * ceil(p * 2^24) (2^32: none) */
static uint64_t threshold(float v) {
    static const float grid[8] = {0.0f, 0.5f, 1.0f, 1.5f, 2.0f, 3.0f, 4.0f, 6.0f};
    const float m = fabsf(v);
    uint32_t k = 0;
    while (k < 7 && grid[k + 1] <= m) ++k;
    const double p = ((double)m - grid[k]) / (grid[k + 1] - grid[k]);
    return 256ull * (uint64_t)ceil(p * 16777216.0);
}

int main(void) {
    long long bad6 = 0, badsr = 0;
#pragma omp parallel for reduction(+ : bad6) schedule(static, 1 << 16)
    for (int64_t b = 0x01000000; b < 0x7F800000; ++b) {
        const float x = f_of((uint32_t)b);
        if (div6_short(x) != x / 6.0f) ++bad6;
    }
#pragma omp parallel for reduction(+ : badsr) schedule(static, 1 << 16)
    for (int64_t b = 0; b < 0x7F800000; ++b) {
        const float v = f_of((uint32_t)b);
        uint32_t us[4];
        int n = 0;
        if (fabsf(v) >= 6.0f) { us[n++] = 0u; us[n++] = 0xFFFFFFFFu; }
        else {
            const uint64_t t = threshold(v);
            if (t > 0) us[n++] = (uint32_t)(t - 1);
            if (t < 0x100000000ull) us[n++] = (uint32_t)t;
        }
        for (int i = 0; i < n; ++i)
            if (sr_short(v, us[i]) != sr_def(v, us[i])) ++badsr;
    }
    printf("div6 %lld\nsr %lld\n", bad6, badsr);
    return 0;
}
