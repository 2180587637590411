/* Exhaustive check of the division method of the 8-bit cache write.
 *
 * The kernel rounds each quotient x / d (x a bf16 or fp16 value, d the
 * group's fp16 scale) as IEEE fp32 division does, but computes it from one
 * correctly rounded reciprocal y = rn(1 / d) per group: q0 = rn(x y), then
 * q = rn(q0 + rn-exact(x - q0 d) y) with fused multiply-adds (Markstein's
 * theorem, "IA-64 and Elementary Functions", ch. 8).  The code stored is
 * clamp(rint(q), -127, 127).  This program runs that method against IEEE
 * division for every finite bf16 and fp16 x and every positive finite fp16 d
 * a group can produce with it (|x / d| < 256, or d = 65504, the saturated
 * scale), and the scale's own division amax / 127 for every finite bf16 and
 * fp16 amax.  It prints the counts and exits 1 on any code that differs.
 * Compile with -ffp-contract=off so that only the fmaf calls fuse (and
 * -fopenmp to spread the scales over the host cores). */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

static float bits_to_f32(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static uint32_t f32_to_bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }

static float f16_to_f32(uint16_t h)
{
    const uint32_t s = (h >> 15) & 1u, e = (h >> 10) & 31u, m = h & 1023u;
    const float v = e == 0 ? ldexpf((float)m, -24) : ldexpf((float)(m | 1024u), (int)e - 25);
    return s ? -v : v;
}

static int code_of(float q)
{
    float r = rintf(q);
    if (r > 127.f) r = 127.f;
    if (r < -127.f) r = -127.f;
    return (int)r;
}

static float quotient(float x, float d, float y)
{
    const float q0 = x * y;
    return fmaf(fmaf(-q0, d, x), y, q0);
}

int main(void)
{
    long pairs = 0, code_diff = 0, quot_diff = 0, scale_diff = 0;
    static float xs[65536];
    for (int dt = 0; dt < 2; ++dt) {          /* 0: bf16 x, 1: fp16 x */
        int nx = 0;
        for (uint32_t p = 0; p < 65536; ++p) {
            const float x = dt == 0 ? bits_to_f32(p << 16) : f16_to_f32((uint16_t)p);
            if (isfinite(x)) xs[nx++] = x;
        }
#pragma omp parallel for schedule(dynamic, 64) reduction(+ : pairs, code_diff, quot_diff)
        for (int hd = 1; hd < 0x7C00; ++hd) {
            const float d = f16_to_f32((uint16_t)hd), y = 1.0f / d;
            /* |x| < 256 d is exactly |x / d| < 256 (256 d is exact) */
            const float lim = hd == 0x7BFF ? INFINITY : 256.0f * d;
            for (int i = 0; i < nx; ++i) {
                const float x = xs[i];
                if (!(fabsf(x) < lim)) continue;
                const float ref = x / d, q = quotient(x, d, y);
                ++pairs;
                if (code_of(q) != code_of(ref)) ++code_diff;
                /* the residual is exact only while it is a normal number: the
                 * quotient may then differ, below 2^-100, where the code is 0 */
                if (f32_to_bits(q) != f32_to_bits(ref) && fabsf(ref) >= 0x1p-100f) ++quot_diff;
            }
        }
    }
    const float y127 = 1.0f / 127.0f;
    for (int dt = 0; dt < 2; ++dt)
        for (uint32_t p = 0; p < 32768; ++p) {           /* non-negative patterns */
            const float a = dt == 0 ? bits_to_f32(p << 16) : f16_to_f32((uint16_t)p);
            if (!isfinite(a)) continue;
            const float ref = a / 127.0f, q = quotient(a, 127.0f, y127);
            /* below 2^-25 the fp16 scale is 0 either way */
            if (ref >= 0x1p-126f ? f32_to_bits(q) != f32_to_bits(ref)
                                 : !(q <= 0x1p-25f && ref <= 0x1p-25f))
                ++scale_diff;
        }
    printf("pairs %ld code_differences %ld quotient_differences %ld scale_differences %ld\n", pairs,
           code_diff, quot_diff, scale_diff);
    return (code_diff || quot_diff || scale_diff) ? 1 : 0;
}
