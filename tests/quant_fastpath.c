/* Exhaustive check of the GPU kernels' activation-code formula against the
 * reading it must reproduce (plain C, IEEE fp32, no contraction).
 *
 * Reading: q = rne(fl(x / s)) with s = fl(amax / 127) (one IEEE division).
 * Kernels: t = fl(x * fl(127 / amax)); q = rne(t), except when t lies within
 * 2^-14 of a half-integer, where they take the division above.
 *
 * For every pair of positive finite fp16 values 0 < x <= amax the two must
 * give the same code (negative x is the mirror image: both formulas are odd
 * in x).  Prints "pairs mismatches fallbacks" and exits 1 on any mismatch. */
#include <math.h>
#include <stdint.h>
#include <stdio.h>

static float half_to_float(uint16_t h) {
    const uint32_t e = (h >> 10) & 0x1Fu, m = h & 0x3FFu;
    if (e == 0) return ldexpf((float)m, -24);                 /* subnormal: m * 2^-24 */
    return ldexpf((float)(m | 0x400u), (int)e - 25);          /* (1024 + m) * 2^(e - 25) */
}

int main(void) {
    static float v[0x7C00];
    const int n = 0x7C00 - 1;                                  /* 1 .. 0x7BFF: positive finite */
    for (int i = 1; i <= n; ++i) v[i - 1] = half_to_float((uint16_t)i);
    const float thr = 0.5f - ldexpf(1.0f, -14);
    unsigned long long pairs = 0, bad = 0, slow = 0;
    for (int ia = 0; ia < n; ++ia) {
        const float a = v[ia];
        volatile float sv = a / 127.0f, rv = 127.0f / a;
        const float s = sv, r = rv;
        for (int ix = 0; ix <= ia; ++ix) {
            const float x = v[ix];
            volatile float qv = x / s, tv = x * r;
            const float exact = rintf(qv), t = tv, c = rintf(t);
            float fast = c;
            if (fabsf(t - c) > thr) {
                fast = exact;
                ++slow;
            }
            if (fast != exact) ++bad;
            ++pairs;
        }
    }
    printf("%llu %llu %llu\n", pairs, bad, slow);
    return bad != 0;
}
