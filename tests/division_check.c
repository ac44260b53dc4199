/* Exhaustive check of the division method the quantiser kernels use (test
 * infrastructure; compiled by tests/test_division_method.py).
 *
 * The kernels form the correctly rounded single-precision quotient t / s from
 * inv = RN(1/s) with one correction step after Markstein (IBM J. Res.
 * Develop. 34(1), 1990): q0 = RN(t*inv), rem = t - q0*s (exact in one fma),
 * y = RN(q0 + rem*inv).  The scale s is always an fp16 value.  This program
 * compares y with IEEE division t / s for every positive finite fp16 s and,
 * for each, every t within `span` floats of the points (k + 1/2) s,
 * k = 0..15 (where a wrong rounding would change a code), plus `nrand` random
 * t in [-s, 16 s].  Prints "checked <n> mismatches <m>". */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

static float f16_value(uint32_t h) {
    int e = (h >> 10) & 31, m = h & 1023;
    return (float)(e ? ldexp(1024.0 + m, e - 25) : ldexp((double)m, -24));
}

static float step(float x, int j) {
    uint32_t u;
    memcpy(&u, &x, 4);
    u = (uint32_t)((int64_t)u + j);
    memcpy(&x, &u, 4);
    return x;
}

static uint64_t rng = 0x9E3779B97F4A7C15ull;
static double uniform(void) {
    rng ^= rng << 13; rng ^= rng >> 7; rng ^= rng << 17;
    return (double)(rng >> 11) / 9007199254740992.0;
}

static int check(float t, float s, float inv) {
    float q0 = t * inv;
    float rem = fmaf(q0, -s, t);
    float y = fmaf(rem, inv, q0);
    float d = t / s;
    return memcmp(&y, &d, 4) != 0;
}

int main(int argc, char** argv) {
    int span = argc > 1 ? atoi(argv[1]) : 200, nrand = argc > 2 ? atoi(argv[2]) : 1000;
    long n = 0, bad = 0;
    for (uint32_t h = 1; h < 0x7C00; ++h) {
        float s = f16_value(h), inv = 1.0f / s;
        for (int k = 0; k < 16; ++k) {
            float mid = (float)((k + 0.5) * (double)s);
            for (int j = -span; j <= span; ++j) {
                bad += check(step(mid, j), s, inv);
                ++n;
            }
        }
        for (int i = 0; i < nrand; ++i) {
            bad += check((float)((uniform() * 17.0 - 1.0) * s), s, inv);
            ++n;
        }
    }
    printf("checked %ld mismatches %ld\n", n, bad);
    return 0;
}
