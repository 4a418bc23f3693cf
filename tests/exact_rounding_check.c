/* Host check of the store kernel's division-free rounding decision (the
 * code_exact step of the dynamic-scale store): for bf16 x and a scale s in
 * [2^-100, 2^120] with r = fl(1/s), the code rne(fl(x/s)) clamped to
 * [-127, 127] follows from n = floor(fl(|x| r)), h = n + 1/2 and the exact
 * remainder d = |x| - h s.  Compared here with one IEEE division per value,
 * over every bf16 x for scales amax/127 from every bf16 amax mantissa, and
 * for random fp32 scales.  Prints the mismatch count; exit status 1 on any. */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

static float f_of(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static uint32_t u_of(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }

static int code_by_division(float x, float s) {
    volatile float t = x / s;
    float q = nearbyintf(t); /* round half to even */
    if (q > 127.0f) q = 127.0f;
    if (q < -127.0f) q = -127.0f;
    return (int)q;
}

static int code_by_remainder(float x, float s, float r) {
    float ax = fabsf(x);
    volatile float y = ax * r;
    int q = 127;
    if (y < 127.0f) {
        float n = floorf(y);
        volatile float h = n + 0.5f;
        float d = fmaf(-h, s, ax);
        float u_hi = f_of((u_of(h) & 0x7F800000u) - (24u << 23));
        volatile float u_lo = h == 0.5f ? u_hi * 0.5f : u_hi;
        volatile float b_hi = s * u_hi, b_lo = s * u_lo;
        int ni = (int)n;
        int on_h = d <= b_hi && d >= -b_lo;
        q = on_h ? ni + (ni & 1) : (d > 0.0f ? ni + 1 : ni);
        if (q > 127) q = 127;
    }
    return x < 0.0f ? -q : q;
}

static uint64_t state = 0x9E3779B97F4A7C15ull;
static uint64_t next(void) {
    state ^= state << 13;
    state ^= state >> 7;
    state ^= state << 17;
    return state;
}

int main(void) {
    long bad = 0, n = 0;
    for (int e = -93; e <= 120; e += 11) { /* amax = (1 + m/128) 2^e */
        for (int m = 0; m < 128; ++m) {
            float amax = f_of(((uint32_t)(e + 127) << 23) | ((uint32_t)m << 16));
            volatile float s = amax / 127.0f;
            if (!(s >= 0x1p-100f && s <= 0x1p+120f)) continue;
            volatile float r = 1.0f / s;
            for (uint32_t xb = 0; xb < 0x7F80; ++xb) {
                float x = f_of(xb << 16);
                if (!(x <= amax)) continue;
                for (int sg = 0; sg < 2; ++sg) {
                    float v = sg ? -x : x;
                    ++n;
                    if (code_by_division(v, s) != code_by_remainder(v, s, r)) {
                        if (bad < 5) printf("mismatch x=%a s=%a\n", v, s);
                        ++bad;
                    }
                }
            }
        }
    }
    for (int it = 0; it < 400; ++it) { /* random scales, |x/s| <= 300 */
        volatile float s = f_of((uint32_t)(next() & 0x7FFFFFu) | ((uint32_t)(27 + next() % 220) << 23));
        if (!(s >= 0x1p-100f && s <= 0x1p+120f)) continue;
        volatile float r = 1.0f / s;
        for (uint32_t xb = 0; xb < 0xFF80; ++xb) {
            if ((xb & 0x7F80u) == 0x7F80u) continue; /* inf / nan */
            float x = f_of(xb << 16);
            if (!(fabsf(x) <= 300.0f * s)) continue;
            ++n;
            if (code_by_division(x, s) != code_by_remainder(x, s, r)) {
                if (bad < 5) printf("mismatch x=%a s=%a\n", x, s);
                ++bad;
            }
        }
    }
    printf("%ld %ld\n", n, bad);
    return bad != 0;
}
