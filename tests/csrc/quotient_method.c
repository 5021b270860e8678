/*
 * Host-side check of the quotient method the vector quantizers use
 * (Markstein's correction: y = RN(1/s), q0 = RN(w y), r = fma(-s, q0, w),
 * q = copysign(RN(q0 + r y), w)), over the whole domain the quantizers feed
 * it: every positive finite bf16 amax with s = RN(amax / 448) >= 2^-92 and
 * every bf16 w with |w| <= amax.  The e4m3 code (nearest-even, saturating,
 * by brute force over the 127 magnitudes) of q must equal the code of the
 * IEEE quotient RN(w / s).  Prints "pairs <n> code_mismatches <m>".
 * Build: -O2 -ffp-contract=off -fopenmp (binary32 IEEE arithmetic).
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

static float bf(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

static double mag[127];

static int enc(float v)
{
    double a = fabs((double)v), bd;
    int neg = signbit(v) ? 1 : 0, best = 0, c;
    if (a >= 448.0)
        return 0x7E | (neg << 7);
    bd = a;
    for (c = 1; c < 127; ++c) {
        double d = fabs(mag[c] - a);
        if (d < bd || (d == bd && !(c & 1))) {
            best = c;
            bd = d;
        }
    }
    return best | (neg << 7);
}

int main(void)
{
    long long total = 0, bad = 0;
    int c;
    for (c = 0; c < 127; ++c) {
        int e = c >> 3, m = c & 7;
        mag[c] = e ? ldexp(8 + m, e - 10) : ldexp(m, -9);
    }
#pragma omp parallel for schedule(dynamic, 64) reduction(+ : total, bad)
    for (int a = 1; a < 0x7F80; ++a) {
        const float amax = bf((uint16_t)a);
        const float s = amax / 448.0f;
        float y;
        if (s < 0x1p-92f)
            continue;
        y = 1.0f / s;
        for (uint32_t wb = 0; wb <= (uint32_t)a; ++wb) {
            int sg;
            for (sg = 0; sg < 2; ++sg) {
                const float w = bf((uint16_t)(wb | ((uint32_t)sg << 15)));
                const float qd = w / s;
                const float q0 = w * y;
                const float r = fmaf(-s, q0, w);
                const float q = copysignf(fmaf(r, y, q0), w);
                total++;
                if ((qd != q || signbit(qd) != signbit(q)) && enc(qd) != enc(q))
                    bad++;
            }
        }
    }
    printf("pairs %lld code_mismatches %lld\n", total, bad);
    return 0;
}
