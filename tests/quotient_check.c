/* Exhaustive host check of the fp8 dispatch's FMA-corrected quotient.
 *
 * The dispatch kernels quantise x to e4m3(x / sc), sc = amax / 448 in fp32,
 * with x and amax bf16 values and |x| <= amax. For sc in [2^-100, 2^120] they
 * form x / sc as q = q0 + rem*r with r = RN(1/sc), q0 = RN(x*r) and
 * rem = RN(x - sc*q0) by FMA (a zero remainder keeps q0). This program walks
 * every positive finite bf16 amax whose scale is in that range and every bf16
 * x of either sign with |x| <= amax, and counts the pairs where q and the IEEE
 * quotient RN(x / sc) could give different e4m3 codes: a different sign, or
 * an e4m3 rounding boundary (a midpoint between two neighbouring e4m3
 * magnitudes, 0 .. 448) inside the closed interval between them. Above 448
 * every value saturates to the same code, so no boundary lies there.
 *
 * Build: cc -O2 -ffp-contract=off [-fopenmp] quotient_check.c -lm
 * Prints: "amax <n> pairs <n> differ <n> violations <n>". */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

static float bf16_value(uint32_t bits)
{
    uint32_t u = bits << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

static uint32_t float_bits(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    return u;
}

static double g_mid[126];   /* midpoints between the 127 e4m3 magnitudes */

static void init_midpoints(void)
{
    double mag[127];
    for (int c = 0; c < 127; ++c) {
        int e = c >> 3, m = c & 7;
        mag[c] = e ? ldexp(1.0 + m / 8.0, e - 7) : ldexp(m / 8.0, -6);
    }
    for (int i = 0; i < 126; ++i)
        g_mid[i] = 0.5 * (mag[i] + mag[i + 1]);
}

static int boundary_between(double lo, double hi)
{
    for (int i = 0; i < 126; ++i)
        if (g_mid[i] >= lo && g_mid[i] <= hi)
            return 1;
    return 0;
}

int main(void)
{
    init_midpoints();
    long long n_amax = 0, pairs = 0, differ = 0, violations = 0;
#pragma omp parallel for schedule(dynamic, 32) reduction(+ : n_amax, pairs, differ, violations)
    for (int a = 1; a < 0x7F80; ++a) {
        const float amax = bf16_value((uint32_t)a);
        const float sc = amax / 448.0f;
        if (!(sc >= 0x1p-100f && sc <= 0x1p120f))
            continue;
        ++n_amax;
        const float r = 1.0f / sc;
        for (int sign = 0; sign < 2; ++sign) {
            for (int xb = 0; xb <= a; ++xb) {
                const float x = bf16_value((uint32_t)xb | (sign ? 0x8000u : 0u));
                const float ieee = x / sc;
                const float q0 = x * r;
                const float rem = fmaf(-q0, sc, x);
                const float q = rem == 0.0f ? q0 : fmaf(rem, r, q0);
                ++pairs;
                if (float_bits(q) == float_bits(ieee))
                    continue;
                ++differ;
                if (signbit(q) != signbit(ieee)) {
                    ++violations;
                    continue;
                }
                double u = fabs((double)q), v = fabs((double)ieee);
                if (boundary_between(u < v ? u : v, u < v ? v : u))
                    ++violations;
            }
        }
    }
    printf("amax %lld pairs %lld differ %lld violations %lld\n", n_amax, pairs, differ, violations);
    return violations != 0;
}
