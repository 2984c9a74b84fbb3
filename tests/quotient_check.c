/* Exhaustive check of the quantizers' fast quotient against IEEE division.
 *
 * The quantizers need fl32(x / s) for every element x of a tile whose scale
 * is s = fl32(amax / 448).  Instead of one IEEE division per element they use
 * Markstein's correction step (IBM J. Res. Dev. 34(1), 1990) on negated
 * quantities, with the per-tile reciprocal nr = -fl32(1 / s):
 *     q0 = fl32(x * nr)            (= -fl32(x r), r = fl32(1/s))
 *     e  = fma(q0, s, x)           (= x - fl32(x r) s, exact)
 *     q  = fma(e, nr, q0)          (= -fl32(x / s) when the theorem holds)
 * and flip the sign of the E4M3 code afterwards.  Tiles with amax < 2^-80
 * take IEEE division instead.
 *
 * This program walks every pair of finite BF16 values (x, amax) with
 * |x| <= amax and amax >= 2^-80, both signs of x, and compares q with
 * -(x / s) computed by IEEE division.  A pair passes when the two FP32
 * results are bit-identical, or when both have magnitude <= 2^-10 and the
 * same sign (E4M3's smallest subnormal is 2^-9, so everything up to 2^-10,
 * the tie included, encodes to a signed zero either way).  It prints the
 * number of pairs checked and the number that fail, and exits 1 on any
 * failure.  argv[1] (optional) = stride over amax values, for a sampled run;
 * argv[2] (optional) = the exponent of the amax cutoff (default -80), so a
 * test can show that a lower cutoff lets wrong quotients through.
 *
 * Build without fast-math or FMA contraction: gcc -O2 -ffp-contract=off
 * -fopenmp quotient_check.c -lm.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

static float bf16_to_f32(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

static uint32_t f32_bits(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    return u;
}

int main(int argc, char** argv) {
    const int stride = argc > 1 ? atoi(argv[1]) : 1;
    const float min_amax = ldexpf(1.0f, argc > 2 ? atoi(argv[2]) : -80);
    const float zero_band = ldexpf(1.0f, -10);
    long long checked = 0, failed = 0;
    /* finite non-negative BF16 values: 0x0000 .. 0x7F7F */
#pragma omp parallel for schedule(dynamic, 64) reduction(+ : checked, failed)
    for (int ha = 0; ha <= 0x7F7F; ha += stride) {
        const float amax = bf16_to_f32((uint16_t)ha);
        if (amax < min_amax) continue;
        const float s = amax / 448.0f;
        const float nr = -(1.0f / s);
        for (int hx = 0; hx <= ha; ++hx) {
            for (int sign = 0; sign < 2; ++sign) {
                const float x = bf16_to_f32((uint16_t)(hx | (sign << 15)));
                const float q0 = x * nr;
                const float e = fmaf(q0, s, x);
                const float q = fmaf(e, nr, q0);
                const float want = -(x / s);
                ++checked;
                if (f32_bits(q) == f32_bits(want)) continue;
                if (fabsf(q) <= zero_band && fabsf(want) <= zero_band && signbit(q) == signbit(want)) continue;
                ++failed;
            }
        }
    }
    printf("checked %lld failed %lld\n", checked, failed);
    return failed != 0;
}
