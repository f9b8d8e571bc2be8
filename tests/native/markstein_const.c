/* Exhaustive check of the constant-divisor quotient used by the kernels'
 * div127 / div255 helpers: q = RN(a y) with y = RN(1/b), r = fma(-b, q, a),
 * q' = fma(r, y, q) must equal the IEEE quotient RN(a / b) for every float a.
 * For a fixed b, scaling a by 2 scales q, r and q' exactly, so the normal
 * binades repeat one pattern; the program checks every float of [1, 2) (both
 * placements of the quotient's binade occur there), the top binade (where
 * overflow could break the pattern) and the binades from 2^-100 (the helpers'
 * lower limit) up.  Prints the number of mismatches per divisor; exit 1 on any.
 * Built without FP contraction; fmaf is the C library's correctly rounded
 * fused multiply-add. */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

static float from_bits(uint32_t u) {
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

static long check_binade(float b, float y, int exp_field) {
  long bad = 0;
  for (uint32_t m = 0; m < (1u << 23); ++m) {
    const float a = from_bits(((uint32_t)exp_field << 23) | m);
    const float q = a * y;
    const float r = fmaf(-b, q, a);
    const float qq = fmaf(r, y, q);
    const float ref = a / b;
    if (memcmp(&qq, &ref, sizeof qq) != 0) ++bad;
  }
  return bad;
}

int main(void) {
  const float divisors[2] = {127.0f, 255.0f};
  int fail = 0;
  for (int i = 0; i < 2; ++i) {
    const float b = divisors[i];
    const float y = 1.0f / b;
    long bad = check_binade(b, y, 127);      /* [1, 2) */
    bad += check_binade(b, y, 254);          /* [2^127, 2^128) */
    bad += check_binade(b, y, 127 - 100);    /* [2^-100, 2^-99) */
    bad += check_binade(b, y, 127 - 99);
    printf("divisor %g: %ld mismatches\n", (double)b, bad);
    if (bad) fail = 1;
  }
  return fail;
}
