/* fp8_quotient_check.c -- exhaustive check of the quotient the fp8_ds_mla
 * write kernel forms instead of an IEEE division per value.
 *
 * The fp8_ds_mla write (656-byte entries; per 128-value tile
 * s = amax / 448, code = e4m3_rn(x / s)) needs x / s correctly rounded in
 * fp32.  The kernel computes, with f = 2^96 when s < 2^-64 (else 1),
 * s2 = s * f and inv = RN(1 / s2):
 *   q0 = RN(x * f * inv), r = x * f - q0 * s2 (one fused multiply-add),
 *   q = copysign(RN(q0 + r * inv), x)
 * (Markstein's correction).  This program compares q with the IEEE
 * quotient x / s for every pair of bf16 values x, amax with |x| <= amax
 * (x of the tile whose maximum magnitude is amax): the fp32 bits must agree,
 * except where both magnitudes are below 2^-11 -- those encode to an e4m3
 * zero -- and there the signs must agree.  It also checks the tile scale
 * itself, formed as RN(q0 + (amax - 448 q0) * RN(1/448)) with
 * q0 = RN(amax * RN(1/448)), against amax / 448 for every positive finite
 * bf16 amax: the bits must agree (the scale is stored).  Exit status 0 when
 * every pair and every scale passes.  Build: gcc -O2 -std=c11 -ffp-contract=off [-fopenmp] ... -lm.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

static float bf16_value(uint16_t b) {
  const uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

static uint32_t float_bits(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  return u;
}

int main(void) {
  long long scales = 0, scale_mismatches = 0;
  const float inv448 = 1.0f / 448.0f;
  for (uint32_t ab = 1; ab < 0x7f80u; ++ab) {
    const float amax = bf16_value((uint16_t)ab);
    const float q0 = amax * inv448;
    const float s = fmaf(fmaf(-q0, 448.0f, amax), inv448, q0);
    ++scales;
    if (float_bits(s) != float_bits(amax / 448.0f)) {
      if (scale_mismatches < 10) printf("scale: amax=%a exact=%a s=%a\n", amax, amax / 448.0f, s);
      ++scale_mismatches;
    }
  }
  printf("scales %lld scale mismatches %lld\n", scales, scale_mismatches);
  long long pairs = 0, mismatches = 0;
#pragma omp parallel for schedule(dynamic, 64) reduction(+ : pairs, mismatches)
  for (uint32_t ab = 1; ab < 0x7f80u; ++ab) {          /* every positive finite bf16 amax */
    const float amax = bf16_value((uint16_t)ab);
    const float s = amax / 448.0f;
    const float f = s < 0x1p-64f ? 0x1p96f : 1.0f;
    const float s2 = s * f;
    const float inv = 1.0f / s2;
    for (uint32_t xb = 0; xb < 0x10000u; ++xb) {
      const float x = bf16_value((uint16_t)xb);
      if (!(fabsf(x) <= amax)) continue;                /* also skips NaN */
      ++pairs;
      const float exact = x / s;
      const float x2 = x * f;
      const float q0 = x2 * inv;
      const float r = fmaf(-q0, s2, x2);
      const float q = copysignf(fmaf(r, inv, q0), x);
      const int both_tiny = fabsf(exact) < 0x1p-11f && fabsf(q) < 0x1p-11f;
      if (float_bits(q) != float_bits(exact) && !(both_tiny && signbit(q) == signbit(exact))) {
        if (mismatches < 10) printf("x=%a amax=%a exact=%a q=%a\n", x, amax, exact, q);
        ++mismatches;
      }
    }
  }
  printf("pairs %lld mismatches %lld\n", pairs, mismatches);
  return mismatches != 0 || scale_mismatches != 0;
}
