/* nvfp4_scale_check.c -- exhaustive check of the NVFP4 group scale the write
 * kernels form without an IEEE division.
 *
 * NVFP4 (16-value groups): sf = e4m3_rn(amax / 6).  The kernels compute the
 * quotient as q0 = RN(amax * RN(1/6)), r = amax - q0 * 6 (one fused
 * multiply-add), q = RN(q0 + r * RN(1/6)) (Markstein's correction), and
 * return amax itself for amax = +inf.  This program compares q with the IEEE
 * quotient amax / 6 for every non-negative finite fp32 amax and +inf: the
 * fp32 bits must agree, except where both are below 2^-11 (an e4m3 zero).
 * Exit status 0 when every value passes.  Build: gcc -O2 -std=c11
 * -ffp-contract=off [-fopenmp] ... -lm.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

static float from_bits(uint32_t u) {
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
  const float inv6 = 1.0f / 6.0f;
  long long values = 0, mismatches = 0;
#pragma omp parallel for schedule(static, 1 << 20) reduction(+ : values, mismatches)
  for (long long i = 0; i <= 0x7f800000LL; ++i) {      /* +0 .. +inf */
    const float amax = from_bits((uint32_t)i);
    ++values;
    const float exact = amax / 6.0f;
    const float q0 = amax * inv6;
    const float r = fmaf(-q0, 6.0f, amax);
    const float q = isinf(amax) ? amax : fmaf(r, inv6, q0);
    const int both_tiny = exact < 0x1p-11f && q < 0x1p-11f;
    if (float_bits(q) != float_bits(exact) && !both_tiny) {
      if (mismatches < 10) printf("amax=%a exact=%a q=%a\n", amax, exact, q);
      ++mismatches;
    }
  }
  printf("values %lld mismatches %lld\n", values, mismatches);
  return mismatches != 0;
}
