/*
 * Exhaustive host check of the e4m3 row quantiser's fast quotient (the GPU kernel divides
 * each element v of a row by the row scale s = RN(amax / 448) as q0 = RN(v * r),
 * r = RN(1 / s), then q = RN(q0 + RN-exact(v - q0 s) * r) with two FMAs -- Markstein's
 * correction -- for scales in [2^-110, 2^110]).
 *
 * For every positive finite bf16 amax whose scale lies in that range and every bf16 v with
 * 0 <= v <= amax (the formula and e4m3 rounding are odd in v, so negative v follow), the
 * e4m3 value of q (round to nearest even, saturating at 448) must equal the e4m3 value of
 * the correctly rounded quotient RN(v / s), which is the decision the definition takes.
 * Prints the number of pairs, of quotient mismatches and of e4m3 mismatches.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

static float bf16_value(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* the e4m3 value nearest to q (ties to the even code), saturating at +-448 */
static float e4m3_value(float q) {
  const float m = fabsf(q);
  float v;
  if (m < 0x1p-6f) {
    v = rintf(m * 0x1p9f) * 0x1p-9f; /* subnormal step 2^-9 */
  } else {
    int e;
    frexpf(m, &e);                      /* m in [2^(e-1), 2^e) */
    const float step = ldexpf(1.0f, e - 4); /* 3 mantissa bits */
    v = rintf(m / step) * step;
  }
  if (v > 448.0f) v = 448.0f;
  return copysignf(v, q);
}

int main(void) {
  long long pairs = 0, quotient_mismatches = 0, e4m3_mismatches = 0;
  for (uint32_t ha = 1; ha < 0x7F80u; ++ha) {
    const float amax = bf16_value((uint16_t)ha);
    const float s = amax / 448.0f;
    if (!(s >= 0x1p-110f && s <= 0x1p110f)) continue;
    const float r = 1.0f / s;
    for (uint32_t hv = 0; hv <= ha; ++hv) {
      const float v = bf16_value((uint16_t)hv);
      const float q0 = v * r;
      const float rem = fmaf(-q0, s, v);
      const float q = fmaf(rem, r, q0);
      const float exact = v / s;
      ++pairs;
      if (q != exact) ++quotient_mismatches;
      if (e4m3_value(q) != e4m3_value(exact)) {
        if (e4m3_mismatches < 5) printf("mismatch amax=%a v=%a q=%a RN(v/s)=%a\n", amax, v, q, exact);
        ++e4m3_mismatches;
      }
    }
  }
  printf("pairs %lld quotient_mismatches %lld e4m3_mismatches %lld\n", pairs,
         quotient_mismatches, e4m3_mismatches);
  return 0;
}
