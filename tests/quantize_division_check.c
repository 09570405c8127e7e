/* Exhaustive check of the division step the E4M3 row quantiser uses: for a
 * row scale s = RN(amax / 448) in [2^-100, FLT_MAX], y = RN(1/s), and a value
 * v with |v| <= amax, q = RN(v y), r = fma(-s, q, v),
 * q' = copysign(fma(r, y, q), v) must equal RN(v / s) bit for bit whenever
 * either has magnitude >= 2^-12, and have its sign below that (such quotients
 * encode as a zero code of that sign). Every positive bf16 amax and every bf16
 * v of either sign up to it is tried. Prints the counts; exits 1 on a
 * mismatch. */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

static float f_of(uint32_t u) {
  float f;
  memcpy(&f, &u, 4);
  return f;
}
static uint32_t u_of(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  return u;
}

int main(void) {
  const float smin = ldexpf(1.0f, -100), qmin = ldexpf(1.0f, -12);
  long long bad = 0, pairs = 0, rows = 0;
#pragma omp parallel for schedule(dynamic, 64) reduction(+ : bad, pairs, rows)
  for (int ab = 1; ab < 0x7F80; ++ab) {
    const float amax = f_of((uint32_t)ab << 16);
    volatile float s = amax / 448.0f;
    if (!(s >= smin)) continue;
    ++rows;
    volatile float y = 1.0f / s;
    for (int vb = 0; vb <= ab; ++vb) {
      for (int neg = 0; neg < 2; ++neg) {
        const float v = f_of(((uint32_t)vb << 16) | ((uint32_t)neg << 31));
        volatile float q = v * y;
        const float r = fmaf(-s, q, v);
        const float q1 = copysignf(fmaf(r, y, q), v);
        volatile float ref = v / s;
        ++pairs;
        const int big = fabsf(ref) >= qmin || fabsf(q1) >= qmin;
        if (big ? u_of(q1) != u_of(ref) : (u_of(q1) >> 31) != (u_of(ref) >> 31)) ++bad;
      }
    }
  }
  printf("rows %lld pairs %lld mismatches %lld\n", rows, pairs, bad);
  return bad != 0;
}
