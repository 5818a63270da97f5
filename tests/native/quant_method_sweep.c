/* Exhaustive check of the dynamic quantiser's division-free code computation over the whole domain
 * the quantiser meets: every positive finite bf16 absmax a whose scale s = RN(a / 127) is at least
 * 2^-120, and every bf16 x with 0 <= x <= a (negative x by symmetry of round-to-nearest).  For each pair
 * it compares rint of the correctly rounded quotient RN(x / s) with
 *   rint(y0),  y0 = RN(x * rs),                         rs = RN(1 / s)
 *   rint(y1),  y1 = RN(y0 + RN(x - y0 * s) * rs) with both steps fused multiply-adds
 * and prints the pair count and the two mismatch counts.  Every operation is an IEEE binary32 operation
 * rounded to nearest, as on the GPU.  Build: cc -O2 -ffp-contract=off -fopenmp ... -lm. */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

static float f_of(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }

int main(void) {
  long long pairs = 0, miss0 = 0, miss1 = 0;
  const float lo = 0x1p-120f;
#pragma omp parallel for schedule(dynamic, 64) reduction(+ : pairs, miss0, miss1)
  for (int a = 1; a <= 0x7F7F; ++a) {
    const float amax = f_of((uint32_t)a << 16);
    volatile float s = amax / 127.0f;
    if (!(s >= lo)) continue;
    volatile float rs = 1.0f / s;
    for (int xb = 0; xb <= a; ++xb) {
      const float x = f_of((uint32_t)xb << 16);
      volatile float q = x / s;
      volatile float y0 = x * rs;
      const float r = fmaf(-y0, s, x);
      const float y1 = fmaf(r, rs, y0);
      const float c = rintf(q);
      ++pairs;
      miss0 += rintf(y0) != c;
      miss1 += rintf(y1) != c;
    }
  }
  printf("%lld %lld %lld\n", pairs, miss0, miss1);
  return 0;
}
