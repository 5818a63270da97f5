/* The SwiGLU exp (Cody-Waite reduction, degree-7 Taylor polynomial, scaling by two powers of two) in two
 * forms: with the specified range selects (x > 89 -> +inf, x < -104 -> +0, NaN -> NaN) after steps run on
 * x clamped to [-104, 89], and with the clamp alone (NaN propagated).  Prints how many of the swept inputs
 * -- every binary32 value in [-112, -100] and [84, 96], and the infinities -- give different bits, and the
 * two boundary results.  Build: cc -O2 -ffp-contract=off ... -lm. */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

static float f_of(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static uint32_t u_of(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
static float pow2i(int k) { return f_of((uint32_t)(k + 127) << 23); }

static float steps(float x) {
  const float log2e = f_of(0x3fb8aa3b), ln2_hi = f_of(0x3f317200), ln2_lo = f_of(0x35bfbe8e);
  const float c7 = f_of(0x39500d01), c6 = f_of(0x3ab60b61), c5 = f_of(0x3c088889), c4 = f_of(0x3d2aaaab),
              c3 = f_of(0x3e2aaaab);
  volatile float t = x * log2e;
  const float n = rintf(t);
  float r = fmaf(-n, ln2_hi, x);
  r = fmaf(-n, ln2_lo, r);
  float p = c7;
  p = fmaf(p, r, c6);
  p = fmaf(p, r, c5);
  p = fmaf(p, r, c4);
  p = fmaf(p, r, c3);
  p = fmaf(p, r, 0.5f);
  p = fmaf(p, r, 1.0f);
  p = fmaf(p, r, 1.0f);
  const int ni = (int)n, n1 = ni / 2, n2 = ni - n1;
  volatile float y1 = p * pow2i(n1);
  volatile float y = y1 * pow2i(n2);
  return y;
}
static float with_selects(float x_in) {
  const float y = steps(fminf(fmaxf(x_in, -104.0f), 89.0f));
  const float hi = x_in > 89.0f ? f_of(0x7f800000) : y;
  const float lo = x_in < -104.0f ? 0.0f : hi;
  return x_in != x_in ? x_in : lo;
}
static float clamp_only(float x_in) { return steps(fminf(fmaxf(x_in, -104.0f), 89.0f)); }

int main(void) {
  long long n = 0, differ = 0;
  const float a[2] = {-112.0f, 84.0f}, b[2] = {-100.0f, 96.0f};
  for (int k = 0; k < 2; ++k)
    for (float x = a[k]; x <= b[k]; x = nextafterf(x, INFINITY), ++n)
      differ += u_of(with_selects(x)) != u_of(clamp_only(x));
  const float inf[2] = {INFINITY, -INFINITY};
  for (int k = 0; k < 2; ++k, ++n) differ += u_of(with_selects(inf[k])) != u_of(clamp_only(inf[k]));
  printf("%lld %lld %08x %08x\n", n, differ, u_of(steps(89.0f)), u_of(steps(-104.0f)));
  return 0;
}
