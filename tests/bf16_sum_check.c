/* bf16_sum_check.c -- host check that one bf16 rounding of the exact difference of two
 * finite bf16 values equals the binary32 difference rounded to bf16, for every pair
 * (4.3e9 pairs; addition is covered too, since negation is exact).  The kernels rely
 * on it when they form residuals bf16(cur - prev) and reconstructions bf16(prev + y)
 * with single bf16x2 instructions; the defined arithmetic is the binary32 one.
 *
 * usage: bf16_sum_check [stride]   (every stride-th b for each a; default 1 = all)
 * prints "pairs <n> mismatches <m>" and exits 0 when m == 0.  Compile without fast-math
 * and without FMA contraction. */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

static float f_of(uint32_t u) { float x; memcpy(&x, &u, 4); return x; }
static uint32_t u_of(float x) { uint32_t v; memcpy(&v, &x, 4); return v; }

/* binary32 -> bf16 bits, nearest even (finite inputs; overflow gives infinity) */
static uint16_t bf16_of_f32(float x) {
  const uint32_t u = u_of(x);
  return (uint16_t)((u + 0x7FFFu + ((u >> 16) & 1u)) >> 16);
}

/* binary64 -> bf16 bits, nearest even, by rounding the scaled significand to an
 * integer (bf16 subnormals share exponent -126); a value past the largest finite bf16
 * by half an ulp or more gives infinity */
static uint16_t bf16_of_f64(double x) {
  const uint16_t s = signbit(x) ? 0x8000 : 0;
  const double a = fabs(x);
  if (a == 0.0) return s;
  int e;
  frexp(a, &e);
  int ue = e - 1;
  if (ue < -126) ue = -126;
  const double q = ldexp(a, 7 - ue);
  const double fl = floor(q), r = q - fl;
  double n = fl;
  if (r > 0.5 || (r == 0.5 && fmod(fl, 2.0) == 1.0)) n = fl + 1.0;
  const double v = ldexp(n, ue - 7);
  if (v > 3.3895313892515355e38) return (uint16_t)(s | 0x7F80); /* past the largest finite bf16 */
  return (uint16_t)(s | (u_of((float)v) >> 16));
}

int main(int argc, char** argv) {
  const uint32_t stride = argc > 1 ? (uint32_t)atoi(argv[1]) : 1u;
  uint64_t n = 0, bad = 0;
  for (uint32_t a = 0; a < 65536; ++a) {
    if (((a >> 7) & 0xFF) == 0xFF) continue; /* infinities and NaNs */
    const float fa = f_of(a << 16);
    for (uint32_t b = a % stride; b < 65536; b += stride) {
      if (((b >> 7) & 0xFF) == 0xFF) continue;
      const float fb = f_of(b << 16);
      const uint16_t via_f32 = bf16_of_f32(fa - fb);
      /* the difference of two bf16 values is exact in binary64 unless their exponents
         differ by more than 45; then the smaller is far below half a bf16 ulp of the
         larger, and rounding the binary64 difference gives the same bf16 as rounding
         the exact one */
      const uint16_t once = bf16_of_f64((double)fa - (double)fb);
      ++n;
      if (via_f32 != once) {
        if (bad < 5) printf("a=%04x b=%04x f32-then-bf16=%04x once=%04x\n", a, b, via_f32, once);
        ++bad;
      }
    }
  }
  printf("pairs %llu mismatches %llu\n", (unsigned long long)n, (unsigned long long)bad);
  return bad == 0 ? 0 : 1;
}
