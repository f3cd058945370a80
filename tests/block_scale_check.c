/* Host check of the NVFP4 block-scale shortcut of the encode kernels.
 *
 * The definition ("feat(kvcache): add nvfp4 kv quantization (FreeToken PR #408)",
 * codec-delta port note: the block scale is an E4M3 value, stored rounded):
 *   t = min((vb / 6) / rs, 448),  code = E4M3 nearest-even of t.
 * The kernels, when rs and vb are at least 2^-120, first form
 *   te = (vb * RN(1/6)) * RN(1/rs),
 *   lo = min(te * (1 - 2^-20), 448),  hi = min(te * (1 + 2^-20), 448)
 * (each product one binary32 rounding) and take the code of lo when lo and hi have
 * the same code; otherwise they divide.  This checks the claim the shortcut rests on:
 * whenever code(lo) == code(hi), code(t) is that code too.
 *
 * The E4M3 encoder here is a brute-force nearest search over the format's 127
 * non-negative finite values (ties to the even code), written from the format
 * definition; it shares nothing with the kernels or the oracle.
 *
 * Inputs: rs = RN(amax / 2688) for amax over 2^-100 .. 2^100, and vb = amax * u; u is
 * uniform, or chosen so that vb / 6 / rs lands within a few ulps of every E4M3
 * rounding midpoint.  With the argument "plant" the bracket is collapsed to te
 * alone, which the check must catch. */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

static double g_val[127];

static void build_table(void) {
  for (int c = 0; c < 127; ++c) { /* 0x00..0x7E: 0x7F is NaN */
    const int e = c >> 3, m = c & 7;
    g_val[c] = e == 0 ? ldexp(m / 8.0, -6) : ldexp(1.0 + m / 8.0, e - 7);
  }
}

/* nearest E4M3 code of t >= 0, ties to the even code, saturating at 448 */
static int e4m3_code(float t) {
  const double x = t;
  int lo = 0, hi = 126;
  if (x >= g_val[126]) return 126;
  while (hi - lo > 1) { /* g_val[lo] <= x < g_val[hi] */
    const int mid = (lo + hi) / 2;
    if (g_val[mid] <= x) lo = mid; else hi = mid;
  }
  const double dl = x - g_val[lo], dh = g_val[hi] - x;
  if (dl < dh) return lo;
  if (dh < dl) return hi;
  return (lo & 1) ? hi : lo;
}

static uint64_t g_rng = 0x2545F4914F6CDD1Dull;
static uint32_t next32(void) {
  g_rng ^= g_rng << 13;
  g_rng ^= g_rng >> 7;
  g_rng ^= g_rng << 17;
  return (uint32_t)(g_rng >> 32);
}
static float uniform01(void) { return (float)((next32() >> 8) + 1) * 0x1p-24f; } /* (0, 1] */

static int g_plant = 0;
static long long g_checked = 0, g_shortcut = 0, g_bad = 0;

static void check(float vb, float rs) {
  if (!(rs >= 0x1p-120f && vb >= 0x1p-120f)) return;
  volatile float v_vb = vb, v_rs = rs; /* keep every operation at run time */
  const float rinv = 1.0f / v_rs;
  const float te = (v_vb * 0x1.555556p-3f) * rinv;
  float lo = fminf(te * 0x1.ffffep-1f, 448.0f), hi = fminf(te * 0x1.00001p+0f, 448.0f);
  if (g_plant) lo = hi = fminf(te, 448.0f);
  const float t = fminf((v_vb / 6.0f) / v_rs, 448.0f);
  ++g_checked;
  const int cl = e4m3_code(lo), ch = e4m3_code(hi);
  if (cl != ch) return;
  ++g_shortcut;
  if (e4m3_code(t) != cl) {
    if (g_bad < 5) printf("vb=%a rs=%a t=%a te=%a code(t)=%d shortcut=%d\n", vb, rs, t, te, e4m3_code(t), cl);
    ++g_bad;
  }
}

int main(int argc, char** argv) {
  g_plant = argc > 1 && strcmp(argv[1], "plant") == 0;
  build_table();
  for (int k = 0; k < 10000000; ++k) { /* uniform fractions of the row maximum */
    const float amax = ldexpf(1.0f + uniform01(), (int)(next32() % 201) - 100);
    const float rs = amax / 2688.0f;
    check(amax * uniform01(), rs);
    check(amax, rs);
  }
  for (int c = 0; c < 126; ++c) { /* every rounding midpoint, a few ulps either side */
    const float mid = (float)((g_val[c] + g_val[c + 1]) / 2);
    for (int k = 0; k < 20000; ++k) {
      const float amax = ldexpf(1.0f + uniform01(), (int)(next32() % 201) - 100);
      const float rs = amax / 2688.0f;
      const int ulps = (int)(next32() % 17) - 8;
      float tt = mid;
      for (int i = 0; i < (ulps < 0 ? -ulps : ulps); ++i) tt = nextafterf(tt, ulps < 0 ? 0.0f : 1e30f);
      check(tt * 6.0f * rs, rs); /* vb near 6 * t * rs */
      check(nextafterf(tt * 6.0f * rs, 0.0f), rs);
      check(nextafterf(tt * 6.0f * rs, 1e30f), rs);
    }
  }
  printf("checked %lld pairs, %lld through the shortcut, %lld wrong\n", g_checked, g_shortcut, g_bad);
  return g_bad == 0 ? 0 : 1;
}
