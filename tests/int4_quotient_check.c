/* int4_quotient_check.c -- host check of the division-free quotients the INT4 encode
 * kernels use (restated here in plain C with the C library's correctly rounded fmaf and
 * IEEE float division; nothing is shared with the kernels or the oracle).
 *
 *   scale:    sc = RN(D / 15) as q0 = RN(D * RN(1/15)), sc = RN(q0 + RN(D - 15 q0) RN(1/15))
 *   quotient: q  = RN(d / sc) with y = RN(1/sc): q0 = RN(d y), q1 = RN(q0 + RN(d - sc q0) y),
 *             q  = RN(q1 + RN(d - sc q1) y)
 *
 * usage: int4_quotient_check scale-binades LO HI   every binary32 D in [2^LO, 2^HI)
 *        int4_quotient_check scale-range            every D in [2^-64, FLT_MAX]
 *        int4_quotient_check quotient N SEED        N structured random (d, sc) pairs
 * prints one line "checked <n> mismatches <m>" and exits 0 when m == 0. */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

static float f_of(uint32_t u) { float x; memcpy(&x, &u, 4); return x; }
static uint32_t u_of(float x) { uint32_t v; memcpy(&v, &x, 4); return v; }

static float scale15(float D) {
  const float y15 = 0x1.111112p-4f;
  const float q0 = D * y15;
  return fmaf(fmaf(-q0, 15.0f, D), y15, q0);
}

static float quotient(float d, float sc) {
  const float y = 1.0f / sc;
  const float q0 = d * y;
  const float q1 = fmaf(fmaf(-q0, sc, d), y, q0);
  return fmaf(fmaf(-q1, sc, d), y, q1);
}

static uint64_t state;
static uint64_t next(void) { state ^= state << 13; state ^= state >> 7; state ^= state << 17; return state; }
static float bf16(float x) { uint32_t v = u_of(x); v = (v + 0x7FFFu + ((v >> 16) & 1u)) & 0xFFFF0000u; return f_of(v); }
static float unit(void) { return (float)(next() >> 40) / 16777216.0f; }

int main(int argc, char** argv) {
  if (argc < 2) return 2;
  volatile float fifteen = 15.0f; /* keep the reference a run-time IEEE division */
  uint64_t n = 0, bad = 0;
  if (!strcmp(argv[1], "scale-binades") || !strcmp(argv[1], "scale-range")) {
    uint32_t lo, hi;
    if (!strcmp(argv[1], "scale-range")) {
      lo = u_of(0x1p-64f);
      hi = 0x7F800000u;
    } else {
      if (argc < 4) return 2;
      lo = u_of(ldexpf(1.0f, atoi(argv[2])));
      hi = u_of(ldexpf(1.0f, atoi(argv[3])));
    }
    for (uint32_t b = lo; b < hi; ++b) {
      const float D = f_of(b);
      if (u_of(scale15(D)) != u_of(D / fifteen)) {
        if (bad < 3) printf("scale mismatch D=%a\n", D);
        ++bad;
      }
      ++n;
    }
  } else if (!strcmp(argv[1], "quotient")) {
    if (argc < 4) return 2;
    const long N = atol(argv[2]);
    state = 0x9E3779B97F4A7C15ull ^ (uint64_t)atol(argv[3]);
    for (long it = 0; it < N; ++it) {
      float d, sc;
      const int mode = (int)(next() & 3);
      const int e = (int)(next() % 150) - 60;
      if (mode == 0 || mode == 2) { /* a bf16 group: the kernel's d and sc */
        const float mn = bf16(ldexpf(2.0f * unit() - 1.0f, e));
        const float step = bf16(ldexpf(unit() + 1.0f / 64, e));
        const float mx = bf16(mn + (mode == 2 ? 30.0f * step : 4.0f * step));
        const float x = bf16(mode == 2 ? mn + (float)(next() % 31) * step : mn + (mx - mn) * unit());
        if (!(mx > mn) || x < mn || x > mx) continue;
        d = x - mn;
        sc = (mx - mn) / fifteen;
      } else if (mode == 1) { /* within a few ulps of a half-integer */
        sc = ldexpf(1.0f + unit(), e);
        d = f_of(u_of(((float)(next() & 15) + 0.5f) * sc) + (uint32_t)(next() % 257) - 128u);
      } else {
        sc = ldexpf(1.0f + unit(), e);
        d = 15.0f * sc * unit();
      }
      if (!(sc >= 0x1p-64f) || !(d >= 0.0f) || !(d <= 15.5f * sc) || !isfinite(d)) continue;
      const float want = d / sc, got = quotient(d, sc);
      /* codes must agree everywhere; the quotient itself from 2^-39 up */
      const float K = 12582912.0f;
      if ((u_of(want + K) & 15u) != (u_of(got + K) & 15u) || (want >= 0x1p-39f && u_of(got) != u_of(want))) {
        if (bad < 3) printf("quotient mismatch d=%a sc=%a\n", d, sc);
        ++bad;
      }
      ++n;
    }
  } else {
    return 2;
  }
  printf("checked %llu mismatches %llu\n", (unsigned long long)n, (unsigned long long)bad);
  return bad == 0 ? 0 : 1;
}
