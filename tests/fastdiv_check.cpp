// Host check of kvq::FastDiv, the multiply-shift division of kvq_params.h that the
// kernels use to split row and task indices, against the hardware division over the
// range the kernels use it for (numerators below 2^31).
//
// Divisors: every d in [1, 2^16] and 200,000 random d below 2^31.  Numerators for
// each: 0, 2^31 - 1 and 2^31 - 2; q*d - 1, q*d and q*d + 1 for the 64 smallest q,
// the 64 largest q that keep n below 2^31 and 64 random q; and 64 random n.  Those
// are where a multiply-shift quotient goes wrong first (at multiples of d and near
// the top of the range).
//
// With the argument "plant" the multiplier is lowered by one (a plausible
// off-by-one in its derivation), which the check must catch.
#include <cstdint>
#include <cstdio>
#include <cstring>

#include "kvq_params.h"

static uint64_t g_rng = 0x9E3779B97F4A7C15ull;
static uint32_t next32() {  // xorshift64
  g_rng ^= g_rng << 13;
  g_rng ^= g_rng >> 7;
  g_rng ^= g_rng << 17;
  return static_cast<uint32_t>(g_rng >> 32);
}

int main(int argc, char** argv) {
  const bool plant = argc > 1 && std::strcmp(argv[1], "plant") == 0;
  const uint32_t kMax = (1u << 31) - 1;
  long long checked = 0, bad = 0;
  auto check = [&](const kvq::FastDiv& f, uint32_t n) {
    uint32_t q = 0, r = 0;
    f.divmod(n, q, r);
    ++checked;
    if (q != n / f.d || r != n % f.d) {
      if (bad < 5) std::printf("d=%u n=%u: got q=%u r=%u\n", f.d, n, q, r);
      ++bad;
    }
  };
  auto run = [&](uint32_t d) {
    kvq::FastDiv f(d);
    if (plant) f.m -= 1;
    check(f, 0);
    check(f, kMax);
    check(f, kMax - 1);
    const uint32_t qmax = kMax / d;
    for (uint32_t k = 0; k < 64; ++k) {
      const uint32_t qs[3] = {k, qmax >= k ? qmax - k : 0u, next32() % (qmax + 1)};
      for (uint32_t q : qs) {
        const int64_t base = static_cast<int64_t>(q) * d;
        for (int dr = -1; dr <= 1; ++dr) {
          const int64_t n = base + dr;
          if (n >= 0 && n <= kMax) check(f, static_cast<uint32_t>(n));
        }
      }
    }
    for (int k = 0; k < 64; ++k) check(f, next32() & kMax);
  };
  for (uint32_t d = 1; d <= (1u << 16); ++d) run(d);
  for (int k = 0; k < 200000; ++k) run(1u + next32() % kMax);
  std::printf("checked %lld quotients, %lld wrong\n", checked, bad);
  return bad == 0 ? 0 : 1;
}
