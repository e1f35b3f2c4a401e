// Host check of the stream-K split (SplitK in bws_internal.h): for a range of
// unit counts, CTA counts and lighter tails, every CTA's range is non-empty
// and contiguous, the ranges cover all units in order, and splitk_owner(u)
// names the CTA whose range holds u. Prints the cases checked; exit code 1 on
// the first failure.
#include <cstdio>

#include "bws_internal.h"

using bws::SplitK;

static bool check(const SplitK& s) {
  if (bws::splitk_begin(s, 0) != 0 || bws::splitk_begin(s, s.n_ctas) != s.n_units) return false;
  for (int c = 0; c < s.n_ctas; ++c) {
    const long long b0 = bws::splitk_begin(s, c), b1 = bws::splitk_begin(s, c + 1);
    if (b1 <= b0) return false;
    for (long long u = b0; u < b1; ++u)
      if (bws::splitk_owner(s, u) != c) return false;
  }
  return true;
}

int main() {
  int cases = 0;
  const long long units[] = {1, 7, 60, 303, 304, 305, 960, 1080, 2720, 5440, 7240, 19400, 77600};
  for (long long U : units) {
    const int G = (int)(U < 304 ? U : 304);
    SplitK s = {U, G, G, 1, 1};   // uniform
    if (!check(s)) { std::printf("uniform U=%lld G=%d failed\n", U, G); return 1; }
    ++cases;
    for (int light : {2, 8, 16, 60}) {
      for (int num = 4; num < 16; ++num) {
        if (light >= G / 4) continue;
        const long long w = 16LL * (G - light) + (long long)num * light;
        if ((long long)num * U < w) continue;   // the guard the split's users apply
        SplitK t = {U, G, G - light, num, 16};
        if (!check(t)) { std::printf("U=%lld G=%d light=%d num=%d failed\n", U, G, light, num); return 1; }
        ++cases;
      }
    }
  }
  std::printf("split ok: %d cases\n", cases);
  return 0;
}
