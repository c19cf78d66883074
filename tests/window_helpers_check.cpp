// Brute-force check of the sliding-window helpers the kernels use
// (win_meets, win_covers, win_span, bit_range in bsa_common.h) on every small
// rectangle and window. Host-only; built and run by test_window_helpers.py.
// Exit status 0 = all cases agree.
#include <cstdio>

#include "bsa_common.h"

using namespace bsa;

static bool in_win(long s, long t, long pre, long next) { return s - pre <= t && t <= s + next; }

int main() {
  long bad = 0, cases = 0;
  const long pres[] = {-6, -1, 0, 1, 3, 9, 40, 1L << 40};
  const long nexts[] = {-6, -1, 0, 2, 5, 11, 40, 1L << 40};
  for (long pre : pres)
    for (long next : nexts) {
      if (pre + next < 0) continue;
      for (long s0 = 0; s0 < 12; ++s0)
        for (long s1 = s0 + 1; s1 <= 14; ++s1)
          for (long t0 = 0; t0 < 12; ++t0)
            for (long t1 = t0 + 1; t1 <= 14; ++t1) {
              bool any = false, all = true;
              for (long s = s0; s < s1; ++s)
                for (long t = t0; t < t1; ++t) {
                  const bool w = in_win(s, t, pre, next);
                  any |= w;
                  all &= w;
                }
              ++cases;
              if (win_meets(s0, s1, t0, t1, pre, next) != any ||
                  win_covers(s0, s1, t0, t1, pre, next) != all) {
                if (bad < 5)
                  std::printf("rect s[%ld,%ld) t[%ld,%ld) pre %ld next %ld\n", s0, s1, t0, t1, pre,
                              next);
                ++bad;
              }
            }
      // spans of a query row (keys) and of a key row (queries), tile base 0..300
      for (long pos = 0; pos < 400; pos += 7)
        for (long base = 0; base < 400; base += 64) {
          const int2 q = win_span(pos, base, -pre, next);
          const int2 k = win_span(pos, base, -next, pre);
          for (int x = 0; x < 128; ++x) {
            const bool want_q = in_win(pos, base + x, pre, next);
            const bool want_k = in_win(base + x, pos, pre, next);
            ++cases;
            if ((x >= q.x && x < q.y) != want_q || (x >= k.x && x < k.y) != want_k) {
              if (bad < 5) std::printf("span pos %ld base %ld x %d\n", pos, base, x);
              ++bad;
            }
          }
        }
    }
  for (int lo = -40; lo <= 70; ++lo)
    for (int hi = -40; hi <= 70; ++hi) {
      const uint32_t m = bit_range(lo, hi);
      for (int b = 0; b < 32; ++b) {
        ++cases;
        if ((((m >> b) & 1u) != 0) != (b >= lo && b < hi)) ++bad;
      }
    }
  std::printf("%ld cases, %ld disagree\n", cases, bad);
  return bad == 0 ? 0 : 1;
}
