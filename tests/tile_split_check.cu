// Host check of he::TileSplit, the two-group stream-K split the stream kernel
// (ranges) and the merge kernel (owners) must agree on.  For every tile count
// TT, CTA count NC <= TT and every first group (E CTAs over T1 tiles) the host
// may choose (T1 >= E, TT - T1 >= NC - E: at least one tile per CTA):
//   begin(0) = 0, begin(NC) = TT, every range non-empty, and owner(t) = c for
//   every tile t of CTA c's range.
// Prints "ok <cases>" or the first failure.
#include <cstdio>
#include <cstdint>
#include <random>

#include "he_pipeline.cuh"

static bool check(int64_t TT, int64_t NC, int64_t E, int64_t T1) {
  const he::TileSplit sp{TT, NC, E, T1};
  if (sp.begin(0) != 0 || sp.begin(NC) != TT) {
    std::printf("FAIL ends TT=%lld NC=%lld E=%lld T1=%lld\n", (long long)TT, (long long)NC,
                (long long)E, (long long)T1);
    return false;
  }
  for (int64_t c = 0; c < NC; ++c) {
    const int64_t b = sp.begin(c), e = sp.begin(c + 1);
    if (e <= b) {
      std::printf("FAIL empty TT=%lld NC=%lld E=%lld T1=%lld c=%lld\n", (long long)TT,
                  (long long)NC, (long long)E, (long long)T1, (long long)c);
      return false;
    }
    for (int64_t t = b; t < e; ++t)
      if (sp.owner(t) != c) {
        std::printf("FAIL owner TT=%lld NC=%lld E=%lld T1=%lld t=%lld owner=%lld c=%lld\n",
                    (long long)TT, (long long)NC, (long long)E, (long long)T1, (long long)t,
                    (long long)sp.owner(t), (long long)c);
        return false;
      }
  }
  return true;
}

int main() {
  long long cases = 0;
  // every small shape and every admissible first group (E = 0: the even split)
  for (int64_t TT = 1; TT <= 48; ++TT)
    for (int64_t NC = 1; NC <= TT && NC <= 16; ++NC) {
      if (!check(TT, NC, 0, 0)) return 1;
      ++cases;
      for (int64_t E = 1; E < NC; ++E)
        for (int64_t T1 = E; TT - T1 >= NC - E; ++T1) {
          if (!check(TT, NC, E, T1)) return 1;
          ++cases;
        }
    }
  // large shapes of the workloads' kind (296 CTAs, thousands of tiles)
  std::mt19937_64 rng(7);
  for (int i = 0; i < 400; ++i) {
    const int64_t NC = 1 + (int64_t)(rng() % 296);
    const int64_t TT = NC + (int64_t)(rng() % 30000);
    const int64_t E = (int64_t)(rng() % NC);
    const int64_t lo = E, hi = TT - (NC - E);
    const int64_t T1 = E == 0 ? 0 : lo + (int64_t)(rng() % (uint64_t)(hi - lo + 1));
    if (!check(TT, NC, E, T1)) return 1;
    ++cases;
  }
  std::printf("ok %lld\n", cases);
  return 0;
}
