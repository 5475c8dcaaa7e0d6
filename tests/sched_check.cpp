// Brute-force check of the backward kernel's work split (bwd_sched.cuh) on the
// CPU: every (head, key tile, query tile) iteration of the units from u0 on is
// taken by exactly one CTA (and none before u0), pieces that cover a whole key
// tile have no slot, every other piece has a slot of its own, and the shared
// key tiles that sched_shared reports (one boundary each) name exactly the
// CTAs and slots that hold their partial sums.
// Usage: sched_check n BH causal G u0   (exit status 0 when every check holds)
//        sched_check group tiles BH group tail   (the head-group grid order)
#include <cstdio>
#include <cstdlib>
#include <map>
#include <set>
#include <string>
#include <utility>
#include <vector>

#include "bwd_sched.cuh"

using namespace fa;

#define CHECK(c)                                                         \
  do {                                                                   \
    if (!(c)) {                                                          \
      std::fprintf(stderr, "check failed at line %d: %s\n", __LINE__, #c); \
      return 1;                                                          \
    }                                                                    \
  } while (0)

// Grid order (group_order): CTAs 0 .. tiles*BH - 1 visit every (tile, head) once;
// the first BH - tail heads come in groups of `group` (the last smaller) and the
// last `tail` heads in one group after them; a group's CTAs are contiguous and
// tile-major (non-decreasing tile index, heads cycling within the group), and
// group = BH, tail = 0 is the plain order ti = t / BH, bh = t % BH.
static int check_group(int tiles, int BH, int group, int tail) {
  std::set<std::pair<int, int>> seen;
  int prev_g0 = -1, prev_ti = -1;
  const int body = BH - tail;
  for (int t = 0; t < tiles * BH; ++t) {
    int ti, bh;
    group_order(t, tiles, BH, group, tail, ti, bh);
    CHECK(ti >= 0 && ti < tiles && bh >= 0 && bh < BH);
    CHECK(seen.insert({ti, bh}).second);
    int g0, gh;  // the first head of bh's group and the group's size
    if (bh >= body) {
      g0 = body;
      gh = tail;
    } else {
      g0 = bh / group * group;
      gh = body - g0 < group ? body - g0 : group;
    }
    CHECK(t >= g0 * tiles && t < (g0 + gh) * tiles);  // the group's CTAs are contiguous
    if (g0 == prev_g0) CHECK(ti >= prev_ti);           // tile-major within the group
    CHECK(bh - g0 == (t - g0 * tiles) % gh);
    prev_g0 = g0;
    prev_ti = ti;
    if (group == BH && tail == 0) CHECK(ti == t / BH && bh == t % BH);
  }
  CHECK((int)seen.size() == tiles * BH);
  return 0;
}

int main(int argc, char** argv) {
  if (argc == 6 && std::string(argv[1]) == "group")
    return check_group(std::atoi(argv[2]), std::atoi(argv[3]), std::atoi(argv[4]), std::atoi(argv[5]));
  if (argc != 6) return 2;
  const int n = std::atoi(argv[1]), BH = std::atoi(argv[2]), causal = std::atoi(argv[3]),
            G = std::atoi(argv[4]), u0 = std::atoi(argv[5]);
  const Sched s = make_sched(n, BH, causal, G, u0);
  // iteration order: key tile, then head (unit u = kt * BH + bh), then query tile
  long long g = 0;
  for (int u = u0; u < n * BH; ++u) {
    const int kt = u / BH, bh = u % BH;
    CHECK(sched_unit_start(u, n, BH, causal) == s.P0 + g);
    for (int q = causal ? kt : 0; q < n; ++q, ++g) {
      int b2, k2, j2;
      sched_locate(s, g, b2, k2, j2);
      CHECK(b2 == bh && k2 == kt && j2 == q - (causal ? kt : 0));
    }
  }
  CHECK(g == s.T);
  CHECK(sched_start(s, 0) == 0 && sched_start(s, G) == s.T);
  std::vector<int> seen((size_t)BH * n * n, 0);
  // key tile -> {(cta, slot)} of its partial pieces
  std::map<std::pair<int, int>, std::set<std::pair<int, int>>> parts;
  std::set<int> slots;
  for (int c = 0; c < G; ++c) {
    long long gg = sched_start(s, c);
    const long long ge = sched_start(s, c + 1);
    CHECK(ge > gg);  // no CTA without work
    bool first = true;
    Seg sg;
    int pieces = 0;
    std::vector<Seg> mine;
    while (sched_next(s, c, gg, ge, first, sg)) {
      mine.push_back(sg);
      ++pieces;
      CHECK(sg.bh >= 0 && sg.bh < BH && sg.kt >= 0 && sg.kt < n);
      CHECK(sg.q_first >= (causal ? sg.kt : 0) && sg.q_first < sg.q_end && sg.q_end <= n);
      for (int q = sg.q_first; q < sg.q_end; ++q) ++seen[((size_t)sg.bh * n + sg.kt) * n + q];
      const bool whole = sg.q_first == (causal ? sg.kt : 0) && sg.q_end == n;
      CHECK(whole == (sg.slot < 0));
      if (sg.slot >= 0) {
        CHECK(slots.insert(sg.slot).second);
        parts[{sg.bh, sg.kt}].insert({c, sg.slot});
      }
    }
    CHECK(gg == ge && pieces >= 1);
    for (size_t k = 0; k < mine.size(); ++k) {
      if (mine[k].slot < 0) continue;
      if (k == 0) CHECK(mine[k].slot == 2 * c);
      else CHECK(k + 1 == mine.size() && mine[k].slot == 2 * c + 1);
    }
  }
  for (int bh = 0; bh < BH; ++bh)
    for (int kt = 0; kt < n; ++kt)
      for (int q = 0; q < n; ++q)
        CHECK(seen[((size_t)bh * n + kt) * n + q] ==
              ((kt * BH + bh >= u0 && (!causal || q >= kt)) ? 1 : 0));
  // the finalize stage's view of the shared key tiles
  std::map<std::pair<int, int>, std::set<std::pair<int, int>>> fixed;
  for (int c = 0; c + 1 < G; ++c) {
    int bh, kt, c_last, fs;
    if (!sched_shared(s, c, bh, kt, c_last, fs)) continue;
    std::set<std::pair<int, int>> want{{c, fs}};
    for (int cc = c + 1; cc <= c_last; ++cc) want.insert({cc, 2 * cc});
    CHECK(fixed.emplace(std::make_pair(bh, kt), want).second);  // one boundary per key tile
  }
  CHECK(fixed == parts);
  std::printf("ok n=%d BH=%d causal=%d G=%d u0=%d T=%lld shared=%zu\n", n, BH, causal, G, u0, s.T,
              parts.size());
  return 0;
}
