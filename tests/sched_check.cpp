// Brute-force check of the backward main kernel's work split (bwd_sched.cuh)
// on the CPU: for an unmasked problem of n tiles per sequence and BH heads
// spread over G CTAs per wave, plan_slices cuts the units from u0 on into
// slices; every visited (head, key tile, query tile) of those units belongs to
// exactly one slice CTA (and of the units before u0 to none), every slice is
// non-empty and at most P long, the slices of a unit of several slices have
// slots of their own that unit_slots names exactly, a unit of one slice has no
// slot, and the slices fill at most one wave (with fewer key tiles than CTAs)
// or the idle SMs of the last wave.
// Usage: sched_check slices n BH causal G   (exit status 0 when every check holds)
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

static int check_slices(int n, int BH, int causal, long long G) {
  int P = -1, u0 = -1;
  const long long units = (long long)n * BH;
  const long long ctas = plan_slices(n, BH, causal, G, P, u0);
  if (P == 0) {  // every key tile one CTA
    CHECK(ctas == units && u0 == units);
    // slicing would not have shortened the launch: no P < n fits one wave, or
    // the last wave is full, causal, too full to split, or n < 4
    if (units < G) CHECK(slice_total(n, BH, causal, n - 1 > 0 ? n - 1 : 1, 0) > G || n == 1);
    std::printf("ok n=%d BH=%d causal=%d G=%lld: whole key tiles\n", n, BH, causal, G);
    return 0;
  }
  CHECK(P >= 1 && P < n && u0 >= 0 && u0 < units);
  CHECK(!causal || u0 == 0);  // a causal launch slices from the first unit only
  const long long total = slice_total(n, BH, causal, P, u0);
  CHECK(ctas == u0 + total);
  if (units < G) {
    CHECK(u0 == 0 && total <= G);
    if (P > 1) CHECK(slice_total(n, BH, causal, P - 1, 0) > G);  // P is the smallest that fits
  } else {
    CHECK(!causal && u0 == units - units % G && total <= G && P >= 2);
  }
  std::vector<int> seen((size_t)BH * n * n, 0);
  std::map<long long, std::vector<int>> unit_slot_list;  // unit -> slots of its slices
  std::map<long long, int> unit_count;                   // unit -> slices
  std::set<int> used;
  for (long long j = 0; j < total; ++j) {
    const Slice sl = slice_locate(j, n, BH, causal, P, u0);
    CHECK(sl.bh >= 0 && sl.bh < BH && sl.kt >= 0 && sl.kt < n);
    const long long u = (long long)sl.kt * BH + sl.bh;
    CHECK(u >= u0);
    const int base = causal ? sl.kt : 0;
    CHECK(sl.q_first >= base && sl.q_first < sl.q_end && sl.q_end <= n && sl.q_end - sl.q_first <= P);
    for (int q = sl.q_first; q < sl.q_end; ++q) ++seen[((size_t)sl.bh * n + sl.kt) * n + q];
    ++unit_count[u];
    if (sl.slot >= 0) {
      CHECK(sl.slot < total && used.insert(sl.slot).second);
      unit_slot_list[u].push_back(sl.slot);
    }
  }
  for (int bh = 0; bh < BH; ++bh)
    for (int kt = 0; kt < n; ++kt)
      for (int q = 0; q < n; ++q)
        CHECK(seen[((size_t)bh * n + kt) * n + q] ==
              (((long long)kt * BH + bh >= u0 && (!causal || q >= kt)) ? 1 : 0));
  // the finalize stage's view: unit_slots names each unit's slots exactly
  for (long long u = u0; u < units; ++u) {
    long long first;
    int count;
    unit_slots(u, n, BH, causal, P, u0, first, count);
    CHECK(count == unit_count[u]);
    if (count == 1) {
      CHECK(unit_slot_list.count(u) == 0);  // one slice: the whole unit, no slot
    } else {
      std::vector<int> want;
      for (int i = 0; i < count; ++i) want.push_back((int)(first + i));
      CHECK(unit_slot_list[u] == want);
    }
  }
  std::printf("ok n=%d BH=%d causal=%d G=%lld: P=%d u0=%d slices=%lld\n", n, BH, causal, G, P, u0, total);
  return 0;
}

int main(int argc, char** argv) {
  if (argc == 6 && std::string(argv[1]) == "group")
    return check_group(std::atoi(argv[2]), std::atoi(argv[3]), std::atoi(argv[4]), std::atoi(argv[5]));
  if (argc == 6 && std::string(argv[1]) == "slices")
    return check_slices(std::atoi(argv[2]), std::atoi(argv[3]), std::atoi(argv[4]), std::atoll(argv[5]));
  return 2;
}
