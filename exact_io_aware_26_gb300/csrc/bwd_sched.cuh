// bwd_sched.cuh -- how the backward main kernel spreads its work over CTAs, and
// the head-group grid order of the one-CTA-per-tile launches of both passes.
//
// A unit is one key tile of one head; the units are numbered key-tile-major,
// u = kt * (B*H) + bh, and a unit visits query tiles base .. base + vis - 1
// (causal: base = kt and vis = n - kt; else base = 0 and vis = n).  Units
// before u0 each run as one CTA.  The units from u0 on are cut into slices of
// at most P visited query tiles (slices_of(kt) = ceil(vis / P) of them), each
// slice its own CTA: with fewer key tiles than SMs, so that every SM gets work
// (u0 = 0, P chosen so that the slices about fill one wave), and for the key
// tiles of a last, partly filled wave (non-causal only).  A unit cut into
// several slices gets its dK, dV as fp32 partial sums, one slot per slice, that
// the finalize kernel adds up.  With a block mask, whose kept query tiles are
// known on the device only, every unit is one CTA.
#pragma once
#include <cstdint>

#ifndef __CUDACC__  // host-only compilers (the schedule is also checked on the CPU)
#define __host__
#define __device__
#endif

namespace fa {

// Most slices a launch may cut (the workspace holds a partial-sum slot for each).
constexpr int kBwdMaxCtas = 160;

// query tiles key tile kt visits
__host__ __device__ inline int sched_visited(int kt, int n, int causal) {
  return causal ? n - kt : n;
}
// sum of ceil(m / P) over m = 1 .. M
__host__ __device__ inline long long ceil_sum(long long M, int P) {
  const long long q = M / P, r = M % P;
  return (long long)P * q * (q + 1) / 2 + (q + 1) * r;
}
// slices of one unit of key tile kt
__host__ __device__ inline int slices_of(int kt, int n, int causal, int P) {
  return (sched_visited(kt, n, causal) + P - 1) / P;
}
// slices of the units of key tiles 0 .. kt - 1 (all heads); every unit sliced
__host__ __device__ inline long long slices_before(int kt, int n, int BH, int causal, int P) {
  if (!causal) return (long long)BH * kt * ((n + P - 1) / P);
  return (long long)BH * (ceil_sum(n, P) - ceil_sum(n - kt, P));
}

// One sliced CTA's work: key tile kt of head bh, query tiles [q_first, q_end),
// and its partial-sum slot (-1: the slice is the whole unit, whose dK, dV it
// writes itself).
struct Slice {
  int kt, bh, q_first, q_end, slot;
};

// The work of sliced CTA j (0-based, counted from the first sliced unit u0).
// A causal launch slices from u0 = 0 only.
__host__ __device__ inline Slice slice_locate(long long j, int n, int BH, int causal, int P, int u0) {
  int kt, bh, s, k;
  if (!causal) {
    k = (n + P - 1) / P;
    const long long u = u0 + j / k;
    kt = (int)(u / BH);
    bh = (int)(u % BH);
    s = (int)(j % k);
  } else {
    // the key tile: the largest kt with slices_before(kt) <= j (binary search)
    int lo = 0, hi = n - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) / 2;
      if (slices_before(mid, n, BH, causal, P) <= j) lo = mid; else hi = mid - 1;
    }
    kt = lo;
    k = slices_of(kt, n, causal, P);
    const long long r = j - slices_before(kt, n, BH, causal, P);
    bh = (int)(r / k);
    s = (int)(r % k);
  }
  const int base = causal ? kt : 0, vis = sched_visited(kt, n, causal);
  Slice sl;
  sl.kt = kt;
  sl.bh = bh;
  sl.q_first = base + s * P;
  sl.q_end = base + ((s + 1) * P < vis ? (s + 1) * P : vis);
  sl.slot = k > 1 ? (int)j : -1;
  return sl;
}

// Slots of unit u >= u0 (kt-major numbering): the first one and how many (one:
// the unit ran whole and has none).
__host__ __device__ inline void unit_slots(long long u, int n, int BH, int causal, int P, int u0,
                                           long long& first, int& count) {
  const int kt = (int)(u / BH), bh = (int)(u % BH);
  count = slices_of(kt, n, causal, P);
  first = causal ? slices_before(kt, n, BH, causal, P) + (long long)bh * count
                 : (u - u0) * (long long)count;
}

// Sliced CTAs from unit u0 on.
__host__ __device__ inline long long slice_total(int n, int BH, int causal, int P, int u0) {
  if (!causal) return ((long long)n * BH - u0) * ((n + P - 1) / P);
  return slices_before(n, n, BH, causal, P);
}

// The work split of an unmasked backward over G CTAs per wave (one per SM):
// P = 0 when every key tile is one CTA; else the units from u0 on are sliced
// with slice length P.  Returns the CTAs of the launch.
//  - fewer key tiles than CTAs: every key tile is cut into slices of at most P
//    visited query tiles, P the smallest whose slices fit in G CTAs;
//  - non-causal, a grid that ends in a partly filled wave of r key tiles: those
//    r tiles are cut into k slices of at least two query tiles over the SMs the
//    wave leaves idle, so the launch ends about (k - 1) / k of a key tile sooner.
__host__ __device__ inline long long plan_slices(int n, int BH, int causal, long long G, int& P, int& u0) {
  const long long units = (long long)n * BH;
  P = 0;
  u0 = (int)units;
  if (units < G) {
    for (int p = 1; p < n; ++p) {
      const long long total = slice_total(n, BH, causal, p, 0);
      if (total <= G) {
        P = p;
        u0 = 0;
        return total;
      }
    }
  } else if (!causal && units % G != 0 && n >= 4) {
    const long long r = units % G;
    const long long k = (G / r < n / 2) ? G / r : n / 2;
    if (k >= 2) {
      P = (int)((n + k - 1) / k);
      u0 = (int)(units - r);
      return units - r + r * ((n + P - 1) / P);
    }
  }
  return units;
}

// Grid order of a one-CTA-per-tile launch (both passes): CTA t of a grid over
// `tiles` tiles of each of BH heads, the heads taken in groups of `group` (the
// last group may be smaller) and the tiles of a group tile-major, so that the
// CTAs running at any moment share the streamed operands of one group of heads;
// the last `tail` heads (0: none) form one more tile-major group after them, so
// that on a causal problem their heaviest tiles start early enough not to
// finish alone after everything else.  Returns the tile index ti (0 first: the
// caller maps it to its heaviest tile) and the head bh.  group = BH, tail = 0
// is plain tile-major order over all heads.
__host__ __device__ inline void group_order(int t, int tiles, int BH, int group, int tail, int& ti,
                                            int& bh) {
  const int body = BH - tail;  // heads before the tail group
  if (t >= body * tiles) {
    const int r = t - body * tiles;
    ti = r / tail;
    bh = body + r % tail;
    return;
  }
  const int per_group = group * tiles;
  const int g0 = (t / per_group) * group;  // first head of t's group
  const int gh = body - g0 < group ? body - g0 : group;  // heads in that group
  const int r = t - g0 * tiles;
  ti = r / gh;
  bh = g0 + r % gh;
}

}  // namespace fa
