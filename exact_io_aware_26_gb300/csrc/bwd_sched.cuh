// bwd_sched.cuh -- how the backward main kernel splits its work over CTAs, and
// the head-group grid order of the one-CTA-per-tile launches of both passes.
//
// A unit is one key tile of one head; the units are numbered key-tile-major,
// u = kt * (B*H) + bh, and each unit's iterations are its visited query tiles
// (causal: from the key tile's own index up).  The units from u0 on are split
// "stream-K": their iterations, in that order, are cut into G contiguous
// ranges of nearly equal length, one per persistent CTA (G about the SM
// count).  A range may begin or end inside a unit: that key tile's dK, dV are
// then written by each CTA that touched it as fp32 partial sums into a slot
// of its own (slot 2c for CTA c's first range piece, 2c + 1 for its last), and
// the finalize kernel adds the slots.  Units before u0 are whole-key-tile
// CTAs of the one-CTA-per-key-tile kernel (so that only the last, ragged
// wave is split), and with a block mask, whose kept query tiles are known on
// the device only, every unit is.
#pragma once
#include <cmath>
#include <cstdint>

#ifndef __CUDACC__  // host-only compilers (the schedule is also checked on the CPU)
#define __host__
#define __device__
#endif

namespace fa {

struct Sched {
  int n;         // tiles per sequence (ceil(N / 128))
  int BH;        // heads (B * H)
  int causal;    // query tiles before the key tile are skipped
  int G;         // CTAs
  long long P0;  // iterations of the units before u0
  long long T;   // iterations of units u0 .. n*BH - 1
};

// Most CTAs a stream-K launch uses (and that the workspace holds slots for).
constexpr int kBwdMaxCtas = 160;

// iterations of the key tiles before kt in one head
__host__ __device__ inline long long sched_before(int kt, int n, int causal) {
  return causal ? (long long)kt * n - (long long)kt * (kt - 1) / 2 : (long long)kt * n;
}
// query tiles key tile kt visits
__host__ __device__ inline int sched_visited(int kt, int n, int causal) {
  return causal ? n - kt : n;
}
// iterations of the units before unit u
__host__ __device__ inline long long sched_unit_start(long long u, int n, int BH, int causal) {
  const int kt = (int)(u / BH), bh = (int)(u - (long long)kt * BH);
  return (long long)BH * sched_before(kt, n, causal) + (long long)bh * sched_visited(kt, n, causal);
}
__host__ __device__ inline Sched make_sched(int n, int BH, int causal, int G, long long u0 = 0) {
  Sched s;
  s.n = n;
  s.BH = BH;
  s.causal = causal;
  s.G = G;
  s.P0 = sched_unit_start(u0, n, BH, causal);
  s.T = (long long)BH * sched_before(n, n, causal) - s.P0;
  return s;
}
// first iteration of CTA c (c = G gives T), counted from unit u0
__host__ __device__ inline long long sched_start(const Sched& s, int c) {
  return (long long)c * s.T / s.G;
}
// head, key tile and index among the key tile's visited query tiles of iteration g
__host__ __device__ inline void sched_locate(const Sched& s, long long g, int& bh, int& kt, int& j) {
  const long long a = g + s.P0;  // from the first unit
  // the key tile: the largest k with BH * sched_before(k) <= a, i.e. with
  // sched_before(k) <= r
  const long long r = a / s.BH;
  int k;
  if (!s.causal) {
    k = (int)(r / s.n);
  } else {
    // a root of k^2 - (2n+1) k + 2r, then corrected by exact integer comparisons
    const double b2 = 2.0 * s.n + 1.0;
    const double disc = b2 * b2 - 8.0 * (double)r;
    k = (int)((b2 - sqrt(disc > 0.0 ? disc : 0.0)) * 0.5);
  }
  if (k < 0) k = 0;
  if (k > s.n - 1) k = s.n - 1;
  while (k > 0 && sched_before(k, s.n, s.causal) > r) --k;
  while (k + 1 < s.n && sched_before(k + 1, s.n, s.causal) <= r) ++k;
  kt = k;
  const long long rem = a - (long long)s.BH * sched_before(k, s.n, s.causal);
  const int v = sched_visited(k, s.n, s.causal);
  bh = (int)(rem / v);
  j = (int)(rem - (long long)bh * v);
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

// One piece of a CTA's range: key tile kt of head bh, query tiles [q_first, q_end).
struct Seg {
  int bh, kt, q_first, q_end;
  int slot;  // -1: the whole key tile (dK, dV written directly); else the partial-sum slot
};

// The next piece of CTA c's range [g, g_end); advances g.
__host__ __device__ inline bool sched_next(const Sched& s, int c, long long& g, long long g_end,
                                           bool& first, Seg& sg) {
  if (g >= g_end) return false;
  int bh, kt, j;
  sched_locate(s, g, bh, kt, j);
  const int vis = sched_visited(kt, s.n, s.causal);
  const long long left = g_end - g;
  const int j_end = (long long)(vis - j) <= left ? vis : j + (int)left;
  const int qbase = s.causal ? kt : 0;
  sg.bh = bh;
  sg.kt = kt;
  sg.q_first = qbase + j;
  sg.q_end = qbase + j_end;
  sg.slot = (j == 0 && j_end == vis) ? -1 : (first ? 2 * c : 2 * c + 1);
  g += j_end - j;
  first = false;
  return true;
}

// The key tile that CTAs c and c + 1 share, if their boundary falls inside one
// and is the first boundary inside it: its head and key tile, the last CTA that
// shares it, and CTA c's slot for it (its last piece 2c + 1, or its first 2c
// when its range starts at the key tile).  CTAs c + 1 .. c_last hold it in
// their first slots, 2c'.
__host__ __device__ inline bool sched_shared(const Sched& s, int c, int& bh, int& kt, int& c_last,
                                             int& first_slot) {
  const long long p = sched_start(s, c + 1);
  int j;
  sched_locate(s, p, bh, kt, j);
  if (j == 0) return false;  // the boundary is at a key tile's start
  const long long u_start = p - j;
  const long long u_end = u_start + sched_visited(kt, s.n, s.causal);
  const long long c_start = sched_start(s, c);
  if (c_start > u_start) return false;  // an earlier boundary lies inside the key tile
  c_last = c + 1;
  while (c_last + 1 < s.G && sched_start(s, c_last + 1) < u_end) ++c_last;
  first_slot = c_start < u_start ? 2 * c + 1 : 2 * c;
  return true;
}

}  // namespace fa
