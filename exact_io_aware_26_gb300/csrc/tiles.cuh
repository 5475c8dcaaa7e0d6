// tiles.cuh -- the tile grid every pass walks, in one place: the 128-row tile,
// which (query tile, key tile) pairs are visited (the causal rule and the block
// mask), and the backward's per-row statistics as its compute warps use them.
#pragma once
#include "internal.h"

namespace fa {

constexpr int kTile = 128;  // query rows per query tile = keys per key tile

// Whether query tile qt sees key tile kt: not when every key lies after every
// query of the tile ("Le masquage causal est l'endroit où le trading bénéficie
// d'une remise": such a tile is never loaded nor computed), nor when the block
// mask hides it ("Extensão: Block-Sparse FlashAttention").
__device__ __forceinline__ bool tile_kept(const MaskArgs& m, int b, int h, int qt, int kt) {
  if (m.causal && kt > qt) return false;
  if (m.mask) {
    const long long at = (long long)b * m.mask_sb + (long long)h * m.mask_sh +
                         (long long)((qt * kTile) / m.mask_block) * m.mask_cols +
                         (kt * kTile) / m.mask_block;
    return m.mask[at] != 0;
  }
  return true;
}

// First key tile at or after kt that query tile qt sees, or kt_end (forward).
__device__ __forceinline__ int next_kept(const MaskArgs& m, int b, int h, int qt, int kt, int kt_end) {
  while (kt < kt_end && !tile_kept(m, b, h, qt, kt)) ++kt;
  return kt;
}

// First query tile at or after qt that sees key tile kt, or q_end (backward).
__device__ __forceinline__ int next_q(const MaskArgs& m, int b, int h, int qt, int kt, int q_end) {
  while (qt < q_end && !tile_kept(m, b, h, qt, kt)) ++qt;
  return qt;
}

// With a block mask, each CTA walks one row (forward: the key tiles its query
// tile sees) or one column (backward: the query tiles that see its key tile) of
// the mask.  Reading the mask in global memory at every step costs one dependent
// load per hidden tile, which on a sparse mask dominated the step, so the CTA
// first turns its row or column into a bitmask in shared memory (all warps, one
// ballot per 32 tiles) and then walks the bits.  kMaskBits tiles fit (N up to
// kMaskBits * 128 keys); longer sequences read the mask itself.
constexpr int kMaskBits = 4096;
constexpr uint32_t kMaskBitBytes = kMaskBits / 8;

// Bit t % 32 of word t / 32 is kept(t), for t in [0, n); every warp of the CTA
// calls it (a CTA-wide barrier must follow before the bits are read).
template <class Kept>
__device__ __forceinline__ void build_tile_bits(uint32_t* words, int n, int warp, int nwarps, int lane,
                                                Kept kept) {
  for (int wd = warp; wd * 32 < n; wd += nwarps) {
    const int t = wd * 32 + lane;
    const uint32_t bits = __ballot_sync(0xffffffffu, t < n && kept(t));
    if (lane == 0) words[wd] = bits;
  }
}

// First t in [t, t_end) whose bit is set, or t_end.
__device__ __forceinline__ int next_bit(const uint32_t* words, int t, int t_end) {
  while (t < t_end) {
    const uint32_t rest = words[t >> 5] >> (t & 31);
    if (rest != 0u) {
      t += __ffs((int)rest) - 1;
      return t < t_end ? t : t_end;
    }
    t = (t | 31) + 1;
  }
  return t_end;
}

// Row statistics of query q as the backward's compute warps use them: LSE *
// log2(e), with +inf hiding the row (past the end, or a row that saw no key),
// and D = rowsum(dO * O).
__device__ __forceinline__ float lse2_of(const BwdArgs& a, int bh, int q) {
  const float lse = q < a.N ? a.LSE[(size_t)bh * a.N + q] : -INFINITY;
  return (lse == -INFINITY) ? INFINITY : lse * 1.4426950408889634f;
}
__device__ __forceinline__ float d_of(const BwdArgs& a, int bh, int q) {
  return q < a.N ? a.Dsum[(size_t)bh * a.N + q] : 0.f;
}

}  // namespace fa
