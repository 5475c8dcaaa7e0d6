// internal.h -- declarations shared by the C-ABI front end (fa_api.cu) and the
// kernel translation units.  Not part of the public interface.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/fa.h"

namespace fa {

// Library status word in device memory (one per device).  `code` is the first
// device-side error since the last fa_get_status(); `abort_epoch` is the
// highest launch epoch in which some CTA gave up, so that the other CTAs of
// the same launch stop waiting too.
struct DevStatus {
  int code;
  unsigned int abort_epoch;
};

// Index checks of the debug build (FA_DEBUG): `ok` false records FA_ERR_BOUNDS
// in the status word (the first error wins) and the caller skips the access;
// nothing traps, so the context stays usable.  In the release build the checks
// are constant true and compile away.
#ifdef __CUDACC__
#ifdef FA_DEBUG
__device__ __forceinline__ bool fa_bounds(DevStatus* st, bool ok) {
  if (!ok) atomicCAS(&st->code, 0, (int)FA_ERR_BOUNDS);
  return ok;
}
#else
__device__ __forceinline__ constexpr bool fa_bounds(DevStatus*, bool) { return true; }
#endif
#endif

// Where a launch reports to and how long its waits may last.
struct Report {
  DevStatus* st;
  uint32_t epoch;
  uint64_t wait_ns;
};

// Which (query tile, key tile) pairs are visited: causal skips tiles whose
// keys all lie after their queries, and the block mask skips hidden tiles.
struct MaskArgs {
  int causal;
  const uint8_t* mask;  // device, or nullptr
  int mask_block;       // tokens per mask entry (a multiple of the kernel tile)
  int mask_cols;        // ceil(N / mask_block)
  long long mask_sb, mask_sh;
};

// Dropout of the attention weights: weight (query i, key j) of head bh is kept
// and scaled by z = 2^16 / (2^16 - t) when the 16-bit half (j mod 2: low, high)
// of word (j mod 8) / 2 of Philox4x32-10 with counter (j / 8, i, bh, offset) and
// key (key0, key1) is >= t = floor(p 2^16), else dropped.  on = 0: no dropout
// (the kernels without it run).
struct DropArgs {
  uint32_t on;
  uint32_t t;
  float z;
  uint32_t key0, key1;
  uint32_t offset;
};

struct FwdArgs {
  int B, H, N;
  float scale;       // natural-units score scale
  float scale_log2;  // scale * log2(e)
  MaskArgs m;
  void* O;
  float* LSE;
  // split key range: with n_splits > 1, CTA split s covers key tiles
  // [s * split_tiles, (s + 1) * split_tiles) of its query tile, and the
  // n_splits CTAs of a query tile (one cluster) merge their slices into O, LSE
  int n_splits;
  int split_tiles;
  // grid order: the heads are taken in groups of head_group (the last group may
  // be smaller); within a group the CTAs run query-tile-major, the heaviest
  // causal tiles of the group's heads first.  head_group = B*H is one group; a
  // smaller group keeps the K, V that the running CTAs stream within L2.  The
  // last head_tail heads (0: none) form one more group after the others
  int head_group;
  int head_tail;
  DropArgs drop;
  Report rep;
};

struct BwdArgs {
  int B, H, N;
  float scale;
  float scale_log2;
  MaskArgs m;
  const void* O;
  const void* dO;
  const float* LSE;
  void* dK;
  void* dV;
  void* dQ;
  float* Dsum;   // [B*H*N]  rowsum(dO * O)
  float* dQacc;  // [B*H*N*d] fp32 accumulator of dQ / scale
  // Work split (bwd_sched.cuh): units (key tiles, u = kt * B*H + bh) before
  // qs_from run one CTA each; with q_slice = P > 0 the units from qs_from on are
  // cut into slices of at most P visited query tiles, one CTA each, and a unit
  // of several slices writes fp32 partial [dV | dK] sums (dK unscaled) to the
  // slots of its slices, which the finalize kernel adds up.  direct: the CTAs
  // of the launch.
  int direct;
  int qs_from;
  int q_slice;
  float* slots;
  // grid order of a launch whose every unit is its own CTA (q_slice = 0):
  // the heads in groups of head_group, key-tile-major within a group (the
  // heaviest causal key tiles of the group's heads first); B*H is one group.  A
  // smaller group keeps the Q, dO and dQ accumulator the running CTAs stream
  // within L2; the last head_tail heads (0: none) form one more group after the
  // others.  Other launches use the key-tile-major unit numbering.
  int head_group;
  int head_tail;
  DropArgs drop;
  Report rep;
};

// Kernel launchers (one per translation unit).
cudaError_t launch_fwd_f32(const FwdArgs& a, int d, const float* Q, const float* K,
                           const float* V, cudaStream_t s);
cudaError_t launch_fwd_tc(const FwdArgs& a, int d, bool f16, const CUtensorMap* tmaps,
                          cudaStream_t s);
cudaError_t launch_bwd_preprocess(const BwdArgs& a, int d, bool f16, cudaStream_t s);
cudaError_t launch_bwd_tc(const BwdArgs& a, int d, bool f16, const CUtensorMap* tmaps,
                          cudaStream_t s);
cudaError_t launch_bwd_finalize(const BwdArgs& a, int d, bool f16, cudaStream_t s);
cudaError_t launch_wait_selftest(const Report& rep, cudaStream_t s);

// Records the text fa_last_error() returns on this thread.
void set_error_text(const char* text);

}  // namespace fa
