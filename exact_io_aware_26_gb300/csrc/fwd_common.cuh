// fwd_common.cuh -- what the tile-per-CTA forward kernels share whatever their
// operand type (fwd_tc.cu: 16-bit operands; fwd_fp8.cu: FP8 operands): the
// barrier layout, the TMA producer of the K/V ring, the MMA warp's schedule, and
// the per-row steps of the softmax warps that do not touch the operands (masking
// a score row, rescaling O, the packed row sums, storing an O row).
//
// Both kernels run one CTA per 128-row query tile of one (batch, head): warps
// 0-3 softmax (thread t owns query row t = TMEM lane t), warp 4 the TMA producer
// (Q once, then K_j and V_j through a ring of NS stages with separate K and V
// barriers), warp 5 the TMEM owner and MMA issuer.
#pragma once
#include "ptx.cuh"
#include "tiles.cuh"

namespace fa {

// Barriers of a forward CTA: 0 q_full, 1 s_full, 2 p_full (P~_j is in TMEM),
// 3 o_done (P~ V_j has completed), 4 fin (every MMA has completed), 5 s_free (the
// softmax warps have copied S_j out of TMEM), then k_full[NS], v_full[NS],
// k_empty[NS], v_empty[NS].
template <int NS>
struct FwdBars {
  static constexpr int kCount = 6 + 4 * NS;
  uint32_t base;  // shared-memory address of barrier 0 (8-byte aligned)
  __device__ __forceinline__ uint32_t at(int i) const { return base + 8u * (uint32_t)i; }
  __device__ __forceinline__ uint32_t q() const { return at(0); }
  __device__ __forceinline__ uint32_t s() const { return at(1); }
  __device__ __forceinline__ uint32_t p() const { return at(2); }
  __device__ __forceinline__ uint32_t o() const { return at(3); }
  __device__ __forceinline__ uint32_t fin() const { return at(4); }
  __device__ __forceinline__ uint32_t sfree() const { return at(5); }
  __device__ __forceinline__ uint32_t kf(int st) const { return at(6 + st); }
  __device__ __forceinline__ uint32_t vf(int st) const { return at(6 + NS + st); }
  __device__ __forceinline__ uint32_t ke(int st) const { return at(6 + 2 * NS + st); }
  __device__ __forceinline__ uint32_t ve(int st) const { return at(6 + 3 * NS + st); }
  // one thread: p_full and s_free count one arrival per softmax warp
  __device__ __forceinline__ void init() const {
    mbar_init(q(), 1);
    mbar_init(s(), 1);
    mbar_init(p(), 4);
    mbar_init(o(), 1);
    mbar_init(fin(), 1);
    mbar_init(sfree(), 4);
    for (int st = 0; st < NS; ++st) {
      mbar_init(kf(st), 1);
      mbar_init(vf(st), 1);
      mbar_init(ke(st), 1);
      mbar_init(ve(st), 1);
    }
  }
};

// The producer lane's K/V copies: K_j and V_j of key tile kt and of every kept
// tile after it (next(kt + 1) gives the one after kt), while fewer than `limit`
// K copies have been issued; copy n goes to stage n mod NS once the MMAs have
// released that stage.  nk and nv count the K and V copies issued so far
// (limit = NS before the setup barrier: the stages are all free and nothing
// waits).  load_k(stage, kt) and load_v(stage, kt) arm the stage's full barrier
// with its byte count and issue the TMA copies.  Returns the next key tile
// (kt_end once every copy is issued), or -1 if a wait gave up.  N: the
// sequence length (the debug build checks each key tile against it).
template <int NS, class Next, class LoadK, class LoadV>
__device__ __forceinline__ int fwd_produce(const WaitCtx& w, const FwdBars<NS>& b, int kt, int kt_end,
                                           int N, int limit, int& nk, int& nv, Next next, LoadK load_k,
                                           LoadV load_v) {
  for (; kt < kt_end && nk < limit; kt = next(kt + 1)) {
    if (!dbg_check(w, kt >= 0 && kt * kTile < N)) return -1;
    const int st = nk % NS;
    const uint32_t ph = ((nk / NS) - 1) & 1;
    if (nk >= NS && !mbar_wait(w, b.ke(st), ph)) return -1;
    load_k(st, kt);
    ++nk;
    if (nv >= NS && !mbar_wait(w, b.ve(st), ph)) return -1;
    load_v(st, kt);
    ++nv;
  }
  return kt;
}

// Every copy the producer issued must have landed before the CTA may exit.
template <int NS>
__device__ __forceinline__ void fwd_drain_copies(const WaitCtx& w, const FwdBars<NS>& b, int nk, int nv) {
  mbar_drain(w, b.q(), 0);
  for (int st = 0; st < NS; ++st) {
    const int ck = (nk - st + NS - 1) / NS, cv = (nv - st + NS - 1) / NS;  // copies into stage st
    if (ck > 0) mbar_drain(w, b.kf(st), (ck - 1) & 1);
    if (cv > 0) mbar_drain(w, b.vf(st), (cv - 1) & 1);
  }
}

// The MMA warp's schedule over the kept key tiles from kt on (the whole warp
// runs it converged, waits are warp-uniform, one elected lane issues each MMA
// and commit).  S_0 first; then for key tile j: with P~ in TMEM columns of its
// own (PSEP), S_{j+1} as soon as the softmax warps have copied S_j out, so that
// it is computed while their softmax of tile j runs; then P~ V_j once P~_j is
// in TMEM and V_j has landed; without PSEP (P~ written over S) S_{j+1} after
// P~ V_j -- MMAs of one thread execute in issue order, so it lands after P~ V_j
// has read P~.  issue_s(stage) issues the products of S = Q K_stage^T;
// issue_pv(stage, j) those of O += P~ V_stage (O overwritten when j = 0).  At the
// end every MMA issued must have completed before TMEM is released.
template <int NS, bool PSEP, class Next, class IssueS, class IssuePV>
__device__ __forceinline__ void fwd_mma_schedule(const WaitCtx& w, const FwdBars<NS>& b, int kt, int kt_end,
                                                 Next next, IssueS issue_s, IssuePV issue_pv) {
  auto s_tile = [&](int it) -> bool {
    const int st = it % NS;
    if (!warp_wait(w, b.kf(st), (it / NS) & 1)) return false;
    tc_fence_after();
    issue_s(st);
    tc_commit_elect(b.s());
    tc_commit_elect(b.ke(st));
    return true;
  };
  bool ok = warp_wait(w, b.q(), 0);
  if (ok && kt < kt_end) ok = s_tile(0);
  for (int it = 0; ok && kt < kt_end; ++it) {
    const int st = it % NS;
    const int kn = next(kt + 1);
    if (PSEP && kn < kt_end) {
      if (!(ok = warp_wait(w, b.sfree(), it & 1))) break;
      if (!(ok = s_tile(it + 1))) break;
    }
    if (!(ok = warp_wait(w, b.p(), it & 1))) break;
    if (!(ok = warp_wait(w, b.vf(st), (it / NS) & 1))) break;
    tc_fence_after();
    issue_pv(st, it);
    tc_commit_elect(b.o());
    tc_commit_elect(b.ve(st));
    if (!PSEP && kn < kt_end && !(ok = s_tile(it + 1))) break;
    kt = kn;
  }
  tc_commit_elect(b.fin());
  if ((threadIdx.x & 31) == 0) mbar_drain(w, b.fin(), 0);
  __syncwarp();
}

// Hides, in the scores of key tile kt held by query `row`'s thread, the keys
// past the end of the sequence and, on the causal diagonal tile, the keys after
// the query ("Le masquage causal").  Returns whether the tile hides any key
// (for every row of the tile, so the result is warp-uniform).
__device__ __forceinline__ bool mask_score_row(float (&s)[kTile], int kt, int qt, int row, int N,
                                               bool causal) {
  const int k0 = kt * kTile;
  const bool diag = causal && kt == qt;
  if (k0 + kTile <= N && !diag) return false;
  int lim = N - k0;
  if (diag) lim = min(lim, row - k0 + 1);
#pragma unroll
  for (int c = 0; c < kTile; ++c)
    if (c >= lim) s[c] = -INFINITY;
  return true;
}

// Maximum of the 16 scores s[16 j .. 16 j + 15] as one dependency chain of
// three-input maxima.
__device__ __forceinline__ float max16(const float (&s)[kTile], int j) {
  float m = fmax3(s[16 * j], s[16 * j + 1], s[16 * j + 2]);
#pragma unroll
  for (int c = 3; c + 1 < 16; c += 2) m = fmax3(m, s[16 * j + c], s[16 * j + c + 1]);
  return fmaxf(m, s[16 * j + 15]);
}

// The four packed partial sums of a row's P~ added up.
__device__ __forceinline__ float sum_packed4(const uint64_t (&acc)[4]) {
  float s0, s1, s2, s3, s4, s5, s6, s7;
  f2unpack(acc[0], s0, s1);
  f2unpack(acc[1], s2, s3);
  f2unpack(acc[2], s4, s5);
  f2unpack(acc[3], s6, s7);
  return ((s0 + s1) + (s2 + s3)) + ((s4 + s5) + (s6 + s7));
}

// This thread's O row in TMEM (D fp32 columns at tO) times f.
template <int D>
__device__ __forceinline__ void scale_o_row(uint32_t tO, float f) {
  const uint64_t fp = f2pack(f, f);
#pragma unroll
  for (int c0 = 0; c0 < D; c0 += 32) {
    uint32_t o[32];
    tmem_ld32(tO + c0, o);
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
      float y0, y1;
      f2unpack(fmul2(f2pack(__uint_as_float(o[i]), __uint_as_float(o[i + 1])), fp), y0, y1);
      o[i] = __float_as_uint(y0);
      o[i + 1] = __float_as_uint(y1);
    }
    tmem_st32(tO + c0, o);
  }
}

// This thread's O row (TMEM at tO; zeros when !have_o) times `mul`, stored as
// D 16-bit values at dst when `write`.  tcgen05.ld is .sync.aligned: every lane
// of the warp loads (have_o is warp-uniform); only the stores are predicated.
template <int D, bool F16>
__device__ __forceinline__ void store_o_row(uint32_t tO, bool have_o, float mul, bool write, uint16_t* dst) {
#pragma unroll
  for (int c0 = 0; c0 < D; c0 += 32) {
    uint32_t o[32];
    if (have_o) {
      tmem_ld32(tO + c0, o);
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) o[i] = 0u;
    }
    if (write) {
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        uint4 q;
        q.x = pack2<F16>(__uint_as_float(o[v * 8 + 0]) * mul, __uint_as_float(o[v * 8 + 1]) * mul);
        q.y = pack2<F16>(__uint_as_float(o[v * 8 + 2]) * mul, __uint_as_float(o[v * 8 + 3]) * mul);
        q.z = pack2<F16>(__uint_as_float(o[v * 8 + 4]) * mul, __uint_as_float(o[v * 8 + 5]) * mul);
        q.w = pack2<F16>(__uint_as_float(o[v * 8 + 6]) * mul, __uint_as_float(o[v * 8 + 7]) * mul);
        *reinterpret_cast<uint4*>(dst + c0 + v * 8) = q;
      }
    }
  }
}

}  // namespace fa
