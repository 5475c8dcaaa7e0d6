// fwd_persist.cu -- the attention forward as persistent CTAs that split the
// work evenly (bwd_sched.cuh's schedule, with query tiles as the units).
//
// The same tile computation as fwd_tc.cu ("L'algorithme Flash Attention",
// marketmaker.cc; "Método" of the FlashAttention reading guide): for every
// 128-row query tile Q_i, S = Q_i K_j^T, the running max and sum, P~ = exp(...)
// and O += P~ V_j over its key tiles, O / l and LSE = m + ln l at the end.
// Here each of G persistent CTAs (two per SM) takes an equal share of all the
// (query tile, key tile) iterations, numbered query tile by query tile
// (heaviest causal tiles first, keys in order), so the last wave is as full as
// the others.  A CTA's share may begin or end inside a query tile: it then
// writes that piece's normalised fp32 O and its LSE to a slot of its own, and
// a second kernel merges the pieces of each shared query tile with the
// statistics merge of "Rastreamento Incremental do Softmax" (the reading
// guide): LSE = log sum_s exp(LSE_s), O = sum_s exp(LSE_s - LSE) O_s.
//
// Warp roles (192 threads) as in fwd_tc.cu.  The producer walks the schedule:
// per piece it loads Q_i (once the previous piece's last S has read the old
// one) and stages the piece's coordinates next to it; the K_j, V_j ring runs
// on across pieces.  The softmax warps write a piece's result, then release O
// to the next piece's first P~ V.
#include "bwd_sched.cuh"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr int kTile = 128;          // query rows per piece = keys per K/V tile
constexpr float kRescaleThr = 8.f;  // move the running max only past 2^8

template <int D>
struct FwdLayout {
  static constexpr uint32_t TILE = kTile * D * 2;  // one 128-row 16-bit tile
  static constexpr int NS = (D == 64) ? 2 : 1;     // K/V ring depth
  // Q buffers: at d = 64 two, so that the next piece's Q_i loads while this
  // piece runs; at d = 128 one (two CTAs per SM leave no room)
  static constexpr int NQ = (D == 64) ? 2 : 1;
  static constexpr uint32_t Q = 0;                  // Q buffer b at Q + b * TILE
  static constexpr uint32_t K0 = Q + NQ * TILE;     // K stage s at K0 + s * TILE
  static constexpr uint32_t V0 = K0 + NS * TILE;    // V stage s at V0 + s * TILE
  static constexpr uint32_t INFO = V0 + NS * TILE;  // two PieceInfo entries (by piece parity)
  static constexpr uint32_t BAR = INFO + 64;
  // barriers: 0-1 q_full[2], 2 s_full, 3 p_full, 4 o_done, 5 fin, 6 s_free,
  //           7-8 q_free[2] (the piece's last S has read its Q buffer), 9 o_free
  //           (O read out), 10 info_ack (the softmax warps have read the piece's
  //           coordinates), 11.. k_full[NS], v_full[NS], k_empty[NS], v_empty[NS]
  static constexpr uint32_t NBAR = 11 + 4 * NS;
  static constexpr uint32_t TSLOT = BAR + NBAR * 8;
  static constexpr uint32_t ABORT = TSLOT + 4;
  static constexpr uint32_t BYTES = ABORT + 4;
  static constexpr uint32_t TMEM_COLS = 256;
  static constexpr bool PSEP = (D == 64);
  static constexpr uint32_t T_S = 0, T_O = 128, T_P = PSEP ? 192 : 0;
};

// A piece's coordinates {qt, bh, kt_first, kt_end} and {slot, more}.
constexpr int kMorePieces = 1;

// Out of line: called once per piece.
static __device__ __noinline__ bool next_piece(const Sched& sc, int c, long long& g, long long g_end,
                                               bool& first, Seg& sg) {
  return sched_next(sc, c, g, g_end, first, sg);
}

template <int D, bool F16>
__global__ void __launch_bounds__(192, 2)
    fwd_persist_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const FwdArgs a) {
  using L = FwdLayout<D>;
  constexpr int NS = L::NS;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sb = smem_addr(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int BH = a.B * a.H;
  const int n_tiles = (a.N + kTile - 1) / kTile;

  auto bar = [&](int i) { return sb + L::BAR + 8u * (uint32_t)i; };
  const uint32_t bar_s = bar(2), bar_p = bar(3), bar_o = bar(4), bar_fin = bar(5),
                 bar_sfree = bar(6), bar_ofree = bar(9), bar_iack = bar(10);
  // piece pc's Q buffer, its full / free barriers, and the phase of its use of them
  auto qbuf = [&](int pc) { return L::NQ == 2 ? (pc & 1) : 0; };
  auto bar_qf = [&](int pc) { return bar(qbuf(pc)); };
  auto bar_qfree = [&](int pc) { return bar(7 + qbuf(pc)); };
  auto qphase = [&](int pc) { return (uint32_t)((L::NQ == 2 ? pc >> 1 : pc) & 1); };
  auto bar_kf = [&](int s) { return bar(11 + s); };
  auto bar_vf = [&](int s) { return bar(11 + NS + s); };
  auto bar_ke = [&](int s) { return bar(11 + 2 * NS + s); };
  auto bar_ve = [&](int s) { return bar(11 + 3 * NS + s); };
  auto info_a = [&](int pc) { return *reinterpret_cast<const int4*>(smem + L::INFO + (pc & 1) * 32); };
  auto info_b = [&](int pc) { return *reinterpret_cast<const int2*>(smem + L::INFO + (pc & 1) * 32 + 16); };
  volatile int* abort_cta = reinterpret_cast<volatile int*>(smem + L::ABORT);
  const WaitCtx w{abort_cta, a.rep.st, a.rep.epoch, a.rep.wait_ns};

  if ((sb & 1023u) != 0) {  // the swizzled layouts need a 1024-byte aligned base
    if (threadIdx.x == 0) raise_error(w, FA_ERR_CUDA);
    return;
  }
  if (threadIdx.x == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(b), 1 + 1);  // q_full: the TMA transaction arrival + the coordinates
      mbar_init(bar(7 + b), 1);  // q_free
    }
    mbar_init(bar_s, 1);
    mbar_init(bar_p, 4);
    mbar_init(bar_o, 1);
    mbar_init(bar_fin, 1);
    mbar_init(bar_sfree, 4);
    mbar_init(bar_ofree, 4);
    mbar_init(bar_iack, 4);
    for (int s = 0; s < NS; ++s) {
      mbar_init(bar_kf(s), 1);
      mbar_init(bar_vf(s), 1);
      mbar_init(bar_ke(s), 1);
      mbar_init(bar_ve(s), 1);
    }
    *abort_cta = 0;
    fence_barrier_init();
  }
  if (warp == 5) {
    tmem_alloc(sb + L::TSLOT, L::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + L::TSLOT);

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
      const Sched sc = make_sched(n_tiles, BH, a.m.causal, a.G_fwd);
      long long g = sched_start(sc, (int)blockIdx.x);
      const long long g_stop = sched_start(sc, (int)blockIdx.x + 1);
      bool first = true;
      Seg sg;
      int nk = 0, nv = 0;  // K and V copies issued
      int pc = 0;          // pieces
      bool ok = true;
      bool live = next_piece(sc, (int)blockIdx.x, g, g_stop, first, sg);
      while (ok && live) {
        // the schedule's unit u = ukt * BH + bh is query tile n - 1 - ukt; its
        // visited "query tiles" are this query tile's key tiles, from 0
        const int qt = n_tiles - 1 - sg.kt, bh = sg.bh;
        const int qbase = a.m.causal ? sg.kt : 0;
        const int kt0 = sg.q_first - qbase, kt1 = sg.q_end - qbase;
        const int slot = sg.slot;
        Seg nxt;
        const bool more = next_piece(sc, (int)blockIdx.x, g, g_stop, first, nxt);
        // Q_i into its buffer, once the last S of the piece that used the buffer
        // before has read it, and once the softmax warps have taken the previous
        // piece's coordinates (so that no Q barrier runs two phases ahead of them)
        const int prev = pc - L::NQ;  // the piece that used this Q buffer before
        if (prev >= 0 && !(ok = mbar_wait(w, bar_qfree(prev), qphase(prev)))) break;
        if (pc > 0 && !(ok = mbar_wait(w, bar_iack, (pc - 1) & 1))) break;
        *reinterpret_cast<int4*>(smem + L::INFO + (pc & 1) * 32) = make_int4(qt, bh, kt0, kt1);
        *reinterpret_cast<int2*>(smem + L::INFO + (pc & 1) * 32 + 16) = make_int2(slot, more ? kMorePieces : 0);
        mbar_arrive(bar_qf(pc));
        mbar_arrive_expect_tx(bar_qf(pc), L::TILE);
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(sb + L::Q + qbuf(pc) * L::TILE + c * (kTile * 128), &tmQ, bar_qf(pc), c * 64,
                      qt * kTile, bh);
        for (int kt = kt0; kt < kt1; ++kt) {
          const int s = nk % NS;
          const uint32_t ph = ((nk / NS) - 1) & 1;
          if (nk >= NS && !(ok = mbar_wait(w, bar_ke(s), ph))) break;
          mbar_arrive_expect_tx(bar_kf(s), L::TILE);
          for (int c = 0; c < D / 64; ++c)
            tma_load_3d(sb + L::K0 + s * L::TILE + c * (kTile * 128), &tmK, bar_kf(s), c * 64,
                        kt * kTile, bh);
          ++nk;
          if (nv >= NS && !(ok = mbar_wait(w, bar_ve(s), ph))) break;
          mbar_arrive_expect_tx(bar_vf(s), L::TILE);
          for (int c = 0; c < D / 64; ++c)
            tma_load_3d(sb + L::V0 + s * L::TILE + c * (kTile * 128), &tmV, bar_vf(s), c * 64,
                        kt * kTile, bh);
          ++nv;
        }
        ++pc;
        sg = nxt;
        live = more;
      }
      // every copy issued must have landed before the CTA may exit
      for (int p = pc - 1; p >= 0 && p >= pc - L::NQ; --p) mbar_drain(w, bar_qf(p), qphase(p));
      for (int s = 0; s < NS; ++s) {
        const int ck = (nk - s + NS - 1) / NS, cv = (nv - s + NS - 1) / NS;  // copies into stage s
        if (ck > 0) mbar_drain(w, bar_kf(s), (ck - 1) & 1);
        if (cv > 0) mbar_drain(w, bar_vf(s), (cv - 1) & 1);
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t idS = idesc_f16(F16, kTile, kTile, false, false);
    constexpr uint32_t idO = idesc_f16(F16, kTile, D, false, true);
    const uint32_t tS = tmem + L::T_S, tO = tmem + L::T_O;
    const uint64_t dQ0 = desc_kmajor_base(sb + L::Q);
    const uint64_t dK0 = desc_kmajor_base(sb + L::K0);
    const uint64_t dV0 = desc_mnmajor_base(sb + L::V0, kTile);
    uint64_t dQ = dQ0;  // the current piece's Q buffer
    auto issue_s = [&](int it) -> bool {
      const int s = it % NS;
      if (!warp_wait(w, bar_kf(s), (it / NS) & 1)) return false;
      tc_fence_after();
      const uint64_t dK = desc_add(dK0, (uint32_t)s * L::TILE);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        tc_mma_ss_elect(tS, dQ + kmajor_step(kk, kTile), dK + kmajor_step(kk, kTile), idS,
                        kk > 0 ? 1u : 0u);
      tc_commit_elect(bar_s);
      tc_commit_elect(bar_ke(s));
      return true;
    };
    bool ok = true;
    int it = 0, pc = 0;
    for (bool more = true; ok && more; ++pc) {
      if (!(ok = warp_wait(w, bar_qf(pc), qphase(pc)))) break;
      const int4 ia = info_a(pc);
      const int2 ib = info_b(pc);
      const int n = ia.w - ia.z;  // key tiles of the piece (at least one)
      dQ = desc_add(dQ0, (uint32_t)qbuf(pc) * L::TILE);
      more = ib.y & kMorePieces;
      // the piece's first S; at d = 64 it goes into columns the softmax may still
      // be reading the previous piece's last S from (at d = 128 it follows that
      // tile's P~ V in issue order, which follows the read)
      if (L::PSEP && it > 0 && !(ok = warp_wait(w, bar_sfree, (it - 1) & 1))) break;
      if (!(ok = issue_s(it))) break;
      if (n == 1) tc_commit_elect(bar_qfree(pc));  // the piece's only S has been issued
      for (int i = 0; ok && i < n; ++i, ++it) {
        const int s = it % NS;
        // d = 64: S_{j+1} as soon as the softmax has copied S_j out of TMEM
        if (L::PSEP && i + 1 < n) {
          if (!(ok = warp_wait(w, bar_sfree, it & 1))) break;
          if (!(ok = issue_s(it + 1))) break;
          if (i + 2 == n) tc_commit_elect(bar_qfree(pc));  // the piece's last S
        }
        // P~ V_j, with P~ read from TMEM; the piece's first overwrites O, once
        // the previous piece's result has been read out of it
        if (!(ok = warp_wait(w, bar_p, it & 1))) break;
        if (!(ok = warp_wait(w, bar_vf(s), (it / NS) & 1))) break;
        if (i == 0 && pc > 0 && !(ok = warp_wait(w, bar_ofree, (pc - 1) & 1))) break;
        tc_fence_after();
        const uint64_t dV = desc_add(dV0, (uint32_t)s * L::TILE);
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk)
          tc_mma_ts_elect(tO, tmem + L::T_P + (uint32_t)kk * 8u, dV + mnmajor_step(kk), idO,
                          (i > 0 || kk > 0) ? 1u : 0u);
        tc_commit_elect(bar_o);
        tc_commit_elect(bar_ve(s));
        // d = 128: the next score tile goes into the columns P~ V_j reads; MMAs
        // of one thread execute in issue order, so it lands after they are read
        if (!L::PSEP && i + 1 < n) {
          if (!(ok = issue_s(it + 1))) break;
          if (i + 2 == n) tc_commit_elect(bar_qfree(pc));
        }
      }
    }
    // every MMA issued must have completed before TMEM is released
    tc_commit_elect(bar_fin);
    if (lane == 0) mbar_drain(w, bar_fin, 0);
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    const int r = threadIdx.x;  // query row in the tile = TMEM lane
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const uint32_t tS = tmem + L::T_S + lane_off, tO = tmem + L::T_O + lane_off;
    const float c2 = a.scale_log2;
    bool ok = true;
    int it = 0, pc = 0;
    for (bool more = true; ok && more; ++pc) {
      if (!(ok = warp_wait(w, bar_qf(pc), qphase(pc)))) break;
      const int4 ia = info_a(pc);
      const int2 ib = info_b(pc);
      const int qt = ia.x, bh = ia.y, kt0 = ia.z, kt1 = ia.w, slot = ib.x;
      more = ib.y & kMorePieces;
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_iack);
      const int row = qt * kTile + r;
      float m_use = -INFINITY;  // running max in use (exp2 domain)
      float l = 0.f;            // running sum of P~ (fp32)
      int i = 0;
      for (int kt = kt0; kt < kt1; ++kt, ++it, ++i) {
        // d = 128: S_j is complete, and so is every earlier MMA (P~ V_{j-1}
        // included), so O is stable and P~_{j-1} has been consumed.  d = 64 waits
        // for P~ V_{j-1} separately below.
        if (!(ok = warp_wait(w, bar_s, it & 1))) break;
        tc_fence_after();
        float s[kTile];
        {
          uint32_t u[64];
          tmem_ld64(tS, u);
  #pragma unroll
          for (int c = 0; c < 64; ++c) s[c] = __uint_as_float(u[c]);
          tmem_ld64(tS + 64, u);
  #pragma unroll
          for (int c = 0; c < 64; ++c) s[64 + c] = __uint_as_float(u[c]);
        }
        if (L::PSEP) {  // S_j is in registers: the MMA warp may compute S_{j+1}
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_sfree);
        }
        // hide keys past the end of the sequence and, on the diagonal tile,
        // keys after the query ("Le masquage causal")
        const int k0 = kt * kTile;
        if (k0 + kTile > a.N || (a.m.causal && kt == qt)) {
          int lim = a.N - k0;
          if (a.m.causal && kt == qt) lim = min(lim, row - k0 + 1);
  #pragma unroll
          for (int c = 0; c < kTile; ++c)
            if (c >= lim) s[c] = -INFINITY;
        }
        // row max as four independent chains (a single chain of dependent maxes
        // would expose its latency: only two softmax warps share a sub-partition)
        float m4[4];
  #pragma unroll
        for (int j = 0; j < 4; ++j) {
          float mj = fmax3(s[32 * j], s[32 * j + 1], s[32 * j + 2]);
  #pragma unroll
          for (int c = 3; c + 1 < 32; c += 2) mj = fmax3(mj, s[32 * j + c], s[32 * j + c + 1]);
          m4[j] = fmaxf(mj, s[32 * j + 31]);
        }
        const float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
        const float m_tile = mx * c2;
        float alpha = 1.f;
        if (m_tile > m_use + kRescaleThr) {
          alpha = ex2(m_use - m_tile);  // 0 on the first tile that sees a key
          m_use = m_tile;
        }
        const float mneg = (m_use == -INFINITY) ? 0.f : -m_use;
        const uint64_t c2p = f2pack(c2, c2), mp = f2pack(mneg, mneg);
        uint64_t acc[4] = {f2pack(0.f, 0.f), f2pack(0.f, 0.f), f2pack(0.f, 0.f), f2pack(0.f, 0.f)};
        uint32_t plo[32], phi[32];  // P~ as 16-bit pairs: keys [0, 64) and [64, 128)
  #pragma unroll
        for (int c = 0; c < kTile; c += 2) {
          float x0, x1;
          f2unpack(ffma2(f2pack(s[c], s[c + 1]), c2p, mp), x0, x1);
          const float p0 = ex2(x0), p1 = ex2(x1);
          acc[(c >> 1) & 3] = fadd2(acc[(c >> 1) & 3], f2pack(p0, p1));  // four independent sums
          if (c < 64)
            plo[c / 2] = pack2<F16>(p0, p1);
          else
            phi[(c - 64) / 2] = pack2<F16>(p0, p1);
        }
        float sum0, sum1, sum2, sum3, sum4, sum5, sum6, sum7;
        f2unpack(acc[0], sum0, sum1);
        f2unpack(acc[1], sum2, sum3);
        f2unpack(acc[2], sum4, sum5);
        f2unpack(acc[3], sum6, sum7);
        l = l * alpha + (((sum0 + sum1) + (sum2 + sum3)) + ((sum4 + sum5) + (sum6 + sum7)));
        if (L::PSEP && it > 0) {
          // P~ V_{j-1} must be done: it reads the P~ columns and writes O
          if (!(ok = warp_wait(w, bar_o, (it - 1) & 1))) break;
          tc_fence_after();
        }
        // P~ (16-bit pairs); at d = 128 over the first 64 columns of S, all of
        // which is already in registers
        tmem_st32(tmem + L::T_P + lane_off, plo);
        tmem_st32(tmem + L::T_P + lane_off + 32, phi);
        if (i > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
          const uint64_t ap = f2pack(alpha, alpha);
  #pragma unroll
          for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t o[32];
            tmem_ld32(tO + c0, o);
  #pragma unroll
            for (int i = 0; i < 32; i += 2) {
              float y0, y1;
              f2unpack(fmul2(f2pack(__uint_as_float(o[i]), __uint_as_float(o[i + 1])), ap), y0, y1);
              o[i] = __float_as_uint(y0);
              o[i + 1] = __float_as_uint(y1);
            }
            tmem_st32(tO + c0, o);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_p);
      }
      if (!ok) break;
      // ---------------------------------------------------------- the piece's result
      ok = warp_wait(w, bar_o, (it - 1) & 1);  // its last P~ V
      tc_fence_after();
      if (!ok) break;
      const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
      const float lse = (l > 0.f) ? (m_use + __log2f(l)) * 0.693147180559945309f : -INFINITY;
      if (slot < 0) {
        if (row < a.N) a.LSE[(size_t)bh * a.N + row] = lse;
        uint16_t* Orow = reinterpret_cast<uint16_t*>(a.O) + ((size_t)bh * a.N + row) * D;
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t o[32];
          tmem_ld32(tO + c0, o);
          if (row < a.N) {
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              uint4 q;
              q.x = pack2<F16>(__uint_as_float(o[v * 8 + 0]) * inv_l, __uint_as_float(o[v * 8 + 1]) * inv_l);
              q.y = pack2<F16>(__uint_as_float(o[v * 8 + 2]) * inv_l, __uint_as_float(o[v * 8 + 3]) * inv_l);
              q.z = pack2<F16>(__uint_as_float(o[v * 8 + 4]) * inv_l, __uint_as_float(o[v * 8 + 5]) * inv_l);
              q.w = pack2<F16>(__uint_as_float(o[v * 8 + 6]) * inv_l, __uint_as_float(o[v * 8 + 7]) * inv_l);
              *reinterpret_cast<uint4*>(Orow + c0 + v * 8) = q;
            }
          }
        }
      } else {
        // a piece of a query tile that other CTAs share: its normalised fp32 O
        // and its LSE into this CTA's slot, [O rows 0..127 | LSE 0..127]
        float* sl = a.Opart + (size_t)slot * (kTile * D + kTile);
        sl[kTile * D + r] = lse;
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t o[32];
          tmem_ld32(tO + c0, o);
#pragma unroll
          for (int v = 0; v < 8; ++v)
            *reinterpret_cast<float4*>(sl + (size_t)r * D + c0 + v * 4) =
                make_float4(__uint_as_float(o[v * 4 + 0]) * inv_l, __uint_as_float(o[v * 4 + 1]) * inv_l,
                            __uint_as_float(o[v * 4 + 2]) * inv_l, __uint_as_float(o[v * 4 + 3]) * inv_l);
        }
      }
      // O has been read: the next piece's first P~ V may overwrite it
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_ofree);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, L::TMEM_COLS);
  }
}

// One block per CTA boundary of the persistent forward: if a query tile is
// shared there (sched_shared), merge its pieces' slots row by row (thread =
// row) and write its O and LSE.
template <int D, bool F16>
__global__ void __launch_bounds__(128) fwd_persist_merge_kernel(const FwdArgs a) {
  const int BH = a.B * a.H;
  const int n_tiles = (a.N + kTile - 1) / kTile;
  const Sched s = make_sched(n_tiles, BH, a.m.causal, a.G_fwd);
  int bh, ukt, c_last, fs;
  const int c = (int)blockIdx.x;
  if (!sched_shared(s, c, bh, ukt, c_last, fs)) return;
  const int qt = n_tiles - 1 - ukt;
  const int r = (int)threadIdx.x;
  const int row = qt * kTile + r;
  if (row >= a.N) return;
  constexpr size_t STRIDE = (size_t)kTile * D + kTile;
  auto slot_of = [&](int cc) { return cc == c ? fs : 2 * cc; };
  float m = -INFINITY;
  for (int cc = c; cc <= c_last; ++cc) m = fmaxf(m, a.Opart[(size_t)slot_of(cc) * STRIDE + kTile * D + r]);
  float acc[D];
#pragma unroll
  for (int k = 0; k < D; ++k) acc[k] = 0.f;
  float sum = 0.f;
  if (m != -INFINITY) {
    for (int cc = c; cc <= c_last; ++cc) {
      const float* sl = a.Opart + (size_t)slot_of(cc) * STRIDE;
      const float wgt = ex2((sl[kTile * D + r] - m) * 1.4426950408889634f);  // 0 for an empty piece
      sum += wgt;
#pragma unroll
      for (int k = 0; k < D; k += 4) {
        const float4 v = *reinterpret_cast<const float4*>(sl + (size_t)r * D + k);
        acc[k] = fmaf(wgt, v.x, acc[k]);
        acc[k + 1] = fmaf(wgt, v.y, acc[k + 1]);
        acc[k + 2] = fmaf(wgt, v.z, acc[k + 2]);
        acc[k + 3] = fmaf(wgt, v.w, acc[k + 3]);
      }
    }
  }
  const float inv = sum > 0.f ? 1.f / sum : 0.f;
  uint16_t* dst = reinterpret_cast<uint16_t*>(a.O) + ((size_t)bh * a.N + row) * D;
#pragma unroll
  for (int k = 0; k < D; k += 8) {
    uint4 q;
    q.x = pack2<F16>(acc[k] * inv, acc[k + 1] * inv);
    q.y = pack2<F16>(acc[k + 2] * inv, acc[k + 3] * inv);
    q.z = pack2<F16>(acc[k + 4] * inv, acc[k + 5] * inv);
    q.w = pack2<F16>(acc[k + 6] * inv, acc[k + 7] * inv);
    *reinterpret_cast<uint4*>(dst + k) = q;
  }
  a.LSE[(size_t)bh * a.N + row] = sum > 0.f ? m + __logf(sum) : -INFINITY;
}

template <int D, bool F16>
cudaError_t launch_t(const FwdArgs& a, const CUtensorMap* tm, cudaStream_t s) {
  using L = FwdLayout<D>;
  auto kern = fwd_persist_kernel<D, F16>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::BYTES);
  if (e != cudaSuccess) return e;
  kern<<<(unsigned)a.G_fwd, 192, L::BYTES, s>>>(tm[0], tm[1], tm[2], a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (a.G_fwd > 1) fwd_persist_merge_kernel<D, F16><<<(unsigned)(a.G_fwd - 1), kTile, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_persist(const FwdArgs& a, int d, bool f16, const CUtensorMap* tm, cudaStream_t s) {
  if (d == 64) return f16 ? launch_t<64, true>(a, tm, s) : launch_t<64, false>(a, tm, s);
  return f16 ? launch_t<128, true>(a, tm, s) : launch_t<128, false>(a, tm, s);
}

}  // namespace fa
