// bwd_tc.cu -- attention backward main kernel on the 5th-generation tensor cores.
//
// The backward pass keeps only O and the per-row statistic from the forward
// pass and recomputes the scores and probabilities tile by tile ("Passe
// arrière : recalculer au lieu de stocker", marketmaker.cc; "Recomputação no
// Backward Pass", FlashAttention reading guide).  One CTA owns one 128-key
// tile (K_j, V_j) of one (batch, head), keeps it in shared memory, accumulates
// dK_j and dV_j in TMEM, and walks the 128-query tiles i that the causal rule
// and the block mask leave:
//   S^T  = K_j Q_i^T                    (tcgen05, TMEM)
//   P^T  = exp(scale * S^T - LSE_i)      (CUDA cores; thread = key row)
//   dP^T = V_j dO_i^T                    (tcgen05, TMEM)
//   dV  += P^T dO_i                      (tcgen05, P^T read from TMEM)
//   dS^T = P^T * (dP^T - D_i)            (CUDA cores)
//   dK  += dS^T Q_i                      (tcgen05)
//   dQ_i = dS K_j                        (tcgen05, read back, staged in shared
//                                         memory and added to the fp32
//                                         accumulator by a TMA reduce-add)
// The score scale is applied once at the end: dK = scale * sum dS^T Q here,
// dQ = scale * accumulator in the finalize kernel.
//
// Warp roles (32 (4 NG + 2 + NQW) threads): warps 0 .. 4 NG - 1 form NG compute
// warpgroups that split the 128 query columns of every tile into NG groups of
// 128 / NG (TMEM lane = key row; warp w reads the lanes of quadrant w mod 4);
// warp 4 NG is the producer (TMA copies of K_j, V_j once and of Q_i, dO_i
// through a ring, plus each query tile's LSE and D staged by its lanes); warp
// 4 NG + 1 owns TMEM and issues the MMAs; at d = 64, warps 4 NG + 2 .. 4 NG + 5
// read dQ_i out of TMEM and reduce it into the fp32 accumulator.  More compute warps per SM
// sub-partition hide more of the TMEM, shared-memory and barrier latencies of
// the elementwise steps, which (with one CTA per SM) bound the loop.
//
// Grids that would leave SMs idle run the same kernel on slices of key tiles'
// query ranges (a separate instantiation, QS; bwd_sched.cuh): a key tile of
// several slices gets fp32 partial dK, dV sums that the finalize kernel adds up.
#include "bwd_sched.cuh"
#include "ptx.cuh"
#include "tiles.cuh"

namespace fa {
namespace {


template <int D, int NG>
struct BwdLayout {
  static_assert(NG == 2 || NG == 4, "compute warpgroups");
  static_assert(D == 64 || NG == 2, "at d = 128 the dQ staging aliases dS^T per warp only with NG = 2");
  static constexpr int CW = kTile / NG;   // query columns per compute warpgroup
  static constexpr int KPG = CW / 16;     // MMA K steps (16 queries) per warpgroup
  static constexpr int NCW = 4 * NG;      // compute warps
  // d = 64: four dQ warps of their own (one per TMEM quadrant) read dQ_i out of
  // TMEM, stage it and issue its reduce-add, off the compute warps' critical
  // path; at d = 128 the compute warps do it (the staging shares dS^T there)
  static constexpr bool QW = (D == 64);
  static constexpr int NQW = QW ? 4 : 0;
  static constexpr int NT = 32 * (NCW + 2 + NQW);
  // dQ read-out: boxes of 32 query rows x DQC fp32 columns (128-byte rows with
  // the 128-byte swizzle when DQC = 32, 64-byte rows with the 64-byte swizzle
  // when DQC = 16) for the TMA reduce-add; a dQ warp stages the D columns of
  // its 32 rows through one box, D / DQC rounds, else each compute warp its
  // group's DQG columns
  static constexpr int DQG = D / NG;      // dQ columns per warpgroup
  static constexpr int DQC = (QW || NG == 2) ? 32 : 16;
  static constexpr uint32_t BOXB = 32u * DQC * 4u;
  static constexpr int DQ_READERS = QW ? NQW : NCW;  // arrivals on dq_free
  static constexpr uint32_t TILE = kTile * D * 2;
  static constexpr int NS = (D == 64) ? 3 : 2;         // Q/dO ring depth
  static constexpr uint32_t K = 0;
  static constexpr uint32_t V = TILE;
  static constexpr uint32_t QS = 2 * TILE;             // stage s: Q at QS + 2s TILE, dO after it
  // dS^T, 128 x 128 16-bit: at d = 64 two buffers, so that the compute warps
  // write dS_{i+1} while the dK_i and dQ_i MMAs still read dS_i; at d = 128 one
  static constexpr int NDS = (D == 64) ? 2 : 1;
  static constexpr uint32_t DSB = kTile * kTile * 2;    // bytes of one dS^T buffer
  static constexpr uint32_t DST = QS + NS * 2 * TILE;  // dS^T buffer b at DST + b DSB
  // per ring stage, the query tile's row statistics: [128] LSE*log2e then [128] D
  static constexpr uint32_t STAT = DST + NDS * DSB;
  // dQ staging: at d = 64 a buffer of its own, one 32 x 32 fp32 box per dQ warp
  // (16 KiB; each warp stages its 64 columns in two rounds); at d = 128 shared
  // memory is full and the dS^T buffer doubles as staging, one box per compute
  // warp
  static constexpr bool STG_SEP = (D == 64);
  static constexpr uint32_t STG_BYTES = QW ? NQW * BOXB : NCW * BOXB;
  static constexpr uint32_t STG = STG_SEP ? STAT + NS * 256 * 4 : DST;
  static_assert(STG_SEP || STG_BYTES == DSB, "staging size");
  static constexpr uint32_t BAR = STAT + NS * 256 * 4 + (STG_SEP ? STG_BYTES : 0);
  // barriers: 0 kv_full, 1 s_full, 2 dp_full, 3 dp_free, 4 p_full, 5 ds_full,
  //           6 dq_full, 7 dq_free, 8 done, 9 pt_free (d = 64: dV_i has finished
  //           reading P^T_i), 10.. q_full[NS], 10+NS.. q_empty[NS],
  //           10+2NS.. ds_free[NDS]
  static constexpr uint32_t NBAR = 10 + 2 * NS + NDS;
  static constexpr uint32_t TSLOT = BAR + NBAR * 8;
  static constexpr uint32_t ABORT = TSLOT + 4;
  static constexpr uint32_t QBITS = ABORT + 4;  // the query tiles that see this key tile (block mask)
  static constexpr uint32_t BYTES = QBITS + kMaskBitBytes;
  static_assert(BYTES <= 232448, "shared memory per CTA");
  static constexpr uint32_t TMEM_COLS = 512;
  // TMEM columns.  S^T [0,128) (warpgroup g reads [CW g, CW g + CW)), dP^T
  // [128,256), dV and dK d columns each.  At d = 64, dQ [384,448) and the 16-bit
  // P^T [448,512) have columns of their own; at d = 128 the 512 columns are
  // full, so dQ goes over dP^T and warpgroup g writes its P^T over the first
  // CW / 2 of its own S^T columns (which it has read by then).
  static constexpr uint32_t T_S = 0, T_DP = 128, T_DV = 256, T_DK = 256 + D;
  static constexpr bool ALIAS = (D == 128);
  static constexpr uint32_t T_DQ = ALIAS ? T_DP : 384;
  static constexpr uint32_t T_PT = ALIAS ? T_S : 448;
  // first of the 8 P^T columns that hold queries 16 kk .. 16 kk + 15 (as
  // 16-bit pairs), and the first of the CW / 2 columns warpgroup g writes
  __device__ static constexpr uint32_t pt_col(int kk) {
    return ALIAS ? (uint32_t)CW * (uint32_t)(kk / KPG) + 8u * (uint32_t)(kk % KPG)
                 : T_PT + 8u * (uint32_t)kk;
  }
  __device__ static constexpr uint32_t pt_write_col(int g) {
    return ALIAS ? (uint32_t)CW * (uint32_t)g : T_PT + (uint32_t)(CW / 2) * (uint32_t)g;
  }
};




template <int D, bool F16, int NG, bool DROP, bool QS, bool MASKED>
__global__ void __launch_bounds__(BwdLayout<D, NG>::NT, 1)
    bwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                  const __grid_constant__ CUtensorMap tmdQ, const BwdArgs a) {
  using L = BwdLayout<D, NG>;
  constexpr int NS = L::NS;
  constexpr int kProd = L::NCW, kMma = L::NCW + 1;  // producer and MMA warps
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sb = smem_addr(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int BH = a.B * a.H;
  const int n_tiles = (a.N + kTile - 1) / kTile;
  // this CTA's key tile kt of head bh and its query tiles [qt_begin, q_end)
  int kt, bh, qt_begin, q_end, slot = -1;
  if (QS && (int)blockIdx.x >= a.qs_from) {
    // a sliced launch (QS) from unit qs_from on: one slice of a key tile's
    // visited query tiles; slot >= 0 when the key tile has several slices
    const Slice sl = slice_locate((int)blockIdx.x - a.qs_from, n_tiles, BH, a.m.causal, a.q_slice,
                                  a.qs_from);
    kt = sl.kt;
    bh = sl.bh;
    qt_begin = sl.q_first;
    q_end = sl.q_end;
    slot = sl.slot;
  } else {
    // a whole key tile.  causal: low key tiles see the most queries, so they go
    // first, within groups of head_group heads (a sliced launch keeps the
    // key-tile-major unit numbering of its slices: one group)
    group_order((int)blockIdx.x, n_tiles, BH, QS ? BH : a.head_group, QS ? 0 : a.head_tail, kt, bh);
    qt_begin = a.m.causal ? kt : 0;
    q_end = n_tiles;
  }
  const int b = bh / a.H, h = bh % a.H;

  auto bar = [&](int i) { return sb + L::BAR + 8u * (uint32_t)i; };
  const uint32_t bar_kv = bar(0), bar_s_full = bar(1), bar_dp_full = bar(2), bar_dp_free = bar(3),
                 bar_p_full = bar(4), bar_ds_full = bar(5), bar_dq_full = bar(6), bar_dq_free = bar(7),
                 bar_done = bar(8), bar_pt_free = bar(9);
  auto bar_qf = [&](int s) { return bar(10 + s); };
  auto bar_qe = [&](int s) { return bar(10 + NS + s); };
  auto bar_ds_free = [&](int b) { return bar(10 + 2 * NS + b); };

  volatile int* abort_cta = reinterpret_cast<volatile int*>(smem + L::ABORT);
  const WaitCtx w{abort_cta, a.rep.st, a.rep.epoch, a.rep.wait_ns};

  if ((sb & 1023u) != 0) {
    if (threadIdx.x == 0) raise_error(w, FA_ERR_CUDA);
    return;
  }
  // debug build: the CTA's key tile, head and query range lie inside the problem
  if (!dbg_check(w, kt >= 0 && kt < n_tiles && bh >= 0 && bh < BH && qt_begin >= 0 &&
                        q_end <= n_tiles && (int)blockIdx.x < a.direct))
    return;
  // The producer lane sets up the barriers and, before the block-wide setup
  // barrier, already issues the copies that need no wait (K_j, V_j and the
  // first NS query tiles' Q, dO), so that their latency overlaps the TMEM
  // allocation.  The statistics of those stages are staged after the barrier.
  const bool producer = (warp == kProd && lane == 0);
  int pre = 0;  // producer lane: query-tile stages already being copied
  if (producer) {
    mbar_init(bar_kv, 1);
    mbar_init(bar_s_full, 1);
    mbar_init(bar_dp_full, 1);
    mbar_init(bar_dp_free, L::NCW);
    mbar_init(bar_p_full, L::NCW);
    mbar_init(bar_ds_full, L::NCW);
    for (int b2 = 0; b2 < L::NDS; ++b2) mbar_init(bar_ds_free(b2), 1);
    mbar_init(bar_dq_full, 1);
    mbar_init(bar_dq_free, L::DQ_READERS);
    mbar_init(bar_done, 1);
    mbar_init(bar_pt_free, 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(bar_qf(s), 1 + 32);  // the TMA transaction arrival + every producer lane
      mbar_init(bar_qe(s), 1);
    }
    *abort_cta = 0;
    fence_barrier_init();
    prefetch_tmap(&tmQ);
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
    prefetch_tmap(&tmdO);
    mbar_arrive_expect_tx(bar_kv, 2 * L::TILE);
    for (int c = 0; c < D / 64; ++c) {
      tma_load_3d(sb + L::K + c * (kTile * 128), &tmK, bar_kv, c * 64, kt * kTile, bh);
      tma_load_3d(sb + L::V + c * (kTile * 128), &tmV, bar_kv, c * 64, kt * kTile, bh);
    }
    for (int qt = next_q(a.m, b, h, qt_begin, kt, q_end); qt < q_end && pre < NS;
         qt = next_q(a.m, b, h, qt + 1, kt, q_end), ++pre) {
      if (!dbg_check(w, qt * kTile < a.N)) break;
      const uint32_t dst = sb + L::QS + (uint32_t)pre * 2u * L::TILE;
      mbar_arrive_expect_tx(bar_qf(pre), 2 * L::TILE);
      for (int c = 0; c < D / 64; ++c) {
        tma_load_3d(dst + c * (kTile * 128), &tmQ, bar_qf(pre), c * 64, qt * kTile, bh);
        tma_load_3d(dst + L::TILE + c * (kTile * 128), &tmdO, bar_qf(pre), c * 64, qt * kTile, bh);
      }
    }
  }
  // block mask (its own instantiation, MASKED, so that launches without one run
  // unchanged code): the column of query tiles that see this key tile, as bits in
  // shared memory
  uint32_t* qbits = reinterpret_cast<uint32_t*>(smem + L::QBITS);
  const bool use_bits = MASKED && n_tiles <= kMaskBits;
  if (use_bits)
    build_tile_bits(qbits, n_tiles, warp, L::NT / 32, lane, [&](int t) { return tile_kept(a.m, b, h, t, kt); });
  if (warp == kMma) {
    tmem_alloc(sb + L::TSLOT, L::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  // the next query tile at or after qt that sees this key tile (after the setup barrier)
  auto next_qt = [&](int qt) {
    return use_bits ? next_bit(qbits, qt, q_end) : next_q(a.m, b, h, qt, kt, q_end);
  };
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + L::TSLOT);

  if (warp == kProd) {
    // ------------------------------------------------------------ producer
    // Lane 0 issues the TMA copies; every lane also stages four rows of the
    // query tile's statistics into the ring stage, so that the stage's full
    // barrier covers Q, dO and the statistics together.
    pre = __shfl_sync(0xffffffffu, pre, 0);
    int it = 0;
    for (int qt = next_qt(qt_begin); qt < q_end;
         qt = next_qt(qt + 1)) {
      const int s = it % NS;
      // the tile's statistics, negated as the compute warps use them (-LSE*log2(e)
      // and -D), loaded before waiting for the stage to be free, so that their
      // global-memory latency overlaps that wait
      float4 l4, d4;
      l4.x = -lse2_of(a, bh, qt * kTile + lane * 4 + 0);
      l4.y = -lse2_of(a, bh, qt * kTile + lane * 4 + 1);
      l4.z = -lse2_of(a, bh, qt * kTile + lane * 4 + 2);
      l4.w = -lse2_of(a, bh, qt * kTile + lane * 4 + 3);
      d4.x = -d_of(a, bh, qt * kTile + lane * 4 + 0);
      d4.y = -d_of(a, bh, qt * kTile + lane * 4 + 1);
      d4.z = -d_of(a, bh, qt * kTile + lane * 4 + 2);
      d4.w = -d_of(a, bh, qt * kTile + lane * 4 + 3);
      if (it >= NS && !warp_wait(w, bar_qe(s), ((it / NS) - 1) & 1)) break;
      if (!__all_sync(0xffffffffu, dbg_check(w, qt >= 0 && qt * kTile < a.N))) break;
      if (lane == 0 && it >= pre) {
        const uint32_t dst = sb + L::QS + (uint32_t)s * 2u * L::TILE;
        mbar_arrive_expect_tx(bar_qf(s), 2 * L::TILE);
        for (int c = 0; c < D / 64; ++c) {
          tma_load_3d(dst + c * (kTile * 128), &tmQ, bar_qf(s), c * 64, qt * kTile, bh);
          tma_load_3d(dst + L::TILE + c * (kTile * 128), &tmdO, bar_qf(s), c * 64, qt * kTile, bh);
        }
      }
      float* st = reinterpret_cast<float*>(smem + L::STAT) + s * 256;
      reinterpret_cast<float4*>(st)[lane] = l4;
      reinterpret_cast<float4*>(st + 128)[lane] = d4;
      mbar_arrive(bar_qf(s));
      ++it;
    }
    if (lane == 0) {
      mbar_drain(w, bar_kv, 0);
      const int issued = it > pre ? it : pre;  // stages copied (some before the loop)
      for (int s = 0; s < NS; ++s) {
        const int n = (issued - s + NS - 1) / NS;  // loads issued into stage s
        if (n > 0) mbar_drain(w, bar_qf(s), (n - 1) & 1);
      }
    }
  } else if (warp == kMma) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs this loop converged (waits are warp-uniform); one
    // elected lane issues each MMA and commit.
    // Per query tile i (the next tile's Q/dO sit in another ring stage):
    //   d = 64:  S^T_{i+1}, dV_i, dP^T_{i+1}, then dQ_i, dK_i
    //   d = 128: dV_i, S^T_{i+1} (over P^T), then dQ_i, dK_i, dP^T_{i+1} (over dQ_i)
    // so the next score tile is computed while the compute warps form dS_i, and
    // dQ_i is ready for them right after the next tile's exponentials.
    {
      constexpr uint32_t idS = idesc_f16(F16, kTile, kTile, false, false);  // K-major x K-major
      constexpr uint32_t idKV = idesc_f16(F16, kTile, D, false, true);      // K-major x MN-major
      constexpr uint32_t idQ = idesc_f16(F16, kTile, D, true, true);        // MN-major x MN-major
      constexpr int KS = D / 16;                                            // K steps of S^T, dP^T
      const uint32_t tS = tmem + L::T_S, tDP = tmem + L::T_DP, tDV = tmem + L::T_DV,
                     tDK = tmem + L::T_DK, tDQ = tmem + L::T_DQ;
      // base descriptors; per-step descriptors are one add away
      const uint64_t dK_k = desc_kmajor_base(sb + L::K), dV_k = desc_kmajor_base(sb + L::V);
      const uint64_t dK_mn = desc_mnmajor_base(sb + L::K, kTile);
      // dS^T buffer of query tile i: it mod NDS
      const uint64_t dS_k = desc_kmajor_base(sb + L::DST);
      const uint64_t dS_mn = desc_mnmajor_base(sb + L::DST, kTile);
      auto ds_off = [&](int it) { return (uint32_t)(it % L::NDS) * L::DSB; };
      const uint64_t dQ_k0 = desc_kmajor_base(sb + L::QS), dQ_mn0 = desc_mnmajor_base(sb + L::QS, kTile);
      auto stage_off = [&](int it) { return (uint32_t)(it % NS) * 2u * L::TILE; };
      auto mma_s = [&](int it, int kk) {
        tc_mma_ss_elect(tS, dK_k + kmajor_step(kk, kTile),
                        desc_add(dQ_k0, stage_off(it)) + kmajor_step(kk, kTile), idS, kk > 0 ? 1u : 0u);
      };
      auto mma_dp = [&](int it, int kk) {
        tc_mma_ss_elect(tDP, dV_k + kmajor_step(kk, kTile),
                        desc_add(dQ_k0, stage_off(it) + L::TILE) + kmajor_step(kk, kTile), idS,
                        kk > 0 ? 1u : 0u);
      };
      auto mma_dv = [&](int it, int kk) {
        tc_mma_ts_elect(tDV, tmem + L::pt_col(kk),
                        desc_add(dQ_mn0, stage_off(it) + L::TILE) + mnmajor_step(kk), idKV,
                        (it > 0 || kk > 0) ? 1u : 0u);
      };
      auto mma_dk = [&](int it, int kk) {
        tc_mma_ss_elect(tDK, desc_add(dS_k, ds_off(it)) + kmajor_step(kk, kTile),
                        desc_add(dQ_mn0, stage_off(it)) + mnmajor_step(kk), idKV, (it > 0 || kk > 0) ? 1u : 0u);
      };
      auto mma_dq = [&](int it, int kk) {
        tc_mma_ss_elect(tDQ, desc_add(dS_mn, ds_off(it)) + mnmajor_step(kk), dK_mn + mnmajor_step(kk), idQ,
                        kk > 0 ? 1u : 0u);
      };
      bool ok = warp_wait(w, bar_kv, 0);
      int qt = next_qt(qt_begin);
      if (ok && qt < q_end && (ok = warp_wait(w, bar_qf(0), 0))) {
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
          mma_s(0, kk);
          mma_dp(0, kk);
        }
        tc_commit_elect(bar_s_full);
        tc_commit_elect(bar_dp_full);
      }
      for (int it = 0; ok && qt < q_end; ++it) {
        const int qn = next_qt(qt + 1);
        const bool next = qn < q_end;
        // Within each group the MMA the compute warps wait for next goes first
        // (MMAs execute in issue order).
        if (!(ok = warp_wait(w, bar_p_full, it & 1))) break;
        if (next && !(ok = warp_wait(w, bar_qf((it + 1) % NS), ((it + 1) / NS) & 1))) break;
        tc_fence_after();
        if (!L::ALIAS) {
          // S^T_{i+1}, then dV += P^T dO_i (P^T has columns of its own)
          if (next) {
#pragma unroll
            for (int kk = 0; kk < KS; ++kk) mma_s(it + 1, kk);
            tc_commit_elect(bar_s_full);
          }
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk) mma_dv(it, kk);
          // P^T_{i+1} may be written once dV_i has read P^T_i; s_full (committed
          // before dV_i) does not cover that
          tc_commit_elect(bar_pt_free);
          // dP^T_{i+1} as soon as the compute warps have read dP^T_i (before
          // they form dS_i), so that the next dS finds it ready
          if (next) {
            if (!(ok = warp_wait(w, bar_dp_free, it & 1))) break;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < KS; ++kk) mma_dp(it + 1, kk);
            tc_commit_elect(bar_dp_full);
          }
        } else {
          // d = 128: S^T_{i+1} overwrites P^T, so it follows dV in issue order
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk) mma_dv(it, kk);
          if (next) {
#pragma unroll
            for (int kk = 0; kk < KS; ++kk) mma_s(it + 1, kk);
            tc_commit_elect(bar_s_full);
          }
        }
        // dQ_i = dS K_j (read out next by the compute warps), then dK += dS^T Q_i
        if (!(ok = warp_wait(w, bar_ds_full, it & 1))) break;
        if (!L::ALIAS && it > 0 && !(ok = warp_wait(w, bar_dq_free, (it - 1) & 1))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk) mma_dq(it, kk);
        // at d = 64 dQ_i may be read out while dK_i runs; at d = 128 the dQ staging
        // reuses the dS^T buffer that dK_i reads, so dq_full waits for dK_i too
        if (L::STG_SEP) tc_commit_elect(bar_dq_full);
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk) mma_dk(it, kk);
        if (!L::STG_SEP) tc_commit_elect(bar_dq_full);
        tc_commit_elect(bar_ds_free(it % L::NDS));
        tc_commit_elect(bar_qe(it % NS));
        if (L::ALIAS && next) {
          // dP^T_{i+1} goes over dQ_i: wait until it has been read out
          if (!(ok = warp_wait(w, bar_dp_free, it & 1))) break;
          if (!(ok = warp_wait(w, bar_dq_free, it & 1))) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < KS; ++kk) mma_dp(it + 1, kk);
          tc_commit_elect(bar_dp_full);
        }
        qt = qn;
      }
      tc_commit_elect(bar_done);
      if (lane == 0) mbar_drain(w, bar_done, 0);
      __syncwarp();
    }
  } else if (warp > kMma) {
    if constexpr (L::QW) {
      // ------------------------------------------------------------ dQ warps
      // Warp of TMEM quadrant qd: query rows 32 qd .. 32 qd + 31 of each tile's
      // dQ_i = dS K_j (TMEM lane = query row), all D columns, read out as soon as
      // the MMA completes, staged in its own 128-byte-swizzled boxes of 32 rows x
      // 32 fp32 columns and added into the fp32 accumulator by TMA reduce-adds (L2
      // performs the adds).  A box is rewritten only after the previous tile's
      // reduces have finished reading it.
      const int qd = warp & 3;
      const uint32_t lane_off = (uint32_t)(qd * 32) << 16;
      const uint32_t stg = sb + L::STG + (uint32_t)qd * L::BOXB;  // this warp's box
      bool pend = false;  // a reduce may still be reading the box
      bool ok = true;
      int it = 0;
      for (int qt = next_qt(qt_begin); qt < q_end;
           qt = next_qt(qt + 1), ++it) {
        if (!(ok = warp_wait(w, bar_dq_full, it & 1))) break;
        tc_fence_after();
        // one box (DQC columns) at a time: out of TMEM, into the box once the
        // previous reduce has finished reading it, then reduced into the
        // accumulator
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += L::DQC) {
          uint32_t dq[L::DQC];
          tmem_ld_n<L::DQC>(tmem + L::T_DQ + lane_off + (uint32_t)c0, dq);
          if (c0 + L::DQC == D) {  // all of dQ_i is in registers: the next dQ may be computed
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_dq_free);
          }
          if (pend) {
            if (lane == 0) bulk_wait_group_read0();
            __syncwarp();
          }
          // row `lane` of the box: 16-byte chunk x at x ^ (row mod 8) (the map's
          // 128-byte swizzle)
#pragma unroll
          for (int x = 0; x < L::DQC / 4; ++x)
            st_shared_v4(stg + (uint32_t)lane * 128u + (uint32_t)((x ^ (lane & 7)) * 16), dq[4 * x],
                         dq[4 * x + 1], dq[4 * x + 2], dq[4 * x + 3]);
          fence_async_smem();
          __syncwarp();
          if (lane == 0 && dbg_check(w, qt * kTile < a.N)) {
            tma_reduce_add_3d(&tmdQ, stg, c0, qt * kTile + qd * 32, bh);
            bulk_commit_group();
          }
          pend = true;
        }
      }
      if (lane == 0) bulk_wait_group0();  // this warp's dQ reductions fully done
    }
  } else {
    // ------------------------------------------------------------ compute warpgroups
    // Software-pipelined per query tile i:  dS_i | P_{i+1} | dQ_i (dQ_i only
    // without dQ warps), so that the exponentials of the next tile run while the
    // tensor core computes dK_i, dQ_i and dP^T_{i+1}.
    constexpr int CW = L::CW;
    const int g = warp >> 2;                 // query columns [CW g, CW g + CW)
    const int r = (warp & 3) * 32 + lane;    // key row in the tile = TMEM lane
    const int key = kt * kTile + r;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint64_t c2p = f2pack(a.scale_log2, a.scale_log2);
    const bool rows_out = __any_sync(0xffffffffu, key >= a.N);  // a tail key tile
    // dQ staging: this warp's box {DQC columns, 32 rows} of the dQ accumulator
    // map, with that map's swizzle.  Each warp reduces its own box, so no warp
    // waits for another.  The TMA reduce reads the box asynchronously; the box
    // is released lazily, when it is about to be written again.
    const uint32_t stg = sb + L::STG + (uint32_t)warp * L::BOXB;
    bool pend = false;  // a reduce may still be reading the box
    auto stg_acquire = [&]() {
      if (pend) {
        if (lane == 0) bulk_wait_group_read0();
        __syncwarp();
        pend = false;
      }
    };
    auto stat = [&](int it) {
      return reinterpret_cast<const float*>(smem + L::STAT) + (it % NS) * 256;
    };
    float p[CW];
    // dropout keep bits of this key row for the tile's CW queries (bit c of
    // kbits[c / 32] for query q0 + c): drawn with P, used again for dS
    uint32_t kbits[CW / 32];
#pragma unroll
    for (int i = 0; i < CW / 32; ++i) kbits[i] = ~0u;
    auto keep = [&](int c) -> bool { return (kbits[c >> 5] >> (c & 31)) & 1u; };
    // S^T -> P^T: fp32 in p[] for dS, 16-bit into TMEM for dV; then p_full
    auto p_phase = [&](int it, int qtile) -> bool {
      if constexpr (DROP) {  // drawn while the tile's S^T may still be in flight
#pragma unroll
        for (int i = 0; i < CW / 32; ++i)
          kbits[i] = drop_keep_col32(a.drop, (uint32_t)key, (uint32_t)(qtile * kTile + CW * g + 32 * i),
                                      (uint32_t)bh);
      }
      // the stage's statistics (staged by the producer with Q and dO)
      if (!warp_wait(w, bar_qf(it % NS), (it / NS) & 1)) return false;
      if (!warp_wait(w, bar_s_full, it & 1)) return false;
      tc_fence_after();
      {
        uint32_t u[CW];
        tmem_ld_n<CW>(tmem + L::T_S + lane_off + CW * g, u);
#pragma unroll
        for (int c = 0; c < CW; ++c) p[c] = __uint_as_float(u[c]);
      }
      const float4* nl4 = reinterpret_cast<const float4*>(stat(it) + CW * g);  // -LSE*log2(e)
      const int q0 = qtile * kTile + CW * g;
      const bool diag = a.m.causal && qtile == kt;
      uint32_t pk[CW / 2];
#pragma unroll
      for (int c = 0; c < CW; c += 4) {
        const float4 nl = nl4[c / 4];
        float x0, x1, x2, x3;
        f2unpack(ffma2(f2pack(p[c], p[c + 1]), c2p, f2pack(nl.x, nl.y)), x0, x1);
        f2unpack(ffma2(f2pack(p[c + 2], p[c + 3]), c2p, f2pack(nl.z, nl.w)), x2, x3);
        p[c] = ex2(x0);
        p[c + 1] = ex2(x1);
        p[c + 2] = ex2(x2);
        p[c + 3] = ex2(x3);
      }
      if (rows_out || diag) {  // warp-uniform: only tail and diagonal tiles mask
#pragma unroll
        for (int c = 0; c < CW; ++c)
          if (key >= a.N || (diag && q0 + c < key)) p[c] = 0.f;
      }
      // P^T for dV: with dropout the kept weights times 1 / (1 - p), else 0 (p[]
      // keeps the undropped weights for dS)
#pragma unroll
      for (int c = 0; c < CW; c += 2) {
        if constexpr (DROP)
          pk[c / 2] = pack2<F16>(keep(c) ? p[c] * a.drop.z : 0.f, keep(c + 1) ? p[c + 1] * a.drop.z : 0.f);
        else
          pk[c / 2] = pack2<F16>(p[c], p[c + 1]);
      }
      if constexpr (!L::ALIAS) {
        // d = 64: P^T has one buffer; dV of the previous tile must be done with it
        // (at d = 128 P^T goes over S^T, which s_full already orders after dV)
        if (it > 0) {
          if (!warp_wait(w, bar_pt_free, (it - 1) & 1)) return false;
          tc_fence_after();
        }
      }
      tmem_st_n<CW / 2>(tmem + L::pt_write_col(g) + lane_off, pk);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_p_full);
      return true;
    };
    bool ok = true;
    int it = 0;
    int qt = next_qt(qt_begin);
    if (qt < q_end) ok = p_phase(0, qt);
    for (; ok && qt < q_end; ++it) {
      const int qn = next_qt(qt + 1);
      // ---- dS_i = P_i * (dP_i - D), with dropout P_i * (z_i dP_i - D)
      if (!(ok = warp_wait(w, bar_dp_full, it & 1))) break;
      tc_fence_after();
      uint32_t pk[CW / 2];
      // in two halves of CW / 2 columns, so that only half of dP^T is held in
      // registers at a time; the MMA may overwrite dP^T once both are loaded
      const float4* nd4 = reinterpret_cast<const float4*>(stat(it) + 128 + CW * g);  // -D
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        constexpr int HW = CW / 2;
        uint32_t u[HW];
        tmem_ld_n<HW>(tmem + L::T_DP + lane_off + CW * g + HW * hf, u);
        if (hf == 1) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_dp_free);
        }
        if constexpr (DROP) {
#pragma unroll
          for (int c = 0; c < HW; ++c)
            u[c] = __float_as_uint(keep(HW * hf + c) ? __uint_as_float(u[c]) * a.drop.z : 0.f);
        }
#pragma unroll
        for (int c = 0; c < HW; c += 4) {
          const int cc = HW * hf + c;  // column within the warp's CW
          const float4 nd = nd4[cc / 4];
          float y0, y1, y2, y3;
          f2unpack(fmul2(f2pack(p[cc], p[cc + 1]),
                         fadd2(f2pack(__uint_as_float(u[c]), __uint_as_float(u[c + 1])), f2pack(nd.x, nd.y))),
                   y0, y1);
          f2unpack(fmul2(f2pack(p[cc + 2], p[cc + 3]),
                         fadd2(f2pack(__uint_as_float(u[c + 2]), __uint_as_float(u[c + 3])), f2pack(nd.z, nd.w))),
                   y2, y3);
          pk[cc / 2] = pack2<F16>(y0, y1);
          pk[cc / 2 + 1] = pack2<F16>(y2, y3);
        }
      }
      // the dS^T buffer of this tile (it mod NDS) must have been read by the dK and
      // dQ MMAs of its previous use, tile it - NDS
      if (it >= L::NDS && !(ok = warp_wait(w, bar_ds_free(it % L::NDS), ((it / L::NDS) - 1) & 1))) break;
      // at d = 128 the last dQ reduction must have finished reading this region
      if (!L::STG_SEP) stg_acquire();
#pragma unroll
      for (int ch = 0; ch < CW / 8; ++ch)
        st_shared_v4(sb + L::DST + (uint32_t)(it % L::NDS) * L::DSB + sw128_chunk_offset(r, (CW / 8) * g + ch, kTile),
                     pk[ch * 4 + 0],
                     pk[ch * 4 + 1], pk[ch * 4 + 2], pk[ch * 4 + 3]);
      fence_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_ds_full);

      // ---- P of the next query tile, while dK_i, dQ_i, dP^T_{i+1} run
      if (qn < q_end && !(ok = p_phase(it + 1, qn))) break;

      // ---- dQ_i (TMEM lane = query row) -> fp32 accumulator by TMA reduce-add
      // (the dQ warps' job when there are dQ warps)
      if constexpr (L::QW) {
        qt = qn;
        continue;
      }
      if (!(ok = warp_wait(w, bar_dq_full, it & 1))) break;
      tc_fence_after();
      uint32_t dq[L::DQG];
      tmem_ld_n<L::DQG>(tmem + L::T_DQ + lane_off + g * L::DQG, dq);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_dq_free);
#pragma unroll
      for (int c0 = 0; c0 < L::DQG; c0 += L::DQC) {
        stg_acquire();
        // row `lane` of this warp's 32: with 128-byte rows, 16-byte chunk x at
        // x ^ (row mod 8); with 64-byte rows, at x ^ ((row / 2) mod 4) (the two
        // swizzles of the map, address bits 4-6 or 4-5 xor bits 7-9 or 7-8)
#pragma unroll
        for (int x = 0; x < L::DQC / 4; ++x) {
          const uint32_t off = (L::DQC == 32) ? (uint32_t)lane * 128u + (uint32_t)((x ^ (lane & 7)) * 16)
                                              : (uint32_t)lane * 64u + (uint32_t)((x ^ ((lane >> 1) & 3)) * 16);
          st_shared_v4(stg + off, dq[c0 + 4 * x], dq[c0 + 4 * x + 1], dq[c0 + 4 * x + 2], dq[c0 + 4 * x + 3]);
        }
        fence_async_smem();
        __syncwarp();
        if (lane == 0 && dbg_check(w, g * L::DQG + c0 + L::DQC <= D && qt * kTile < a.N)) {
          tma_reduce_add_3d(&tmdQ, stg, g * L::DQG + c0, qt * kTile + (warp & 3) * 32, bh);
          bulk_commit_group();
        }
        pend = true;
      }
      if (!ok) break;
      qt = qn;
    }
    if (lane == 0) bulk_wait_group0();  // this warp's dQ reductions fully done
    // ------------------------------------------------------------ dK, dV epilogue
    bool have = false;
    if (ok) {
      ok = warp_wait(w, bar_done, 0);
      tc_fence_after();
      have = ok && it > 0;
    }
    // tcgen05.ld is .sync.aligned: every lane of the warp loads (the condition
    // `ok`/`have` is warp-uniform); only the stores are predicated on the row
    if (QS && slot >= 0) {
      if (ok) {
        // one of several slices of the key tile's query tiles: fp32 partial
        // sums, dK unscaled
        float* slotp = a.slots + (size_t)slot * (2 * kTile * D);
        for (int which = 0; which < 2; ++which) {
          const uint32_t col = (which == 0 ? L::T_DV : L::T_DK) + g * L::DQG;
          float* dst = slotp + (size_t)which * (kTile * D) + (size_t)r * D + g * L::DQG;
          constexpr int EC = L::DQG < 32 ? L::DQG : 32;
#pragma unroll
          for (int c0 = 0; c0 < L::DQG; c0 += EC) {
            uint32_t u[EC];
            if (have) {
              tmem_ld_n<EC>(tmem + col + lane_off + c0, u);
            } else {
#pragma unroll
              for (int i = 0; i < EC; ++i) u[i] = 0u;
            }
#pragma unroll
            for (int v = 0; v < EC / 4; ++v)
              *reinterpret_cast<float4*>(dst + c0 + v * 4) =
                  make_float4(__uint_as_float(u[4 * v]), __uint_as_float(u[4 * v + 1]),
                              __uint_as_float(u[4 * v + 2]), __uint_as_float(u[4 * v + 3]));
          }
        }
      }
    } else if (ok) {
      const bool store = key < a.N && dbg_check(w, (size_t)bh * a.N + key < (size_t)BH * a.N);
      constexpr int EC = L::DQG < 32 ? L::DQG : 32;  // columns per TMEM load
      uint16_t* dVrow = reinterpret_cast<uint16_t*>(a.dV) + ((size_t)bh * a.N + key) * D + g * L::DQG;
      uint16_t* dKrow = reinterpret_cast<uint16_t*>(a.dK) + ((size_t)bh * a.N + key) * D + g * L::DQG;
      for (int which = 0; which < 2; ++which) {
        const uint32_t col = (which == 0 ? L::T_DV : L::T_DK) + g * L::DQG;
        const float mul = which == 0 ? 1.f : a.scale;
        uint16_t* dst = which == 0 ? dVrow : dKrow;
#pragma unroll
        for (int c0 = 0; c0 < L::DQG; c0 += EC) {
          uint32_t u[EC];
          if (have) {
            tmem_ld_n<EC>(tmem + col + lane_off + c0, u);
          } else {
#pragma unroll
            for (int i = 0; i < EC; ++i) u[i] = 0u;
          }
#pragma unroll
          for (int v = 0; v < EC / 8; ++v) {
            uint4 pq;
            pq.x = pack2<F16>(__uint_as_float(u[v * 8 + 0]) * mul, __uint_as_float(u[v * 8 + 1]) * mul);
            pq.y = pack2<F16>(__uint_as_float(u[v * 8 + 2]) * mul, __uint_as_float(u[v * 8 + 3]) * mul);
            pq.z = pack2<F16>(__uint_as_float(u[v * 8 + 4]) * mul, __uint_as_float(u[v * 8 + 5]) * mul);
            pq.w = pack2<F16>(__uint_as_float(u[v * 8 + 6]) * mul, __uint_as_float(u[v * 8 + 7]) * mul);
            if (store) *reinterpret_cast<uint4*>(dst + c0 + v * 8) = pq;
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMma) {
    tc_fence_after();
    tmem_dealloc(tmem, L::TMEM_COLS);
  }
}

template <int D, bool F16>
cudaError_t launch_t(const BwdArgs& a, const CUtensorMap* tm, cudaStream_t s) {
  // four compute warpgroups at d = 64; two at d = 128, where the dQ staging
  // shares the dS^T buffer: with two, the dS^T rows a warp writes are exactly
  // its own staging box (so waiting for its own reduce to finish reading is
  // enough); with four they would fall into other warps' boxes
  constexpr int NG = (D == 64) ? 4 : 2;
  using L = BwdLayout<D, NG>;
  // sliced launches (their own instantiation, QS) have no block mask
  auto kern = a.q_slice > 0 ? (a.drop.on ? bwd_tc_kernel<D, F16, NG, true, true, false>
                                         : bwd_tc_kernel<D, F16, NG, false, true, false>)
              : a.m.mask ? (a.drop.on ? bwd_tc_kernel<D, F16, NG, true, false, true>
                                      : bwd_tc_kernel<D, F16, NG, false, false, true>)
                         : (a.drop.on ? bwd_tc_kernel<D, F16, NG, true, false, false>
                                      : bwd_tc_kernel<D, F16, NG, false, false, false>);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::BYTES);
  if (e != cudaSuccess) return e;
  // the dQ accumulator map whose box matches the staging: {32, 32} with the
  // 128-byte swizzle (tm[4]) or {16, 32} with the 64-byte swizzle (tm[5])
  kern<<<(unsigned)a.direct, L::NT, L::BYTES, s>>>(tm[0], tm[1], tm[2], tm[3], tm[L::DQC == 32 ? 4 : 5], a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_tc(const BwdArgs& a, int d, bool f16, const CUtensorMap* tm, cudaStream_t s) {
  if (d == 64) return f16 ? launch_t<64, true>(a, tm, s) : launch_t<64, false>(a, tm, s);
  return f16 ? launch_t<128, true>(a, tm, s) : launch_t<128, false>(a, tm, s);
}

}  // namespace fa
