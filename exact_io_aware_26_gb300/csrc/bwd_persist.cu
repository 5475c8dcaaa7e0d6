// bwd_persist.cu -- the attention backward main kernel as persistent CTAs that
// split the work evenly (used when one CTA per key tile would leave SMs idle).
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
// The CTAs are persistent and split the iterations evenly (bwd_sched.cuh): a
// CTA walks a sequence of (key tile, query tile) tiles that covers one or more
// pieces of key tiles.  Only the producer runs the
// schedule; it stages each tile's coordinates with its Q, dO and statistics,
// and the other roles read them from there.  At d = 64 K_j, V_j are double
// buffered and the pipeline runs on across key tiles (the next key tile's
// first score tile is computed while the last one of the current key tile is
// finished); at d = 128 shared memory holds one K_j, V_j, so the pipeline
// drains at each key tile and refills after the reload.
//
// Warp roles (320 threads): warps 0-3 and 4-7 are two compute warpgroups that
// split the 128 query columns of every tile (TMEM lane = key row); warp 8 is
// the producer (TMA copies of K_j, V_j and of Q_i, dO_i through a ring, plus
// each query tile's LSE, D and coordinates staged by its lanes); warp 9 owns
// TMEM and issues the MMAs.
#include "bwd_sched.cuh"
#include "ptx.cuh"
#include "tiles.cuh"

namespace fa {
namespace {


template <int D>
struct BwdLayout {
  static constexpr uint32_t TILE = kTile * D * 2;
  // d = 64: two K_j, V_j buffers, so that the next key tile loads while the
  // current one is finished; d = 128: one (shared memory is full)
  static constexpr bool KV2 = (D == 64);
  static constexpr int NKV = KV2 ? 2 : 1;
  // Q and dO rings.  Q_i is read by S^T_i and, last, by dK_i at the end of
  // iteration i; dO_i by dP^T_i and, last, by dV_i early in iteration i, so its
  // stage frees sooner and a shallower ring keeps it as far ahead
  static constexpr int NQ = (D == 64) ? 3 : 2;
  static constexpr int NO = 2;
  __device__ static constexpr uint32_t K(int b) { return (uint32_t)b * 2u * TILE; }
  __device__ static constexpr uint32_t V(int b) { return (uint32_t)b * 2u * TILE + TILE; }
  static constexpr uint32_t QR = NKV * 2 * TILE;       // Q stage s at QR + s TILE
  static constexpr uint32_t OR = QR + NQ * TILE;       // dO stage s at OR + s TILE
  static constexpr uint32_t DST = OR + NO * TILE;      // dS^T, 128 x 128 16-bit
  // per Q stage: [128] -LSE*log2e, [128] -D of the query tile, then its
  // coordinates (TileInfo)
  static constexpr uint32_t STAT = DST + kTile * kTile * 2;
  static constexpr uint32_t STAT_STRIDE = 256 * 4 + 32;
  // dQ staging (fp32, two 128 x 32 boxes): a buffer of its own at d = 64; at
  // d = 128 shared memory is full and the dS^T buffer doubles as staging
  static constexpr bool STG_SEP = (D == 64);
  static constexpr uint32_t STG = STG_SEP ? (STAT + NQ * STAT_STRIDE + 1023) & ~1023u : DST;  // 1024-aligned (swizzle)
  static constexpr uint32_t BAR = STG_SEP ? STG + 2 * kTile * 128 : (STAT + NQ * STAT_STRIDE + 7) & ~7u;
  // barriers: 0-1 kv_full[2], 2-3 kv_empty[2], 4 s_full, 5 dp_full, 6 dp_free, 7 p_full,
  //           8 ds_full, 9 ds_free, 10 dq_full, 11 dq_free, 12 acc_full (a piece's dK, dV
  //           complete), 13 acc_free (read out), 14 pt_free (dV_i has read P^T_i),
  //           15.. q_full[NQ], q_empty[NQ], o_full[NO], o_empty[NO]
  static constexpr uint32_t NBAR = 15 + 2 * NQ + 2 * NO;
  static constexpr uint32_t TSLOT = BAR + NBAR * 8;
  static constexpr uint32_t ABORT = TSLOT + 4;
  static constexpr uint32_t BYTES = ABORT + 4;
  static constexpr uint32_t TMEM_COLS = 512;
  // TMEM columns.  S^T [0,128) (warpgroup g reads [64g, 64g+64)), dP^T [128,256),
  // dV and dK d columns each.  At d = 64, dQ [384,448) and the 16-bit P^T
  // [448,512) have columns of their own; at d = 128 the 512 columns are full, so
  // dQ goes over dP^T and warpgroup g writes its P^T over [64g, 64g+32) of S^T.
  static constexpr uint32_t T_S = 0, T_DP = 128, T_DV = 256, T_DK = 256 + D;
  static constexpr bool ALIAS = (D == 128);
  static constexpr uint32_t T_DQ = ALIAS ? T_DP : 384;
  static constexpr uint32_t T_PT = ALIAS ? T_S : 448;
  // column of P^T that holds query pair kk*8 .. kk*8+7 (16 queries), and the
  // columns warpgroup g writes
  __device__ static constexpr uint32_t pt_col(int kk) {
    return ALIAS ? 64u * (uint32_t)(kk >> 2) + 8u * (uint32_t)(kk & 3) : T_PT + 8u * (uint32_t)kk;
  }
  __device__ static constexpr uint32_t pt_write_col(int g) {
    return ALIAS ? 64u * (uint32_t)g : T_PT + 32u * (uint32_t)g;
  }
};
static_assert(BwdLayout<64>::BYTES <= 232448 && BwdLayout<128>::BYTES <= 232448, "shared memory");
static_assert(BwdLayout<64>::STG % 1024 == 0 && BwdLayout<64>::DST % 1024 == 0 &&
                  BwdLayout<128>::DST % 1024 == 0 && BwdLayout<64>::OR % 1024 == 0,
              "swizzled buffers need 1024-byte alignment");

// A tile's coordinates, staged by the producer next to its statistics.
struct TileInfo {
  int kt, bh, qt, slot;  // key tile, head, query tile, partial-sum slot of its piece (-1: none)
  int pc;                // piece counter within the CTA
  int flags;             // kFirst, kLast: the tile opens / closes its piece; kMore: a tile follows
};
constexpr int kFirst = 1, kLast = 2, kMore = 4;




// Out of line: called once per piece, and inlined into the producer it would
// cost registers in its loop.
static __device__ __noinline__ bool next_piece(const Sched& sc, int c, long long& g, long long g_end,
                                               bool& first, Seg& sg) {
  return sched_next(sc, c, g, g_end, first, sg);
}

template <int D, bool F16, bool DROP>
__global__ void __launch_bounds__(320, 1)
    bwd_persist_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                  const __grid_constant__ CUtensorMap tmdQ, const BwdArgs a) {
  using L = BwdLayout<D>;
  constexpr int NQ = L::NQ, NO = L::NO;
  constexpr bool KV2 = L::KV2;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sb = smem_addr(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int BH = a.B * a.H;
  const int n_tiles = (a.N + kTile - 1) / kTile;
  // With a block mask (one key tile per CTA) the tile may see no query at all:
  // then dK = dV = 0 and no role has anything to wait for.
  bool empty = false;
  if (a.G == 0) {
    const int kt = (int)(blockIdx.x / BH), bh = (int)(blockIdx.x % BH);
    empty = next_q(a.m, bh / a.H, bh % a.H, a.m.causal ? kt : 0, kt, n_tiles) >= n_tiles;
  }

  auto bar = [&](int i) { return sb + L::BAR + 8u * (uint32_t)i; };
  auto bar_kv_full = [&](int b) { return bar(b); };
  auto bar_kv_empty = [&](int b) { return bar(2 + b); };
  const uint32_t bar_s_full = bar(4), bar_dp_full = bar(5), bar_dp_free = bar(6),
                 bar_p_full = bar(7), bar_ds_full = bar(8), bar_ds_free = bar(9),
                 bar_dq_full = bar(10), bar_dq_free = bar(11), bar_acc_full = bar(12),
                 bar_acc_free = bar(13), bar_pt_free = bar(14);
  auto bar_qf = [&](int s) { return bar(15 + s); };
  auto bar_qe = [&](int s) { return bar(15 + NQ + s); };
  auto bar_of = [&](int s) { return bar(15 + 2 * NQ + s); };
  auto bar_oe = [&](int s) { return bar(15 + 2 * NQ + NO + s); };
  // K/V buffer of piece pc and the phase of its use of that buffer
  auto kv_buf = [&](int pc) { return KV2 ? (pc & 1) : 0; };
  auto kv_phase = [&](int pc) { return (uint32_t)(KV2 ? (pc >> 1) & 1 : pc & 1); };
  // tile it's coordinates {kt, bh, qt, slot} and {pc, flags}: plain vector
  // loads, read only after the stage's full barrier (whose wait orders them)
  auto info_a = [&](int it) {
    return *reinterpret_cast<const int4*>(smem + L::STAT + (it % NQ) * L::STAT_STRIDE + 1024);
  };
  auto info_b = [&](int it) {
    return *reinterpret_cast<const int2*>(smem + L::STAT + (it % NQ) * L::STAT_STRIDE + 1040);
  };

  volatile int* abort_cta = reinterpret_cast<volatile int*>(smem + L::ABORT);
  const WaitCtx w{abort_cta, a.rep.st, a.rep.epoch, a.rep.wait_ns};
  // waits for tile it's Q stage (with its statistics and coordinates) and dO stage
  auto q_ready = [&](int it) { return warp_wait(w, bar_qf(it % NQ), (it / NQ) & 1); };
  auto o_ready = [&](int it) { return warp_wait(w, bar_of(it % NO), (it / NO) & 1); };

  if ((sb & 1023u) != 0) {
    if (threadIdx.x == 0) raise_error(w, FA_ERR_CUDA);
    return;
  }
  if (threadIdx.x == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_kv_full(b), 1);
      mbar_init(bar_kv_empty(b), 1);
    }
    mbar_init(bar_s_full, 1);
    mbar_init(bar_dp_full, 1);
    mbar_init(bar_dp_free, 8);
    mbar_init(bar_p_full, 8);
    mbar_init(bar_ds_full, 8);
    mbar_init(bar_ds_free, 1);
    mbar_init(bar_dq_full, 1);
    mbar_init(bar_dq_free, 8);
    mbar_init(bar_acc_full, 1);
    mbar_init(bar_acc_free, 8);
    mbar_init(bar_pt_free, 1);
    for (int s = 0; s < NQ; ++s) {
      mbar_init(bar_qf(s), 1 + 32);  // the TMA transaction arrival + every producer lane
      mbar_init(bar_qe(s), 1);
    }
    for (int s = 0; s < NO; ++s) {
      mbar_init(bar_of(s), 1);
      mbar_init(bar_oe(s), 1);
    }
    *abort_cta = 0;
    fence_barrier_init();
  }
  if (warp == 9) {
    tmem_alloc(sb + L::TSLOT, L::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + L::TSLOT);

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    // Walks the schedule.  Lane 0 issues the TMA copies; every lane stages four
    // rows of the query tile's statistics, lane 0 the tile's coordinates, into
    // the ring stage, so that the stage's full barrier covers them all.  A
    // piece's K_j, V_j are loaded when its first tile is reached, into the
    // buffer its piece before last has released.
    if (lane == 0) {
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
      prefetch_tmap(&tmdO);
    }
    const Sched sc = make_sched(n_tiles, BH, a.m.causal, a.G > 0 ? a.G : 1, a.u0);
    long long g = a.G > 0 ? sched_start(sc, (int)blockIdx.x) : 0;
    const long long g_stop = a.G > 0 ? sched_start(sc, (int)blockIdx.x + 1) : 1;
    bool first_piece = true;
    Seg sg;
    auto open = [&]() -> bool {  // the next piece, into sg
      if (a.G > 0) return next_piece(sc, (int)blockIdx.x, g, g_stop, first_piece, sg);
      if (g >= g_stop || empty) return false;
      g = g_stop;
      sg.kt = (int)(blockIdx.x / BH);
      sg.bh = (int)(blockIdx.x % BH);
      sg.q_first = a.m.causal ? sg.kt : 0;
      sg.q_end = n_tiles;
      sg.slot = -1;
      return true;
    };
    int it = 0, pc = 0;
    bool ok = true;
    bool live = open();
    int qt = live ? next_q(a.m, sg.bh / a.H, sg.bh % a.H, sg.q_first, sg.kt, sg.q_end) : 0;
    bool at_start = true;
    // the next tile's statistics, loaded one tile ahead so that their latency
    // hides behind the previous tile's copies: -LSE*log2(e) and -D of rows
    // 4 lane .. 4 lane + 3, negated as the compute warps use them
    float4 l4, d4;
    auto load_stats = [&](int bh, int q0) {
      l4 = make_float4(-lse2_of(a, bh, q0 + lane * 4 + 0), -lse2_of(a, bh, q0 + lane * 4 + 1),
                       -lse2_of(a, bh, q0 + lane * 4 + 2), -lse2_of(a, bh, q0 + lane * 4 + 3));
      d4 = make_float4(-d_of(a, bh, q0 + lane * 4 + 0), -d_of(a, bh, q0 + lane * 4 + 1),
                       -d_of(a, bh, q0 + lane * 4 + 2), -d_of(a, bh, q0 + lane * 4 + 3));
    };
    if (live) load_stats(sg.bh, qt * kTile);
    while (ok && live) {
      // this tile, and whether another follows (in this piece or the next)
      const int kt = sg.kt, bh = sg.bh, slot = sg.slot;
      // debug build: the piece the schedule handed out lies inside the problem and
      // its slot inside the workspace's slots (two per CTA)
      if (!(ok = __all_sync(0xffffffffu, dbg_check(w, kt >= 0 && kt < n_tiles && bh >= 0 && bh < BH &&
                                                        qt >= sg.q_first && qt < sg.q_end &&
                                                        sg.q_end <= n_tiles && slot >= -1 &&
                                                        slot < 2 * (a.G > 0 ? a.G : 1)))))
        break;
      const int qn = next_q(a.m, bh / a.H, bh % a.H, qt + 1, kt, sg.q_end);
      const bool last = qn >= sg.q_end;
      const bool first = at_start;
      if (first) {
        const int b = kv_buf(pc);
        const int prev = KV2 ? pc - 2 : pc - 1;  // the piece that used the buffer before
        if (prev >= 0 && !(ok = warp_wait(w, bar_kv_empty(b), kv_phase(prev)))) break;
        if (lane == 0) {
          mbar_arrive_expect_tx(bar_kv_full(b), 2 * L::TILE);
          for (int c = 0; c < D / 64; ++c) {
            tma_load_3d(sb + L::K(b) + c * (kTile * 128), &tmK, bar_kv_full(b), c * 64, kt * kTile, bh);
            tma_load_3d(sb + L::V(b) + c * (kTile * 128), &tmV, bar_kv_full(b), c * 64, kt * kTile, bh);
          }
        }
      }
      const int this_pc = pc;
      const int this_qt = qt;
      if (last) {
        live = open();
        if (live) {
          ++pc;
          qt = next_q(a.m, sg.bh / a.H, sg.bh % a.H, sg.q_first, sg.kt, sg.q_end);
        }
        at_start = true;
      } else {
        qt = qn;
        at_start = false;
      }
      const int s = it % NQ;
      if (it >= NQ && !(ok = warp_wait(w, bar_qe(s), ((it / NQ) - 1) & 1))) break;
      if (lane == 0) {
        const uint32_t dst = sb + L::QR + (uint32_t)s * L::TILE;
        mbar_arrive_expect_tx(bar_qf(s), L::TILE);
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(dst + c * (kTile * 128), &tmQ, bar_qf(s), c * 64, this_qt * kTile, bh);
      }
      float* st = reinterpret_cast<float*>(smem + L::STAT + s * L::STAT_STRIDE);
      reinterpret_cast<float4*>(st)[lane] = l4;
      reinterpret_cast<float4*>(st + 128)[lane] = d4;
      if (lane == 0) {
        *reinterpret_cast<int4*>(st + 256) = make_int4(kt, bh, this_qt, slot);
        *reinterpret_cast<int2*>(st + 260) =
            make_int2(this_pc, (first ? kFirst : 0) | (last ? kLast : 0) | (live ? kMore : 0));
      }
      mbar_arrive(bar_qf(s));
      if (live) load_stats(sg.bh, qt * kTile);  // the next tile's
      const int os = it % NO;
      if (it >= NO && !(ok = warp_wait(w, bar_oe(os), ((it / NO) - 1) & 1))) break;
      if (lane == 0) {
        const uint32_t dst = sb + L::OR + (uint32_t)os * L::TILE;
        mbar_arrive_expect_tx(bar_of(os), L::TILE);
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(dst + c * (kTile * 128), &tmdO, bar_of(os), c * 64, this_qt * kTile, bh);
      }
      ++it;
    }
    // every copy issued has landed before the CTA may exit
    if (lane == 0) {
      const int pieces = it > 0 ? pc + 1 : 0;
      for (int p = pieces - 1; p >= 0 && p >= pieces - L::NKV; --p)
        mbar_drain(w, bar_kv_full(kv_buf(p)), kv_phase(p));
      for (int s = 0; s < NQ; ++s) {
        const int n = (it - s + NQ - 1) / NQ;  // loads issued into Q stage s
        if (n > 0) mbar_drain(w, bar_qf(s), (n - 1) & 1);
      }
      for (int s = 0; s < NO; ++s) {
        const int n = (it - s + NO - 1) / NO;  // into dO stage s
        if (n > 0) mbar_drain(w, bar_of(s), (n - 1) & 1);
      }
    }
    __syncwarp();
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs this loop converged (waits are warp-uniform); one
    // elected lane issues each MMA and commit.
    // Per tile i (the next tile's Q/dO sit in the other ring stage):
    //   d = 64:  S^T_{i+1}, dV_i, dP^T_{i+1}, then dQ_i, dK_i
    //   d = 128: dV_i, S^T_{i+1} (over P^T), then dQ_i, dK_i, dP^T_{i+1} (over dQ_i)
    // so the next score tile is computed while the compute warps form dS_i, and
    // dQ_i is ready for them right after the next tile's exponentials.  Tile
    // i+1 may belong to the next piece (d = 64 only): its S^T and dP^T use the
    // other K/V buffer.
    constexpr uint32_t idS = idesc_f16(F16, kTile, kTile, false, false);  // K-major x K-major
    constexpr uint32_t idKV = idesc_f16(F16, kTile, D, false, true);      // K-major x MN-major
    constexpr uint32_t idQ = idesc_f16(F16, kTile, D, true, true);        // MN-major x MN-major
    constexpr int KS = D / 16;                                            // K steps of S^T, dP^T
    const uint32_t tS = tmem + L::T_S, tDP = tmem + L::T_DP, tDV = tmem + L::T_DV,
                   tDK = tmem + L::T_DK, tDQ = tmem + L::T_DQ;
    // base descriptors; per-step descriptors are one add away
    const uint64_t dS_k = desc_kmajor_base(sb + L::DST);
    const uint64_t dS_mn = desc_mnmajor_base(sb + L::DST, kTile);
    const uint64_t dQ_k0 = desc_kmajor_base(sb + L::QR), dQ_mn0 = desc_mnmajor_base(sb + L::QR, kTile);
    const uint64_t dO_k0 = desc_kmajor_base(sb + L::OR), dO_mn0 = desc_mnmajor_base(sb + L::OR, kTile);
    const uint64_t dK_k0 = desc_kmajor_base(sb + L::K(0)), dV_k0 = desc_kmajor_base(sb + L::V(0));
    const uint64_t dK_mn0 = desc_mnmajor_base(sb + L::K(0), kTile);
    const uint32_t kv_off = 2u * L::TILE;  // second K/V buffer
    auto q_off = [&](int it) { return (uint32_t)(it % NQ) * L::TILE; };
    auto o_off = [&](int it) { return (uint32_t)(it % NO) * L::TILE; };
    auto mma_s = [&](int it, int b, int kk) {
      tc_mma_ss_elect(tS, desc_add(dK_k0, b ? kv_off : 0u) + kmajor_step(kk, kTile),
                      desc_add(dQ_k0, q_off(it)) + kmajor_step(kk, kTile), idS, kk > 0 ? 1u : 0u);
    };
    auto mma_dp = [&](int it, int b, int kk) {
      tc_mma_ss_elect(tDP, desc_add(dV_k0, b ? kv_off : 0u) + kmajor_step(kk, kTile),
                      desc_add(dO_k0, o_off(it)) + kmajor_step(kk, kTile), idS, kk > 0 ? 1u : 0u);
    };
    // dV, dK start afresh (accumulate = 0) at the first tile of each piece
    auto mma_dv = [&](int it, int kk, bool acc) {
      tc_mma_ts_elect(tDV, tmem + L::pt_col(kk), desc_add(dO_mn0, o_off(it)) + mnmajor_step(kk), idKV,
                      (acc || kk > 0) ? 1u : 0u);
    };
    auto mma_dk = [&](int it, int kk, bool acc) {
      tc_mma_ss_elect(tDK, dS_k + kmajor_step(kk, kTile), desc_add(dQ_mn0, q_off(it)) + mnmajor_step(kk),
                      idKV, (acc || kk > 0) ? 1u : 0u);
    };
    auto mma_dq = [&](int b, int kk) {
      tc_mma_ss_elect(tDQ, dS_mn + mnmajor_step(kk), desc_add(dK_mn0, b ? kv_off : 0u) + mnmajor_step(kk),
                      idQ, kk > 0 ? 1u : 0u);
    };
    bool ok = !empty;
    int it = 0, pieces = 0;
    while (ok) {
      if (!(ok = q_ready(it))) break;
      const int2 ib = info_b(it);
      const int pc = ib.x, fl = ib.y;
      const int b = kv_buf(pc);
      const bool first = fl & kFirst, last = fl & kLast, more = fl & kMore;
      if (first) pieces = pc + 1;
      if (first && (it == 0 || !KV2)) {
        // (re)fill the pipeline: S^T_i, dP^T_i once K_j, V_j have landed and,
        // after an earlier piece, its last dP^T (and at d = 128 its last dQ,
        // which dP^T overwrites) has been read
        if (!(ok = warp_wait(w, bar_kv_full(b), kv_phase(pc)))) break;
        if (!(ok = o_ready(it))) break;
        if (it > 0) {
          if (!(ok = warp_wait(w, bar_dp_free, (it - 1) & 1))) break;
          if (L::ALIAS && !(ok = warp_wait(w, bar_dq_free, (it - 1) & 1))) break;
        }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
          mma_s(it, b, kk);
          mma_dp(it, b, kk);
        }
        tc_commit_elect(bar_s_full);
        tc_commit_elect(bar_dp_full);
      }
      // the next tile, if it is computed ahead: always at d = 64, within the
      // piece at d = 128
      const bool ahead = KV2 ? more : (more && !last);
      int nb = b;
      // Within each group the MMA the compute warps wait for next goes first
      // (MMAs execute in issue order).
      if (!(ok = warp_wait(w, bar_p_full, it & 1))) break;
      if (ahead) {
        if (!(ok = q_ready(it + 1))) break;
        const int npc = info_b(it + 1).x;
        nb = kv_buf(npc);
        if (npc != pc && !(ok = warp_wait(w, bar_kv_full(nb), kv_phase(npc)))) break;
      }
      if (first && pc > 0) {
        // the previous piece's dK, dV have been read out of TMEM
        if (!(ok = warp_wait(w, bar_acc_free, (pc - 1) & 1))) break;
      }
      tc_fence_after();
      if (!L::ALIAS) {
        // S^T_{i+1}, then dV += P^T dO_i (P^T has columns of its own)
        if (ahead) {
#pragma unroll
          for (int kk = 0; kk < KS; ++kk) mma_s(it + 1, nb, kk);
          tc_commit_elect(bar_s_full);
        }
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk) mma_dv(it, kk, !first);
        // P^T_{i+1} may be written once dV_i has read P^T_i; s_full (committed
        // before dV_i) does not cover that.  dO_i is not read after dV_i.
        tc_commit_elect(bar_pt_free);
        tc_commit_elect(bar_oe(it % NO));
        // dP^T_{i+1} as soon as the compute warps have read dP^T_i (before
        // they form dS_i), so that the next dS finds it ready
        if (ahead) {
          if (!(ok = warp_wait(w, bar_dp_free, it & 1))) break;
          if (!(ok = o_ready(it + 1))) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < KS; ++kk) mma_dp(it + 1, nb, kk);
          tc_commit_elect(bar_dp_full);
        }
      } else {
        // d = 128: S^T_{i+1} overwrites P^T, so it follows dV in issue order
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk) mma_dv(it, kk, !first);
        tc_commit_elect(bar_oe(it % NO));
        if (ahead) {
#pragma unroll
          for (int kk = 0; kk < KS; ++kk) mma_s(it + 1, nb, kk);
          tc_commit_elect(bar_s_full);
        }
      }
      // dQ_i = dS K_j (read out next by the compute warps), then dK += dS^T Q_i
      if (!(ok = warp_wait(w, bar_ds_full, it & 1))) break;
      if (!L::ALIAS && it > 0 && !(ok = warp_wait(w, bar_dq_free, (it - 1) & 1))) break;
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < kTile / 16; ++kk) mma_dq(b, kk);
      // at d = 64 dQ_i may be read out while dK_i runs; at d = 128 the dQ staging
      // reuses the dS^T buffer that dK_i reads, so dq_full waits for dK_i too
      if (L::STG_SEP) tc_commit_elect(bar_dq_full);
#pragma unroll
      for (int kk = 0; kk < kTile / 16; ++kk) mma_dk(it, kk, !first);
      if (!L::STG_SEP) tc_commit_elect(bar_dq_full);
      tc_commit_elect(bar_ds_free);
      tc_commit_elect(bar_qe(it % NQ));
      if (last) {
        // the piece's dK, dV are complete, and its K_j, V_j no longer read
        tc_commit_elect(bar_acc_full);
        tc_commit_elect(bar_kv_empty(b));
      }
      if (L::ALIAS && ahead) {
        // dP^T_{i+1} goes over dQ_i: wait until it has been read out
        if (!(ok = warp_wait(w, bar_dp_free, it & 1))) break;
        if (!(ok = warp_wait(w, bar_dq_free, it & 1))) break;
        if (!(ok = o_ready(it + 1))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) mma_dp(it + 1, nb, kk);
        tc_commit_elect(bar_dp_full);
      }
      ++it;
      if (!more) break;
    }
    if (lane == 0 && pieces > 0) {
      mbar_drain(w, bar_acc_full, (pieces - 1) & 1);
      for (int p = pieces - 1; p >= 0 && p >= pieces - L::NKV; --p)
        mbar_drain(w, bar_kv_empty(kv_buf(p)), kv_phase(p));
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ compute warpgroups
    // Software-pipelined per tile i:  dS_i | P_{i+1} | dQ_i, so that the
    // exponentials of the next tile run while the tensor core computes dK_i,
    // dQ_i and dP^T_{i+1}.  After the last tile of a piece: its dK, dV.
    const int g = warp >> 2;                 // 0: query columns 0-63, 1: 64-127
    const int r = (warp & 3) * 32 + lane;    // key row in the tile = TMEM lane
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint64_t c2p = f2pack(a.scale_log2, a.scale_log2);
    // dQ staging: this warp's 4 KiB, laid out as the 128-byte-swizzled box
    // {32 columns, 32 rows} of tmdQ.  Each warp reduces its own box, so no warp
    // waits for another.  The TMA reduce reads the box asynchronously; the box
    // is released lazily, when it is about to be written again.
    const uint32_t stg = sb + L::STG + (uint32_t)g * (kTile * 128) + (uint32_t)(warp & 3) * 4096u;
    bool pend = false;  // a reduce may still be reading the box
    auto stg_acquire = [&]() {
      if (pend) {
        if (lane == 0) bulk_wait_group_read0();
        __syncwarp();
        pend = false;
      }
    };
    auto stat = [&](int it) {
      return reinterpret_cast<const float*>(smem + L::STAT + (it % NQ) * L::STAT_STRIDE);
    };
    float p[64];
    // dropout keep bits of this key row for the tile's 64 queries (bit c of
    // kbits[c / 32] for query q0 + c): drawn with P, used again for dS
    uint32_t kbits[2] = {~0u, ~0u};
    auto keep = [&](int c) -> bool { return (kbits[c >> 5] >> (c & 31)) & 1u; };
    // S^T -> P^T of tile it: fp32 in p[] for dS, 16-bit into TMEM for dV; then p_full
    auto p_phase = [&](int it) -> bool {
      // the stage's statistics and coordinates (staged by the producer with Q and dO)
      if (!q_ready(it)) return false;
      const int4 ia = info_a(it);
      const int kt = ia.x, qtile = ia.z;
      const int key = kt * kTile + r;
      if constexpr (DROP) {
#pragma unroll
        for (int i = 0; i < 2; ++i)
          kbits[i] = drop_keep_col32(a.drop, (uint32_t)key, (uint32_t)(qtile * kTile + 64 * g + 32 * i),
                                      (uint32_t)ia.y);
      }
      // a tail key tile: some row of this warp's 32 lies past N (warp-uniform)
      const bool rows_out = kt * kTile + (warp & 3) * 32 + 31 >= a.N;
      if (!warp_wait(w, bar_s_full, it & 1)) return false;
      tc_fence_after();
      {
        uint32_t u[64];
        tmem_ld64(tmem + L::T_S + lane_off + 64 * g, u);
#pragma unroll
        for (int c = 0; c < 64; ++c) p[c] = __uint_as_float(u[c]);
      }
      const float4* nl4 = reinterpret_cast<const float4*>(stat(it) + 64 * g);  // -LSE*log2(e)
      const int q0 = qtile * kTile + 64 * g;
      const bool diag = a.m.causal && qtile == kt;
      uint32_t pk[32];
#pragma unroll
      for (int c = 0; c < 64; c += 4) {
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
        for (int c = 0; c < 64; ++c)
          if (key >= a.N || (diag && q0 + c < key)) p[c] = 0.f;
      }
      // P^T for dV: with dropout the kept weights times the keep scale z, else 0
#pragma unroll
      for (int c = 0; c < 64; c += 2) {
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
      tmem_st32(tmem + L::pt_write_col(g) + lane_off, pk);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_p_full);
      return true;
    };
    // dK, dV of the piece that ended with tile it (key tile kt of head bh)
    auto write_piece = [&](int kt, int bh, int slot, bool have) {
      const int key = kt * kTile + r;
      if (slot < 0) {
        // the whole key tile: dK = scale * sum dS^T Q, dV, in the 16-bit type
        const bool store = key < a.N;
        uint16_t* dVrow = reinterpret_cast<uint16_t*>(a.dV) + ((size_t)bh * a.N + key) * D + g * (D / 2);
        uint16_t* dKrow = reinterpret_cast<uint16_t*>(a.dK) + ((size_t)bh * a.N + key) * D + g * (D / 2);
        for (int which = 0; which < 2; ++which) {
          const uint32_t col = (which == 0 ? L::T_DV : L::T_DK) + g * (D / 2);
          const float mul = which == 0 ? 1.f : a.scale;
          uint16_t* dst = which == 0 ? dVrow : dKrow;
#pragma unroll
          for (int c0 = 0; c0 < D / 2; c0 += 32) {
            uint32_t u[32];
            if (have) {
              tmem_ld32(tmem + col + lane_off + c0, u);
            } else {
#pragma unroll
              for (int i = 0; i < 32; ++i) u[i] = 0u;
            }
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              uint4 pq;
              pq.x = pack2<F16>(__uint_as_float(u[v * 8 + 0]) * mul, __uint_as_float(u[v * 8 + 1]) * mul);
              pq.y = pack2<F16>(__uint_as_float(u[v * 8 + 2]) * mul, __uint_as_float(u[v * 8 + 3]) * mul);
              pq.z = pack2<F16>(__uint_as_float(u[v * 8 + 4]) * mul, __uint_as_float(u[v * 8 + 5]) * mul);
              pq.w = pack2<F16>(__uint_as_float(u[v * 8 + 6]) * mul, __uint_as_float(u[v * 8 + 7]) * mul);
              if (store) *reinterpret_cast<uint4*>(dst + c0 + v * 8) = pq;
            }
          }
        }
      } else {
        // part of a key tile shared with other CTAs: fp32 partial sums of dV
        // and of dK / scale into this CTA's slot, [dV rows 0..127 | dK rows 0..127]
        float* sl = a.slots + (size_t)slot * (2 * kTile * D);
        for (int which = 0; which < 2; ++which) {
          const uint32_t col = (which == 0 ? L::T_DV : L::T_DK) + g * (D / 2);
          float* dst = sl + (size_t)which * kTile * D + (size_t)r * D + g * (D / 2);
#pragma unroll
          for (int c0 = 0; c0 < D / 2; c0 += 32) {
            uint32_t u[32];
            tmem_ld32(tmem + col + lane_off + c0, u);
#pragma unroll
            for (int v = 0; v < 8; ++v)
              *reinterpret_cast<float4*>(dst + c0 + v * 4) =
                  make_float4(__uint_as_float(u[v * 4 + 0]), __uint_as_float(u[v * 4 + 1]),
                              __uint_as_float(u[v * 4 + 2]), __uint_as_float(u[v * 4 + 3]));
          }
        }
      }
    };
    if (empty) {
      // a key tile that no query sees (block mask): dK = dV = 0
      write_piece((int)(blockIdx.x / BH), (int)(blockIdx.x % BH), -1, false);
    } else {
      bool ok = p_phase(0);
      for (int it = 0; ok; ++it) {
        // this tile's coordinates (its stage is not reused before dK_i completes)
        const int4 ia = info_a(it);
        const int2 ib = info_b(it);
        const int kt = ia.x, bh = ia.y, qt = ia.z, slot = ia.w;
        const int pc = ib.x, fl = ib.y;
        const bool last = fl & kLast, more = fl & kMore;
        // ---- dS_i = P_i * (dP_i - D)
        if (!(ok = warp_wait(w, bar_dp_full, it & 1))) break;
        tc_fence_after();
        uint32_t pk[32];
        {
          uint32_t u[64];
          tmem_ld64(tmem + L::T_DP + lane_off + 64 * g, u);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_dp_free);
          if constexpr (DROP) {  // dS = P (z dP - D)
#pragma unroll
            for (int c = 0; c < 64; ++c)
              u[c] = __float_as_uint(keep(c) ? __uint_as_float(u[c]) * a.drop.z : 0.f);
          }
          const float4* nd4 = reinterpret_cast<const float4*>(stat(it) + 128 + 64 * g);  // -D
#pragma unroll
          for (int c = 0; c < 64; c += 4) {
            const float4 nd = nd4[c / 4];
            float y0, y1, y2, y3;
            f2unpack(fmul2(f2pack(p[c], p[c + 1]),
                           fadd2(f2pack(__uint_as_float(u[c]), __uint_as_float(u[c + 1])), f2pack(nd.x, nd.y))),
                     y0, y1);
            f2unpack(fmul2(f2pack(p[c + 2], p[c + 3]),
                           fadd2(f2pack(__uint_as_float(u[c + 2]), __uint_as_float(u[c + 3])), f2pack(nd.z, nd.w))),
                     y2, y3);
            pk[c / 2] = pack2<F16>(y0, y1);
            pk[c / 2 + 1] = pack2<F16>(y2, y3);
          }
        }
        if (it > 0 && !(ok = warp_wait(w, bar_ds_free, (it - 1) & 1))) break;
        // at d = 128 the last dQ reduction must have finished reading this region
        if (!L::STG_SEP) stg_acquire();
#pragma unroll
        for (int ch = 0; ch < 8; ++ch)
          st_shared_v4(sb + L::DST + sw128_chunk_offset(r, 8 * g + ch, kTile), pk[ch * 4 + 0],
                       pk[ch * 4 + 1], pk[ch * 4 + 2], pk[ch * 4 + 3]);
        fence_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_ds_full);

        // ---- P of the next tile, while dK_i, dQ_i, dP^T_{i+1} run (at d = 128
        // only within the piece: the next piece's first P follows its reload)
        const bool ahead = KV2 ? more : (more && !last);
        if (ahead && !(ok = p_phase(it + 1))) break;

        // ---- dQ_i (TMEM lane = query row) -> fp32 accumulator by TMA reduce-add
        if (!(ok = warp_wait(w, bar_dq_full, it & 1))) break;
        tc_fence_after();
        uint32_t dq[D / 2];
        if constexpr (D == 64) {
          tmem_ld32(tmem + L::T_DQ + lane_off + g * (D / 2), *reinterpret_cast<uint32_t(*)[32]>(dq));
        } else {
          tmem_ld64(tmem + L::T_DQ + lane_off + g * (D / 2), *reinterpret_cast<uint32_t(*)[64]>(dq));
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_dq_free);
#pragma unroll
        for (int c0 = 0; c0 < D / 2; c0 += 32) {
          stg_acquire();
          // row `lane` of this warp's 32, 16-byte chunk x at x ^ (row & 7)
#pragma unroll
          for (int x = 0; x < 8; ++x)
            st_shared_v4(stg + (uint32_t)lane * 128u + (uint32_t)((x ^ (lane & 7)) * 16), dq[c0 + 4 * x],
                         dq[c0 + 4 * x + 1], dq[c0 + 4 * x + 2], dq[c0 + 4 * x + 3]);
          fence_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_reduce_add_3d(&tmdQ, stg, g * (D / 2) + c0, qt * kTile + (warp & 3) * 32, bh);
            bulk_commit_group();
          }
          pend = true;
        }

        if (last) {
          // ---- the piece's dK, dV
          if (!(ok = warp_wait(w, bar_acc_full, pc & 1))) break;
          tc_fence_after();
          // tcgen05.ld is .sync.aligned: every lane of the warp loads; only the
          // stores are predicated on the row
          write_piece(kt, bh, slot, true);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_acc_free);
          // d = 128: the next piece's first P, after its K_j, V_j reload
          if (!KV2 && more && !(ok = p_phase(it + 1))) break;
        }
        if (!more) break;
      }
    }
    if (lane == 0) bulk_wait_group0();  // this warp's dQ reductions fully done
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, L::TMEM_COLS);
  }
}

template <int D, bool F16>
cudaError_t launch_t(const BwdArgs& a, const CUtensorMap* tm, cudaStream_t s) {
  using L = BwdLayout<D>;
  auto kern = a.drop.on ? bwd_persist_kernel<D, F16, true> : bwd_persist_kernel<D, F16, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::BYTES);
  if (e != cudaSuccess) return e;
  const int n_tiles = (a.N + kTile - 1) / kTile;
  const unsigned grid = a.G > 0 ? (unsigned)a.G : (unsigned)(n_tiles * a.B * a.H);
  kern<<<grid, 320, L::BYTES, s>>>(tm[0], tm[1], tm[2], tm[3], tm[4], a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_persist(const BwdArgs& a, int d, bool f16, const CUtensorMap* tm, cudaStream_t s) {
  if (d == 64) return f16 ? launch_t<64, true>(a, tm, s) : launch_t<64, false>(a, tm, s);
  return f16 ? launch_t<128, true>(a, tm, s) : launch_t<128, false>(a, tm, s);
}

}  // namespace fa
