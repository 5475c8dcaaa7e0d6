// fwd_tc.cu -- attention forward on the 5th-generation tensor cores (sm_103a).
//
// One CTA owns one 128-row query tile Q_i of one (batch, head) and walks the
// 128-key tiles (K_j, V_j) that the causal rule and the block mask leave,
// following "L'algorithme Flash Attention" (marketmaker.cc) and "Método" of the
// FlashAttention reading guide, with the deferred normalisation of "FA2 :
// parallélisme":
//   S   = Q_i K_j^T                      tcgen05.mma, f32 accumulator in TMEM
//   m'  = max(m, rowmax(scale * S))      one thread per row (TMEM lane)
//   P~  = exp(scale * S - m')            exp2 with log2(e) folded into scale
//   l   = l * e^(m - m') + rowsum(P~)
//   O   = O * e^(m - m') + P~ V_j        P~ written to TMEM as 16-bit, then
//                                        tcgen05.mma with A read from TMEM
// and at the end O / l and LSE = m + ln l are written out.
//
// The running max is only moved when a row's new maximum exceeds the one in
// use by more than 2^8 (in the exp2 domain): until then P~ <= 2^8, which fp32
// sums and the 16-bit P~ hold exactly as well, and O and l keep sharing the
// same stale max, so the result is unchanged while most tiles skip the O
// rescale.
//
// At d = 64 P~ has TMEM columns of its own, so S_{j+1} is computed while the
// softmax of tile j runs; at d = 128 P~ overwrites S and the schedule is
// serial (S_j, softmax, P~V_j, S_{j+1}).  Two CTAs share each SM (256 TMEM
// columns and at most 100 KiB of shared memory each), so one CTA's
// exponentials run on the CUDA cores while the other's MMAs run on the tensor
// core ("FA3 : Mécanique de la trémie", point 2, realised across CTAs).
//
// Split-KV (a separate instantiation, SPLIT): the key range of a query tile is
// cut into slices run by the CTAs of one thread-block cluster, which merge
// their running statistics and partial O through distributed shared memory.
//
// Dropout (a separate instantiation): after the exponentials of a tile, each
// weight whose 16-bit Philox4x32-10 draw is below the threshold is replaced by 0 and
// each other one is multiplied by the keep scale before P~ V; l sums the undropped
// weights, so O / l and LSE are those of the dropped-out attention and of the
// undropped scores respectively.
//
// Warp roles (192 threads): warps 0-3 softmax (thread t owns query row t =
// TMEM lane t); warp 4 TMA producer (Q once, K_j and V_j through a ring of
// NS stages with separate K and V barriers); warp 5 TMEM owner and MMA
// issuer.  Tiles hidden by the causal rule or the block mask are never
// loaded ("Le masquage causal ...": "jamais chargée et jamais calculée").
#include "bwd_sched.cuh"
#include "fwd_common.cuh"

namespace fa {
namespace {

constexpr float kRescaleThr = 8.f;  // move the running max only past 2^8
constexpr int kMaxSplits = FA_MAX_SPLITS;  // key-range slices of a query tile: one cluster

template <int D>
struct FwdLayout {
  static constexpr uint32_t TILE = kTile * D * 2;  // one 128-row 16-bit tile
  static constexpr int NS = (D == 64) ? 2 : 1;     // K/V ring depth
  static constexpr uint32_t Q = 0;
  static constexpr uint32_t K0 = Q + TILE;          // K stage s at K0 + s * TILE
  static constexpr uint32_t V0 = K0 + NS * TILE;    // V stage s at V0 + s * TILE
  static constexpr uint32_t BAR = V0 + NS * TILE;  // FwdBars<NS>
  static constexpr uint32_t TSLOT = BAR + FwdBars<NS>::kCount * 8;
  static constexpr uint32_t ABORT = TSLOT + 4;
  static constexpr uint32_t KBITS = ABORT + 4;  // the key tiles this query tile sees (block mask)
  // split launches: each row's (running max, sum) for the cluster's merge
  static constexpr uint32_t MST = (KBITS + kMaskBitBytes + 7) & ~7u;
  static constexpr uint32_t BYTES = MST + kTile * 8;
  // split launches: the weighted partial O, fp32 [128][D], over the K/V stages
  // once every copy and product has completed
  static constexpr uint32_t OBUF = K0;
  static_assert(kTile * D * 4 <= 2 * NS * TILE, "merge buffer");
  // TMEM (256 columns): S at [0, 128), O at [128, 128 + D).  At d = 64 the 16-bit
  // P~ has columns of its own, [192, 256), so S_{j+1} can be computed while the
  // softmax of tile j runs; at d = 128 P~ is written over the first 64 columns of S
  // and the schedule is serial.
  static constexpr uint32_t TMEM_COLS = 256;
  static constexpr bool PSEP = (D == 64);
  static constexpr uint32_t T_S = 0, T_O = 128, T_P = PSEP ? 192 : 0;
};



template <int D, bool F16, bool DROP, bool MASKED, bool SPLIT>
__global__ void __launch_bounds__(192, 2)
    fwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const FwdArgs a) {
  using L = FwdLayout<D>;
  constexpr int NS = L::NS;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sb = smem_addr(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int BH = a.B * a.H;
  const int n_tiles = (a.N + kTile - 1) / kTile;
  const int split = (int)(blockIdx.x % a.n_splits);
  const int tile = (int)(blockIdx.x / a.n_splits);
  // heads in groups of head_group; within a group the heaviest (causal) query
  // tiles of all its heads first
  int qt, bh;
  group_order(tile, n_tiles, BH, a.head_group, a.head_tail, qt, bh);
  qt = n_tiles - 1 - qt;
  const int b = bh / a.H, h = bh % a.H;
  // this CTA's key tiles: [kt_begin, kt_end)
  const int kt_begin = split * a.split_tiles;
  int kt_end = min(a.m.causal ? min(qt + 1, n_tiles) : n_tiles, kt_begin + a.split_tiles);

  const FwdBars<NS> bars{sb + L::BAR};
  volatile int* abort_cta = reinterpret_cast<volatile int*>(smem + L::ABORT);
  const WaitCtx w{abort_cta, a.rep.st, a.rep.epoch, a.rep.wait_ns};

  if ((sb & 1023u) != 0) {  // the swizzled layouts need a 1024-byte aligned base
    if (threadIdx.x == 0) raise_error(w, FA_ERR_CUDA);
    return;
  }
  // debug build: the CTA's tile, head and key range lie inside the problem.  A
  // CTA of a split launch must reach its cluster's barriers even then: it keeps
  // an empty key range and writes nothing.
  const bool cta_ok = dbg_check(w, qt >= 0 && qt < n_tiles && bh >= 0 && bh < BH && kt_begin >= 0 &&
                                       kt_end <= n_tiles && split < a.n_splits);
  if (!cta_ok) {
    if (!SPLIT) return;
    kt_end = kt_begin;
  }
  // The producer lane sets up the barriers and, before the block-wide setup
  // barrier, already issues the copies that need no wait (Q and the first NS
  // K, V tiles), so that their latency overlaps the TMEM allocation.
  const bool producer = (warp == 4 && lane == 0);
  int nk = 0, nv = 0;  // producer lane: K and V copies issued
  int kt_next = kt_end;  // producer lane: the next key tile to copy
  // K_j, V_j of key tile kt into ring stage st: D / 64 boxes of 64 columns each
  auto load_k = [&](int st, int kt) {
    mbar_arrive_expect_tx(bars.kf(st), L::TILE);
    for (int c = 0; c < D / 64; ++c)
      tma_load_3d(sb + L::K0 + st * L::TILE + c * (kTile * 128), &tmK, bars.kf(st), c * 64, kt * kTile, bh);
  };
  auto load_v = [&](int st, int kt) {
    mbar_arrive_expect_tx(bars.vf(st), L::TILE);
    for (int c = 0; c < D / 64; ++c)
      tma_load_3d(sb + L::V0 + st * L::TILE + c * (kTile * 128), &tmV, bars.vf(st), c * 64, kt * kTile, bh);
  };
  if (producer) {
    bars.init();
    *abort_cta = 0;
    fence_barrier_init();
    prefetch_tmap(&tmQ);
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
    mbar_arrive_expect_tx(bars.q(), L::TILE);
    for (int c = 0; c < D / 64; ++c)
      tma_load_3d(sb + L::Q + c * (kTile * 128), &tmQ, bars.q(), c * 64, qt * kTile, bh);
    kt_next = fwd_produce(w, bars, next_kept(a.m, b, h, qt, kt_begin, kt_end), kt_end, a.N, NS, nk, nv,
                          [&](int kt) { return next_kept(a.m, b, h, qt, kt, kt_end); }, load_k, load_v);
  }
  // block mask (its own instantiation, MASKED, so that launches without one run
  // unchanged code): this query tile's row of kept key tiles as bits in shared memory
  uint32_t* kbits = reinterpret_cast<uint32_t*>(smem + L::KBITS);
  const bool use_bits = MASKED && n_tiles <= kMaskBits;
  if (use_bits)
    build_tile_bits(kbits, n_tiles, warp, 6, lane, [&](int t) { return tile_kept(a.m, b, h, qt, t); });
  if (warp == 5) {
    tmem_alloc(sb + L::TSLOT, L::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  // the next kept key tile at or after kt (after the setup barrier)
  auto next_k = [&](int kt) {
    return use_bits ? next_bit(kbits, kt, kt_end) : next_kept(a.m, b, h, qt, kt, kt_end);
  };
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + L::TSLOT);
  // split launches: what the softmax thread of row r hands to the cluster merge
  float m_fin = -INFINITY, l_fin = 0.f;  // running max (exp2 domain) and sum
  bool o_fin = false, ok_fin = false;    // O holds products; no wait gave up

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      // the rest of the K, V tiles, each into a stage once it is released
      if (kt_next >= 0) fwd_produce(w, bars, kt_next, kt_end, a.N, 1 << 30, nk, nv, next_k, load_k, load_v);
      fwd_drain_copies(w, bars, nk, nv);
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t idS = idesc_f16(F16, kTile, kTile, false, false);
    constexpr uint32_t idO = idesc_f16(F16, kTile, D, false, true);
    const uint32_t tS = tmem + L::T_S, tO = tmem + L::T_O;
    const uint64_t dQ = desc_kmajor_base(sb + L::Q);
    const uint64_t dK0 = desc_kmajor_base(sb + L::K0);
    const uint64_t dV0 = desc_mnmajor_base(sb + L::V0, kTile);
    fwd_mma_schedule<NS, L::PSEP>(
        w, bars, next_k(kt_begin), kt_end, next_k,
        [&](int st) {  // S = Q K^T: D / 16 products of K = 16
          const uint64_t dK = desc_add(dK0, (uint32_t)st * L::TILE);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            tc_mma_ss_elect(tS, dQ + kmajor_step(kk, kTile), dK + kmajor_step(kk, kTile), idS,
                            kk > 0 ? 1u : 0u);
        },
        [&](int st, int it) {  // O += P~ V, P~ read from TMEM: 8 products of K = 16 keys
          const uint64_t dV = desc_add(dV0, (uint32_t)st * L::TILE);
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk)
            tc_mma_ts_elect(tO, tmem + L::T_P + (uint32_t)kk * 8u, dV + mnmajor_step(kk), idO,
                            (it > 0 || kk > 0) ? 1u : 0u);
        });
  } else {
    // ------------------------------------------------------------ softmax
    const int r = threadIdx.x;  // query row in the tile = TMEM lane
    const int row = qt * kTile + r;
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const uint32_t tS = tmem + L::T_S + lane_off, tO = tmem + L::T_O + lane_off;
    const float c2 = a.scale_log2;
    float m_use = -INFINITY;  // running max in use (exp2 domain)
    float l = 0.f;            // running sum of P~ (fp32)
    bool ok = true;
    int it = 0;
    for (int kt = next_k(kt_begin); kt < kt_end; kt = next_k(kt + 1), ++it) {
      // d = 128: S_j is complete, and so is every earlier MMA (P~ V_{j-1}
      // included), so O is stable and P~_{j-1} has been consumed.  d = 64 waits
      // for P~ V_{j-1} separately below.
      // dropout: keep bits of the tile's 128 keys for this row (bit c of kb[c / 32]),
      // drawn while S_j is still being computed
      uint32_t kb[4] = {~0u, ~0u, ~0u, ~0u};
      if constexpr (DROP) {
        // one 32-key word at a time (four counters in flight), written by
        // selects so that kb stays in registers
#pragma unroll 1
        for (int w4 = 0; w4 < 4; ++w4) {
          const uint32_t bits =
              drop_keep32(a.drop, (uint32_t)kt * (kTile / 32) + (uint32_t)w4, (uint32_t)row, (uint32_t)bh);
#pragma unroll
          for (int i = 0; i < 4; ++i) kb[i] = (w4 == i) ? bits : kb[i];
        }
      }
      if (!(ok = warp_wait(w, bars.s(), it & 1))) break;
      tc_fence_after();
      float s[kTile];
      float m8[8];
      {
        uint32_t u[64], v[64];
        tmem_ld64(tS, u);
        tmem_ld64_nowait(tS + 64, v);
#pragma unroll
        for (int c = 0; c < 64; ++c) s[c] = __uint_as_float(u[c]);
#pragma unroll
        for (int j = 0; j < 4; ++j) m8[j] = max16(s, j);  // the first half's maxima while the second half arrives
        tmem_wait_ld64(v);
#pragma unroll
        for (int c = 0; c < 64; ++c) s[64 + c] = __uint_as_float(v[c]);
      }
      if (L::PSEP) {  // S_j is in registers: the MMA warp may compute S_{j+1}
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bars.sfree());
      }
      // the rest of the row max as four more independent chains of sixteen (eight
      // chains keep the dependent-max latency short: only two softmax warps share
      // an SM sub-partition); on a tile that masks keys the first four are redone
      // on the masked values
      if (mask_score_row(s, kt, qt, row, a.N, a.m.causal)) {
#pragma unroll
        for (int j = 0; j < 4; ++j) m8[j] = max16(s, j);
      }
#pragma unroll
      for (int j = 4; j < 8; ++j) m8[j] = max16(s, j);
      const float mx = fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
      const float m_tile = mx * c2;
      float alpha = 1.f;
      if (m_tile > m_use + kRescaleThr) {
        alpha = ex2(m_use - m_tile);  // 0 on the first tile that sees a key
        m_use = m_tile;
      }
      const float mneg = (m_use == -INFINITY) ? 0.f : -m_use;
      const uint64_t c2p = f2pack(c2, c2), mp = f2pack(mneg, mneg);
      uint64_t acc[4] = {f2pack(0.f, 0.f), f2pack(0.f, 0.f), f2pack(0.f, 0.f), f2pack(0.f, 0.f)};
      // The tile's exponentials in four chunks of 32 keys; each chunk's 16-bit P~
      // goes to TMEM as soon as it is formed (16 columns), so the stores overlap
      // the next chunk's arithmetic instead of waiting at the end.
      bool o_ready = !(L::PSEP && it > 0);  // P~ V_{j-1} done (d = 128: implied by S_j)
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        uint32_t pk[16];
#pragma unroll
        for (int pr = 0; pr < 16; ++pr) {
          const int c = 32 * ch + 2 * pr;
          float x0, x1;
          f2unpack(ffma2(f2pack(s[c], s[c + 1]), c2p, mp), x0, x1);
          float p0 = ex2(x0), p1 = ex2(x1);
          acc[pr & 3] = fadd2(acc[pr & 3], f2pack(p0, p1));  // four independent sums
          if constexpr (DROP) {  // l sums the undropped weights; P~ V takes the dropped ones
            p0 = ((kb[c >> 5] >> (c & 31)) & 1u) ? p0 * a.drop.z : 0.f;
            p1 = ((kb[(c + 1) >> 5] >> ((c + 1) & 31)) & 1u) ? p1 * a.drop.z : 0.f;
          }
          pk[pr] = pack2<F16>(p0, p1);
        }
        if (!o_ready) {
          // P~ V_{j-1} must be done: it reads the P~ columns and writes O
          if (!(ok = warp_wait(w, bars.o(), (it - 1) & 1))) break;
          tc_fence_after();
          o_ready = true;
        }
        // P~ (16-bit pairs); at d = 128 over the first 64 columns of S, all of
        // which is already in registers
        tmem_st16(tmem + L::T_P + lane_off + 16 * ch, pk);
      }
      if (!ok) break;
      l = l * alpha + sum_packed4(acc);
      if (it > 0 && __any_sync(0xffffffffu, alpha != 1.f)) scale_o_row<D>(tO, alpha);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bars.p());
    }
    // ------------------------------------------------------------ epilogue
    bool have_o = false;
    if (ok && it > 0) {
      // the o_done barrier is at most one phase behind the last P~ V: at d = 64
      // the loop waited every earlier phase, at d = 128 each earlier P~ V
      // completed before the next S did
      ok = warp_wait(w, bars.o(), (it - 1) & 1);
      tc_fence_after();
      have_o = ok;
    }
    const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
    const float lse = (l > 0.f) ? (m_use + __log2f(l)) * 0.693147180559945309f : -INFINITY;
    // debug build: the row's outputs lie inside O and LSE
    if (row < a.N && ok) ok = dbg_check(w, (size_t)bh * a.N + row < (size_t)BH * a.N);
    if constexpr (!SPLIT) {
      if (row < a.N && ok) a.LSE[(size_t)bh * a.N + row] = lse;
      store_o_row<D, F16>(tO, have_o, inv_l, row < a.N && ok,
                          reinterpret_cast<uint16_t*>(a.O) + ((size_t)bh * a.N + row) * D);
    } else {
      // a slice of the key range: the cluster merges the slices below
      m_fin = m_use;
      l_fin = l;
      o_fin = have_o;
      ok_fin = ok;
    }
  }

  if constexpr (SPLIT) {
    // The n_splits CTAs of a query tile form one cluster and merge their slices
    // with the running-statistics merge of "Rastreamento Incremental do Softmax"
    // (FlashAttention reading guide): with M = max_s m_s and L = sum_s l_s 2^(m_s - M),
    // O = sum_s 2^(m_s - M) O_s / L and LSE = (M + log2 L) ln 2 (an empty slice has
    // l_s = 0 and weighs nothing).  Every thread of the cluster reaches the three
    // cluster barriers, after waits that are bounded, and none leaves early.
    const uint32_t rank = cluster_rank();
    const int ks = a.n_splits;
    const int r = (int)threadIdx.x;
    constexpr int CPR = D / 4;  // 16-byte chunks of an O row
    if (warp < 4) reinterpret_cast<float2*>(smem + L::MST)[r] = make_float2(m_fin, l_fin);
    cluster_sync();  // every slice's statistics are visible
    if (warp < 4) {
      float2 st[kMaxSplits];
      float M = -INFINITY, Ls = 0.f;
#pragma unroll
      for (int sp = 0; sp < kMaxSplits; ++sp) {
        st[sp] = make_float2(-INFINITY, 0.f);
        if (sp < ks) st[sp] = ld_cluster_f32x2(cluster_map(sb + L::MST + 8u * (uint32_t)r, (uint32_t)sp));
        if (st[sp].y > 0.f) M = fmaxf(M, st[sp].x);
      }
#pragma unroll
      for (int sp = 0; sp < kMaxSplits; ++sp)
        if (st[sp].y > 0.f) Ls += st[sp].y * ex2(st[sp].x - M);
      const float wgt = (l_fin > 0.f && Ls > 0.f) ? ex2(m_fin - M) / Ls : 0.f;
      const int row = qt * kTile + r;
      if (rank == 0 && row < a.N && cta_ok)
        a.LSE[(size_t)bh * a.N + row] = Ls > 0.f ? (M + __log2f(Ls)) * 0.693147180559945309f : -INFINITY;
      // this slice's weighted O row into the merge buffer (16-byte chunks XOR-
      // swizzled by row, so that a warp's stores spread over the banks)
      const uint32_t tO = tmem + L::T_O + ((uint32_t)(warp * 32) << 16);
      float* ob = reinterpret_cast<float*>(smem + L::OBUF) + (size_t)r * D;
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t o[32];
        if (o_fin) {
          tmem_ld32(tO + c0, o);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = 0u;
        }
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          const int c = c0 / 4 + v;
          *reinterpret_cast<float4*>(ob + 4 * (c ^ (r & (CPR - 1)))) =
              make_float4(__uint_as_float(o[4 * v]) * wgt, __uint_as_float(o[4 * v + 1]) * wgt,
                          __uint_as_float(o[4 * v + 2]) * wgt, __uint_as_float(o[4 * v + 3]) * wgt);
        }
      }
    }
    cluster_sync();  // every slice's weighted O is visible
    if (warp < 4) {
      // CTA `rank` sums its share of the rows over the cluster and writes them
      const int per = (kTile + ks - 1) / ks;
      const int r0 = (int)rank * per, r1 = min(kTile, r0 + per);
      uint16_t* Ob = reinterpret_cast<uint16_t*>(a.O) + ((size_t)bh * a.N + (size_t)qt * kTile) * D;
      for (int e = r; e < (r1 - r0) * CPR; e += kTile) {
        const int rr = r0 + e / CPR, c = e % CPR;
        const uint32_t off = L::OBUF + 4u * (uint32_t)(rr * D + 4 * (c ^ (rr & (CPR - 1))));
        float4 acc = ld_cluster_f32x4(cluster_map(sb + off, 0));
        for (int sp = 1; sp < ks; ++sp) {
          const float4 v = ld_cluster_f32x4(cluster_map(sb + off, (uint32_t)sp));
          acc.x += v.x;
          acc.y += v.y;
          acc.z += v.z;
          acc.w += v.w;
        }
        if (qt * kTile + rr < a.N && cta_ok) {
          uint2 pk;
          pk.x = pack2<F16>(acc.x, acc.y);
          pk.y = pack2<F16>(acc.z, acc.w);
          *reinterpret_cast<uint2*>(Ob + (size_t)rr * D + 4 * c) = pk;
        }
      }
    }
    cluster_sync();  // no CTA leaves while another reads its shared memory
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, L::TMEM_COLS);
  }
}

template <int D, bool F16, bool SPLIT>
cudaError_t launch_t(const FwdArgs& a, const CUtensorMap* tm, cudaStream_t s) {
  using L = FwdLayout<D>;
  auto kern = a.m.mask ? (a.drop.on ? fwd_tc_kernel<D, F16, true, true, SPLIT> : fwd_tc_kernel<D, F16, false, true, SPLIT>)
                       : (a.drop.on ? fwd_tc_kernel<D, F16, true, false, SPLIT> : fwd_tc_kernel<D, F16, false, false, SPLIT>);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::BYTES);
  if (e != cudaSuccess) return e;
  const int n_tiles = (a.N + kTile - 1) / kTile;
  const unsigned grid = (unsigned)(n_tiles * a.B * a.H * a.n_splits);
  if constexpr (!SPLIT) {
    kern<<<grid, 192, L::BYTES, s>>>(tm[0], tm[1], tm[2], a);
    return cudaGetLastError();
  }
  // the key-range slices of a query tile (consecutive CTAs) form one cluster
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(192);
  cfg.dynamicSmemBytes = L::BYTES;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)a.n_splits;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tm[0], tm[1], tm[2], a);
}

template <int D, bool F16>
cudaError_t launch_d(const FwdArgs& a, const CUtensorMap* tm, cudaStream_t s) {
  // split launches (clusters that merge their slices) are their own instantiation
  return a.n_splits > 1 ? launch_t<D, F16, true>(a, tm, s) : launch_t<D, F16, false>(a, tm, s);
}

}  // namespace

cudaError_t launch_fwd_tc(const FwdArgs& a, int d, bool f16, const CUtensorMap* tm, cudaStream_t s) {
  if (d == 64) return f16 ? launch_d<64, true>(a, tm, s) : launch_d<64, false>(a, tm, s);
  return f16 ? launch_d<128, true>(a, tm, s) : launch_d<128, false>(a, tm, s);
}

}  // namespace fa
