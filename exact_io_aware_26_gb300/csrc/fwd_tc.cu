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
//   O   = O * e^(m - m') + P~ V_j        rescale in TMEM, then tcgen05.mma
// and at the end O / l and LSE = m + ln l are written out.
//
// Warp roles (192 threads):
//   warps 0-3  softmax: thread t owns query row t = TMEM lane t;
//   warp 4     TMA producer: Q once, then K_j / V_j through a 2-stage ring;
//   warp 5     TMEM allocator and MMA issuer (one thread).
// The MMA thread issues S_{j+1} as soon as the softmax warps have copied S_j
// into registers, so the tensor core computes the next score tile while the
// exponentials of the current one run on the CUDA cores ("FA3 : Mécanique de
// la trémie", point 2).  Tiles hidden by the causal rule or the block mask
// are never loaded ("Le masquage causal ...": "jamais chargée et jamais
// calculée").
#include "ptx.cuh"

namespace fa {
namespace {

constexpr int kTile = 128;  // query rows per CTA = keys per K/V tile

template <int D>
struct FwdLayout {
  static constexpr uint32_t TILE = kTile * D * 2;     // one 128-row 16-bit tile
  static constexpr uint32_t Q = 0;
  static constexpr uint32_t K0 = Q + TILE;            // K stage s at K0 + s * TILE
  static constexpr uint32_t V0 = K0 + 2 * TILE;       // V stage s at V0 + s * TILE
  static constexpr uint32_t P = V0 + 2 * TILE;        // 128 x 128 16-bit probabilities
  static constexpr uint32_t BAR = P + kTile * kTile * 2;
  // barriers: 0 q_full, 1-2 k_full, 3-4 v_full, 5-6 kv_empty, 7 s_full,
  //           8 s_free, 9 p_full, 10 o_done, 11 fin
  static constexpr uint32_t NBAR = 12;
  static constexpr uint32_t TSLOT = BAR + NBAR * 8;
  static constexpr uint32_t ABORT = TSLOT + 4;
  static constexpr uint32_t BYTES = ABORT + 4;
  static constexpr uint32_t TMEM_COLS = 256;          // S: 128 columns, O: D columns
};

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

template <int D, bool F16>
__global__ void __launch_bounds__(192, (D == 64 ? 2 : 1))
    fwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const FwdArgs a) {
  using L = FwdLayout<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sb = smem_addr(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int BH = a.B * a.H;
  const int n_tiles = (a.N + kTile - 1) / kTile;
  const int qt = n_tiles - 1 - (int)(blockIdx.x / BH);  // heaviest (causal) tiles first
  const int bh = (int)(blockIdx.x % BH);
  const int b = bh / a.H, h = bh % a.H;
  const int kt_end = a.m.causal ? min(qt + 1, n_tiles) : n_tiles;

  const uint32_t bar_q = sb + L::BAR;
  auto bar_k = [&](int s) { return sb + L::BAR + 8u * (1 + s); };
  auto bar_v = [&](int s) { return sb + L::BAR + 8u * (3 + s); };
  auto bar_e = [&](int s) { return sb + L::BAR + 8u * (5 + s); };
  const uint32_t bar_s_full = sb + L::BAR + 8u * 7;
  const uint32_t bar_s_free = sb + L::BAR + 8u * 8;
  const uint32_t bar_p = sb + L::BAR + 8u * 9;
  const uint32_t bar_o = sb + L::BAR + 8u * 10;
  const uint32_t bar_fin = sb + L::BAR + 8u * 11;
  volatile int* abort_cta = reinterpret_cast<volatile int*>(smem + L::ABORT);
  const WaitCtx w{abort_cta, a.rep.st, a.rep.epoch, a.rep.wait_ns};

  if ((sb & 1023u) != 0) {  // the swizzled layouts need a 1024-byte aligned base
    if (threadIdx.x == 0) raise_error(w, FA_ERR_CUDA);
    return;
  }
  if (threadIdx.x == 0) {
    mbar_init(bar_q, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar_k(s), 1);
      mbar_init(bar_v(s), 1);
      mbar_init(bar_e(s), 1);
    }
    mbar_init(bar_s_full, 1);
    mbar_init(bar_s_free, 4);
    mbar_init(bar_p, 4);
    mbar_init(bar_o, 1);
    mbar_init(bar_fin, 1);
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
  const uint32_t tS = tmem;          // columns [0, 128)
  const uint32_t tO = tmem + kTile;  // columns [128, 128 + D)

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
      mbar_arrive_expect_tx(bar_q, L::TILE);
      for (int c = 0; c < D / 64; ++c)
        tma_load_3d(sb + L::Q + c * (kTile * 128), &tmQ, bar_q, c * 64, qt * kTile, bh);
      int it = 0;
      for (int kt = 0; kt < kt_end; ++kt) {
        if (!tile_kept(a.m, b, h, qt, kt)) continue;
        const int s = it & 1;
        if (it >= 2 && !mbar_wait(w, bar_e(s), ((it >> 1) - 1) & 1)) break;
        mbar_arrive_expect_tx(bar_k(s), L::TILE);
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(sb + L::K0 + s * L::TILE + c * (kTile * 128), &tmK, bar_k(s), c * 64,
                      kt * kTile, bh);
        mbar_arrive_expect_tx(bar_v(s), L::TILE);
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(sb + L::V0 + s * L::TILE + c * (kTile * 128), &tmV, bar_v(s), c * 64,
                      kt * kTile, bh);
        ++it;
      }
      // every copy issued must have landed before the CTA may exit
      mbar_drain(w, bar_q, 0);
      for (int s = 0; s < 2; ++s) {
        const int n = (it + 1 - s) / 2;  // loads issued into stage s
        if (n > 0) {
          mbar_drain(w, bar_k(s), (n - 1) & 1);
          mbar_drain(w, bar_v(s), (n - 1) & 1);
        }
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idS = idesc_f16(F16, kTile, kTile, false, false);
      constexpr uint32_t idO = idesc_f16(F16, kTile, D, false, true);
      auto issue_pv = [&](int t) -> bool {
        const int s = t & 1;
        if (!mbar_wait(w, bar_p, t & 1)) return false;
        if (!mbar_wait(w, bar_v(s), (t >> 1) & 1)) return false;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk)
          tc_mma_ss(tO, desc_kmajor(sb + L::P, kk, kTile),
                    desc_mnmajor(sb + L::V0 + s * L::TILE, kk, kTile), idO,
                    (t > 0 || kk > 0) ? 1u : 0u);
        tc_commit(bar_o);
        tc_commit(bar_e(s));
        return true;
      };
      bool ok = mbar_wait(w, bar_q, 0);
      int it = 0;
      for (int kt = 0; ok && kt < kt_end; ++kt) {
        if (!tile_kept(a.m, b, h, qt, kt)) continue;
        const int s = it & 1;
        if (!(ok = mbar_wait(w, bar_k(s), (it >> 1) & 1))) break;
        if (it > 0 && !(ok = mbar_wait(w, bar_s_free, (it - 1) & 1))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          tc_mma_ss(tS, desc_kmajor(sb + L::Q, kk, kTile),
                    desc_kmajor(sb + L::K0 + s * L::TILE, kk, kTile), idS, kk > 0 ? 1u : 0u);
        tc_commit(bar_s_full);
        if (it > 0 && !(ok = issue_pv(it - 1))) break;
        ++it;
      }
      if (ok && it > 0) issue_pv(it - 1);
      // every MMA issued must have completed before TMEM is released
      tc_commit(bar_fin);
      mbar_drain(w, bar_fin, 0);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int r = threadIdx.x;  // query row in the tile = TMEM lane
    const int row = qt * kTile + r;
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const float c2 = a.scale_log2;
    float m2 = -INFINITY;  // running max of scale*log2(e)*S, log2 units
    float l = 0.f;         // running sum of exp2(...) in fp32
    bool ok = true;
    int it = 0;
    for (int kt = 0; kt < kt_end; ++kt) {
      if (!tile_kept(a.m, b, h, qt, kt)) continue;
      if (!(ok = warp_wait(w, bar_s_full, it & 1))) break;
      tc_fence_after();
      float s[kTile];
      {
        uint32_t u[64];
        tmem_ld64(tS + lane_off, u);
#pragma unroll
        for (int c = 0; c < 64; ++c) s[c] = __uint_as_float(u[c]);
        tmem_ld64(tS + lane_off + 64, u);
#pragma unroll
        for (int c = 0; c < 64; ++c) s[64 + c] = __uint_as_float(u[c]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_s_free);

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
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < kTile; ++c) mx = fmaxf(mx, s[c]);
      const float m_new = fmaxf(m2, mx * c2);
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = ex2(m2 - m_use);
      float sum = 0.f;
#pragma unroll
      for (int c = 0; c < kTile; ++c) {
        s[c] = ex2(fmaf(s[c], c2, -m_use));
        sum += s[c];
      }
      l = l * alpha + sum;

      if (it > 0) {
        // P~ V of the previous tile must be done: it read the P buffer and
        // wrote the O accumulator that is rescaled now
        if (!(ok = warp_wait(w, bar_o, (it - 1) & 1))) break;
        tc_fence_after();
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
          for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t o[32];
            tmem_ld32(tO + lane_off + c0, o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st32(tO + lane_off + c0, o);
          }
          tmem_st_wait();
        }
      }
      // P~ (16-bit) -> shared memory, K-major 128-byte-swizzled, row r
#pragma unroll
      for (int ch = 0; ch < kTile / 8; ++ch) {
        st_shared_v4(sb + L::P + sw128_chunk_offset(r, ch, kTile),
                     pack2<F16>(s[ch * 8 + 0], s[ch * 8 + 1]),
                     pack2<F16>(s[ch * 8 + 2], s[ch * 8 + 3]),
                     pack2<F16>(s[ch * 8 + 4], s[ch * 8 + 5]),
                     pack2<F16>(s[ch * 8 + 6], s[ch * 8 + 7]));
      }
      fence_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_p);
      m2 = m_new;
      ++it;
    }
    // ------------------------------------------------------------ epilogue
    bool have_o = false;
    if (ok && it > 0) {
      ok = warp_wait(w, bar_o, (it - 1) & 1);
      tc_fence_after();
      have_o = ok;
    }
    const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
    if (row < a.N && ok) {
      a.LSE[(size_t)bh * a.N + row] =
          (l > 0.f) ? (m2 + __log2f(l)) * 0.693147180559945309f : -INFINITY;
    }
    typedef uint16_t elem_t;
    elem_t* Orow = reinterpret_cast<elem_t*>(a.O) + ((size_t)bh * a.N + row) * D;
#pragma unroll
    for (int c0 = 0; c0 < D; c0 += 32) {
      uint32_t o[32];
      if (have_o) {
        tmem_ld32(tO + lane_off + c0, o);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] = 0u;
      }
      if (row < a.N && ok) {
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          uint4 pk;
          pk.x = pack2<F16>(__uint_as_float(o[v * 8 + 0]) * inv_l, __uint_as_float(o[v * 8 + 1]) * inv_l);
          pk.y = pack2<F16>(__uint_as_float(o[v * 8 + 2]) * inv_l, __uint_as_float(o[v * 8 + 3]) * inv_l);
          pk.z = pack2<F16>(__uint_as_float(o[v * 8 + 4]) * inv_l, __uint_as_float(o[v * 8 + 5]) * inv_l);
          pk.w = pack2<F16>(__uint_as_float(o[v * 8 + 6]) * inv_l, __uint_as_float(o[v * 8 + 7]) * inv_l);
          *reinterpret_cast<uint4*>(Orow + c0 + v * 8) = pk;
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, L::TMEM_COLS);
  }
}

template <int D, bool F16>
cudaError_t launch_t(const FwdArgs& a, const CUtensorMap* tm, cudaStream_t s) {
  using L = FwdLayout<D>;
  auto kern = fwd_tc_kernel<D, F16>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::BYTES);
  if (e != cudaSuccess) return e;
  const int n_tiles = (a.N + kTile - 1) / kTile;
  const unsigned grid = (unsigned)(n_tiles * a.B * a.H);
  kern<<<grid, 192, L::BYTES, s>>>(tm[0], tm[1], tm[2], a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_tc(const FwdArgs& a, int d, bool f16, const CUtensorMap* tm, cudaStream_t s) {
  if (d == 64) return f16 ? launch_t<64, true>(a, tm, s) : launch_t<64, false>(a, tm, s);
  return f16 ? launch_t<128, true>(a, tm, s) : launch_t<128, false>(a, tm, s);
}

}  // namespace fa
