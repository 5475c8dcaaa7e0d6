// fwd_fp8.cu -- attention forward on FP8 operands with incoherent processing
// ("Trois idées pour FA3", marketmaker.cc, point 3: rotate the query and key
// vectors at random before quantising them block by block, so that an outlier
// coordinate's magnitude is spread over all coordinates).
//
// Two kernels.
//
// fp8_quant_kernel: one CTA per (tensor, head, 128-row block).  Q and K rows are
// multiplied by D = diag(signs) and by the Sylvester Hadamard matrix H (a fast
// Walsh-Hadamard butterfly in fp32: three stages inside a thread's 8 columns,
// log2(d / 8) across the lanes that share a row), Q^ = Q D H / d and K^ = K D H,
// so that Q^ K^^T = Q K^T (H H^T = d I).  Each block then takes the smallest
// power of two sigma with amax / sigma <= 448 and is stored as e4m3 codes of
// x / sigma (round to nearest even, saturating).  V is not rotated; its codes
// are written transposed ([d][keys]) so that both operands of P~ V are K-major.
//
// fwd_fp8_kernel: the schedule of the 16-bit forward (warps 0-3 softmax, one
// query row per thread; warp 4 TMA producer with a two-stage K/V ring; warp 5
// TMEM owner and MMA issuer; two CTAs per SM; the same grid order over heads and
// the same block-mask bitmask), with
//   S   = Q8 K8^T              tcgen05.mma kind::f8f6f4 (e4m3 x e4m3, f32 in TMEM)
//   s   = S * scale * sigma_q * sigma_k,j   (powers of two: exact)
//   P~  = exp(s - m) against the exact running max m, so that P~ <= 1,
//         quantised as e4m3(256 P~) and stored four codes per TMEM column
//   O   = O * e^(m_old - m) * (u_old / sigma_v,j) + Pq V8_j   with O held in
//         units u = sigma_v of the latest key block (power-of-two changes of
//         unit are exact)
//   l   = l * e^(m_old - m) + rowsum(P~)   (the unquantised fp32 P~)
// and at the end O * u / (256 l) and LSE = m + ln l.  With d = 64 the Q and K
// rows are 64 bytes (64-byte swizzle); with d = 128 they are 128 bytes (128-byte
// swizzle).  P~ has TMEM columns of its own at d = 64; at d = 128 it overwrites
// S and the schedule is serial, as in the 16-bit kernel.
#include "bwd_sched.cuh"
#include "fp8.h"
#include "fwd_common.cuh"

namespace fa {
namespace {

constexpr int kT = kTile;  // rows per block = query rows per CTA = keys per key tile

// ---------------------------------------------------------------- helpers

// Instruction descriptor of tcgen05.mma kind::f8f6f4 with both operands e4m3
// (format 0), both K-major, f32 accumulator: bits 4-5 D format (1 = f32), 7-9 A
// format, 10-12 B format, 17-22 N >> 3, 24-28 M >> 4.
__host__ __device__ constexpr uint32_t idesc_e4m3(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Shared-memory descriptor of a K-major tile whose rows are ROWB bytes, the
// layout a TMA box with the matching swizzle writes: 128-byte rows use the
// 128-byte swizzle (mode 2), 64-byte rows the 64-byte swizzle (mode 4); groups
// of 8 rows are 8 * ROWB bytes apart.  An MMA step of 32 bytes of contraction
// adds 32 bytes (2 units) to the start address.
template <int ROWB>
__device__ __forceinline__ uint64_t desc_k(uint32_t addr) {
  static_assert(ROWB == 64 || ROWB == 128, "64- or 128-byte rows");
  constexpr uint64_t mode = ROWB == 128 ? 2ull : 4ull;
  constexpr uint32_t sbo = 8u * ROWB;
  return (uint64_t)((addr & 0x3FFFFu) >> 4) | (1ull << 16) | ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) |
         (1ull << 46) | (mode << 61);
}

__device__ __forceinline__ void mma_f8_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred e, p;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_f8_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred e, p;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Four values to four e4m3 codes (round to nearest even, saturating to +-448),
// x0 in the lowest byte.  The packed conversion puts its first source in the
// upper byte of each pair.
__device__ __forceinline__ uint32_t pack4_e4m3(float x0, float x1, float x2, float x3) {
  uint16_t lo, hi;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(x1), "f"(x0));
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(x3), "f"(x2));
  return (uint32_t)lo | ((uint32_t)hi << 16);
}

// The smallest power of two sigma with amax / sigma <= 448 = 1.75 * 2^8, read
// off the bits of amax = (1 + f) 2^e: sigma = 2^(e - 8) when 1 + f <= 1.75, else
// 2^(e - 7); 1 for amax = 0 (or NaN).  Returns sigma and sets inv = 1 / sigma
// (both exact).  Blocks with amax below 2^-118 take sigma = 2^-126.
__device__ __forceinline__ float pow2_scale(float amax, float& inv) {
  int k = 0;
  if (amax > 0.f) {
    const uint32_t u = __float_as_uint(amax);
    const int e = (int)((u >> 23) & 0xFFu) - 127;
    k = ((u & 0x7FFFFFu) <= 0x600000u) ? e - 8 : e - 7;
    k = max(k, -126);
  }
  inv = __uint_as_float((uint32_t)(127 - k) << 23);
  return __uint_as_float((uint32_t)(127 + k) << 23);
}



// ---------------------------------------------------------------- quantise

// blockIdx.x = head * T + block, blockIdx.y = tensor (0 Q, 1 K, 2 V).  2d threads:
// d / 8 lanes share a row, each holding 8 consecutive columns (one 16-byte load),
// so a warp covers 256 / d rows per step and 8 steps cover its share of the
// block's 128 rows.  All eight loads of a thread are issued before any of them is
// used.  V's codes go row-major into shared memory (8-byte stores), and each
// 32-byte piece of a transposed row (32 keys of one column) is then gathered with
// byte reads in which consecutive lanes take consecutive columns.
template <int D, bool F16>
__global__ void __launch_bounds__(2 * D) fp8_quant_kernel(const Fp8QuantArgs a) {
  constexpr int NT = 2 * D, NW = NT / 32;
  constexpr int LPR = D / 8;       // lanes per row
  constexpr int RPI = 32 / LPR;    // rows per warp step
  constexpr int RPW = kT / NW;     // rows per warp
  constexpr int IT = RPW / RPI;    // steps
  static_assert(IT == 8, "eight steps of eight columns per thread");
  __shared__ float wmax[NW];
  __shared__ __align__(16) uint8_t vrm[kT * D];  // V block codes, row-major [row][column]

  const int which = blockIdx.y;
  const int bh = blockIdx.x / a.T, t = blockIdx.x % a.T;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ch = lane % LPR, rsub = lane / LPR;
  const uint16_t* src =
      static_cast<const uint16_t*>(which == 0 ? a.Q : which == 1 ? a.K : a.V) + (size_t)bh * a.N * D;
  const bool rotate = which < 2 && a.signs != nullptr;

  uint4 raw[IT];
#pragma unroll
  for (int it = 0; it < IT; ++it) {
    const int r = t * kT + warp * RPW + it * RPI + rsub;
    raw[it] = make_uint4(0u, 0u, 0u, 0u);
    if (r < a.N) raw[it] = __ldg(reinterpret_cast<const uint4*>(src + (size_t)r * D + ch * 8));
  }
  float sg[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) sg[e] = rotate ? a.signs[ch * 8 + e] : 1.f;
  const float post = (rotate && which == 0) ? 1.f / (float)D : 1.f;

  float x[IT][8];
  float amax = 0.f;
#pragma unroll
  for (int it = 0; it < IT; ++it) {
    float v[8];
    {
      const float2 p0 = unpack2<F16>(raw[it].x), p1 = unpack2<F16>(raw[it].y),
                   p2 = unpack2<F16>(raw[it].z), p3 = unpack2<F16>(raw[it].w);
      v[0] = p0.x, v[1] = p0.y, v[2] = p1.x, v[3] = p1.y, v[4] = p2.x, v[5] = p2.y, v[6] = p3.x, v[7] = p3.y;
    }
    if (rotate) {
#pragma unroll
      for (int e = 0; e < 8; ++e) v[e] *= sg[e];
      // butterflies over column bits 0-2 (inside the thread) ...
#pragma unroll
      for (int s = 1; s < 8; s <<= 1)
#pragma unroll
        for (int e = 0; e < 8; ++e)
          if (!(e & s)) {
            const float lo = v[e], hi = v[e + s];
            v[e] = lo + hi;
            v[e + s] = lo - hi;
          }
      // ... and over column bits 3 and up (lane bits inside the row's lane group)
#pragma unroll
      for (int s = 1; s < LPR; s <<= 1) {
        const bool upper = (ch & s) != 0;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float o = __shfl_xor_sync(0xffffffffu, v[e], s);
          v[e] = upper ? o - v[e] : v[e] + o;
        }
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) v[e] *= post;
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      x[it][e] = v[e];
      amax = fmaxf(amax, fabsf(v[e]));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if (lane == 0) wmax[warp] = amax;
  __syncthreads();
  float bmax = wmax[0];
#pragma unroll
  for (int w = 1; w < NW; ++w) bmax = fmaxf(bmax, wmax[w]);
  float inv;
  const float sigma = pow2_scale(bmax, inv);

  if (which < 2) {
    uint8_t* dst = (which == 0 ? a.q8 : a.k8) + (size_t)bh * a.N * D;
#pragma unroll
    for (int it = 0; it < IT; ++it) {
      const int r = t * kT + warp * RPW + it * RPI + rsub;
      if (r < a.N) {
        uint2 w;
        w.x = pack4_e4m3(x[it][0] * inv, x[it][1] * inv, x[it][2] * inv, x[it][3] * inv);
        w.y = pack4_e4m3(x[it][4] * inv, x[it][5] * inv, x[it][6] * inv, x[it][7] * inv);
        *reinterpret_cast<uint2*>(dst + (size_t)r * D + ch * 8) = w;
      }
    }
  } else {
#pragma unroll
    for (int it = 0; it < IT; ++it) {
      const int rl = warp * RPW + it * RPI + rsub;  // row in the block (rows past N hold 0)
      uint2 w;
      w.x = pack4_e4m3(x[it][0] * inv, x[it][1] * inv, x[it][2] * inv, x[it][3] * inv);
      w.y = pack4_e4m3(x[it][4] * inv, x[it][5] * inv, x[it][6] * inv, x[it][7] * inv);
      *reinterpret_cast<uint2*>(vrm + rl * D + ch * 8) = w;
    }
    __syncthreads();
    // piece (c, k32): keys [32 k32, 32 k32 + 32) of column c; c runs fastest over the
    // threads, so the byte reads of a warp hit consecutive bytes of one row
    uint8_t* dst = a.vt8 + (size_t)bh * D * a.ld;
    for (int i = threadIdx.x; i < D * (kT / 32); i += NT) {
      const int c = i % D, k32 = i / D;
      const int col = t * kT + k32 * 32;
      uint32_t wds[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const uint8_t* b = vrm + (k32 * 32 + q * 4) * D + c;
        wds[q] = (uint32_t)b[0] | ((uint32_t)b[D] << 8) | ((uint32_t)b[2 * D] << 16) | ((uint32_t)b[3 * D] << 24);
      }
      uint8_t* out = dst + (size_t)c * a.ld + col;
      if (col < a.ld) *reinterpret_cast<uint4*>(out) = make_uint4(wds[0], wds[1], wds[2], wds[3]);
      if (col + 16 < a.ld) *reinterpret_cast<uint4*>(out + 16) = make_uint4(wds[4], wds[5], wds[6], wds[7]);
    }
  }
  if (threadIdx.x == 0) (which == 0 ? a.sq : which == 1 ? a.sk : a.sv)[(size_t)bh * a.T + t] = sigma;
}

// ---------------------------------------------------------------- forward

template <int D>
struct F8Layout {
  static constexpr uint32_t TQ = kT * D;  // a Q8 or K8 tile: 128 rows of D bytes
  static constexpr uint32_t TV = D * kT;  // a Vt8 tile: D rows of 128 bytes
  static constexpr int NS = 2;            // K/V ring depth
  static constexpr uint32_t Q = 0;
  static constexpr uint32_t K0 = Q + TQ;
  static constexpr uint32_t V0 = K0 + NS * TQ;
  static constexpr uint32_t BAR = V0 + NS * TV;  // FwdBars<NS>
  static constexpr uint32_t TSLOT = BAR + FwdBars<NS>::kCount * 8;
  static constexpr uint32_t ABORT = TSLOT + 4;
  static constexpr uint32_t KBITS = ABORT + 4;  // the key tiles this query tile sees (block mask)
  static constexpr uint32_t BYTES = KBITS + kMaskBitBytes;
  // TMEM (256 columns): S [0, 128), O [128, 128 + D); the e4m3 P~ (128 keys, four
  // per column) at [192, 224) for d = 64, over the first 32 columns of S for d = 128
  static constexpr uint32_t TMEM_COLS = 256;
  static constexpr bool PSEP = (D == 64);
  static constexpr uint32_t T_S = 0, T_O = 128, T_P = PSEP ? 192 : 0;
};

template <int D, bool F16, bool MASKED>
__global__ void __launch_bounds__(192, 2)
    fwd_fp8_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const Fp8FwdArgs a) {
  using L = F8Layout<D>;
  constexpr int NS = L::NS;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sb = smem_addr(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int BH = a.B * a.H;
  const int n_tiles = a.T;
  // heads in groups of head_group; within a group the heaviest (causal) query
  // tiles of all its heads first
  int qt, bh;
  group_order((int)blockIdx.x, n_tiles, BH, a.head_group, a.head_tail, qt, bh);
  qt = n_tiles - 1 - qt;
  const int b = bh / a.H, h = bh % a.H;
  const int kt_end = a.m.causal ? min(qt + 1, n_tiles) : n_tiles;

  const FwdBars<NS> bars{sb + L::BAR};
  volatile int* abort_cta = reinterpret_cast<volatile int*>(smem + L::ABORT);
  const WaitCtx w{abort_cta, a.rep.st, a.rep.epoch, a.rep.wait_ns};

  if ((sb & 1023u) != 0) {  // the swizzled layouts need a 1024-byte aligned base
    if (threadIdx.x == 0) raise_error(w, FA_ERR_CUDA);
    return;
  }
  const bool producer = (warp == 4 && lane == 0);
  int nk = 0, nv = 0;  // producer lane: K and V copies issued
  int kt_next = kt_end;  // producer lane: the next key tile to copy
  // the next kept key tile at or after kt, from the mask in device memory (the
  // producer's first copies, before the setup barrier) ...
  auto next_mem = [&](int kt) { return next_kept(a.m, b, h, qt, kt, kt_end); };
  // K8_j (128 keys x D bytes) and Vt8_j (D rows x 128 keys) of key tile kt into stage st
  auto load_k = [&](int st, int kt) {
    mbar_arrive_expect_tx(bars.kf(st), L::TQ);
    tma_load_3d(sb + L::K0 + st * L::TQ, &tmK, bars.kf(st), 0, kt * kT, bh);
  };
  auto load_v = [&](int st, int kt) {
    mbar_arrive_expect_tx(bars.vf(st), L::TV);
    tma_load_3d(sb + L::V0 + st * L::TV, &tmV, bars.vf(st), kt * kT, 0, bh);
  };
  if (producer) {
    bars.init();
    *abort_cta = 0;
    fence_barrier_init();
    prefetch_tmap(&tmQ);
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
    mbar_arrive_expect_tx(bars.q(), L::TQ);
    tma_load_3d(sb + L::Q, &tmQ, bars.q(), 0, qt * kT, bh);
    kt_next = fwd_produce(w, bars, next_mem(0), kt_end, a.N, NS, nk, nv, next_mem, load_k, load_v);
  }
  // block mask (its own instantiation, MASKED): this query tile's row of kept key
  // tiles as bits in shared memory
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
  // ... and from the bitmask after the setup barrier
  auto next = [&](int kt) { return use_bits ? next_bit(kbits, kt, kt_end) : next_mem(kt); };
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + L::TSLOT);

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      if (kt_next >= 0) fwd_produce(w, bars, kt_next, kt_end, a.N, 1 << 30, nk, nv, next, load_k, load_v);
      fwd_drain_copies(w, bars, nk, nv);
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t idS = idesc_e4m3(kT, kT);
    constexpr uint32_t idO = idesc_e4m3(kT, D);
    const uint32_t tS = tmem + L::T_S, tO = tmem + L::T_O;
    const uint64_t dQ = desc_k<D>(sb + L::Q);
    const uint64_t dK0 = desc_k<D>(sb + L::K0);
    const uint64_t dV0 = desc_k<128>(sb + L::V0);
    fwd_mma_schedule<NS, L::PSEP>(
        w, bars, next(0), kt_end, next,
        [&](int st) {  // S = Q8 K8^T: D / 32 products of K = 32 bytes
          const uint64_t dK = dK0 + (uint64_t)((st * L::TQ) >> 4);
#pragma unroll
          for (int kk = 0; kk < D / 32; ++kk)
            mma_f8_ss(tS, dQ + (uint64_t)(kk * 2), dK + (uint64_t)(kk * 2), idS, kk > 0 ? 1u : 0u);
        },
        [&](int st, int it) {  // O += Pq Vt8^T, Pq read from TMEM: 4 products of 32 keys
          const uint64_t dV = dV0 + (uint64_t)((st * L::TV) >> 4);
#pragma unroll
          for (int kk = 0; kk < kT / 32; ++kk)
            mma_f8_ts(tO, tmem + L::T_P + (uint32_t)kk * 8u, dV + (uint64_t)(kk * 2), idO,
                      (it > 0 || kk > 0) ? 1u : 0u);
        });
  } else {
    // ------------------------------------------------------------ softmax
    const int r = threadIdx.x;
    const int row = qt * kT + r;
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const uint32_t tS = tmem + L::T_S + lane_off, tO = tmem + L::T_O + lane_off;
    const float* sk_h = a.sk + (size_t)bh * a.T;
    const float* sv_h = a.sv + (size_t)bh * a.T;
    const float c2q = a.scale_log2 * a.sq[(size_t)bh * a.T + qt];
    float m_use = -INFINITY;  // running max (exp2 domain)
    float l = 0.f;            // running sum of the unquantised P~
    float unit = 0.f;         // O is held in units of this V scale
    bool ok = true;
    int it = 0;
    for (int kt = next(0); kt < kt_end; kt = next(kt + 1), ++it) {
      const float c2 = c2q * sk_h[kt];
      const float sv = sv_h[kt];
      if (!(ok = warp_wait(w, bars.s(), it & 1))) break;
      tc_fence_after();
      float s[kT];
      {
        uint32_t u[64];
        tmem_ld64(tS, u);
#pragma unroll
        for (int c = 0; c < 64; ++c) s[c] = __uint_as_float(u[c]);
        tmem_ld64(tS + 64, u);
#pragma unroll
        for (int c = 0; c < 64; ++c) s[64 + c] = __uint_as_float(u[c]);
      }
      if (L::PSEP) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bars.sfree());
      }
      mask_score_row(s, kt, qt, row, a.N, a.m.causal);
      float m8[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) m8[j] = max16(s, j);
      const float m_tile =
          fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7])) * c2;
      const float m_new = fmaxf(m_use, m_tile);
      const float alpha = (m_new > m_use) ? ex2(m_use - m_new) : 1.f;  // 0 when m_use = -inf
      m_use = m_new;
      // O moves to this key block's V unit: a power-of-two factor, exact
      const float f = (it > 0 && unit != sv) ? alpha * (unit / sv) : alpha;
      unit = sv;
      const float mneg = (m_use == -INFINITY) ? 0.f : -m_use;
      const uint64_t c2p = f2pack(c2, c2), mp = f2pack(mneg, mneg);
      uint64_t acc[4] = {f2pack(0.f, 0.f), f2pack(0.f, 0.f), f2pack(0.f, 0.f), f2pack(0.f, 0.f)};
      uint32_t pc[32];  // e4m3 codes of 256 P~, four keys per word
#pragma unroll
      for (int c = 0; c < kT; c += 4) {
        float x0, x1, x2, x3;
        f2unpack(ffma2(f2pack(s[c], s[c + 1]), c2p, mp), x0, x1);
        f2unpack(ffma2(f2pack(s[c + 2], s[c + 3]), c2p, mp), x2, x3);
        const float p0 = ex2(x0), p1 = ex2(x1), p2 = ex2(x2), p3 = ex2(x3);
        acc[(c >> 2) & 3] = fadd2(acc[(c >> 2) & 3], fadd2(f2pack(p0, p1), f2pack(p2, p3)));
        pc[c / 4] = pack4_e4m3(p0 * 256.f, p1 * 256.f, p2 * 256.f, p3 * 256.f);
      }
      l = l * alpha + sum_packed4(acc);
      if (L::PSEP && it > 0) {
        if (!(ok = warp_wait(w, bars.o(), (it - 1) & 1))) break;
        tc_fence_after();
      }
      tmem_st32(tmem + L::T_P + lane_off, pc);
      if (it > 0 && __any_sync(0xffffffffu, f != 1.f)) scale_o_row<D>(tO, f);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bars.p());
    }
    // ------------------------------------------------------------ epilogue
    bool have_o = false;
    if (ok && it > 0) {
      ok = warp_wait(w, bars.o(), (it - 1) & 1);
      tc_fence_after();
      have_o = ok;
    }
    const float inv = (l > 0.f) ? unit / (256.f * l) : 0.f;
    const float lse = (l > 0.f) ? (m_use + __log2f(l)) * 0.693147180559945309f : -INFINITY;
    if (row < a.N && ok) a.LSE[(size_t)bh * a.N + row] = lse;
    store_o_row<D, F16>(tO, have_o, inv, row < a.N && ok,
                        reinterpret_cast<uint16_t*>(a.O) + ((size_t)bh * a.N + row) * D);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, L::TMEM_COLS);
  }
}

template <int D, bool F16>
cudaError_t quant_t(const Fp8QuantArgs& a, cudaStream_t s) {
  const dim3 grid((unsigned)(a.BH * a.T), 3u);
  fp8_quant_kernel<D, F16><<<grid, 2 * D, 0, s>>>(a);
  return cudaGetLastError();
}

template <int D, bool F16>
cudaError_t fwd_t(const Fp8FwdArgs& a, const CUtensorMap* tm, cudaStream_t s) {
  using L = F8Layout<D>;
  // the block-mask bitmask is its own instantiation
  auto kern = a.m.mask ? fwd_fp8_kernel<D, F16, true> : fwd_fp8_kernel<D, F16, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::BYTES);
  if (e != cudaSuccess) return e;
  const unsigned grid = (unsigned)(a.T * a.B * a.H);
  kern<<<grid, 192, L::BYTES, s>>>(tm[0], tm[1], tm[2], a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fp8_quantize(const Fp8QuantArgs& a, int d, bool f16, cudaStream_t s) {
  if (d == 64) return f16 ? quant_t<64, true>(a, s) : quant_t<64, false>(a, s);
  return f16 ? quant_t<128, true>(a, s) : quant_t<128, false>(a, s);
}

cudaError_t launch_fwd_fp8(const Fp8FwdArgs& a, int d, bool f16, const CUtensorMap* tm, cudaStream_t s) {
  if (d == 64) return f16 ? fwd_t<64, true>(a, tm, s) : fwd_t<64, false>(a, tm, s);
  return f16 ? fwd_t<128, true>(a, tm, s) : fwd_t<128, false>(a, tm, s);
}

}  // namespace fa
