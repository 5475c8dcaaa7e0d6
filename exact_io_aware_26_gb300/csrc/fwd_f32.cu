// fwd_f32.cu -- attention forward in fp32 arithmetic on the CUDA cores.
//
// The tensor cores have no fp32 mode (tf32 rounds the inputs to 10 mantissa
// bits, far outside a 1e-5 error budget), so fp32 inputs take this SIMT path.
// It is the same tiled online-softmax recurrence as the tensor-core kernel
// ("L'algorithme Flash Attention", marketmaker.cc; "Rastreamento Incremental
// do Softmax", FlashAttention reading guide), on 64 x 64 tiles staged in
// shared memory: S = Q_i K_j^T with a 4 x 4 register block per thread, the
// running max / sum per row (4 threads per row), then O = O e^(m-m') + P V_j.
// O / l and LSE = m + ln l are written at the end.  With dropout, the weights
// that enter P V_j are the kept ones times the keep scale and the dropped ones 0
// (Philox4x32-10 keep bits, as in the tensor-core kernels); l sums them all.
#include <cmath>

#include "ptx.cuh"

namespace fa {
namespace {

constexpr int BR = 64, BC = 64, NT = 256;

__device__ __forceinline__ bool tile_kept64(const MaskArgs& m, int b, int h, int qt, int kt) {
  if (m.causal && kt > qt) return false;
  if (m.mask) {
    const long long at = (long long)b * m.mask_sb + (long long)h * m.mask_sh +
                         (long long)((qt * BR) / m.mask_block) * m.mask_cols +
                         (kt * BC) / m.mask_block;
    return m.mask[at] != 0;
  }
  return true;
}

template <int D>
__global__ void __launch_bounds__(NT) fwd_f32_kernel(const float* __restrict__ Q,
                                                     const float* __restrict__ K,
                                                     const float* __restrict__ V, const FwdArgs a) {
  extern __shared__ float sm[];
  float* sQ = sm;                    // [BR][D+1]
  float* sK = sQ + BR * (D + 1);     // [BC][D+1]
  float* sV = sK + BC * (D + 1);     // [BC][D]
  float* sS = sV + BC * D;           // [BR][BC+1]
  float* sRow = sS + BR * (BC + 1);  // [BR] per-row factor

  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  const int BH = a.B * a.H;
  const int n_tiles = (a.N + BR - 1) / BR;
  const int qt = n_tiles - 1 - (int)(blockIdx.x / BH);
  const int bh = (int)(blockIdx.x % BH);
  const int b = bh / a.H, h = bh % a.H;
  const int q0 = qt * BR;
  const size_t base = (size_t)bh * a.N * D;

  for (int e = tid; e < BR * D; e += NT) {
    const int r = e / D, c = e % D;
    sQ[r * (D + 1) + c] = (q0 + r < a.N) ? Q[base + (size_t)(q0 + r) * D + c] : 0.f;
  }

  // softmax state of row sr (4 threads per row keep identical copies)
  const int sr = tid >> 2, part = tid & 3;
  float m = -INFINITY, l = 0.f;
  constexpr int CJ = D / 16;
  float o[4][CJ];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < CJ; ++j) o[i][j] = 0.f;

  const int kt_end = a.m.causal ? min(qt + 1, n_tiles) : n_tiles;
  for (int kt = 0; kt < kt_end; ++kt) {
    if (!tile_kept64(a.m, b, h, qt, kt)) continue;
    const int k0 = kt * BC;
    __syncthreads();
    for (int e = tid; e < BC * D; e += NT) {
      const int r = e / D, c = e % D;
      const bool in = k0 + r < a.N;
      sK[r * (D + 1) + c] = in ? K[base + (size_t)(k0 + r) * D + c] : 0.f;
      sV[r * D + c] = in ? V[base + (size_t)(k0 + r) * D + c] : 0.f;
    }
    __syncthreads();
    // S = Q_i K_j^T, rows ty + 16 i, columns tx + 16 j
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
    for (int k = 0; k < D; ++k) {
      float qa[4], kb[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) qa[i] = sQ[(ty + 16 * i) * (D + 1) + k];
#pragma unroll
      for (int j = 0; j < 4; ++j) kb[j] = sK[(tx + 16 * j) * (D + 1) + k];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(qa[i], kb[j], acc[i][j]);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int r = ty + 16 * i, c = tx + 16 * j;
        const bool hide = (k0 + c >= a.N) || (a.m.causal && k0 + c > q0 + r);
        sS[r * (BC + 1) + c] = hide ? -INFINITY : acc[i][j] * a.scale;
      }
    __syncthreads();
    // running max / sum of row sr over its 16 columns, reduced over 4 lanes
    float* srow = sS + sr * (BC + 1) + part * 16;
    float mx = -INFINITY;
#pragma unroll
    for (int c = 0; c < 16; ++c) mx = fmaxf(mx, srow[c]);
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    const float m_new = fmaxf(m, mx);
    const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
    const float alpha = expf(m - m_use);
    uint32_t kb16 = 0xFFFFu;  // dropout keep bits of this thread's 16 columns
    if (a.drop.on) {
      uint4 c[2];
#pragma unroll
      for (int g = 0; g < 2; ++g)
        c[g] = make_uint4((uint32_t)((k0 + part * 16) / 8 + g), (uint32_t)(q0 + sr), (uint32_t)bh, a.drop.offset);
      philox4x32_10_n<2>(c, a.drop.key0, a.drop.key1);
      kb16 = keep_bits8(c[0], a.drop.t) | (keep_bits8(c[1], a.drop.t) << 8);
    }
    float sum = 0.f;
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      const float p = expf(srow[c] - m_use);
      srow[c] = a.drop.on ? (((kb16 >> c) & 1u) ? p * a.drop.z : 0.f) : p;
      sum += p;
    }
    sum += __shfl_xor_sync(0xffffffffu, sum, 1);
    sum += __shfl_xor_sync(0xffffffffu, sum, 2);
    l = l * alpha + sum;
    m = m_new;
    if (part == 0) sRow[sr] = alpha;
    __syncthreads();
    // O = O * alpha + P V_j
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float al = sRow[ty + 16 * i];
#pragma unroll
      for (int j = 0; j < CJ; ++j) o[i][j] *= al;
    }
    for (int k = 0; k < BC; ++k) {
      float pa[4], vb[CJ];
#pragma unroll
      for (int i = 0; i < 4; ++i) pa[i] = sS[(ty + 16 * i) * (BC + 1) + k];
#pragma unroll
      for (int j = 0; j < CJ; ++j) vb[j] = sV[k * D + tx + 16 * j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < CJ; ++j) o[i][j] = fmaf(pa[i], vb[j], o[i][j]);
    }
  }
  __syncthreads();
  if (part == 0) {
    sRow[sr] = l;
    if (q0 + sr < a.N)
      a.LSE[(size_t)bh * a.N + q0 + sr] = (l > 0.f) ? m + logf(l) : -INFINITY;
  }
  __syncthreads();
  float* O = reinterpret_cast<float*>(a.O);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = ty + 16 * i;
    if (q0 + r >= a.N) continue;
    const float lr = sRow[r];
    const float inv = (lr > 0.f) ? 1.f / lr : 0.f;
#pragma unroll
    for (int j = 0; j < CJ; ++j) O[base + (size_t)(q0 + r) * D + tx + 16 * j] = o[i][j] * inv;
  }
}

template <int D>
cudaError_t launch_t(const FwdArgs& a, const float* Q, const float* K, const float* V,
                     cudaStream_t s) {
  const size_t bytes = sizeof(float) * (size_t)(BR * (D + 1) + BC * (D + 1) + BC * D +
                                                BR * (BC + 1) + BR);
  auto kern = fwd_f32_kernel<D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e != cudaSuccess) return e;
  const int n_tiles = (a.N + BR - 1) / BR;
  kern<<<(unsigned)(n_tiles * a.B * a.H), NT, bytes, s>>>(Q, K, V, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_f32(const FwdArgs& a, int d, const float* Q, const float* K, const float* V,
                           cudaStream_t s) {
  return d == 64 ? launch_t<64>(a, Q, K, V, s) : launch_t<128>(a, Q, K, V, s);
}

}  // namespace fa
