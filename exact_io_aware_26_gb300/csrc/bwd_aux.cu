// bwd_aux.cu -- the memory-bound stages around the backward main kernel, and
// the barrier-timeout self-test.
//
//   preprocess: D_i = sum_k dO_ik O_ik (fp32) for every row, and the fp32 dQ
//               accumulator zeroed.  D_i equals sum_j P_ij dP_ij, the row term
//               of dS = P * (dP - D), because O_i = sum_j P_ij v_j.
//   finalize:   dQ = scale * accumulator, rounded to the 16-bit output type;
//               and, after a sliced main kernel, dK and dV of every key tile
//               cut into several slices: the sum of their fp32 partial slots
//               (bwd_sched.cuh).
// Both are plain streaming kernels: 16-byte vector loads/stores, coalesced,
// grid sized to a multiple of the SM count.
#include "bwd_sched.cuh"
#include "ptx.cuh"

namespace fa {
namespace {

template <int D, bool F16>
__global__ void __launch_bounds__(256) bwd_preprocess_kernel(const uint4* __restrict__ O,
                                                             const uint4* __restrict__ dO,
                                                             float* __restrict__ Dsum,
                                                             float4* __restrict__ dQacc,
                                                             long long rows) {
  constexpr int TPR = D / 8;  // threads per row, 8 elements (16 bytes) each
  const long long nthreads = (long long)gridDim.x * blockDim.x;
  const long long total = rows * TPR;
  const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
  for (long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x; t - (threadIdx.x & 31) < total;
       t += nthreads) {
    const bool in = t < total;
    float acc = 0.f;
    if (in) {
      const uint4 o = O[t], g = dO[t];
      const uint32_t ov[4] = {o.x, o.y, o.z, o.w}, gv[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 a = unpack2<F16>(ov[i]), b = unpack2<F16>(gv[i]);
        acc = fmaf(a.x, b.x, acc);
        acc = fmaf(a.y, b.y, acc);
      }
      dQacc[2 * t] = z;
      dQacc[2 * t + 1] = z;
    }
#pragma unroll
    for (int off = TPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (in && (t % TPR) == 0) Dsum[t / TPR] = acc;
  }
}

template <bool F16>
__global__ void __launch_bounds__(256) bwd_finalize_kernel(const float4* __restrict__ acc,
                                                           uint4* __restrict__ dQ, float scale,
                                                           long long n8) {
  const long long nthreads = (long long)gridDim.x * blockDim.x;
  for (long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x; t < n8; t += nthreads) {
    const float4 a = acc[2 * t], b = acc[2 * t + 1];
    uint4 o;
    o.x = pack2<F16>(a.x * scale, a.y * scale);
    o.y = pack2<F16>(a.z * scale, a.w * scale);
    o.z = pack2<F16>(b.x * scale, b.y * scale);
    o.w = pack2<F16>(b.z * scale, b.w * scale);
    dQ[t] = o;
  }
}

// Fixup blocks per sliced key tile: each adds one part of the key tile's slots,
// so that enough loads are in flight to hide their latency.
constexpr int kFixupParts = 8;

// Block `part` of unit `unit` (a key tile of a sliced main kernel): if the unit
// was cut into several slices, the block adds its part of their partial slots
// and writes that part of the key tile's dV and dK (dK times the score scale).
template <int D, bool F16>
__device__ void slices_key_tile(const BwdArgs& a, long long unit, int part) {
  const int BH = a.B * a.H;
  const int n = (a.N + 127) / 128;
  long long first;
  int count;
  unit_slots(unit, n, BH, a.m.causal, a.q_slice, a.qs_from, first, count);
  if (count < 2) return;  // a whole key tile: written by its CTA
  const int kt = (int)(unit / BH), bh = (int)(unit % BH);
  constexpr int PER = 2 * 128 * D / 4;  // float4 per slot ([dV | dK])
  constexpr int PART = PER / kFixupParts;
  const float4* base = reinterpret_cast<const float4*>(a.slots) + (size_t)first * PER;
  for (int e = part * PART + (int)threadIdx.x; e < (part + 1) * PART; e += blockDim.x) {
    float4 acc = base[e];
    for (int sp = 1; sp < count; ++sp) {
      const float4 v = base[(size_t)sp * PER + e];
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
    const int f = e * 4;              // first float of the four
    const int which = f / (128 * D);  // 0: dV, 1: dK
    const int row = (f / D) % 128;
    const int col = f % D;
    const int key = kt * 128 + row;
    if (key >= a.N) continue;
    const float mul = which == 0 ? 1.f : a.scale;
    uint16_t* dst = reinterpret_cast<uint16_t*>(which == 0 ? a.dV : a.dK) + ((size_t)bh * a.N + key) * D + col;
    uint2 o;
    o.x = pack2<F16>(acc.x * mul, acc.y * mul);
    o.y = pack2<F16>(acc.z * mul, acc.w * mul);
    *reinterpret_cast<uint2*>(dst) = o;
  }
}

// Blocks [0, dq_blocks) convert the dQ accumulator; blocks after them,
// kFixupParts per unit from qs_from on, add up the sliced key tiles' partial
// dK, dV.
template <int D, bool F16>
__global__ void __launch_bounds__(256) bwd_finalize_slices_kernel(const BwdArgs a, int dq_blocks) {
  if ((int)blockIdx.x >= dq_blocks) {
    const long long k = (long long)blockIdx.x - dq_blocks;
    slices_key_tile<D, F16>(a, a.qs_from + k / kFixupParts, (int)(k % kFixupParts));
    return;
  }
  const long long n8 = (long long)a.B * a.H * a.N * D / 8;
  const float4* acc = reinterpret_cast<const float4*>(a.dQacc);
  uint4* dQ = reinterpret_cast<uint4*>(a.dQ);
  const long long nthreads = (long long)dq_blocks * blockDim.x;
  for (long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x; t < n8; t += nthreads) {
    const float4 x = acc[2 * t], y = acc[2 * t + 1];
    uint4 o;
    o.x = pack2<F16>(x.x * a.scale, x.y * a.scale);
    o.y = pack2<F16>(x.z * a.scale, x.w * a.scale);
    o.z = pack2<F16>(y.x * a.scale, y.y * a.scale);
    o.w = pack2<F16>(y.z * a.scale, y.w * a.scale);
    dQ[t] = o;
  }
}

__global__ void wait_selftest_kernel(Report rep) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_cta;
  if (threadIdx.x == 0) {
    mbar_init(smem_addr(&bar), 1);
    abort_cta = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const WaitCtx w{&abort_cta, rep.st, rep.epoch, rep.wait_ns};
    // nothing arrives on this barrier: the wait must run out and report
    mbar_wait(w, smem_addr(&bar), 0);
  }
  __syncthreads();
}

int grid_for(long long work, int per_block) {
  int dev = 0, sms = 152;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  long long blocks = (work + per_block - 1) / per_block;
  const long long cap = (long long)sms * 8;
  if (blocks > cap) blocks = cap;
  return (int)(blocks < 1 ? 1 : blocks);
}

template <int D, bool F16>
cudaError_t pre_t(const BwdArgs& a, cudaStream_t s) {
  const long long rows = (long long)a.B * a.H * a.N;
  bwd_preprocess_kernel<D, F16><<<grid_for(rows * (D / 8), 256), 256, 0, s>>>(
      reinterpret_cast<const uint4*>(a.O), reinterpret_cast<const uint4*>(a.dO), a.Dsum,
      reinterpret_cast<float4*>(a.dQacc), rows);
  return cudaGetLastError();
}

template <int D, bool F16>
cudaError_t fin_slices_t(const BwdArgs& a, int dq_blocks, cudaStream_t s) {
  const long long units = (long long)a.B * a.H * ((a.N + 127) / 128);  // sliced: [qs_from, units)
  bwd_finalize_slices_kernel<D, F16><<<(unsigned)(dq_blocks + (units - a.qs_from) * kFixupParts), 256, 0, s>>>(
      a, dq_blocks);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_preprocess(const BwdArgs& a, int d, bool f16, cudaStream_t s) {
  if (d == 64) return f16 ? pre_t<64, true>(a, s) : pre_t<64, false>(a, s);
  return f16 ? pre_t<128, true>(a, s) : pre_t<128, false>(a, s);
}

cudaError_t launch_bwd_finalize(const BwdArgs& a, int d, bool f16, cudaStream_t s) {
  const long long n8 = (long long)a.B * a.H * a.N * d / 8;
  const int grid = grid_for(n8, 256);
  if (a.q_slice > 0) {
    // sliced main kernel: the same launch adds up the sliced key tiles' partial dK, dV
    if (d == 64) return f16 ? fin_slices_t<64, true>(a, grid, s) : fin_slices_t<64, false>(a, grid, s);
    return f16 ? fin_slices_t<128, true>(a, grid, s) : fin_slices_t<128, false>(a, grid, s);
  }
  if (f16)
    bwd_finalize_kernel<true><<<grid, 256, 0, s>>>(reinterpret_cast<const float4*>(a.dQacc),
                                                   reinterpret_cast<uint4*>(a.dQ), a.scale, n8);
  else
    bwd_finalize_kernel<false><<<grid, 256, 0, s>>>(reinterpret_cast<const float4*>(a.dQacc),
                                                    reinterpret_cast<uint4*>(a.dQ), a.scale, n8);
  return cudaGetLastError();
}

cudaError_t launch_wait_selftest(const Report& rep, cudaStream_t s) {
  wait_selftest_kernel<<<1, 32, 0, s>>>(rep);
  return cudaGetLastError();
}

}  // namespace fa
