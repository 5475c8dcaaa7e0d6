// fa_api.cu -- the C ABI of libfa.so (declared in include/fa.h): argument
// validation, TMA tensor-map encoding, the device status word, and the kernel
// launches.  Everything here is host code except the status word.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "bwd_sched.cuh"
#include "fp8.h"
#include "internal.h"

#include <nvtx3/nvToolsExt.h>

using namespace fa;

namespace {
// An NVTX range around each call that launches work, so that a profiler's
// timeline names the library call every kernel belongs to.  Header-only NVTX:
// without a profiler attached each push and pop is a cheap no-op.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};
}  // namespace

namespace {
void set_err(const char* fmt, ...);
}

void fa::set_error_text(const char* text) { set_err("%s", text); }

namespace {

__device__ DevStatus g_status;  // per device: first error code + abort epoch

thread_local char g_err[512] = "";

void set_err(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
}

fa_status cuda_fail(cudaError_t e, const char* what) {
  set_err("%s: %s", what, cudaGetErrorString(e));
  return FA_ERR_CUDA;
}

std::atomic<uint32_t> g_epoch{0};
std::atomic<unsigned long long> g_wait_ns{2000000000ull};
std::atomic<int> g_bwd_ctas{0};  // backward CTAs per wave; 0 = one per SM

constexpr int kMaxDev = 64;
struct DevState {
  bool checked = false;
  bool supported = false;
  int sms = 0;
  int l2_bytes = 0;
  DevStatus* st = nullptr;
};
DevState g_dev[kMaxDev];
std::mutex g_mu;

// The current device must be sm_103; resolves the status word's address once.
fa_status device_ready(DevStatus** st) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDev) {
    set_err("device ordinal %d out of range", dev);
    return FA_ERR_DEVICE;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  DevState& d = g_dev[dev];
  if (!d.checked) {
    int major = 0, minor = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute");
    if ((e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute");
    d.supported = (major == 10 && minor == 3);
    if ((e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute");
    if ((e = cudaDeviceGetAttribute(&d.l2_bytes, cudaDevAttrL2CacheSize, dev)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute");
    if (d.supported) {
      void* p = nullptr;
      if ((e = cudaGetSymbolAddress(&p, g_status)) != cudaSuccess)
        return cuda_fail(e, "cudaGetSymbolAddress(status)");
      d.st = static_cast<DevStatus*>(p);
    }
    d.checked = true;
    if (!d.supported) {
      set_err("device %d is sm_%d%d; this library is built for sm_103a", dev, major, minor);
    }
  }
  if (!d.supported) return FA_ERR_DEVICE;
  *st = d.st;
  return FA_OK;
}

// SM count of the current device (after device_ready).
int device_sms() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return 1;
  std::lock_guard<std::mutex> lock(g_mu);
  return g_dev[dev].sms > 0 ? g_dev[dev].sms : 1;
}

// L2 size of the current device in bytes (after device_ready).
long long device_l2_bytes() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return 0;
  std::lock_guard<std::mutex> lock(g_mu);
  return g_dev[dev].l2_bytes;
}

// How many heads' CTAs a launch runs together (see group_order in bwd_sched.cuh).
// In tile-major order over all heads the CTAs running at any moment belong to
// every head, so every head's streamed operands -- the forward's K and V, the
// backward's Q, dO and fp32 dQ accumulator -- compete for L2 at once; when they
// do not fit, most tiles are re-read from DRAM by every CTA that needs them (the
// block-sparse B2 H16 N16384 d128 problem moved 5.7 GB per forward and 20 GB per
// backward instead of 0.5 and 1.3).  Then the launch runs head by head (one head
// per group).  Measured on GB300: the forward keeps tile-major order while its K,
// V fit in three quarters of L2 (the causal N = 23400, 12-head forward is 12%
// faster that way than head by head, its heaviest tiles all running first); the
// backward goes head by head beyond half of L2 (faster there than groups sized
// to fit L2, and than tile-major order).  Head by head, a causal launch would
// end with the last head's heaviest tiles running alone (they start last), so
// its last heads -- as many as fit the same budget -- form one tile-major group.
struct HeadOrder {
  int group, tail;
};
// per_head: the streamed bytes of one head (forward: K and V; backward: Q, dO and
// the fp32 dQ accumulator)
HeadOrder head_order_bytes(const fa_params* p, long long per_head, bool backward) {
  const long long bh = (long long)p->B * p->H;
  const long long l2 = device_l2_bytes();
  const long long budget = backward ? l2 / 2 : l2 * 3 / 4;
  if (l2 <= 0 || bh * per_head <= budget) return {(int)bh, 0};
  long long tail = p->causal ? budget / per_head : 0;
  if (tail < 2) tail = 0;
  return {1, (int)tail};
}
HeadOrder head_order(const fa_params* p, bool backward) {
  const long long e = p->dtype == FA_F32 ? 4 : 2;
  const long long nd = (long long)p->N * p->d;
  return head_order_bytes(p, backward ? nd * (2 * e + 4) : nd * 2 * e, backward);
}

Report make_report(DevStatus* st) {
  Report r;
  r.st = st;
  r.epoch = g_epoch.fetch_add(1) + 1;
  r.wait_ns = g_wait_ns.load();
  return r;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// ---------------------------------------------------------------- TMA maps

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// A [B*H][N][d] 16-bit tensor as a 3-D TMA map {d, N, B*H}; box {64, 128, 1},
// 128-byte swizzle; rows past N read as zero.
fa_status encode_bhnd(CUtensorMap* m, const void* ptr, const fa_params* p) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) {
    set_err("cuTensorMapEncodeTiled is not available from the driver");
    return FA_ERR_CUDA;
  }
  const cuuint64_t dims[3] = {(cuuint64_t)p->d, (cuuint64_t)p->N, (cuuint64_t)p->B * p->H};
  const cuuint64_t strides[2] = {(cuuint64_t)p->d * 2, (cuuint64_t)p->N * p->d * 2};
  const cuuint32_t box[3] = {64, 128, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapDataType dt =
      p->dtype == FA_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  CUresult r = fn(m, dt, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_err("cuTensorMapEncodeTiled failed (CUresult %d)", (int)r);
    return FA_ERR_CUDA;
  }
  return FA_OK;
}

// The fp32 dQ accumulator [B*H][N][d] as a 3-D TMA map {d, N, B*H}; box
// {cols, 32, 1} (one warp's slice of 32 rows): 32 columns (128-byte rows) with
// the 128-byte swizzle or 16 columns (64-byte rows) with the 64-byte swizzle;
// rows past N are not written.
fa_status encode_dqacc(CUtensorMap* m, const float* ptr, const fa_params* p, int cols) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) {
    set_err("cuTensorMapEncodeTiled is not available from the driver");
    return FA_ERR_CUDA;
  }
  const cuuint64_t dims[3] = {(cuuint64_t)p->d, (cuuint64_t)p->N, (cuuint64_t)p->B * p->H};
  const cuuint64_t strides[2] = {(cuuint64_t)p->d * 4, (cuuint64_t)p->N * p->d * 4};
  const cuuint32_t box[3] = {(cuuint32_t)cols, 32, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(ptr), dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  cols == 32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_err("cuTensorMapEncodeTiled (dQ accumulator) failed (CUresult %d)", (int)r);
    return FA_ERR_CUDA;
  }
  return FA_OK;
}

// An 8-bit tensor {x, y, z} (x contiguous) as a 3-D TMA map with box {bx, by, 1}
// and the given swizzle; reads past the extents give zero.
fa_status encode_u8(CUtensorMap* m, const void* ptr, uint64_t x, uint64_t y, uint64_t z, uint32_t bx,
                    uint32_t by, CUtensorMapSwizzle sw) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) {
    set_err("cuTensorMapEncodeTiled is not available from the driver");
    return FA_ERR_CUDA;
  }
  const cuuint64_t dims[3] = {(cuuint64_t)x, (cuuint64_t)y, (cuuint64_t)z};
  const cuuint64_t strides[2] = {(cuuint64_t)x, (cuuint64_t)(x * y)};
  const cuuint32_t box[3] = {bx, by, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_err("cuTensorMapEncodeTiled (8-bit operand) failed (CUresult %d)", (int)r);
    return FA_ERR_CUDA;
  }
  return FA_OK;
}

MaskArgs mask_args(const fa_params* p) {
  MaskArgs m;
  m.causal = p->causal ? 1 : 0;
  m.mask = p->block_mask;
  m.mask_block = p->block_mask ? p->mask_block : 128;
  m.mask_cols = (p->N + m.mask_block - 1) / m.mask_block;
  m.mask_sb = p->mask_stride_b;
  m.mask_sh = p->mask_stride_h;
  return m;
}

// The dropout arguments the kernels take: threshold t = floor(p * 2^16) on a
// 16-bit half of a Philox word, keep scale 2^16 / (2^16 - t) (the inverse of the
// keep probability), the key and the counter's last word.
DropArgs drop_args(const fa_params* p) {
  DropArgs d;
  std::memset(&d, 0, sizeof(d));
  if (p->dropout_p > 0.f) {
    const double t = std::floor((double)p->dropout_p * 65536.0);
    d.on = 1;
    d.t = t >= 65535.0 ? 65535u : (uint32_t)t;
    d.z = (float)(65536.0 / (65536.0 - (double)d.t));
    d.key0 = (uint32_t)(p->dropout_seed & 0xFFFFFFFFull);
    d.key1 = (uint32_t)(p->dropout_seed >> 32);
    d.offset = p->dropout_offset;
  }
  return d;
}

BwdArgs bwd_args(const fa_params* p, void* ws) {
  BwdArgs a;
  std::memset(&a, 0, sizeof(a));
  a.B = p->B;
  a.H = p->H;
  a.N = p->N;
  a.scale = p->scale;
  a.scale_log2 = p->scale * 1.4426950408889634f;
  a.m = mask_args(p);
  a.drop = drop_args(p);
  a.head_group = p->B * p->H;
  const size_t rows = (size_t)p->B * p->H * p->N;
  a.Dsum = static_cast<float*>(ws);
  a.dQacc = reinterpret_cast<float*>(static_cast<char*>(ws) + align256(rows * 4));
  a.slots = reinterpret_cast<float*>(static_cast<char*>(ws) + align256(rows * 4) +
                                     align256(rows * (size_t)p->d * 4));
  const int n = (p->N + 127) / 128;
  const long long units = (long long)p->B * p->H * n;
  a.direct = (int)units;  // one CTA per key tile ...
  a.qs_from = (int)units;
  a.q_slice = 0;
  if (!p->block_mask) {
    // ... unless that leaves SMs idle (plan_slices; G: CTAs per wave, one per
    // SM, at most kBwdMaxCtas, or the count set by fa_set_bwd_ctas)
    long long G = device_sms();
    if (G > kBwdMaxCtas) G = kBwdMaxCtas;
    const int cap = g_bwd_ctas.load();
    if (cap > 0 && cap < G) G = cap;
    int P = 0, u0 = 0;
    const long long ctas = plan_slices(n, p->B * p->H, p->causal ? 1 : 0, G, P, u0);
    if (P > 0) {
      a.q_slice = P;
      a.qs_from = u0;
      a.direct = (int)ctas;
    }
  }
  // every key tile its own CTA: in groups of heads whose streamed operands fit
  // in L2 together
  if (a.q_slice == 0) {
    const HeadOrder ho = head_order(p, true);
    a.head_group = ho.group;
    a.head_tail = ho.tail;
  }
  return a;
}

fa_status check_ws(const fa_params* p, const void* ws, size_t bytes) {
  const size_t need = fa_bwd_workspace_size(p);
  if (!ws || bytes < need || !aligned(ws, 256)) {
    set_err("workspace %p of %zu bytes; need %zu bytes, 256-byte aligned", ws, bytes, need);
    return FA_ERR_WORKSPACE;
  }
  return FA_OK;
}

fa_status need16(const void* ptr, const char* name) {
  if (!ptr) {
    set_err("%s is NULL", name);
    return FA_ERR_INVALID;
  }
  if (!aligned(ptr, 16)) {
    set_err("%s is not 16-byte aligned", name);
    return FA_ERR_INVALID;
  }
  return FA_OK;
}

#define FA_TRY(x)                    \
  do {                               \
    fa_status _s = (x);              \
    if (_s != FA_OK) return _s;      \
  } while (0)

}  // namespace

extern "C" {

int fa_version(void) { return 100; }

int fa_fp8_vt_cols(int N) { return N < 1 ? 0 : (N + 15) / 16 * 16; }

namespace {
fa_status fp8_check(const fa_params* p) {
  FA_TRY(fa_check(p, 0));
  if (p->dtype == FA_F32) {
    set_err("the FP8 path takes fp16 or bf16 tensors");
    return FA_ERR_UNSUPPORTED;
  }
  if (p->dropout_p > 0.f) {
    set_err("the FP8 forward has no dropout");
    return FA_ERR_UNSUPPORTED;
  }
  return FA_OK;
}

fa_status need_scales(const float* a, const float* b, const float* c) {
  for (const float* x : {a, b, c})
    if (!x || !aligned(x, 4)) {
      set_err("a block-scale array is NULL or not 4-byte aligned");
      return FA_ERR_INVALID;
    }
  return FA_OK;
}
}  // namespace

fa_status fa_fp8_quantize(const fa_params* p, const void* Q, const void* K, const void* V,
                          const float* signs, void* q8, void* k8, void* vt8, float* sq, float* sk,
                          float* sv, void* stream) {
  NvtxRange nvtx_range("fa_fp8_quantize");
  FA_TRY(fp8_check(p));
  FA_TRY(need16(Q, "Q"));
  FA_TRY(need16(K, "K"));
  FA_TRY(need16(V, "V"));
  FA_TRY(need16(q8, "q8"));
  FA_TRY(need16(k8, "k8"));
  FA_TRY(need16(vt8, "vt8"));
  FA_TRY(need_scales(sq, sk, sv));
  DevStatus* st = nullptr;
  FA_TRY(device_ready(&st));
  if (signs) {  // read by the kernel: it must be device memory
    cudaPointerAttributes at{};
    if (!aligned(signs, 4) || cudaPointerGetAttributes(&at, signs) != cudaSuccess ||
        (at.type != cudaMemoryTypeDevice && at.type != cudaMemoryTypeManaged)) {
      cudaGetLastError();
      set_err("signs must be 4-byte aligned device memory (d floats) or NULL");
      return FA_ERR_INVALID;
    }
  }
  Fp8QuantArgs a;
  std::memset(&a, 0, sizeof(a));
  a.BH = p->B * p->H;
  a.N = p->N;
  a.T = (p->N + 127) / 128;
  a.ld = fa_fp8_vt_cols(p->N);
  a.Q = Q;
  a.K = K;
  a.V = V;
  a.signs = signs;
  a.q8 = static_cast<uint8_t*>(q8);
  a.k8 = static_cast<uint8_t*>(k8);
  a.vt8 = static_cast<uint8_t*>(vt8);
  a.sq = sq;
  a.sk = sk;
  a.sv = sv;
  const cudaError_t e = launch_fp8_quantize(a, p->d, p->dtype == FA_F16, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "FP8 quantise launch");
  return FA_OK;
}

fa_status fa_fwd_fp8(const fa_params* p, const void* q8, const void* k8, const void* vt8,
                     const float* sq, const float* sk, const float* sv, void* O, float* LSE,
                     void* stream) {
  NvtxRange nvtx_range("fa_fwd_fp8");
  FA_TRY(fp8_check(p));
  FA_TRY(need16(q8, "q8"));
  FA_TRY(need16(k8, "k8"));
  FA_TRY(need16(vt8, "vt8"));
  FA_TRY(need16(O, "O"));
  FA_TRY(need_scales(sq, sk, sv));
  if (!LSE || !aligned(LSE, 4)) {
    set_err("LSE is NULL or misaligned");
    return FA_ERR_INVALID;
  }
  DevStatus* st = nullptr;
  FA_TRY(device_ready(&st));
  const uint64_t BH = (uint64_t)p->B * p->H, d = (uint64_t)p->d;
  CUtensorMap tm[3];
  const CUtensorMapSwizzle sw = p->d == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B;
  FA_TRY(encode_u8(&tm[0], q8, d, (uint64_t)p->N, BH, (uint32_t)d, 128, sw));
  FA_TRY(encode_u8(&tm[1], k8, d, (uint64_t)p->N, BH, (uint32_t)d, 128, sw));
  FA_TRY(encode_u8(&tm[2], vt8, (uint64_t)fa_fp8_vt_cols(p->N), d, BH, 128, (uint32_t)d,
                   CU_TENSOR_MAP_SWIZZLE_128B));
  Fp8FwdArgs a;
  std::memset(&a, 0, sizeof(a));
  a.B = p->B;
  a.H = p->H;
  a.N = p->N;
  a.T = (p->N + 127) / 128;
  a.scale_log2 = p->scale * 1.4426950408889634f;
  a.m = mask_args(p);
  a.sq = sq;
  a.sk = sk;
  a.sv = sv;
  a.O = O;
  a.LSE = LSE;
  // the FP8 K and V: one byte per element
  const HeadOrder ho = head_order_bytes(p, 2LL * p->N * p->d, false);
  a.head_group = ho.group;
  a.head_tail = ho.tail;
  a.rep = make_report(st);
  const cudaError_t e = launch_fwd_fp8(a, p->d, p->dtype == FA_F16, tm, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "FP8 forward launch");
  return FA_OK;
}

const char* fa_last_error(void) { return g_err; }

const char* fa_status_string(int s) {
  switch (s) {
    case FA_OK: return "ok";
    case FA_ERR_INVALID: return "invalid argument";
    case FA_ERR_UNSUPPORTED: return "unsupported configuration";
    case FA_ERR_CUDA: return "CUDA error";
    case FA_ERR_TIMEOUT: return "kernel barrier wait timed out";
    case FA_ERR_WORKSPACE: return "workspace missing or too small";
    case FA_ERR_DEVICE: return "device is not sm_103";
    case FA_ERR_BOUNDS: return "index check failed in a kernel (debug build)";
    default: return "unknown status";
  }
}

fa_status fa_check(const fa_params* p, int for_backward) {
  if (!p) {
    set_err("params is NULL");
    return FA_ERR_INVALID;
  }
  if (p->B < 1 || p->H < 1 || p->N < 1 || p->d < 1) {
    set_err("B, H, N, d must be >= 1 (got %d, %d, %d, %d)", p->B, p->H, p->N, p->d);
    return FA_ERR_INVALID;
  }
  if (p->dtype != FA_F32 && p->dtype != FA_F16 && p->dtype != FA_BF16) {
    set_err("dtype %d is not an fa_dtype", p->dtype);
    return FA_ERR_INVALID;
  }
  if (!(std::isfinite(p->scale) && p->scale > 0.f)) {
    set_err("scale must be positive and finite");
    return FA_ERR_INVALID;
  }
  if (p->d != 64 && p->d != 128) {
    set_err("head size %d is not supported (64 or 128)", p->d);
    return FA_ERR_UNSUPPORTED;
  }
  const long long elems = (long long)p->B * p->H * p->N * p->d;
  if (elems >= (1ll << 31)) {
    set_err("B*H*N*d = %lld exceeds 2^31 - 1", elems);
    return FA_ERR_UNSUPPORTED;
  }
  if (p->block_mask) {
    if (p->mask_block <= 0 || p->mask_stride_b < 0 || p->mask_stride_h < 0) {
      set_err("mask_block must be positive and mask strides non-negative");
      return FA_ERR_INVALID;
    }
    if (p->mask_block % 128 != 0) {
      set_err("mask_block %d is not a multiple of the 128-token tile", p->mask_block);
      return FA_ERR_UNSUPPORTED;
    }
  }
  if (for_backward && p->dtype == FA_F32) {
    set_err("the backward pass takes fp16 or bf16 tensors");
    return FA_ERR_UNSUPPORTED;
  }
  if (!(p->dropout_p >= 0.f && p->dropout_p < 1.f)) {
    set_err("dropout_p must lie in [0, 1)");
    return FA_ERR_INVALID;
  }
  return FA_OK;
}


unsigned long long fa_set_wait_limit_ns(unsigned long long ns) {
  if (ns == 0) ns = 1;
  return g_wait_ns.exchange(ns);
}

fa_status fa_fwd(const fa_params* p, const void* Q, const void* K, const void* V, void* O,
                 float* LSE, void* stream) {
  NvtxRange nvtx_range("fa_fwd");
  FA_TRY(fa_check(p, 0));
  FA_TRY(need16(Q, "Q"));
  FA_TRY(need16(K, "K"));
  FA_TRY(need16(V, "V"));
  FA_TRY(need16(O, "O"));
  if (!LSE || !aligned(LSE, 4)) {
    set_err("LSE is NULL or misaligned");
    return FA_ERR_INVALID;
  }
  DevStatus* st = nullptr;
  FA_TRY(device_ready(&st));
  FwdArgs a;
  std::memset(&a, 0, sizeof(a));
  a.B = p->B;
  a.H = p->H;
  a.N = p->N;
  a.scale = p->scale;
  a.scale_log2 = p->scale * 1.4426950408889634f;
  a.m = mask_args(p);
  a.drop = drop_args(p);
  a.O = O;
  a.LSE = LSE;
  a.n_splits = 1;
  a.split_tiles = (p->N + 127) / 128;
  const HeadOrder ho = head_order(p, false);
  a.head_group = ho.group;
  a.head_tail = ho.tail;
  a.rep = make_report(st);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (p->dtype == FA_F32) {
    e = launch_fwd_f32(a, p->d, static_cast<const float*>(Q), static_cast<const float*>(K),
                       static_cast<const float*>(V), s);
  } else {
    CUtensorMap tm[3];
    FA_TRY(encode_bhnd(&tm[0], Q, p));
    FA_TRY(encode_bhnd(&tm[1], K, p));
    FA_TRY(encode_bhnd(&tm[2], V, p));
    e = launch_fwd_tc(a, p->d, p->dtype == FA_F16, tm, s);
  }
  if (e != cudaSuccess) return cuda_fail(e, "forward launch");
  return FA_OK;
}

namespace {
// key tiles per slice and the number of non-empty slices for a request of
// `splits` slices over n_tiles key tiles
void split_shape(int n_tiles, int splits, int* per, int* used) {
  *per = (n_tiles + splits - 1) / splits;
  *used = (n_tiles + *per - 1) / *per;
}

fa_status check_splits(const fa_params* p, int num_splits) {
  const int n_tiles = (p->N + 127) / 128;
  if (num_splits < 1 || num_splits > FA_MAX_SPLITS || num_splits > n_tiles) {
    set_err("num_splits out of range [1, min(FA_MAX_SPLITS, ceil(N / 128))]");
    return FA_ERR_INVALID;
  }
  if (num_splits > 1 && p->dtype == FA_F32) {
    set_err("split forward needs fp16 or bf16");
    return FA_ERR_UNSUPPORTED;
  }
  return FA_OK;
}
}  // namespace

int fa_fwd_num_splits(const fa_params* p, int num_sms) {
  if (fa_check(p, 0) != FA_OK) return 0;
  if (p->dtype == FA_F32) return 1;
  if (num_sms <= 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        num_sms <= 0) {
      cudaGetLastError();
      return 1;
    }
  }
  // Model: two CTAs share an SM, so a launch runs in waves of 2 * num_sms
  // CTAs, and a wave lasts about as long as its CTAs' key tiles plus two tiles
  // for loading Q, writing the partial result and merging it.  A grid that
  // fills the first wave is left whole (splitting it would only trade a tail
  // for the partials' extra traffic); otherwise pick the split count with the
  // lowest modelled time (ties to fewer splits).
  const long long n_tiles = (p->N + 127) / 128;
  const long long ctas = (long long)p->B * p->H * n_tiles;
  const long long slots = 2LL * num_sms;
  if (ctas >= slots) return 1;
  const int max_s = (int)std::min<long long>(FA_MAX_SPLITS, n_tiles);
  int best = 1;
  long long best_cost = -1;
  for (int sp = 1; sp <= max_s; ++sp) {
    int per = 0, used = 0;
    split_shape((int)n_tiles, sp, &per, &used);
    if (used != sp) continue;  // a split count that leaves a slice empty
    const long long waves = (ctas * sp + slots - 1) / slots;
    const long long cost = waves * (per + 2);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = sp;
    }
  }
  return best;
}

fa_status fa_fwd_split(const fa_params* p, const void* Q, const void* K, const void* V, void* O,
                       float* LSE, int num_splits, void* stream) {
  NvtxRange nvtx_range("fa_fwd_split");
  FA_TRY(fa_check(p, 0));
  FA_TRY(check_splits(p, num_splits));
  if (num_splits == 1) return fa_fwd(p, Q, K, V, O, LSE, stream);
  FA_TRY(need16(Q, "Q"));
  FA_TRY(need16(K, "K"));
  FA_TRY(need16(V, "V"));
  FA_TRY(need16(O, "O"));
  if (!LSE || !aligned(LSE, 4)) {
    set_err("LSE is NULL or misaligned");
    return FA_ERR_INVALID;
  }
  DevStatus* st = nullptr;
  FA_TRY(device_ready(&st));
  const int n_tiles = (p->N + 127) / 128;
  int per = 0, used = 0;
  split_shape(n_tiles, num_splits, &per, &used);
  FwdArgs a;
  std::memset(&a, 0, sizeof(a));
  a.B = p->B;
  a.H = p->H;
  a.N = p->N;
  a.scale = p->scale;
  a.scale_log2 = p->scale * 1.4426950408889634f;
  a.m = mask_args(p);
  a.drop = drop_args(p);
  a.O = O;
  a.LSE = LSE;
  a.n_splits = used;
  a.split_tiles = per;
  const HeadOrder ho = head_order(p, false);
  a.head_group = ho.group;
  a.head_tail = ho.tail;
  a.rep = make_report(st);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  CUtensorMap tm[3];
  FA_TRY(encode_bhnd(&tm[0], Q, p));
  FA_TRY(encode_bhnd(&tm[1], K, p));
  FA_TRY(encode_bhnd(&tm[2], V, p));
  cudaError_t e = launch_fwd_tc(a, p->d, p->dtype == FA_F16, tm, s);
  if (e != cudaSuccess) return cuda_fail(e, "split forward launch");
  return FA_OK;
}

size_t fa_bwd_workspace_size(const fa_params* p) {
  if (fa_check(p, 0) != FA_OK) return 0;
  const size_t rows = (size_t)p->B * p->H * p->N;
  size_t slots = 0;
  if (!p->block_mask) {
    // an fp32 [dV | dK] partial-sum slot of 128 x d each per slice CTA: at most
    // kBwdMaxCtas, and at most one per visited (key tile, query tile) pair
    const int n = (p->N + 127) / 128;
    const long long T = (long long)p->B * p->H * (p->causal ? (long long)n * (n + 1) / 2 : (long long)n * n);
    const long long G = T < kBwdMaxCtas ? T : kBwdMaxCtas;
    slots = align256((size_t)G * 2 * 128 * (size_t)p->d * 4);
  }
  return align256(rows * 4) + align256(rows * (size_t)p->d * 4) + slots;
}

int fa_set_bwd_ctas(int n) { return g_bwd_ctas.exchange(n < 0 ? 0 : n); }

fa_status fa_bwd_preprocess(const fa_params* p, const void* O, const void* dO, void* ws,
                            size_t ws_bytes, void* stream) {
  NvtxRange nvtx_range("fa_bwd_preprocess");
  FA_TRY(fa_check(p, 1));
  FA_TRY(need16(O, "O"));
  FA_TRY(need16(dO, "dO"));
  FA_TRY(check_ws(p, ws, ws_bytes));
  DevStatus* st = nullptr;
  FA_TRY(device_ready(&st));
  BwdArgs a = bwd_args(p, ws);
  a.O = O;
  a.dO = dO;
  a.rep = make_report(st);
  cudaError_t e = launch_bwd_preprocess(a, p->d, p->dtype == FA_F16, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "backward preprocess launch");
  return FA_OK;
}

fa_status fa_bwd_main(const fa_params* p, const void* Q, const void* K, const void* V,
                      const void* dO, const float* LSE, void* dK, void* dV, void* ws,
                      size_t ws_bytes, void* stream) {
  NvtxRange nvtx_range("fa_bwd_main");
  FA_TRY(fa_check(p, 1));
  FA_TRY(need16(Q, "Q"));
  FA_TRY(need16(K, "K"));
  FA_TRY(need16(V, "V"));
  FA_TRY(need16(dO, "dO"));
  FA_TRY(need16(dK, "dK"));
  FA_TRY(need16(dV, "dV"));
  if (!LSE || !aligned(LSE, 4)) {
    set_err("LSE is NULL or misaligned");
    return FA_ERR_INVALID;
  }
  FA_TRY(check_ws(p, ws, ws_bytes));
  DevStatus* st = nullptr;
  FA_TRY(device_ready(&st));
  BwdArgs a = bwd_args(p, ws);
  a.dO = dO;
  a.LSE = LSE;
  a.dK = dK;
  a.dV = dV;
  a.rep = make_report(st);
  CUtensorMap tm[6];
  FA_TRY(encode_bhnd(&tm[0], Q, p));
  FA_TRY(encode_bhnd(&tm[1], K, p));
  FA_TRY(encode_bhnd(&tm[2], V, p));
  FA_TRY(encode_bhnd(&tm[3], dO, p));
  FA_TRY(encode_dqacc(&tm[4], a.dQacc, p, 32));
  FA_TRY(encode_dqacc(&tm[5], a.dQacc, p, 16));
  cudaError_t e = cudaSuccess;
  if (a.direct > 0) e = launch_bwd_tc(a, p->d, p->dtype == FA_F16, tm, static_cast<cudaStream_t>(stream));
  if (e == cudaErrorNotSupported) {
    set_err("backward main kernel not available in this build");
    return FA_ERR_UNSUPPORTED;
  }
  if (e != cudaSuccess) return cuda_fail(e, "backward main launch");
  return FA_OK;
}

fa_status fa_bwd_finalize(const fa_params* p, void* dQ, void* dK, void* dV, void* ws,
                          size_t ws_bytes, void* stream) {
  NvtxRange nvtx_range("fa_bwd_finalize");
  FA_TRY(fa_check(p, 1));
  FA_TRY(need16(dQ, "dQ"));
  FA_TRY(need16(dK, "dK"));
  FA_TRY(need16(dV, "dV"));
  FA_TRY(check_ws(p, ws, ws_bytes));
  DevStatus* st = nullptr;
  FA_TRY(device_ready(&st));
  BwdArgs a = bwd_args(p, ws);
  a.dQ = dQ;
  a.dK = dK;
  a.dV = dV;
  a.rep = make_report(st);
  cudaError_t e = launch_bwd_finalize(a, p->d, p->dtype == FA_F16, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "backward finalize launch");
  return FA_OK;
}

fa_status fa_bwd(const fa_params* p, const void* Q, const void* K, const void* V, const void* O,
                 const void* dO, const float* LSE, void* dQ, void* dK, void* dV, void* ws,
                 size_t ws_bytes, void* stream) {
  NvtxRange nvtx_range("fa_bwd");
  FA_TRY(fa_check(p, 1));
  FA_TRY(need16(dQ, "dQ"));
  FA_TRY(fa_bwd_preprocess(p, O, dO, ws, ws_bytes, stream));
  FA_TRY(fa_bwd_main(p, Q, K, V, dO, LSE, dK, dV, ws, ws_bytes, stream));
  return fa_bwd_finalize(p, dQ, dK, dV, ws, ws_bytes, stream);
}

fa_status fa_get_status(void* stream) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  DevStatus* st = nullptr;
  FA_TRY(device_ready(&st));
  int code = 0;
  if ((e = cudaMemcpy(&code, &st->code, sizeof(int), cudaMemcpyDeviceToHost)) != cudaSuccess)
    return cuda_fail(e, "reading the status word");
  if (code != 0) {
    if ((e = cudaMemset(&st->code, 0, sizeof(int))) != cudaSuccess)
      return cuda_fail(e, "clearing the status word");
    set_err("device reported: %s", fa_status_string(code));
  }
  return static_cast<fa_status>(code);
}

fa_status fa_selftest_timeout(void* stream) {
  NvtxRange nvtx_range("fa_selftest_timeout");
  DevStatus* st = nullptr;
  FA_TRY(device_ready(&st));
  cudaError_t e = launch_wait_selftest(make_report(st), static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "self-test launch");
  return FA_OK;
}

}  // extern "C"
