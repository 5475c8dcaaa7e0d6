// fa_noalloc.cu -- fa_bwd_noalloc: the backward pass with its scratch in a
// fixed device array that belongs to this library instead of a caller workspace.
//
// Some callers cannot allocate device memory at the point where they run the
// backward pass: a plugin that its host application gives a fixed memory
// budget, an engine that plans every buffer ahead of time and forbids
// allocation on its execution path, or code that must not enter the CUDA
// allocator while other work holds it.  For them the backward pass takes its
// fp32 scratch (D = rowsum(dO * O) and the dQ accumulator) from the array
// below.  The array is part of the library image, so every GPU that loads the
// library holds FA_NOALLOC_SCRATCH_BYTES of device memory for it until the
// process exits.  With the runtime's default lazy module loading, the driver
// commits that memory when this file's module is first used on a device, i.e. at
// the first fa_bwd_noalloc call's address lookup (with eager loading, at context
// creation): callers should make that first call during set-up.  Nothing in this
// file calls cudaMalloc, cudaFree or any other allocating routine.  The cached
// address is the primary context's; other driver contexts are not supported.
#include <mutex>

#include "internal.h"

namespace {

static __device__ __align__(256) unsigned char g_bwd_scratch[FA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDev = 64;
void* g_scratch_addr[kMaxDev] = {};
std::mutex g_scratch_mu;

// Device address of g_bwd_scratch on the current device.  In host code the
// array's name only stands for it (a kernel handed that name would fault, or
// silently use host memory), so the address is looked up once per device,
// with that device current, and cached.
fa_status scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    fa::set_error_text("fa_bwd_noalloc: cudaGetDevice failed");
    return FA_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDev) {
    fa::set_error_text("fa_bwd_noalloc: device ordinal out of range");
    return FA_ERR_DEVICE;
  }
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_bwd_scratch);
    if (e != cudaSuccess || p == nullptr) {
      fa::set_error_text("fa_bwd_noalloc: cudaGetSymbolAddress of the scratch array failed");
      return FA_ERR_CUDA;
    }
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return FA_OK;
}

}  // namespace

extern "C" fa_status fa_bwd_noalloc(const fa_params* p, const void* Q, const void* K,
                                    const void* V, const void* O, const void* dO,
                                    const float* LSE, void* dQ, void* dK, void* dV,
                                    void* stream) {
  fa_status s = fa_check(p, 1);
  if (s != FA_OK) return s;
  if (fa_bwd_workspace_size(p) > (size_t)FA_NOALLOC_SCRATCH_BYTES) {
    fa::set_error_text(
        "fa_bwd_noalloc: this problem needs more scratch than the library's fixed "
        "FA_NOALLOC_SCRATCH_BYTES array; call fa_bwd with a caller workspace instead");
    return FA_ERR_WORKSPACE;
  }
  void* scratch = nullptr;
  if ((s = scratch_address(&scratch)) != FA_OK) return s;
  // fa_bwd's first stage rewrites D and zeroes the dQ accumulator before the
  // main kernel reads either, and the main stage stores every partial-sum slot
  // of a sliced key tile in full before the finalize stage reads it (no slot is
  // accumulated into), so the array's previous contents never matter
  return fa_bwd(p, Q, K, V, O, dO, LSE, dQ, dK, dV, scratch, (size_t)FA_NOALLOC_SCRATCH_BYTES,
                stream);
}
