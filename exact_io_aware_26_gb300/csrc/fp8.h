// fp8.h -- arguments and launchers of the FP8 forward (fwd_fp8.cu), shared with
// the C-ABI front end.  Not part of the public interface.
#pragma once
#include "internal.h"

namespace fa {

// Rotation and block quantisation: Q^ = Q D H / d, K^ = K D H (D = diag(signs),
// H the Sylvester Hadamard matrix; no rotation when signs is null) and V, each
// quantised to e4m3 with one power-of-two scale per 128-row block.
struct Fp8QuantArgs {
  int BH, N;
  int T;   // ceil(N / 128): blocks per head
  int ld;  // row length of vt8: N rounded up to a multiple of 16
  const void* Q;
  const void* K;
  const void* V;
  const float* signs;  // [d] of +-1, or nullptr
  uint8_t* q8;         // [BH][N][d]
  uint8_t* k8;         // [BH][N][d]
  uint8_t* vt8;        // [BH][d][ld]
  float* sq;           // [BH][T]
  float* sk;
  float* sv;
};

struct Fp8FwdArgs {
  int B, H, N, T;
  float scale_log2;  // softmax scale * log2(e)
  MaskArgs m;
  const float* sq;
  const float* sk;
  const float* sv;
  void* O;     // [B*H][N][d], 16-bit
  float* LSE;  // [B*H][N]
  // grid order, as in the 16-bit forward: heads in groups of head_group, query-
  // tile-major within a group, the last head_tail heads one more group
  int head_group;
  int head_tail;
  Report rep;
};

cudaError_t launch_fp8_quantize(const Fp8QuantArgs& a, int d, bool f16, cudaStream_t s);
// tm: Q8, K8 ({d, N, B*H} bytes, box {d, 128}) and Vt8 ({ld, d, B*H}, box {128, d})
cudaError_t launch_fwd_fp8(const Fp8FwdArgs& a, int d, bool f16, const CUtensorMap* tm,
                           cudaStream_t s);

}  // namespace fa
