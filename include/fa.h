/*
 * fa.h -- C ABI of libfa.so: exact tiled scaled-dot-product attention on one
 * GB300 GPU (sm_103a), forward and backward.
 *
 * The operation is O = softmax(scale * Q K^T) V for every batch b and head h,
 * as stated in "Pourquoi l'attention est liée à la mémoire" (marketmaker.cc,
 * "Un contexte d'une journée complète bat-il un contexte de dix minutes ?")
 * and in "Problema e motivação" of the FlashAttention reading guide
 * (xyznot.com, arXiv 2205.14135).  The score matrix is never written to
 * device memory: the forward pass streams key/value tiles through on-chip
 * memory with the running-max / running-sum recurrence ("La récurrence
 * softmax en ligne"; "Rastreamento Incremental do Softmax"), and the backward
 * pass recomputes the scores and probabilities tile by tile from Q, K, V and
 * the saved per-row statistic ("Passe arrière : recalculer au lieu de
 * stocker").
 *
 * Conventions shared by every call:
 *   - Tensors Q, K, V, O, dO, dQ, dK, dV are device buffers of shape
 *     [B][H][N][d], contiguous, in the element type `dtype`; their base
 *     addresses must be 16-byte aligned.  LSE is a device fp32 buffer [B][H][N].
 *   - The caller owns every buffer.  The library allocates no device memory of
 *     its own apart from one small status word per device.
 *   - Calls are asynchronous on `stream` (a cudaStream_t, or NULL for the
 *     legacy default stream).  Argument errors are returned before anything is
 *     launched; a failed launch returns FA_ERR_CUDA; a kernel that gives up
 *     waiting on an on-chip barrier records FA_ERR_TIMEOUT in the status word,
 *     which fa_get_status() returns.
 *   - Only the current CUDA device is used; it must be compute capability 10.3.
 *   - A debug build of the library (compiled with FA_DEBUG defined: libfa_debug.so)
 *     checks, in the kernels, every global-memory index it stores to and every
 *     tile coordinate it copies from against the tensor's bounds; a failed check
 *     skips the access and records FA_ERR_BOUNDS in the status word (no trap, so
 *     the context stays usable).  The release build compiles the checks away.
 */
#ifndef FA_H
#define FA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID = -1,     /* null pointer, size out of range, misaligned buffer, bad scale */
  FA_ERR_UNSUPPORTED = -2, /* well-formed request this library does not implement */
  FA_ERR_CUDA = -3,        /* a CUDA runtime or driver call failed */
  FA_ERR_TIMEOUT = -4,     /* a kernel gave up waiting on a barrier (via fa_get_status) */
  FA_ERR_WORKSPACE = -5,   /* workspace missing or smaller than required */
  FA_ERR_DEVICE = -6,      /* the current device is not compute capability 10.3 */
  FA_ERR_BOUNDS = -7       /* debug build only: a kernel's index check failed (via fa_get_status) */
} fa_status;

typedef enum { FA_F32 = 0, FA_F16 = 1, FA_BF16 = 2 } fa_dtype;

/*
 * Problem description.
 *   B, H, N, d  batch, heads, sequence length (queries = keys), head size.
 *               N >= 1 (any value: tails that are not a multiple of the tile
 *               are masked); d in {64, 128}; B*H*N*d < 2^31.
 *   dtype       element type of Q, K, V, O, dO, dQ, dK, dV (fa_dtype).
 *               FA_F32 runs the fp32 forward only.
 *   scale       positive finite factor applied to Q K^T before the softmax
 *               (1/sqrt(d) for standard attention).
 *   causal      nonzero: query i only sees keys j <= i ("Le masquage causal
 *               est l'endroit où le trading bénéficie d'une remise").
 *   block_mask  device uint8 matrix or NULL ("Extensão: Block-Sparse
 *               FlashAttention"): entry [i / mask_block][j / mask_block]
 *               keeps (nonzero) or hides (0) the pair (query i, key j).  Each
 *               (b, h) uses the T x T row-major matrix at
 *               block_mask + b * mask_stride_b + h * mask_stride_h, with
 *               T = ceil(N / mask_block); strides in elements, 0 broadcasts.
 *               Combined with `causal` by AND.  Hidden tiles are never loaded.
 *   mask_block  tokens per mask entry; a positive multiple of 128 when
 *               block_mask is set (ignored otherwise).
 *   dropout_p   probability in [0, 1) of dropping each attention weight (the
 *               softmax output, after masking); kept weights are scaled by the
 *               inverse of the keep probability.  Dropout is fused into the
 *               kernels ("Fusão de Kernels", reading guide, "Ideias centrais").
 *               0 = none.
 *   dropout_seed, dropout_offset
 *               the keep decision of weight (query i, key j) of head
 *               bh = b * H + h is the 16-bit half (low for even j, high for
 *               odd j) of word (j mod 8) / 2 of Philox4x32-10 (Salmon et al.,
 *               SC 2011) with counter (j / 8, i, bh, dropout_offset) and key
 *               (seed mod 2^32, seed / 2^32): kept when the half is at least
 *               t = floor(p * 2^16), i.e. with probability 1 - t / 2^16 (p to
 *               within 2^-16), and then scaled by 2^16 / (2^16 - t).  The
 *               backward regenerates the same decisions from the same three
 *               values instead of storing them.
 * A query row whose allowed key set is empty gets O = 0 and LSE = -inf, and
 * contributes nothing to the gradients.  With dropout, O is the dropped and
 * rescaled weights times V, while LSE stays the log-sum-exp of the undropped
 * scores (it is what the backward recomputes the weights from).
 */
typedef struct {
  int B, H, N, d;
  int dtype;
  float scale;
  int causal;
  const uint8_t* block_mask;
  int mask_block;
  long long mask_stride_b, mask_stride_h;
  float dropout_p;
  unsigned long long dropout_seed;
  unsigned int dropout_offset;
} fa_params;

/* Host-only validation of `p` (no CUDA call).  for_backward selects the
 * backward's extra limits.  Returns FA_OK, FA_ERR_INVALID or
 * FA_ERR_UNSUPPORTED. */
fa_status fa_check(const fa_params* p, int for_backward);

/*
 * Forward: O = softmax(scale * Q K^T [masked]) V and
 * LSE[b,h,i] = m_i + ln(l_i), the natural-log log-sum-exp of row i of the
 * scaled, masked scores (the running max m and running sum l of "L'algorithme
 * Flash Attention", folded into one number).  O is written in `dtype`; LSE in
 * fp32.  fp16/bf16 run on the tensor cores (tcgen05, fp32 accumulation);
 * fp32 runs a SIMT kernel in fp32 arithmetic.
 */
fa_status fa_fwd(const fa_params* p, const void* Q, const void* K, const void* V, void* O,
                 float* LSE, void* stream);

/* Largest split count fa_fwd_split accepts (the slices of a query tile run as
 * one thread-block cluster, at most 8 CTAs in a portable cluster). */
#define FA_MAX_SPLITS 8

/*
 * Split-KV forward: the same O and LSE as fa_fwd, computed with the key range
 * of every 128-row query tile cut into `num_splits` slices of
 * ceil(ceil(N / 128) / num_splits) key tiles, one CTA per (query tile, slice),
 * so that a problem with few query tiles (one long sequence, few heads) still
 * fills the GPU.  Each slice keeps its own running max m_s and sum l_s; the
 * slices of a query tile run as one thread-block cluster and merge in shared
 * memory with the statistics merge of "Rastreamento Incremental do Softmax"
 * (the reading guide to the FlashAttention paper): m = max_s m_s,
 * l = sum_s exp(m_s - m) l_s, O = sum_s exp(m_s - m) O_s / l and
 * LSE = m + log l, each slice's O_s unnormalised.  Nothing goes through device
 * memory but Q, K, V, O and LSE.  The key-scan parallelism of the decode
 * kernels mentioned in "Что это изменило на практике" ("Почему Flash Attention
 * быстрее") is the same idea.
 *
 * num_splits in [1, min(FA_MAX_SPLITS, ceil(N / 128))], else FA_ERR_INVALID;
 * a count that would leave trailing slices empty runs with the non-empty ones
 * only.  num_splits = 1 is fa_fwd.  fp16/bf16 only for num_splits > 1 (FA_F32
 * -> FA_ERR_UNSUPPORTED).  Results match fa_fwd up to rounding order (the
 * fp32 slices are rounded to `dtype` once, after the merge).
 */
fa_status fa_fwd_split(const fa_params* p, const void* Q, const void* K, const void* V, void* O,
                       float* LSE, int num_splits, void* stream);

/* Split count for fa_fwd_split on a GPU with `num_sms` SMs (<= 0: ask the
 * current device; 1 if that fails).  1 when the unsplit grid of B*H*ceil(N/128)
 * CTAs already fills one wave of 2 * num_sms (two CTAs per SM); otherwise the
 * count with the fewest modelled waves x (key tiles per CTA + 2).  1 for
 * FA_F32, 0 on invalid p.  Host-only when num_sms > 0. */
int fa_fwd_num_splits(const fa_params* p, int num_sms);

/* Bytes of device workspace fa_bwd needs, each part 256-byte aligned.  The
 * backward of "Passe arrière : recalculer au lieu de stocker" (marketmaker.cc)
 * keeps only O and the per-row statistic of the forward and recomputes the rest;
 * what it needs besides is linear in N ("Análise de Complexidade", reading
 * guide: O(N) extra memory): fp32
 * D = rowsum(dO * O) [B*H*N], the fp32 dQ accumulator [B*H*N*d] and, without a
 * block mask, the fp32 partial-sum slots of a sliced main kernel (2 x 128 x d
 * values for each of up to min(160, pairs) slices, where pairs = B*H*T^2 or
 * B*H*T(T+1)/2 causal, T = ceil(N / 128)).  0 on invalid p. */
size_t fa_bwd_workspace_size(const fa_params* p);

/*
 * Backward of the forward above for the loss whose gradient at O is dO, as
 * "Passe arrière : recalculer au lieu de stocker" (marketmaker.cc) and the
 * recomputation bullet of "Ideias centrais" (reading guide) describe it: the
 * score and probability tiles are recomputed block by block from Q, K and the
 * saved LSE instead of being stored.  The formulas (the pages give none) are the
 * derivative of the definition:
 *   P = exp(scale * S - LSE), dV = P^T dO, dP = dO V^T, D = rowsum(dO * O),
 *   dS = P * (dP - D), dQ = scale * dS K, dK = scale * dS^T Q.
 * Q, K, V, O, LSE must be those of the forward call (same params).  dQ, dK, dV
 * are written in `dtype`.  `workspace` is a device buffer of at least
 * fa_bwd_workspace_size(p) bytes, 256-byte aligned, owned by the caller; its
 * contents on entry do not matter.  fp16/bf16 only (FA_F32 -> UNSUPPORTED).
 * Runs fa_bwd_preprocess, fa_bwd_main and fa_bwd_finalize in that order.
 */
fa_status fa_bwd(const fa_params* p, const void* Q, const void* K, const void* V, const void* O,
                 const void* dO, const float* LSE, void* dQ, void* dK, void* dV, void* workspace,
                 size_t workspace_bytes, void* stream);

/* The three stages of fa_bwd, exported so that each can be timed on its own.
 * preprocess: D = rowsum(dO * O) into the workspace, dQ accumulator zeroed.
 * main: recompute P tile by tile, accumulate dK, dV per key tile and add
 *       scale-free dQ contributions into the accumulator.  One CTA per key
 *       tile, whose dK, dV it writes.  Without a block mask, when that would
 *       leave SMs idle, key tiles are cut into slices of their query tiles,
 *       one CTA each, a key tile of several slices getting fp32 partial dK, dV
 *       in the workspace: with fewer key tiles than SMs every key tile (slices
 *       as short as fill one wave), and, non-causal, the key tiles of a last,
 *       partly filled wave (over the SMs that wave leaves idle).
 * finalize: dQ = scale * accumulator, converted to `dtype`, and dK, dV of the
 *       shared key tiles from their partial sums.  Must follow the main stage
 *       of the same call sequence (same p, workspace and fa_set_bwd_ctas). */
fa_status fa_bwd_preprocess(const fa_params* p, const void* O, const void* dO, void* workspace,
                            size_t workspace_bytes, void* stream);
fa_status fa_bwd_main(const fa_params* p, const void* Q, const void* K, const void* V,
                      const void* dO, const float* LSE, void* dK, void* dV, void* workspace,
                      size_t workspace_bytes, void* stream);
fa_status fa_bwd_finalize(const fa_params* p, void* dQ, void* dK, void* dV, void* workspace,
                          size_t workspace_bytes, void* stream);

/* The CTAs per wave that the backward main kernel plans its slices for (0, the
 * default: one per SM, at most 160; n > 0: min(n, that)).  Applies to backward
 * calls made after it; do not change it between the main and finalize stages
 * of one backward pass.  Returns the previous value.  The tests use it to make
 * small problems cut their key tiles into slices. */
int fa_set_bwd_ctas(int n);

/*
 * Maximum workspace, in bytes, that fa_bwd_noalloc can serve (64 MiB); e.g.
 * B=4, H=12, N=2048, d=64 needs about 34 MiB (fa_bwd_workspace_size).
 */
#define FA_NOALLOC_SCRATCH_BYTES (64ull << 20)

/*
 * The backward pass for callers that cannot allocate device memory where they
 * run it -- a plugin handed a fixed memory budget by its host application, an
 * engine that plans every buffer ahead of time and forbids allocation on its
 * execution path, or code that must not enter the CUDA allocator while other
 * work holds it.  The pages have no counterpart of this call; it exists for
 * those callers only.
 *
 * Same arguments and results as fa_bwd without the workspace: the fp32 scratch
 * (D, the dQ accumulator and the partial-sum slots) comes from a FA_NOALLOC_SCRATCH_BYTES array that
 * is part of the library image, so every GPU that loads libfa.so holds that
 * memory until the process exits.  No call here allocates or frees device
 * memory.  A problem whose workspace (fa_bwd_workspace_size) exceeds the array
 * is rejected with FA_ERR_WORKSPACE before anything is launched.
 *
 * The first call on each device looks up the array's device address (with
 * that device current) and caches it; make that first call before any stream
 * capture.  Under the CUDA runtime's default lazy module loading the driver
 * commits the array's device memory at that first lookup (under eager loading,
 * when the context is created), so that first call is where an out-of-memory
 * error can appear: make it during set-up, not on the execution path.  The
 * cached address is that of the runtime's primary context on each device;
 * callers that run the library under another driver context are not served.
 * Every call, on every stream, shares the one array: calls that can overlap on
 * the GPU race on it and must be serialised by the caller.  Each call rewrites
 * all the scratch it reads: D and the dQ accumulator (zeroed first) in the first
 * stage, and the fp32 partial-sum slots of key tiles cut into several slices,
 * each stored in full by the main stage before the finalize stage reads it.  So
 * nothing left by an earlier call affects a call's results.
 */
fa_status fa_bwd_noalloc(const fa_params* p, const void* Q, const void* K, const void* V,
                         const void* O, const void* dO, const float* LSE, void* dQ, void* dK,
                         void* dV, void* stream);

/* Synchronises `stream`, returns the device-side status recorded since the
 * previous call (FA_OK or FA_ERR_TIMEOUT) and clears it; FA_ERR_CUDA if the
 * synchronisation itself fails.  The pages have no counterpart: it reports the
 * library's own failure detection (every on-chip barrier wait of every kernel is
 * bounded in time, so a kernel that cannot proceed gives up and records the
 * error instead of hanging), which guards the custom low-level CUDA that
 * "Limitações e questões em aberto" (reading guide) names as the method's cost. */
fa_status fa_get_status(void* stream);

/* Upper bound, in nanoseconds, on any single barrier wait inside the kernels
 * launched after this call (default 2e9).  Returns the previous value. */
unsigned long long fa_set_wait_limit_ns(unsigned long long ns);

/* Launches one CTA that waits on a barrier nothing will complete, so that the
 * wait limit runs out and FA_ERR_TIMEOUT is recorded; used to test the
 * failure path without faulting the GPU.  Returns the launch status. */
fa_status fa_selftest_timeout(void* stream);

/* Static description of a status code. */
const char* fa_status_string(int status);

/* Text of the last CUDA or validation failure seen by this thread. */
const char* fa_last_error(void);

/* Library interface version (major * 100 + minor). */
int fa_version(void);

/* ------------------------------------------------------------------------
 * FP8 forward with incoherent processing ("Trois idées pour FA3",
 * marketmaker.cc, point 3: naive FP8 attention suffers from outlier
 * coordinates; rotating the query and key vectors at random before block
 * quantisation spreads an outlier over all coordinates).  Two calls, so that
 * the quantised operands can be produced once and reused:
 *
 *   fa_fp8_quantize  Q^ = Q D H / d and K^ = K D H, with H the d x d Sylvester
 *                    Hadamard matrix (H_ab = (-1)^popcount(a & b)) and
 *                    D = diag(signs); Q^ K^^T = Q K^T since H H^T = d I.  With
 *                    signs = NULL there is no rotation (Q^ = Q, K^ = K).  V is
 *                    not rotated.  Each block of 128 rows of one head of Q^, K^
 *                    and V gets the smallest power-of-two scale sigma with
 *                    max|x| / sigma <= 448 (1 for an all-zero block; 2^-126 at
 *                    least), and its values become e4m3 codes of x / sigma
 *                    (round to nearest even, saturating to +-448; the rotated
 *                    values are formed in fp32).
 *   fa_fwd_fp8       the forward on those codes: scores
 *                    scale * sigma_q * sigma_k * (q8 . k8) accumulated in fp32
 *                    on the tensor cores, the online softmax against the exact
 *                    running max m, the weights P~ = exp(s - m) <= 1 quantised
 *                    as e4m3(256 P~) for the P~ V product, the row sum l of the
 *                    unquantised P~; O = sum sigma_v P~q V8 / (256 l) in the
 *                    dtype of p, LSE = m + ln l (natural log, fp32).
 *
 * Buffers (device memory, owned by the caller, 16-byte aligned except the
 * scales, which are 4-byte aligned):
 *   q8, k8      uint8 [B*H][N][d]     e4m3 codes of Q^ and K^
 *   vt8         uint8 [B*H][d][ld]    e4m3 codes of V transposed (row c holds
 *                                     column c of V over the keys), ld =
 *                                     fa_fp8_vt_cols(N); entries past N are 0
 *   sq, sk, sv  float [B*H][ceil(N / 128)]  the block scales (powers of two)
 *   signs       float [d]             +-1 (device memory), or NULL
 * p: dtype FA_F16 or FA_BF16 (of Q, K, V and of O), d 64 or 128, causal and
 * block masks as for fa_fwd; dropout and FA_F32 give FA_ERR_UNSUPPORTED.  Both
 * calls are asynchronous on `stream`; validation errors return before any
 * launch.  Codes made elsewhere (any e4m3 values with power-of-two scales in
 * this layout) may be passed to fa_fwd_fp8.
 * ------------------------------------------------------------------------ */
int fa_fp8_vt_cols(int N);
fa_status fa_fp8_quantize(const fa_params* p, const void* Q, const void* K, const void* V,
                          const float* signs, void* q8, void* k8, void* vt8, float* sq, float* sk,
                          float* sv, void* stream);
fa_status fa_fwd_fp8(const fa_params* p, const void* q8, const void* k8, const void* vt8,
                     const float* sq, const float* sk, const float* sv, void* O, float* LSE,
                     void* stream);

#ifdef __cplusplus
}
#endif

#endif /* FA_H */
