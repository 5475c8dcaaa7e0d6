// ptx.cuh -- inline-PTX building blocks for sm_103a kernels: mbarriers with
// bounded waits, TMA tiled loads, tcgen05 (TMEM allocation, MMA, commit,
// TMEM load/store) and the shared-memory / instruction descriptors of the
// 5th-generation tensor cores.  Written from the public PTX ISA.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"

namespace fa {

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ----------------------------------------------------------------- clusters

// This CTA's rank in its thread-block cluster.
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Cluster-wide barrier of all threads, with release / acquire of the memory
// operations before / after it (shared memory of the cluster's CTAs included).
// The wait is a hardware barrier without a time limit: callers reach it on
// every path, after waits that are themselves bounded.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The shared::cluster address of `addr` (a shared::cta address of this CTA's
// layout) in the shared memory of the cluster's CTA `rank`.
__device__ __forceinline__ uint32_t cluster_map(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

__device__ __forceinline__ float2 ld_cluster_f32x2(uint32_t addr) {
  float2 v;
  asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr) : "memory");
  return v;
}

__device__ __forceinline__ float4 ld_cluster_f32x4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

// ----------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Makes barrier initialisation visible to the async proxy (TMA, tcgen05.commit).
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ uint32_t mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok;
}

// Non-blocking test of whether the phase with the given parity has completed.
__device__ __forceinline__ uint32_t mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok;
}

// Everything a bounded wait needs: the CTA's abort word (shared memory), the
// library status word, the launch's epoch and the time limit.
struct WaitCtx {
  volatile int* abort_cta;
  DevStatus* st;
  uint32_t epoch;
  uint64_t limit_ns;
};

__device__ __forceinline__ void raise_error(const WaitCtx& w, int code) {
  *w.abort_cta = 1;
  atomicCAS(&w.st->code, 0, code);
  atomicMax(&w.st->abort_epoch, w.epoch);
}

// Index check of the debug build (FA_DEBUG): a failed check aborts the launch
// the way a timed-out wait does, with FA_ERR_BOUNDS in the status word (the first
// error wins), and the caller skips the access; nothing traps.  The release build
// compiles it to `true`.
__device__ __forceinline__ bool dbg_check(const WaitCtx& w, bool ok) {
#ifdef FA_DEBUG
  if (!ok) raise_error(w, FA_ERR_BOUNDS);
  return ok;
#else
  (void)w;
  (void)ok;
  return true;
#endif
}

// Wait until the phase with the given parity has completed.  Gives up (returns
// false) when the time limit passes -- recording FA_ERR_TIMEOUT -- or when
// another thread of this CTA or another CTA of this launch has given up.
// Inlined: a call would save and restore live registers through local memory
// on every wait, which costs hundreds of cycles even when the phase is done.
__device__ __forceinline__ bool mbar_wait(const WaitCtx& w, uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  uint64_t t0 = 0;
#pragma unroll 1
  for (uint32_t n = 1;; ++n) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((n & 63u) == 0) {
      if (*w.abort_cta) return false;
      if (*(volatile uint32_t*)&w.st->abort_epoch >= w.epoch) {
        *w.abort_cta = 1;
        return false;
      }
      const uint64_t now = globaltimer_ns();
      if (t0 == 0) {
        t0 = now;
      } else if (now - t0 > w.limit_ns) {
        raise_error(w, FA_ERR_TIMEOUT);
        return false;
      }
    }
  }
}

// Drain wait used on the way out: ignores the abort word (copies or MMAs that
// are in flight must land before shared memory or TMEM is released) but still
// ends after the time limit.
static __device__ __noinline__ bool mbar_drain(const WaitCtx& w, uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t n = 0;; ++n) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((n & 63u) == 63u && globaltimer_ns() - t0 > w.limit_ns) {
      raise_error(w, FA_ERR_TIMEOUT);
      return false;
    }
  }
}

// Warp-uniform wait: every lane polls, and the warp proceeds only if all lanes
// saw the phase complete, so that the .sync.aligned tcgen05 instructions after
// it are executed by a converged warp.
__device__ __forceinline__ bool warp_wait(const WaitCtx& w, uint32_t bar, uint32_t parity) {
  bool ok = mbar_wait(w, bar, parity);
  return __all_sync(0xffffffffu, ok);
}

// ----------------------------------------------------------------- TMA

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

// Element-wise add of a shared-memory tile into global memory (the L2 does the
// additions), tracked by this thread's bulk-async group.
__device__ __forceinline__ void tma_reduce_add_3d(const CUtensorMap* map, uint32_t src, int c0, int c1,
                                                  int c2) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group"
      " [%0, {%1, %2, %3}], [%4];" ::"l"(reinterpret_cast<uint64_t>(map)),
      "r"(c0), "r"(c1), "r"(c2), "r"(src)
      : "memory");
}
__device__ __forceinline__ void bulk_commit_group() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Wait until every bulk copy committed by this thread has completed.
__device__ __forceinline__ void bulk_wait_group0() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
// Wait until every bulk copy committed by this thread has finished reading its
// shared-memory source.
__device__ __forceinline__ void bulk_wait_group_read0() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Generic-proxy shared-memory writes -> visible to the async proxy (tcgen05.mma).
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

__device__ __forceinline__ void named_barrier_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ----------------------------------------------------------------- tcgen05

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Arrive (once) on the mbarrier when every tcgen05 op issued so far by this
// thread has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// D[tmem] (+)= A[smem] * B[smem], kind::f16 (f16/bf16 in, f32 accumulate).
__device__ __forceinline__ void tc_mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem], kind::f16.  A (M x K, 16-bit) lives in TMEM
// with row m in lane m and elements 2c, 2c+1 of the K index packed into column c;
// one MMA (K = 16) reads 8 columns.
__device__ __forceinline__ void tc_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// The same two MMAs and a commit, issued by one lane elected from a converged
// warp: the whole warp runs the issuing loop, so descriptors and addresses stay
// warp-uniform, and the instruction is predicated onto the elected lane.
// (Issuing from divergent single-lane code costs tens of cycles per MMA.)
__device__ __forceinline__ void tc_mma_ss_elect(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                                uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred e, p;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void tc_mma_ts_elect(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                                uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred e, p;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void tc_commit_elect(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n}\n" ::"r"(bar)
      : "memory");
}

// Instruction descriptor of tcgen05.mma kind::f16 with an f32 accumulator.
//   bits 4-5 D format (1 = f32); 7-9 A format, 10-12 B format (0 = f16, 1 = bf16);
//   bit 15 A major (0 = K-major, 1 = MN-major); bit 16 B major;
//   bits 17-22 N >> 3; bits 24-28 M >> 4.
__host__ __device__ constexpr uint32_t idesc_f16(bool f16, int M, int N, bool a_mn, bool b_mn) {
  return (1u << 4) | ((f16 ? 0u : 1u) << 7) | ((f16 ? 0u : 1u) << 10) | ((a_mn ? 1u : 0u) << 15) |
         ((b_mn ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Shared-memory matrix descriptor, 128-byte swizzle.
//   bits 0-13 start address >> 4; 16-29 leading-dimension byte offset >> 4;
//   32-45 stride-dimension byte offset >> 4; 46-48 fixed 0b001;
//   61-63 swizzle mode (2 = 128-byte swizzle).
__device__ __forceinline__ uint64_t desc_sw128(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// Operand tiles in shared memory are built from 128-byte-swizzled atoms of
// `rows` rows x 64 16-bit elements (rows * 128 bytes each, 1024-byte aligned),
// the layout a TMA box of {64, rows} with 128-byte swizzle writes.
//
// K-major operand (the contraction index runs along the 64-element rows):
// MMA step kk covers contraction elements [16 kk, 16 kk + 16).
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t tile, int kk, int rows) {
  return desc_sw128(tile + (uint32_t)(kk >> 2) * (uint32_t)(rows * 128) + (uint32_t)(kk & 3) * 32u,
                    16u, 1024u);
}

// MN-major operand (the contraction index runs down the rows, the M/N index
// along them): MMA step kk covers rows [16 kk, 16 kk + 16); successive 64-wide
// M/N atoms are `rows * 128` bytes apart (leading offset), successive groups of
// 8 rows 1024 bytes apart (stride offset).
__device__ __forceinline__ uint64_t desc_mnmajor(uint32_t tile, int kk, int rows) {
  return desc_sw128(tile + (uint32_t)kk * 2048u, (uint32_t)(rows * 128), 1024u);
}

// Base descriptors of a tile and the per-step increments to add to them (the
// start-address field is the low 14 bits, in 16-byte units, and tiles lie below
// 256 KiB, so adding an offset never carries out of the field).
__device__ __forceinline__ uint64_t desc_kmajor_base(uint32_t tile) { return desc_sw128(tile, 16u, 1024u); }
__device__ __forceinline__ uint64_t desc_mnmajor_base(uint32_t tile, int rows) {
  return desc_sw128(tile, (uint32_t)(rows * 128), 1024u);
}
__host__ __device__ constexpr uint32_t kmajor_step(int kk, int rows) {
  return (uint32_t)(((kk >> 2) * rows * 128 + (kk & 3) * 32) >> 4);
}
__host__ __device__ constexpr uint32_t mnmajor_step(int kk) { return (uint32_t)(kk * 2048 >> 4); }
__device__ __forceinline__ uint64_t desc_add(uint64_t desc, uint32_t bytes) { return desc + (bytes >> 4); }

// Byte offset of 16-byte chunk `ch` (8 elements) of row `r` inside a tile of
// 128-byte-swizzled atoms with `rows` rows: chunk ch lives in atom ch / 8.
__device__ __forceinline__ uint32_t sw128_chunk_offset(int r, int ch, int rows) {
  return (uint32_t)(ch >> 3) * (uint32_t)(rows * 128) + (uint32_t)r * 128u +
         ((uint32_t)((ch & 7) ^ (r & 7)) << 4);
}

#define FA_R8(i) "=r"(r[i]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), "=r"(r[i + 4]), \
                 "=r"(r[i + 5]), "=r"(r[i + 6]), "=r"(r[i + 7])
#define FA_W8(i) "r"(r[i]), "r"(r[i + 1]), "r"(r[i + 2]), "r"(r[i + 3]), "r"(r[i + 4]), \
                 "r"(r[i + 5]), "r"(r[i + 6]), "r"(r[i + 7])

// TMEM loads and stores are .sync.aligned: all 32 lanes of the warp must execute
// them together, so they may only sit under warp-uniform conditions (predicate
// the global stores that follow, never the TMEM access itself).
//
// 32 consecutive TMEM columns of this thread's lane -> 32 registers, and wait
// for the load in the same asm statement so that no use can be scheduled
// before the data has arrived.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : FA_R8(0), FA_R8(8), FA_R8(16), FA_R8(24)
      : "r"(taddr)
      : "memory");
}

// 16 consecutive TMEM columns of this thread's lane -> 16 registers.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : FA_R8(0), FA_R8(8)
      : "r"(taddr)
      : "memory");
}

// Two 32-column loads issued back to back, one wait.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, uint32_t (&r)[64]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31}, [%64];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%32, %33, %34, %35, %36, %37, %38, %39, %40, "
      "%41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, "
      "%58, %59, %60, %61, %62, %63}, [%65];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : FA_R8(0), FA_R8(8), FA_R8(16), FA_R8(24), FA_R8(32), FA_R8(40), FA_R8(48), FA_R8(56)
      : "r"(taddr), "r"(taddr + 32u)
      : "memory");
}

// Two 32-column loads issued without waiting; tmem_wait_ld64 on the same array
// waits for them (its operands tie the registers to the wait, so that no use is
// scheduled before it).
__device__ __forceinline__ void tmem_ld64_nowait(uint32_t taddr, uint32_t (&r)[64]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31}, [%64];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%32, %33, %34, %35, %36, %37, %38, %39, %40, "
      "%41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, "
      "%58, %59, %60, %61, %62, %63}, [%65];"
      : FA_R8(0), FA_R8(8), FA_R8(16), FA_R8(24), FA_R8(32), FA_R8(40), FA_R8(48), FA_R8(56)
      : "r"(taddr), "r"(taddr + 32u)
      : "memory");
}
#define FA_RW8(i) "+r"(r[i]), "+r"(r[i + 1]), "+r"(r[i + 2]), "+r"(r[i + 3]), "+r"(r[i + 4]), \
                  "+r"(r[i + 5]), "+r"(r[i + 6]), "+r"(r[i + 7])
__device__ __forceinline__ void tmem_wait_ld64(uint32_t (&r)[64]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : FA_RW8(0), FA_RW8(8), FA_RW8(16), FA_RW8(24), FA_RW8(32), FA_RW8(40), FA_RW8(48),
                 FA_RW8(56)
               :
               : "memory");
}
#undef FA_RW8

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31, %32};" ::"r"(taddr),
      FA_W8(0), FA_W8(8), FA_W8(16), FA_W8(24)
      : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      FA_W8(0), FA_W8(8)
      : "memory");
}

// N (16, 32 or 64) consecutive TMEM columns of this thread's lane, with the wait.
template <int N>
__device__ __forceinline__ void tmem_ld_n(uint32_t taddr, uint32_t (&r)[N]) {
  static_assert(N == 16 || N == 32 || N == 64, "TMEM load width");
  if constexpr (N == 16) tmem_ld16(taddr, r);
  else if constexpr (N == 32) tmem_ld32(taddr, r);
  else tmem_ld64(taddr, r);
}
template <int N>
__device__ __forceinline__ void tmem_st_n(uint32_t taddr, const uint32_t (&r)[N]) {
  static_assert(N == 16 || N == 32, "TMEM store width");
  if constexpr (N == 16) tmem_st16(taddr, r);
  else tmem_st32(taddr, r);
}

__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

#undef FA_R8
#undef FA_W8

// ----------------------------------------------------------------- dropout
// Philox4x32-10 (Salmon, Moraes, Dror and Shaw, "Parallel random numbers: as
// easy as 1, 2, 3", SC 2011): ten rounds of
//   (x0, x1, x2, x3) -> (hi(M1 x2) ^ x1 ^ k0, lo(M1 x2), hi(M0 x0) ^ x3 ^ k1, lo(M0 x0))
// with the key bumped by the Weyl constants between rounds.  K counters are
// advanced round by round in lockstep: the rounds of one counter depend on each
// other, so independent counters keep the multiply and logic pipes busy.
template <int K>
__device__ __forceinline__ void philox4x32_10_n(uint4 (&c)[K], uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
#pragma unroll
    for (int j = 0; j < K; ++j) {
      const uint32_t hi0 = __umulhi(0xD2511F53u, c[j].x), lo0 = 0xD2511F53u * c[j].x;
      const uint32_t hi1 = __umulhi(0xCD9E8D57u, c[j].z), lo1 = 0xCD9E8D57u * c[j].z;
      c[j] = make_uint4(hi1 ^ c[j].y ^ k0, lo1, hi0 ^ c[j].w ^ k1, lo0);
    }
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
}

// The eight keep decisions of one draw: bit b (for key 8 g + b of the counter
// (g, ...)) from the 16-bit half b mod 2 (low, high) of word b / 2.
__device__ __forceinline__ uint32_t keep_bits8(const uint4& w, uint32_t t) {
  const uint32_t v[4] = {w.x, w.y, w.z, w.w};
  uint32_t bits = 0;
#pragma unroll
  for (int k = 0; k < 4; ++k)
    bits |= ((uint32_t)((v[k] & 0xFFFFu) >= t) << (2 * k)) | ((uint32_t)((v[k] >> 16) >= t) << (2 * k + 1));
  return bits;
}

// Keep bits of keys 32 w .. 32 w + 31 (bit c for key 32 w + c) of query row i in
// head bh: four counters (w * 4 .. w * 4 + 3, i, bh, offset) drawn together.
__device__ __forceinline__ uint32_t drop_keep32(const DropArgs& dr, uint32_t w, uint32_t i, uint32_t bh) {
  uint4 c[4];
#pragma unroll
  for (int g = 0; g < 4; ++g) c[g] = make_uint4(4u * w + (uint32_t)g, i, bh, dr.offset);
  philox4x32_10_n<4>(c, dr.key0, dr.key1);
  uint32_t bits = 0;
#pragma unroll
  for (int g = 0; g < 4; ++g) bits |= keep_bits8(c[g], dr.t) << (8 * g);
  return bits;
}

// Keep bits, for the key row of this lane (keys are consecutive across lanes, so
// lanes 8a .. 8a + 7 share one key group), of the 32 queries q0 .. q0 + 31: bit c
// for query q0 + c.  The eight lanes of a group each draw the counter of one
// query of every 8 and pass the words round, so no counter is drawn twice.  All
// 32 lanes must call it together.
__device__ __forceinline__ uint32_t drop_keep_col32(const DropArgs& dr, uint32_t key, uint32_t q0,
                                                    uint32_t bh) {
  const uint32_t lane = threadIdx.x & 31u, r = lane & 7u;
  uint4 c[4];
#pragma unroll
  for (int m = 0; m < 4; ++m) c[m] = make_uint4(key >> 3, q0 + 8u * m + r, bh, dr.offset);
  philox4x32_10_n<4>(c, dr.key0, dr.key1);
  const uint32_t sh = 16u * (r & 1u);  // this key's half of a word
  uint32_t bits = 0;
#pragma unroll
  for (int m = 0; m < 4; ++m) {
#pragma unroll
    for (uint32_t t = 0; t < 8; ++t) {
      // offer the word that lane (r - t) mod 8 of the group needs for its key; take
      // from lane (r + t) mod 8, whose draw is for query 8m + ((r + t) mod 8), the
      // word of this lane's key
      const uint32_t k = ((r - t) & 7u) >> 1;
      const uint32_t offer = k == 0 ? c[m].x : k == 1 ? c[m].y : k == 2 ? c[m].z : c[m].w;
      const uint32_t got = t == 0 ? offer : __shfl_sync(0xffffffffu, offer, (lane & ~7u) | ((r + t) & 7u));
      bits |= (uint32_t)(((got >> sh) & 0xFFFFu) >= dr.t) << (8u * m + ((r + t) & 7u));
    }
  }
  return bits;
}

// ----------------------------------------------------------------- math

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Packed two-lane fp32 arithmetic (one instruction for two values).
__device__ __forceinline__ uint64_t f2pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t fmul2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

template <bool F16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (F16) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  } else {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
}

template <bool F16>
__device__ __forceinline__ float2 unpack2(uint32_t v) {
  if constexpr (F16) {
    __half2 h = *reinterpret_cast<__half2*>(&v);
    return __half22float2(h);
  } else {
    __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162*>(&v);
    return __bfloat1622float2(h);
  }
}

}  // namespace fa
