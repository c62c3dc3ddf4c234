// Device-side building blocks for the sm_103a attention kernels: mbarriers,
// TMA tile loads, tcgen05 (UMMA) issue/commit, TMEM allocation and loads,
// shared-memory matrix descriptors and bounded waits.
//
// Everything here is inline PTX written from the public PTX ISA description of
// these instructions; no CUTLASS/CuTe is used.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pfa_internal.h"

namespace pfa {

// ----------------------------------------------------------------------------
// Small helpers
// ----------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Programmatic dependent launch. A kernel launched with launch_pdl() may start
// while the kernel before it on the stream is still running; it runs its setup
// (barriers, TMEM) and then calls grid_dependency_wait() before its first access
// to global memory, which returns once that kernel has completed and its writes
// are visible (immediately when there is none). grid_launch_dependents() lets
// the next kernel on the stream be scheduled onto SMs as this one's CTAs leave.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;"); }

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float lg2_approx(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Three-input maximum (one instruction on sm_100 and later).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Packed FP32x2 arithmetic: two lanes of work per instruction.
__device__ __forceinline__ void fma2(float& y0, float& y1, float x0, float x1, float a, float b) {
  asm("{\n\t.reg .b64 xa, aa, ba, ya;\n\t"
      "mov.b64 xa, {%2, %3};\n\tmov.b64 aa, {%4, %4};\n\tmov.b64 ba, {%5, %5};\n\t"
      "fma.rn.f32x2 ya, xa, aa, ba;\n\tmov.b64 {%0, %1}, ya;\n\t}"
      : "=f"(y0), "=f"(y1)
      : "f"(x0), "f"(x1), "f"(a), "f"(b));
}
// y = x * a + b lane-wise, with per-lane a and b.
__device__ __forceinline__ void fma2v(float& y0, float& y1, float x0, float x1, float a0, float a1,
                                      float b0, float b1) {
  asm("{\n\t.reg .b64 xa, aa, ba, ya;\n\t"
      "mov.b64 xa, {%2, %3};\n\tmov.b64 aa, {%4, %5};\n\tmov.b64 ba, {%6, %7};\n\t"
      "fma.rn.f32x2 ya, xa, aa, ba;\n\tmov.b64 {%0, %1}, ya;\n\t}"
      : "=f"(y0), "=f"(y1)
      : "f"(x0), "f"(x1), "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}
__device__ __forceinline__ void mul2v(float& y0, float& y1, float x0, float x1, float a0, float a1) {
  asm("{\n\t.reg .b64 xa, aa, ya;\n\t"
      "mov.b64 xa, {%2, %3};\n\tmov.b64 aa, {%4, %5};\n\t"
      "mul.rn.f32x2 ya, xa, aa;\n\tmov.b64 {%0, %1}, ya;\n\t}"
      : "=f"(y0), "=f"(y1)
      : "f"(x0), "f"(x1), "f"(a0), "f"(a1));
}
__device__ __forceinline__ void add2(float& s0, float& s1, float x0, float x1) {
  asm("{\n\t.reg .b64 sa, xa;\n\t"
      "mov.b64 sa, {%0, %1};\n\tmov.b64 xa, {%2, %3};\n\t"
      "add.rn.f32x2 sa, sa, xa;\n\tmov.b64 {%0, %1}, sa;\n\t}"
      : "+f"(s0), "+f"(s1)
      : "f"(x0), "f"(x1));
}
__device__ __forceinline__ void mul2(float& y0, float& y1, float a) {
  asm("{\n\t.reg .b64 ya, aa;\n\t"
      "mov.b64 ya, {%0, %1};\n\tmov.b64 aa, {%2, %2};\n\t"
      "mul.rn.f32x2 ya, ya, aa;\n\tmov.b64 {%0, %1}, ya;\n\t}"
      : "+f"(y0), "+f"(y1)
      : "f"(a));
}

// Two FP32 values -> packed BF16x2 (round to nearest even); `lo` goes to bits 0..15.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}
// The FP32 pair (a, b) rounded to the nearest FP8 E4M3 values (ties to even,
// saturating at 448), returned as FP32 (exact: E4M3 values are FP16 values).
__device__ __forceinline__ void e4m3_round2(float& a, float& b) {
  uint32_t h;
  asm("{\n\t.reg .b16 t;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 t, %1, %2;\n\t"   // upper byte from the first source
      "cvt.rn.f16x2.e4m3x2 %0, t;\n\t}"               // lower byte to the lower half
      : "=r"(h)
      : "f"(b), "f"(a));
  a = __half2float(__ushort_as_half(static_cast<unsigned short>(h & 0xFFFFu)));
  b = __half2float(__ushort_as_half(static_cast<unsigned short>(h >> 16)));
}
// The FP32 pair (a, b) rounded to the nearest FP4 E2M1 values (0, 0.5, 1, 1.5, 2,
// 3, 4, 6; ties to even, saturating at 6), returned as FP32.
__device__ __forceinline__ void e2m1_round2(float& a, float& b) {
  uint32_t h;
  asm("{\n\t.reg .b8 t;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\t"   // upper nibble from the first source
      "cvt.rn.f16x2.e2m1x2 %0, t;\n\t}"               // lower nibble to the lower half
      : "=r"(h)
      : "f"(b), "f"(a));
  a = __half2float(__ushort_as_half(static_cast<unsigned short>(h & 0xFFFFu)));
  b = __half2float(__ushort_as_half(static_cast<unsigned short>(h >> 16)));
}

// x rounded to the nearest BF16 value (ties to even), returned as FP32.
__device__ __forceinline__ float bf16_round(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }
__device__ __forceinline__ float bf16lo_to_f32(uint32_t p) { return __uint_as_float(p << 16); }
__device__ __forceinline__ float bf16hi_to_f32(uint32_t p) { return __uint_as_float(p & 0xFFFF0000u); }

// Read-only global load that stays where it is written: a prefetch issued one
// tile ahead must not be moved down to its use by the compiler.
__device__ __forceinline__ float ld_global_early(const float* p) {
  float v;
  asm volatile("ld.global.nc.f32 %0, [%1];" : "=f"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

// Writes made by ordinary stores to shared memory become visible to the async
// proxy (TMA, tensor core) once this fence has executed in the writing thread.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ----------------------------------------------------------------------------
// mbarrier
// ----------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
// Warp-collective: every lane calls it with the same arguments; one elected lane arrives.
__device__ __forceinline__ void mbar_arrive_expect_tx_warp(uint32_t bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n\t}" ::"r"(bar),
      "r"(bytes)
      : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Per-CTA control block for bounded waits. `abort` lives in shared memory; once
// any thread gives up on a wait it is set and every other wait returns false
// promptly, so all roles reach the common teardown. The first wait to give up
// in a launch also records where: kernel id, barrier offset, parity and block.
struct WaitCtl {
  volatile int* abort;           // shared memory
  int* err;                      // global error word (may be null)
  unsigned long long* site;      // global error-site word (may be null)
  uint32_t smem_base;            // shared address of the CTA's dynamic shared memory
  uint32_t kernel;               // 1 forward, 2 backward, 3 delta via dP o P
};

// Wait budget per wait: a correct pipeline waits micro-seconds; a stuck one
// is abandoned after about a second.
constexpr uint64_t kWaitLimitNs = 1000ull * 1000ull * 1000ull;

// Error site encoding: bit 63 set, kernel in bits 56-59, bit 55 drain wait,
// bit 54 parity, barrier byte offset in bits 32-53, blockIdx.x in bits 0-31.
__device__ __forceinline__ void raise_error(const WaitCtl& c, int code, uint32_t bar, uint32_t parity,
                                            bool drain) {
  *c.abort = 1;
  if (c.err) atomicOr(c.err, code);
  if (c.site) {
    const unsigned long long w = (1ull << 63) | (static_cast<unsigned long long>(c.kernel & 15u) << 56) |
                                 (static_cast<unsigned long long>(drain ? 1u : 0u) << 55) |
                                 (static_cast<unsigned long long>(parity & 1u) << 54) |
                                 (static_cast<unsigned long long>((bar - c.smem_base) & 0x3FFFFFu) << 32) |
                                 static_cast<unsigned long long>(blockIdx.x);
    atomicCAS(c.site, 0ull, w);
  }
}

// The same wait with acquire semantics at cluster scope: for a barrier that
// threads of the other CTA of a cluster arrive on (their writes before the
// arrival become visible to this CTA).
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// ----------------------------------------------------------------------------
// Clusters of two CTAs (the cta_group::2 tensor-core pairing)
// ----------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Shared::cluster address of the variable at shared address `addr` in CTA `rank`
// of this cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
// Arrive on an mbarrier given by its shared::cluster address (possibly in the other
// CTA), releasing this thread's prior writes at cluster scope.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}
// Every thread of both CTAs of the cluster (also a barrier within the CTA).
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

// Whole-warp wait with a warp-uniform result (all 32 lanes must call it).
// CLUSTER: acquire at cluster scope (mbar_try_wait_cluster).
template <bool CLUSTER = false>
__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity, const WaitCtl& c) {
  auto try_wait = [&]() { return CLUSTER ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity); };
  if (__all_sync(0xFFFFFFFFu, try_wait())) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    const bool done = try_wait();
    if (__all_sync(0xFFFFFFFFu, done)) return true;
    if ((it & 15u) == 0) {
      int give_up = 0;
      if ((threadIdx.x & 31) == 0) {
        if (*c.abort) {
          give_up = 1;
        } else if (global_timer_ns() - t0 > kWaitLimitNs) {
          raise_error(c, PFA_DEVERR_TIMEOUT, bar, parity, false);
          give_up = 1;
        }
      }
      if (__shfl_sync(0xFFFFFFFFu, give_up, 0)) return false;
    }
  }
}

// Teardown wait that ignores the abort flag: used to let in-flight TMA copies
// and MMAs finish before the CTA releases its shared memory and TMEM.
__device__ __forceinline__ bool wait_drain(uint32_t bar, uint32_t parity, const WaitCtl& c) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > kWaitLimitNs) {
      raise_error(c, PFA_DEVERR_TIMEOUT, bar, parity, true);
      return false;
    }
  }
  return true;
}

// ----------------------------------------------------------------------------
// TMA
// ----------------------------------------------------------------------------
// Issue from a whole warp. The TMA and tcgen05 issue instructions below are
// warp-collective wrappers: all 32 lanes of the warp call them together with
// warp-uniform arguments and one lane, chosen by elect.sync, issues. Issuing
// from a branch that only one lane takes instead leaves the compiler unable to
// treat the operands as uniform, which was measured at roughly 65 cycles per
// tcgen05.mma against 32-64 cycles of tensor work.
__device__ __forceinline__ void tma_prefetch_desc_warp(const CUtensorMap* m) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e prefetch.tensormap [%0];\n\t}" ::"l"(reinterpret_cast<uint64_t>(m))
      : "memory");
}

// 3-D tiled load: coordinates (x innermost, y, z) in elements; x must be a
// multiple of 8 for 16-bit data (16-byte rule), which the callers guarantee by
// only using x in {0, 64}.
__device__ __forceinline__ void tma_load_3d_warp(uint32_t dst, const CUtensorMap* m, uint32_t bar,
                                                 int x, int y, int z) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];\n\t}" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(x), "r"(y), "r"(z)
      : "memory");
}

// 3-D tiled reduce-add of a shared-memory box into global memory (FP32 add
// for an FP32 tensor map). Elements outside the tensor's extent are skipped.
// The coordinates must be non-negative and x x 4 bytes a multiple of 16.
// Warp-collective; the elected lane also commits the copy to its bulk group.
__device__ __forceinline__ void tma_reduce_add_3d_warp(const CUtensorMap* m, uint32_t src, int x, int y,
                                                       int z) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group"
      " [%0, {%2, %3, %4}], [%1];\n\t"
      "@e cp.async.bulk.commit_group;\n\t}" ::"l"(reinterpret_cast<uint64_t>(m)),
      "r"(src), "r"(x), "r"(y), "r"(z)
      : "memory");
}
// 3-D tiled store of a shared-memory box into global memory; elements outside
// the tensor's extent are not written. The coordinates must be non-negative and
// x x the element size a multiple of 16 bytes. Warp-collective; the elected lane
// also commits the copy to its bulk group.
__device__ __forceinline__ void tma_store_3d_warp(const CUtensorMap* m, uint32_t src, int x, int y, int z) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group"
      " [%0, {%2, %3, %4}], [%1];\n\t"
      "@e cp.async.bulk.commit_group;\n\t}" ::"l"(reinterpret_cast<uint64_t>(m)),
      "r"(src), "r"(x), "r"(y), "r"(z)
      : "memory");
}
// The elected lane waits until its committed bulk copies have finished reading
// shared memory (read) or have completed (all); then the warp reconverges.
__device__ __forceinline__ void bulk_wait_read_warp() {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e cp.async.bulk.wait_group.read 0;\n\t}" ::
          : "memory");
  __syncwarp();
}
__device__ __forceinline__ void bulk_wait_all_warp() {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e cp.async.bulk.wait_group 0;\n\t}" ::
          : "memory");
  __syncwarp();
}

// Prefetch a 3-D tile into L2 (no shared memory, no completion to wait for);
// warp-collective like the loads.
__device__ __forceinline__ void tma_prefetch_l2_3d_warp(const CUtensorMap* m, int x, int y, int z) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];\n\t}" ::"l"(
          reinterpret_cast<uint64_t>(m)),
      "r"(x), "r"(y), "r"(z)
      : "memory");
}

// ----------------------------------------------------------------------------
// tcgen05: TMEM allocation, MMA, commit, loads/stores
// ----------------------------------------------------------------------------
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

// D[tmem] (+)= A[smem] * B[smem], BF16 inputs, FP32 accumulate (warp-collective).
__device__ __forceinline__ void umma_bf16_warp(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                               uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]: A is read from tensor memory (one row per lane,
// two BF16 values per 32-bit column, lower K index in the low half). Warp-collective.
__device__ __forceinline__ void umma_bf16_tmem_a_warp(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                                      uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on `bar` when every tcgen05.mma issued so far by the elected lane
// has completed (warp-collective; the same lane is elected for every call of a
// converged warp, so it covers all MMAs the warp issued).
__device__ __forceinline__ void umma_commit_warp(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar)
      : "memory");
}

// The pairing of two CTAs on one product (cta_group::2). One warp of each CTA of
// the pair allocates and frees the same TMEM columns together. The MMA is issued
// by the even CTA alone: M = 256, rows 0-127 of A (and of D) in the even CTA's
// shared memory (TMEM), rows 128-255 in the odd CTA's at the same addresses;
// columns 0 .. N/2 - 1 of B in the even CTA's shared memory, N/2 .. N - 1 in the
// odd CTA's at the same address. The commit arrives on the barrier at the same
// shared address in every CTA of `mask`.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void umma_pair_bf16_warp(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                                    uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void umma_pair_bf16_tmem_a_warp(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void umma_pair_commit_mc_warp(uint32_t bar, uint16_t mask) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;\n\t}" ::"r"(bar),
      "h"(mask)
      : "memory");
}
__device__ __forceinline__ void umma_pair_commit_warp(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar)
      : "memory");
}

// Instruction descriptor for kind::f16 with BF16 A/B and FP32 D.
//   bits 4-5 D format (1 = F32), 7-9 A format (1 = BF16), 10-12 B format (1 = BF16),
//   15 A major (0 = K-major, 1 = MN-major), 16 B major, 17-22 N>>3, 24-28 M>>4.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn_major, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn_major ? 1u : 0u) << 15) |
         ((b_mn_major ? 1u : 0u) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// Shared-memory matrix descriptor, 128-byte swizzle (the layout TMA writes with
// CU_TENSOR_MAP_SWIZZLE_128B into a 1024-byte aligned buffer):
//   bits 0-13 start address >> 4, 16-29 leading byte offset >> 4,
//   32-45 stride byte offset >> 4, 46-48 fixed 0b001, 61-63 swizzle (2 = 128B).
// K-major: rows of 128 bytes (64 BF16 along K), 8-row groups SBO = 1024 bytes
//          apart; LBO unused. Advancing along K inside the 128-byte row is done by
//          adding the byte offset to the start address.
// MN-major: 64 BF16 along M/N per 128-byte row, 8 K-rows per 1024-byte group;
//          LBO = distance between 64-wide M/N blocks, SBO = distance between
//          8-deep K groups.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t smem_addr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((smem_addr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// Byte offset of the 16-byte chunk `c` (0..7) of row `r` inside a 128B-swizzled
// K-major panel (rows of 128 bytes): the chunk index is XORed with r mod 8.
__device__ __forceinline__ uint32_t sw128_offset(uint32_t r, uint32_t c) {
  return r * 128u + ((c ^ (r & 7u)) << 4);
}

// TMEM loads: 32 lanes (one per thread of the warp) x N consecutive 32-bit columns.
// The wait variant ties the destination registers to tcgen05.wait::ld so that no
// use can be scheduled before the data has arrived.
#define PFA_R8(i) "=r"(r[i + 0]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), \
                  "=r"(r[i + 4]), "=r"(r[i + 5]), "=r"(r[i + 6]), "=r"(r[i + 7])
#define PFA_W8(i) "+r"(r[i + 0]), "+r"(r[i + 1]), "+r"(r[i + 2]), "+r"(r[i + 3]), \
                  "+r"(r[i + 4]), "+r"(r[i + 5]), "+r"(r[i + 6]), "+r"(r[i + 7])
#define PFA_S8(i) "r"(r[i + 0]), "r"(r[i + 1]), "r"(r[i + 2]), "r"(r[i + 3]), \
                  "r"(r[i + 4]), "r"(r[i + 5]), "r"(r[i + 6]), "r"(r[i + 7])

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : PFA_R8(0), PFA_R8(8), PFA_R8(16), PFA_R8(24)
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tmem_ld_wait32(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : PFA_W8(0), PFA_W8(8), PFA_W8(16), PFA_W8(24)
               :
               : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      PFA_S8(0), PFA_S8(8), PFA_S8(16), PFA_S8(24)
      : "memory");
}

#define PFA_R64 PFA_R8(0), PFA_R8(8), PFA_R8(16), PFA_R8(24), PFA_R8(32), PFA_R8(40), PFA_R8(48), PFA_R8(56)
#define PFA_W64 PFA_W8(0), PFA_W8(8), PFA_W8(16), PFA_W8(24), PFA_W8(32), PFA_W8(40), PFA_W8(48), PFA_W8(56)

// 32 lanes x 64 consecutive 32-bit columns into r[0..63].
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,"
      "%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
      "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];"
      : PFA_R64
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_ld_wait64(uint32_t* r) {
  asm volatile("tcgen05.wait::ld.sync.aligned;" : PFA_W64 : : "memory");
}

#define PFA_S64 PFA_S8(0), PFA_S8(8), PFA_S8(16), PFA_S8(24), PFA_S8(32), PFA_S8(40), PFA_S8(48), PFA_S8(56)
// r[0..63] into 32 lanes x 64 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_st64(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x64.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,"
      "%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,"
      "%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63,%64};" ::"r"(taddr),
      PFA_S64
      : "memory");
}

// 32 lanes x 16 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : PFA_R8(0), PFA_R8(8)
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_ld_wait16(uint32_t (&r)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;" : PFA_W8(0), PFA_W8(8) : : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      PFA_S8(0), PFA_S8(8)
      : "memory");
}

__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

}  // namespace pfa
