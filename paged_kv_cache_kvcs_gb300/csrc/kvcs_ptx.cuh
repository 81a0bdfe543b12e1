// kvcs_ptx.cuh -- thin inline-PTX wrappers for sm_103a: mbarriers, the bulk
// (TMA, non-tensor) global->shared copy, L2 cache policies and the global
// timer.  Hand-written; no library headers beyond the CUDA runtime.
#pragma once

#include <cstdint>

namespace kvcs {
namespace ptx {

typedef unsigned long long u64;
typedef unsigned int u32;

__device__ __forceinline__ u32 smem_addr(const void *p) {
  return static_cast<u32>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(u32 bar, u32 count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count)
               : "memory");
}

// Make barrier initialisation visible to the async (bulk-copy) proxy.
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(u32 bar) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar)
      : "memory");
}

// Arrive and add `tx` bytes to the phase's expected transaction count.
__device__ __forceinline__ void mbar_arrive_expect_tx(u32 bar, u32 tx) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(bar),
      "r"(tx)
      : "memory");
}

// One probe of phase `parity`; the hardware may suspend the thread briefly.
__device__ __forceinline__ bool mbar_try_wait(u32 bar, u32 parity) {
  u32 ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ u64 globaltimer_ns() {
  u64 t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait for phase `parity` of barrier `bar`: gives up (returns false)
// after `limit_ns` of wall time or 2^26 probes, whichever comes first, so a
// lost arrival can never hang the GPU.
__device__ __forceinline__ bool mbar_wait_bounded(u32 bar, u32 parity,
                                                  u64 limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const u64 t0 = globaltimer_ns();
  for (u32 i = 0; i < (1u << 26); ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 15u) == 15u && globaltimer_ns() - t0 > limit_ns) return false;
  }
  return false;
}

// 8-byte asynchronous copy from global to shared memory (both addresses
// 8-byte aligned); it completes in the background like a bulk copy.
__device__ __forceinline__ void cp_async8(u32 dst, const void *src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst), "l"(src) : "memory");
}

// One arrival on `bar` once every cp.async this thread issued before has
// completed (the barrier's pending count is raised first, so the current
// phase waits for that arrival too).
__device__ __forceinline__ void cp_async_mbar_arrive(u32 bar) {
  asm volatile("cp.async.mbarrier.arrive.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

// Programmatic dependent launch.  grid_dep_launch lets the next kernel of
// the stream (launched with programmatic stream serialization) start before
// this one ends; grid_dep_wait makes the calling thread wait until the grids
// it depends on have finished and their writes are visible (at once when the
// kernel was launched without such a dependency).
__device__ __forceinline__ void grid_dep_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void grid_dep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// L2 policy for data read exactly once.
__device__ __forceinline__ u64 policy_evict_first() {
  u64 pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;"
               : "=l"(pol));
  return pol;
}

// Bulk copy of `bytes` (multiple of 16; both addresses 16-byte aligned) from
// global memory into this CTA's shared memory; completion is signalled on
// `bar` as transaction bytes.
__device__ __forceinline__ void bulk_g2s(u32 dst, const void *src, u32 bytes,
                                         u32 bar, u64 policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::"
      "cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

}  // namespace ptx
}  // namespace kvcs
