// Inline-PTX wrappers for the barriers and bulk memory operations the sampler uses on
// sm_103a: mbarriers (local and remote arrive, cluster-scope acquire), the 1-D TMA bulk
// copy global -> shared (optionally with an L2 eviction policy) and the TMA bulk
// prefetch into L2.  Every wait is bounded.
#pragma once

#include <cstdint>

namespace clsample {

// Polls of an mbarrier before a wait gives up (each try_wait may itself suspend the
// thread for a short, hardware-defined time).
constexpr uint32_t kSpinLimit = 1u << 22;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(unsigned long long* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

// Makes mbarrier initialisations visible to the async proxy and to the cluster.
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(unsigned long long* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_local(unsigned long long* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Arrive, with release semantics at cluster scope, on the mbarrier at the same shared
// offset in CTA `rank` of this cluster.
__device__ __forceinline__ void mbar_arrive_remote(unsigned long long* bar, uint32_t rank) {
  asm volatile(
      "{\n\t.reg .b32 ra;\n\t"
      "mapa.shared::cluster.u32 ra, %0, %1;\n\t"
      "mbarrier.arrive.release.cluster.shared::cluster.b64 _, [ra];\n\t}" ::"r"(smem_addr(bar)),
      "r"(rank)
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(unsigned long long* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ bool mbar_try_wait_cluster(unsigned long long* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// One poll that may suspend the thread for up to kSuspendNs before it reports the
// phase as incomplete, so a waiting warp does not take issue slots from the others.
constexpr uint32_t kSuspendNs = 20000;
constexpr uint32_t kSleepLimit = 1u << 16;  // suspending polls before a wait gives up
__device__ __forceinline__ bool mbar_try_wait_sleep(unsigned long long* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity), "r"(kSuspendNs)
      : "memory");
  return ok != 0;
}

// Bounded waits: false when the phase did not complete within kSpinLimit polls.
__device__ __forceinline__ bool mbar_wait(unsigned long long* bar, uint32_t parity) {
  for (uint32_t i = 0; i < kSpinLimit; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}
// Bounded wait by suspending polls (at most kSleepLimit of them, about a second).
__device__ __forceinline__ bool mbar_wait_sleep(unsigned long long* bar, uint32_t parity) {
  for (uint32_t i = 0; i < kSleepLimit; ++i)
    if (mbar_try_wait_sleep(bar, parity)) return true;
  return false;
}
__device__ __forceinline__ bool mbar_wait_cluster(unsigned long long* bar, uint32_t parity) {
  for (uint32_t i = 0; i < kSpinLimit; ++i)
    if (mbar_try_wait_cluster(bar, parity)) return true;
  return false;
}

// 1-D bulk copy (TMA) of `bytes` from global memory into this CTA's shared memory,
// completing on `bar` (complete_tx).  Both addresses 16-byte aligned, bytes a multiple
// of 16.
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes,
                                              unsigned long long* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// The same copy with an L2 eviction policy (from make_policy_evict_first or
// make_policy_evict_normal) for the lines it brings into L2.
__device__ __forceinline__ void bulk_copy_g2s_hint(void* dst, const void* src, uint32_t bytes,
                                                   unsigned long long* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
      "%4;" ::"r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// L2 policies: lines a stream reads once go first when L2 needs room; normal lines stay
// as long as the usual replacement keeps them.
__device__ __forceinline__ uint64_t make_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t make_policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Asks the TMA unit to bring `bytes` of global memory into L2 (no completion signal;
// later loads of those lines hit L2 or join the fetch in flight).  The address must be
// 16-byte aligned and bytes a multiple of 16.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

}  // namespace clsample
