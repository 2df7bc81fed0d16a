// tma.cuh -- 1-D bulk copies (cp.async.bulk, the TMA engine) into shared
// memory and the mbarrier operations that track them, with bounded waits.
//
// Every wait gives up after kWaitLimitNs of %globaltimer time and returns
// false; callers then record ECHO_ERR_TIMEOUT in the status word, wait once
// more (also bounded) so that copies in flight land before the block exits,
// and return.
#pragma once

#include <stdint.h>

namespace echo {

constexpr uint64_t kWaitLimitNs = 1000ull * 1000ull * 1000ull;  // 1 s

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(bar), "r"(count) : "memory");
}

// Makes barrier initialisation visible to the async proxy (the TMA engine).
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Orders this thread's earlier generic-proxy shared-memory accesses before
// later async-proxy (bulk copy) accesses to the same memory.
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
               :: "r"(bar), "r"(bytes) : "memory");
}

// Global -> shared bulk copy completing on `bar`.  dst, src 16-byte aligned,
// bytes a multiple of 16.  `policy` is an L2 cache policy (createpolicy).
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;"
      :: "r"(dst), "l"(src), "r"(bytes), "r"(bar), "l"(policy) : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}

#ifndef ECHO_CODES_EVICT_LAST
#define ECHO_CODES_EVICT_LAST 1
#endif
// Codes written by one kernel for the next are stored with L2 evict_last.
constexpr bool kCodesPolicyLast = ECHO_CODES_EVICT_LAST != 0;

__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done) : "r"(bar), "r"(parity) : "memory");
  return done != 0;
}

// Wait for phase `parity` of the barrier, giving up after kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_ns() - t0 > kWaitLimitNs) return false;
  }
  return true;
}

// Bounded wait whose outcome is the same for the whole warp: every lane waits
// (bounded) and the lanes then agree by vote, so that if any lane gave up,
// all of them take the give-up path together.
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity) {
  return __all_sync(0xFFFFFFFFu, mbar_wait_bounded(bar, parity)) != 0;
}

// The same for the whole block (contains a __syncthreads: every thread of the
// block must call it).
__device__ __forceinline__ bool mbar_wait_block(uint32_t bar, uint32_t parity) {
  return __syncthreads_and(mbar_wait_bounded(bar, parity) ? 1 : 0) != 0;
}

// Global stores with an L2 cache policy (createpolicy): the codes written by
// one kernel and read by the next are kept in L2 with evict_last.
__device__ __forceinline__ void st_hint_u32(void* p, uint32_t v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.b32 [%0], %1, %2;" :: "l"(p), "r"(v), "l"(pol) : "memory");
}
__device__ __forceinline__ void st_hint_u64(void* p, uint64_t v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.b64 [%0], %1, %2;" :: "l"(p), "l"(v), "l"(pol) : "memory");
}

}  // namespace echo
