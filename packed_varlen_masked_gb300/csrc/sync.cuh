// Shared-memory barriers and bounded waits for the library's kernels
// (mbarrier phases completed by thread arrivals and by the byte counts of
// bulk asynchronous copies).  Every wait a kernel makes is bounded in time:
// on expiry it records PK_ERR_TIMEOUT in the caller's status word and raises
// a CTA-local abort flag, so the kernel can drain and return instead of
// spinning forever.
#pragma once
#include <cstdint>

#include "pk.h"

namespace pk {
namespace dev {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
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
// try_wait that may suspend the thread for up to `ns` nanoseconds while the
// phase is incomplete (it resumes as soon as the phase completes).
__device__ __forceinline__ bool mbar_try_wait_hint(uint32_t bar, uint32_t parity, uint32_t ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(ns)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

struct WaitCtl {
  volatile int* abort_flag;  // CTA-local, shared memory
  int32_t* status;           // device status word, may be null
  uint64_t limit_ns;
};

// Bound of the drain waits on the abort path.  A drain waits for copies and
// MMAs the CTA has already issued (to validated addresses), which always
// complete, so its bound is fixed and generous: the user's wait limit, which
// may be set to a few nanoseconds to force the abort path, does not apply.
constexpr uint64_t kDrainLimitNs = 5000000000ull;

// Slow path of a bounded wait: poll until the phase completes, the CTA has
// aborted, or the time limit passes (then record the timeout and abort).
// Inlined: an out-of-line call inside the softmax loop constrains its
// register allocation, which measured about 1% slower.
static __device__ __forceinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity, WaitCtl c,
                                            bool honour_abort) {
  const uint64_t t0 = globaltimer_ns();
  const uint64_t limit = honour_abort ? c.limit_ns : kDrainLimitNs;
  for (uint32_t n = 1;; ++n) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((n & 15u) == 0) {
      if (honour_abort && *c.abort_flag) return false;
      if (globaltimer_ns() - t0 > limit) {
        *c.abort_flag = 1;
        if (c.status) atomicCAS(c.status, 0, (int32_t)PK_ERR_TIMEOUT);
        return false;
      }
    }
  }
}
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, const WaitCtl& c) {
  if (mbar_try_wait(bar, parity)) return true;
  return mbar_wait_slow(bar, parity, c, true);
}
// Drain wait, used on the abort path and for the MMA issuers' final commit:
// ignores the abort flag, bounded by kDrainLimitNs.
__device__ __forceinline__ bool mbar_wait_drain(uint32_t bar, uint32_t parity, const WaitCtl& c) {
  if (mbar_try_wait(bar, parity)) return true;
  return mbar_wait_slow(bar, parity, c, false);
}

// Drain wait on a ring barrier of a head-pair cluster (two CTAs filling and
// emptying each other's ring stages).  After an abort the other CTA may
// never send its half of a stage or read it, so the awaited phase may never
// complete; what can still be in flight (this CTA's own copies, the other
// CTA's last commit arrivals) lands within microseconds.  So the wait is
// bounded by kDrainLimitNs, or, once the CTA has aborted, by
// kClusterAbortDrainNs from its start.
constexpr uint64_t kClusterAbortDrainNs = 2000000ull;
__device__ __forceinline__ bool mbar_wait_cluster_drain(uint32_t bar, uint32_t parity,
                                                        const WaitCtl& c) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t n = 1;; ++n) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((n & 15u) == 0) {
      const uint64_t dt = globaltimer_ns() - t0;
      const bool aborted = *c.abort_flag != 0;
      if (aborted && dt > kClusterAbortDrainNs) return false;
      if (dt > kDrainLimitNs) {
        *c.abort_flag = 1;
        if (c.status) atomicCAS(c.status, 0, (int32_t)PK_ERR_TIMEOUT);
        return false;
      }
    }
  }
}

// Bounded wait for a waiter with nothing else to do (the epilogue warps
// between units): each try suspends the thread for up to 2 us, so the
// waiting warps take no issue slots from the softmax warps on the same SM
// sub-partitions.
__device__ __forceinline__ bool mbar_wait_sleep(uint32_t bar, uint32_t parity, const WaitCtl& c) {
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (mbar_try_wait_hint(bar, parity, 2000u)) return true;
    if (*c.abort_flag) return false;
    if (globaltimer_ns() - t0 > c.limit_ns) {
      *c.abort_flag = 1;
      if (c.status) atomicCAS(c.status, 0, (int32_t)PK_ERR_TIMEOUT);
      return false;
    }
  }
}

}  // namespace dev
}  // namespace pk
