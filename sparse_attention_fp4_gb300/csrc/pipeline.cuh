// Bounded waits shared by the warp-specialised logits kernels (logits_mxf4.cu,
// logits_fp8.cu).  Every wait gives up after ctl.timeout_ns: it then raises the CTA's
// abort flag and records FP4IDX_ERR_TIMEOUT in the caller's status word, and the kernel
// winds down in order (in-flight copies land, tensor memory is freed) instead of hanging.
#pragma once

#include <stdint.h>

#include "fp4idx_internal.cuh"
#include "ptx.cuh"

namespace fp4idx {
namespace pipe {

constexpr unsigned kFull = 0xFFFFFFFFu;
constexpr uint32_t kSuspendNs = 20000;  // upper bound of one suspended probe

struct Ctl {
  volatile int32_t* abort;  // the CTA's abort flag (shared memory)
  int32_t* status;          // the caller's status word (nullable)
  uint64_t timeout_ns;      // how long one wait may last
};

__device__ __forceinline__ bool give_up(const Ctl& c) {
  *c.abort = 1;
  record_error(c.status, FP4IDX_ERR_TIMEOUT);
  return false;
}

// Bounded poll of an mbarrier phase by the calling thread.  False on timeout (which
// raises the abort flag) or, when honor_abort, once another warp has aborted.  A waiting
// thread stays suspended between probes (up to kSuspendNs each) instead of spinning, so
// that waiters leave their scheduler's issue slots to the working warps.
__device__ __forceinline__ bool poll(uint32_t bar, uint32_t parity, const Ctl& c, bool honor_abort) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (ptx::mbar_try_wait_sleep(bar, parity, kSuspendNs)) return true;
    if ((it & 7u) == 0) {
      if (honor_abort && *c.abort) return false;
      if (ptx::globaltimer() - t0 > c.timeout_ns) return give_up(c);
    }
  }
}

// Bounded wait, by one thread, until the shared-memory counter at `a` has reached
// need_a and the one at `b` need_b (wrap-safe comparisons); both loads are issued before
// either is tested.  Pass b = a, need_b = need_a to wait on one counter.
__device__ __forceinline__ bool wait_counts(uint32_t a, uint32_t need_a, uint32_t b, uint32_t need_b, const Ctl& c) {
  auto ready = [&]() {
    const uint32_t va = ptx::smem_ld_acquire(a), vb = ptx::smem_ld_acquire(b);
    return (int32_t)(va - need_a) >= 0 && (int32_t)(vb - need_b) >= 0;
  };
  if (ready()) return true;
  const uint64_t t0 = ptx::globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (ready()) return true;
    if ((it & 63u) == 0) {
      if (*c.abort) return false;
      if (ptx::globaltimer() - t0 > c.timeout_ns) return give_up(c);
    }
  }
}

// Every lane polls (the lanes then read what the barrier guards); uniform result.
__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity, const Ctl& c, bool honor_abort = true) {
  const bool ok = poll(bar, parity, c, honor_abort);
  return __all_sync(kFull, ok);
}

// Lane 0 polls for a warp whose work after the wait is issued by lane 0 alone.
__device__ __forceinline__ bool wait_lane0(uint32_t bar, uint32_t parity, const Ctl& c, bool honor_abort = true) {
  int ok = 1;
  if ((threadIdx.x & 31) == 0) ok = poll(bar, parity, c, honor_abort) ? 1 : 0;
  return __shfl_sync(kFull, ok, 0) != 0;
}

__device__ __forceinline__ void prefetch_l2(const void* a) { asm volatile("prefetch.global.L2 [%0];" ::"l"(a)); }

}  // namespace pipe
}  // namespace fp4idx
