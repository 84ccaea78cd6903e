// Time-bounded mbarrier waits shared by the kernels.  A wait that runs past
// its limit records bit 0 in the device error word, raises the CTA's abort
// flag so the other roles leave their loops too, and returns false: no
// kernel of this library can hang on a barrier.
#pragma once

#include <cstdint>

#include "ptx.cuh"

namespace w4a16 {

struct WaitCtx {
  uint32_t* err;          // device error word (global)
  uint64_t timeout_ns;    // limit of one wait
  int* abort_flag;        // shared-memory flag of this CTA
};

static __device__ __forceinline__ void wait_record_timeout(const WaitCtx& w) {
  *reinterpret_cast<volatile int*>(w.abort_flag) = 1;
  atomicOr(w.err, 1u);
}

// Single-thread wait.  false = gave up (timeout, or another role gave up).
static __device__ __noinline__ bool wait_one_slow(uint64_t* bar, uint32_t parity, const WaitCtx& w) {
  const uint64_t t0 = ptx::globaltimer_ns();
  for (uint32_t spin = 1;; ++spin) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if ((spin & 31) == 0) {
      if (*reinterpret_cast<volatile int*>(w.abort_flag)) return false;
      if (ptx::globaltimer_ns() - t0 > w.timeout_ns) {
        wait_record_timeout(w);
        return false;
      }
    }
  }
}

// Warp-uniform wait: every lane observes the phase; the give-up decision is
// lane 0's and is shared, so the warp stays converged for .sync.aligned ops.
static __device__ __noinline__ bool wait_warp_slow(uint64_t* bar, uint32_t parity, const WaitCtx& w) {
  const int lane = threadIdx.x & 31;
  uint64_t t0 = 0;
  for (uint32_t spin = 0;; ++spin) {
    const bool ok = ptx::mbar_try_wait(bar, parity);
    if (__all_sync(0xffffffffu, ok)) return true;
    if ((spin & 31) == 31) {
      int give_up = 0;
      if (lane == 0) {
        const uint64_t now = ptx::globaltimer_ns();
        if (t0 == 0) t0 = now;
        if (*reinterpret_cast<volatile int*>(w.abort_flag)) {
          give_up = 1;
        } else if (now - t0 > w.timeout_ns) {
          wait_record_timeout(w);
          give_up = 1;
        }
      }
      give_up = __shfl_sync(0xffffffffu, give_up, 0);
      if (give_up) return false;
    }
  }
}

static __device__ __forceinline__ bool wait_one(uint64_t* bar, uint32_t parity, const WaitCtx& w) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  return wait_one_slow(bar, parity, w);
}

static __device__ __forceinline__ bool wait_warp(uint64_t* bar, uint32_t parity, const WaitCtx& w) {
  if (__all_sync(0xffffffffu, ptx::mbar_try_wait(bar, parity))) return true;
  return wait_warp_slow(bar, parity, w);
}

}  // namespace w4a16
