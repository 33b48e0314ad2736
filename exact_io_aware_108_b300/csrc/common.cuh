// common.cuh -- device-side helpers shared by the attention kernels:
// the device error flag and bounded mbarrier waits.
#pragma once
#include "ptx.cuh"

namespace fa {

// A pipeline wait that takes longer than this is a bug; the kernel gives up.
// g_fa_wait_limit_ns holds the limit the kernels use (the host may lower it,
// fa_set_wait_limit_ns); waits that drain copies already in flight after an
// abort always allow kWaitLimitNs, so those copies land before the CTA exits.
constexpr uint64_t kWaitLimitNs = 2000000000ull;
__device__ unsigned long long g_fa_wait_limit_ns = kWaitLimitNs;

// Nonzero: the TMA producer of every attention kernel issues no loads, so
// each CTA's first pipeline wait can only end by running out of time. Set by
// fa_debug_starve_pipelines to exercise the time limit, the abort flag and
// the device error word; zero in normal operation.
__device__ unsigned int g_fa_starve_pipelines = 0;
__device__ __forceinline__ bool pipelines_starved() {
  return *static_cast<volatile unsigned int *>(&g_fa_starve_pipelines) != 0u;
}

// Bits of the device error word.
//   kDevErrTimeout    a pipeline wait ran out of time
//   kDevErrSmemAlign  the dynamic shared-memory base was not 1 KB aligned
//                     (the kernel returned before doing any work)
//   kDevErrRange      a bf16 input value that the backward converts to fp16
//                     was beyond fp16's largest finite value, 65504
enum : uint32_t { kDevErrTimeout = 1u, kDevErrSmemAlign = 2u, kDevErrRange = 4u };

// Device error word, read and cleared by fa_get_device_error(). Kernels and
// the host code that reads it live in one translation unit (fa_lib.cu).
__device__ unsigned int g_fa_device_error = 0;

// Slow path of a wait: poll until the phase completes, the CTA-wide abort
// flag is raised by another role, or the time limit passes (then raise the
// abort flag and the device error word). honor_abort = false is used when
// draining copies in flight after an abort. Inlined: a real call would be
// shared by warpgroups that run under different setmaxnreg register limits.
__device__ __forceinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity,
                                            volatile uint32_t *abort_flag, bool honor_abort) {
  const uint64_t t0 = globaltimer_ns();
  const uint64_t limit =
      honor_abort ? *static_cast<volatile unsigned long long *>(&g_fa_wait_limit_ns) : kWaitLimitNs;
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 127u) == 0) {
      if (honor_abort && *abort_flag) return false;
      if (globaltimer_ns() - t0 > limit) {
        *abort_flag = 1u;
        atomicOr(&g_fa_device_error, kDevErrTimeout);
        return false;
      }
    }
  }
}

// Wait for the phase of `bar` with parity `parity`; false on abort/timeout.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity,
                                          volatile uint32_t *abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  return mbar_wait_slow(bar, parity, abort_flag, true);
}

// Same, called by all 32 lanes of a warp; the result is warp-uniform so the
// warp stays converged for the .sync.aligned tcgen05 instructions after it.
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity,
                                               volatile uint32_t *abort_flag) {
  const bool ok = mbar_wait(bar, parity, abort_flag);
  return __all_sync(0xffffffffu, ok);
}

// Wait for a work-item hand-over between the roles of a persistent kernel:
// bounded like a drain (it ignores the abort flag), so that after a stop the
// roles still walk the remaining items together (writing zeros for them);
// false only when the hand-over itself ran out of time.
__device__ __forceinline__ bool mbar_wait_handoff(uint32_t bar, uint32_t parity,
                                                  volatile uint32_t *abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  return mbar_wait_slow(bar, parity, abort_flag, false);
}

// Bounded wait that ignores the abort flag (used to drain in-flight copies).
__device__ __forceinline__ void mbar_wait_drain(uint32_t bar, uint32_t parity,
                                                volatile uint32_t *abort_flag) {
  if (!mbar_try_wait(bar, parity)) mbar_wait_slow(bar, parity, abort_flag, false);
}

__device__ __forceinline__ uint32_t align_up_1024(uint32_t a) { return (a + 1023u) & ~1023u; }

}  // namespace fa
