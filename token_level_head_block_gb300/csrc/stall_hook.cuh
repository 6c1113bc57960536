// Diagnostic hook for the timeout path of the bounded waits (the host call is
// mhla_debug_stall_waits).  When set, every bounded mbarrier wait made by one
// chosen warp index that does not find its phase complete at the first poll
// behaves as if its barrier never completed: it polls no more, gives up after
// a short limit (or as soon as another role of its CTA
// has given up), raises the CTA's abort flag and sets bit 0 of its file's
// error word -- the same exit a wait on a lost completion takes.  The other
// roles then stop, copies already in flight drain through the separate drain
// waits, tensor memory is released and the kernel returns.  Nothing faults,
// traps or hangs: it only makes the rarely taken exit testable.  Off (zero) by
// default; one copy per translation unit, all set together by the host call.
// The waits look at it only after a first poll has failed, so it costs the
// pipelines nothing while their barriers are ready (a check before every first
// poll was measured at 2.7 us on the DiT-S/2 forward).
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "ptx.cuh"

namespace mhla {

static __constant__ uint32_t c_stall_warp = 0;   // warp index + 1 whose waits stall; 0: none
static __constant__ uint64_t c_stall_ns = 0;     // how long a stalled wait lasts

static __device__ __forceinline__ bool stall_this_warp() {
  return c_stall_warp != 0u && (threadIdx.x >> 5) + 1u == c_stall_warp;
}

// The stalled wait itself: no barrier is polled; returns after c_stall_ns or
// when the CTA's abort flag rises (bounded in time and in iterations).
static __device__ __noinline__ void stalled_wait(volatile uint32_t* abort_flag) {
  const uint64_t t0 = ptx::globaltimer();
  for (uint32_t it = 0; it < (1u << 28); ++it) {
    if ((it & 63u) == 0) {
      if (*abort_flag) return;
      if (ptx::globaltimer() - t0 > c_stall_ns) return;
    }
  }
}

// Host side: this translation unit's copy of the setting.
static inline int set_stall_hook(uint32_t warp_plus_1, uint64_t ns) {
  if (cudaMemcpyToSymbol(c_stall_warp, &warp_plus_1, sizeof(warp_plus_1)) != cudaSuccess) return 4;
  if (cudaMemcpyToSymbol(c_stall_ns, &ns, sizeof(ns)) != cudaSuccess) return 4;
  return 0;
}

}  // namespace mhla

// Defines, in a translation unit with bounded waits, the function the host
// call uses to set that unit's copy.
#define MHLA_DEFINE_STALL_SETTER(fn) \
  int fn(uint32_t warp_plus_1, uint64_t ns) { return set_stall_hook(warp_plus_1, ns); }
