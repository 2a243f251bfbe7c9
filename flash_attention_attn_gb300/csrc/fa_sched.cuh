// fa_sched.cuh -- dynamic work distribution of the persistent kernels.
//
// A persistent kernel launches at most one CTA per SM.  Work units are
// numbered longest first; CTA c starts with unit c and then takes the next
// unclaimed unit from a counter in the workspace (atomicAdd), so that SMs
// that run faster take more units, as the hardware block scheduler would.
// Inside the CTA the producer warp claims the units and hands each one to
// the MMA warp and the compute warps through a small ring of shared-memory
// slots guarded by mbarriers; a unit index >= the unit count ends the loop.
//
// The counter pair {next, done} must be zero when a kernel starts.  The
// workspace is zero-filled before its first use, and every launch leaves the
// pair at zero again: each CTA counts itself out in `done` as it exits, and
// the last one (by then every CTA has made its final claim) resets both.
#pragma once

#include <stdint.h>

#include "sm103_ptx.cuh"

namespace fa {

struct SchedCounter {
  unsigned int next;  // units claimed past the first gridDim.x
  unsigned int done;  // CTAs that have finished
};

constexpr int kSchedSlots = 4;

struct SchedRing {
  uint64_t full[kSchedSlots];   // slot written by the producer (1 arrival)
  uint64_t empty[kSchedSlots];  // slot read by every consumer warp
  int unit[kSchedSlots];
};

__device__ __forceinline__ void sched_init(SchedRing* r, uint32_t consumer_warps) {
  for (int i = 0; i < kSchedSlots; ++i) {
    ptx::mbar_init(&r->full[i], 1);
    ptx::mbar_init(&r->empty[i], consumer_warps);
  }
}

// Producer, lane 0: the unit after the CTA's first, claimed from the counter.
__device__ __forceinline__ int sched_claim(SchedCounter* c) {
  return static_cast<int>(gridDim.x + atomicAdd(&c->next, 1u));
}

// Producer warp (converged): publish unit u in sequence slot i.  Returns
// false if the wait for the slot gave up.
__device__ __forceinline__ bool sched_publish(SchedRing* r, int i, int u, const ptx::Ctl& ctl, unsigned code) {
  const int slot = i % kSchedSlots;
  if (i >= kSchedSlots && !ptx::warp_wait(&r->empty[slot], ((i / kSchedSlots) - 1) & 1, ctl, code)) return false;
  if ((threadIdx.x & 31) == 0) {
    *reinterpret_cast<volatile int*>(&r->unit[slot]) = u;
    ptx::mbar_arrive(&r->full[slot]);
  }
  __syncwarp();
  return true;
}

// Consumer warp (converged): the unit in sequence slot i, or -1 if the wait
// gave up.  The warp releases the slot as soon as it has read it.
__device__ __forceinline__ int sched_next(SchedRing* r, int i, const ptx::Ctl& ctl, unsigned code) {
  const int slot = i % kSchedSlots;
  if (!ptx::warp_wait(&r->full[slot], (i / kSchedSlots) & 1, ctl, code)) return -1;
  const int u = *reinterpret_cast<volatile int*>(&r->unit[slot]);
  ptx::warp_arrive(&r->empty[slot]);
  return u;
}

// One thread per CTA, after every role has finished: count the CTA out; the
// last CTA resets the counter pair for the next launch.
__device__ __forceinline__ void sched_exit(SchedCounter* c) {
  __threadfence();
  if (atomicAdd(&c->done, 1u) == gridDim.x - 1) {
    atomicExch(&c->next, 0u);
    atomicExch(&c->done, 0u);
  }
}

}  // namespace fa
