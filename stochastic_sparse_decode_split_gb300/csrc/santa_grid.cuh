// santa_grid.cuh -- the grid-wide barrier of the single-launch kernels
// (sm_103a, cooperative launch: every CTA is resident).
#pragma once

#include "santa_common.cuh"

namespace santa {

constexpr unsigned long long GRID_WAIT_NS = 2000000000ull;

// ---------------------------------------------------------------------------
// Grid-wide barrier (all CTAs are resident: cooperative launch).  Two
// arrival counters and a generation word in the workspace: a launch uses
// counter (generation & 1), which every CTA increments once without waiting;
// a CTA that needs the others spins until it reaches the grid size.  The
// launch's first CTA clears the other counter for the next launch and, once
// all have arrived, advances the generation.  Waits are bounded; on expiry
// ERR_TIMEOUT is flagged and the CTA proceeds.
// ---------------------------------------------------------------------------
__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release(unsigned* p, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void red_release_add(unsigned* p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// Waiting for every CTA's arrival: thread 0 spins until the counter reaches
// n (bounded), then the CTA proceeds together.
__device__ __forceinline__ void arrivals_wait(const unsigned* count, unsigned n, int* err,
                                             unsigned long long limit_ns = GRID_WAIT_NS) {
  if (threadIdx.x == 0) {
    const unsigned long long t0 = global_ns();
    while (ld_acquire(count) < n) {
      if (global_ns() - t0 > limit_ns) {
        flag_error(err, ERR_TIMEOUT);
        break;
      }
    }
  }
  __syncthreads();
}
// Waiting half: thread 0 spins until the generation moves past g (bounded),
// then the CTA proceeds together.
__device__ __forceinline__ void grid_wait(const unsigned* gen, unsigned g, int* err,
                                          unsigned long long limit_ns = GRID_WAIT_NS) {
  if (threadIdx.x == 0) {
    const unsigned long long t0 = global_ns();
    while (ld_acquire(gen) == g) {
      if (global_ns() - t0 > limit_ns) {
        flag_error(err, ERR_TIMEOUT);
        break;
      }
      __nanosleep(32);
    }
    __threadfence();
  }
  __syncthreads();
}

}  // namespace santa
