// bounded_wait.cuh -- device waits that give up: a wait that runs out records
// MOE_ERR_TIMEOUT and the kernel id in the workspace error word and raises a
// CTA-local abort flag, so that the other roles of the CTA stop waiting too
// and the kernel returns with the context intact.  (mbarrier waits:
// ptx::mbar_wait in tc_ptx.cuh.)
#pragma once

#include <cstdint>

#include "moe_kernels.cuh"
#include "tc_ptx.cuh"

namespace moe {

// where (> 0): which wait of the kernel ran out, recorded as bit `where` of
// err[2]; a wait that ended because the CTA was already winding down (its
// abort flag set) adds no bit.  err[3]: the CTA that recorded the timeout.
__device__ __forceinline__ void raise_timeout(int32_t* err, volatile int* abort_flag, int kern, int where = 0) {
  if (where > 0 && !*abort_flag) atomicOr(err + 2, 1 << where);
  if (atomicCAS(err, 0, kErrTimeout) == 0) {
    atomicExch(err + 1, kern);
    atomicExch(err + 3, static_cast<int32_t>(blockIdx.x));
  }
  *abort_flag = 1;
}

__device__ __forceinline__ int ld_acquire(const int32_t* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release(int32_t* p, int v) {
  asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Bounded wait of one warp for a flag another CTA sets (non-zero); the result
// is warp-uniform.  Gives up after timeout_ns or once *abort_flag is set.
__device__ __forceinline__ bool wait_flag(const int32_t* flag, const volatile int* abort_flag, uint64_t timeout_ns) {
  bool ok = true;
  if ((threadIdx.x & 31) == 0) {
    const uint64_t t0 = ptx::globaltimer_ns();
    while (ld_acquire(flag) == 0) {
      if (*abort_flag || ptx::globaltimer_ns() - t0 > timeout_ns) {
        ok = false;
        break;
      }
      __nanosleep(64);
    }
  }
  ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
  if (ok) (void)ld_acquire(flag);  // every lane acquires before reading what the flag guards
  return ok;
}

}  // namespace moe
