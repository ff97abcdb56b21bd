// pdl.cuh -- device side of programmatic dependent launch.
//
// Convention of this library: a kernel executes pdl_wait() before
// pdl_launch_dependents().  So when a kernel starts, its predecessor may still
// be running, but the kernel before that one has completed: a kernel may read
// its grandparent's outputs (e.g. the routing tables) before its own
// pdl_wait(), and must wait before reading its parent's outputs.
#pragma once

namespace moe {

// Let the next kernel in the stream be scheduled now (its CTAs wait in
// pdl_wait until this grid has completed and its writes are visible).
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Wait until the previous grid in the stream has completed and its memory
// operations are visible.  A no-op when the kernel was launched without a
// programmatic dependency.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

}  // namespace moe
