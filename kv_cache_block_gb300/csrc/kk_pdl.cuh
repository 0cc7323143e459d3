// Programmatic dependent launch for the chained decode-step kernels.
#pragma once

namespace kk {

// A kernel launched with programmatic stream serialisation may start while
// the kernel before it in the stream is still running; it waits here, before
// its first access to global memory, until that kernel has finished and its
// writes are visible (no wait when there is no such kernel). Signalling early
// lets the next kernel of the stream be launched in the meantime, so the
// launch latency of a chain of small kernels overlaps their execution.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

}  // namespace kk
