// Small inline-PTX helpers shared by the library's kernels.
#pragma once
#include <stdint.h>

namespace hpc {

__device__ __forceinline__ float ptx_ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Programmatic dependent launch: wait until the preceding kernel in the
// stream has completed and its memory is visible (a no-op when this kernel
// was launched without the programmatic-serialization attribute).
__device__ __forceinline__ void griddep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
// Let the next kernel in the stream start launching its CTAs.
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

}  // namespace hpc
