// Helpers shared by the forward scans (head dims 64 and 128): 3-input max / min and the barrier
// of the 256 softmax threads (named barrier 1).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace pathattn {

// 3-input max/min.
__device__ __forceinline__ float max3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
__device__ __forceinline__ float min3(float a, float b, float c) {
  float r;
  asm("min.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Barrier 1 over the softmax threads; returns whether q held for any of them.
__device__ __forceinline__ bool softmax_any(bool q) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred pq, pr;\n\t"
      "setp.ne.u32 pq, %1, 0;\n\t"
      "bar.red.or.pred pr, 1, 256, pq;\n\t"
      "selp.u32 %0, 1, 0, pr;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)q)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void softmax_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

}  // namespace pathattn
