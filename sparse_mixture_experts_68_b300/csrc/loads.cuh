// Loads issued where they stand.  A header of its own, next to common.cuh,
// for the small kernels that reduce batches of loaded values.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace moe {

// Loads issued where they stand.  Where a batch of loads feeds additions that
// are each under a bounds test, the compiler may move each load into its test
// and so wait for them one at a time; a volatile asm load stays in place, so
// the batch is in flight together.  Generic addressing (global or shared).
__device__ __forceinline__ float ld_now(const float* p) {
  float v;
  asm volatile("ld.f32 %0, [%1];" : "=f"(v) : "l"(p) : "memory");
  return v;
}
// Global memory, cached in L2 only (data another kernel has just written).
__device__ __forceinline__ float ld_now_cg(const float* p) {
  float v;
  asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(v) : "l"(p) : "memory");
  return v;
}
// Global memory through the read-only path, 16 bytes.
__device__ __forceinline__ uint4 ld_now_nc_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p)
               : "memory");
  return v;
}

}  // namespace moe
