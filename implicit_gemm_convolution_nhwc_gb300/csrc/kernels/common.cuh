// Device helpers shared by the kernels: element loads/stores in the three
// storage types, and a few PTX wrappers.
#pragma once

#include <cstdint>

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "../conv_internal.h"

namespace cig {

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }
__device__ __forceinline__ float to_f32(__half v) { return __half2float(v); }

// Round-to-nearest-even store of an fp32 value into the output type.
__device__ __forceinline__ void store_out(float* p, float v) { *p = v; }
__device__ __forceinline__ void store_out(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }
__device__ __forceinline__ void store_out(__half* p, float v) { *p = __float2half_rn(v); }

// Store of one result element: into slab `sigma` of the workspace when the
// reduction is split, else straight into the output with the final rounding.
template <typename TO>
__device__ __forceinline__ void store_result(TO* out, float* ws, int64_t E, int32_t sigma, int64_t e,
                                             float v) {
  if (ws) {
    ws[(int64_t)sigma * E + e] = v;
  } else {
    store_out(out + e, v);
  }
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte global->shared copy that bypasses L1; src_bytes = 0 zero-fills.
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_u32(smem)), "l"(gmem),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// This CTA's main work is done: the fold, launched as a programmatic
// dependent, may be scheduled (it still waits for this grid to complete).
__device__ __forceinline__ void signal_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

inline int launch_grid_cap(int64_t units, int threads, int sms, int per_sm) {
  int64_t blocks = (units + threads - 1) / threads;
  const int64_t cap = (int64_t)sms * per_sm;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return (int)blocks;
}

}  // namespace cig
