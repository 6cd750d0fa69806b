// Stage 2 of split-K: the fold. out[e] = round(sum_{sigma=0..S-1} slab[sigma][e])
// with the slabs added one after another in slice order, then one
// round-to-nearest-even into the output type ("feat(rocke): split-K forward
// implicit-GEMM convolution on gfx1250", "Two-stage split-K": the reduce
// kernel folds the slabs and casts into D). The bias slabs fold the same way
// in the same launch.
//
// Bandwidth- and latency-bound: the slabs were just written by stage 1 and
// usually sit in L2. Each thread owns 4 consecutive elements (1 when E is
// small or not a multiple of 4) and issues the loads of a batch of B slabs
// (B sized to S, so a small S keeps few registers and a high occupancy)
// before it adds any of them, so every warp keeps a batch of independent
// loads in flight; the adds still happen strictly in slice order.
#include "common.cuh"
#include "../kernel_entry.h"

namespace cig {
namespace {

constexpr int kThreads = 256;

template <int V>
struct Vec;
template <>
struct Vec<1> {
  using T = float;
  static __device__ __forceinline__ T load(const float* p) { return __ldcs(p); }
  static __device__ __forceinline__ void add(T& a, const T& b) { a += b; }
};
template <>
struct Vec<4> {
  using T = float4;
  static __device__ __forceinline__ T load(const float* p) { return __ldcs(reinterpret_cast<const float4*>(p)); }
  static __device__ __forceinline__ void add(T& a, const T& b) {
    a.x += b.x; a.y += b.y; a.z += b.z; a.w += b.w;
  }
};

// Sum of S slabs (stride E floats) at element e, in slice order. Each batch
// of B slabs issues all of its (predicated) loads before its first add, the
// last, partial batch included, so no slab load waits on the previous add.
template <int V, int B>
__device__ __forceinline__ typename Vec<V>::T fold_at(const float* ws, int64_t E, int32_t S, int64_t e) {
  using T = typename Vec<V>::T;
  T acc = Vec<V>::load(ws + e);
  for (int32_t s = 1; s < S; s += B) {
    T v[B];
#pragma unroll
    for (int i = 0; i < B; ++i)
      if (s + i < S) v[i] = Vec<V>::load(ws + (int64_t)(s + i) * E + e);
#pragma unroll
    for (int i = 0; i < B; ++i)
      if (s + i < S) Vec<V>::add(acc, v[i]);
  }
  return acc;
}

template <typename TO>
__device__ __forceinline__ void store_vec(TO* out, int64_t e, float v) { store_out(out + e, v); }
__device__ __forceinline__ void store_vec(float* out, int64_t e, float4 v) {
  *reinterpret_cast<float4*>(out + e) = v;
}
__device__ __forceinline__ void store_vec(__nv_bfloat16* out, int64_t e, float4 v) {
  __nv_bfloat162 h[2] = {__floats2bfloat162_rn(v.x, v.y), __floats2bfloat162_rn(v.z, v.w)};
  *reinterpret_cast<uint2*>(out + e) = *reinterpret_cast<uint2*>(h);
}
__device__ __forceinline__ void store_vec(__half* out, int64_t e, float4 v) {
  __half2 h[2] = {__floats2half2_rn(v.x, v.y), __floats2half2_rn(v.z, v.w)};
  *reinterpret_cast<uint2*>(out + e) = *reinterpret_cast<uint2*>(h);
}

// Units [0, E / V) cover the main slabs, then [0, K) the bias slabs (if any).
template <typename TO, int V, int B>
__global__ void __launch_bounds__(kThreads) fold_kernel(const float* __restrict__ ws, TO* out, int64_t E,
                                                        const float* __restrict__ wsb, TO* db, int64_t K,
                                                        int32_t S) {
  // Launched as a programmatic dependent of stage 1: wait here until stage 1
  // has completed and its slab writes are visible.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int64_t main_units = E / V;
  const int64_t units = main_units + (db ? K : 0);
  const int64_t stride = (int64_t)gridDim.x * kThreads;
  for (int64_t u = (int64_t)blockIdx.x * kThreads + threadIdx.x; u < units; u += stride) {
    if (u < main_units) {
      store_vec(out, u * V, fold_at<V, B>(ws, E, S, u * V));
    } else {
      const int64_t k = u - main_units;
      store_out(db + k, fold_at<1, B>(wsb, K, S, k));
    }
  }
}

// The batch: just above S - 1 (the first slab loads alone) up to 8 (16-byte
// units) or 32 (single floats) slabs, which keeps the registers of a batch
// of float4 loads near 64.
template <typename TO>
cudaError_t launch_b4(const cudaLaunchConfig_t& cfg, const float* ws, TO* out, int64_t E, const float* wsb, TO* db,
                      int64_t K, int32_t S) {
  if (S <= 5) return cudaLaunchKernelEx(&cfg, fold_kernel<TO, 4, 4>, ws, out, E, wsb, db, K, S);
  return cudaLaunchKernelEx(&cfg, fold_kernel<TO, 4, 8>, ws, out, E, wsb, db, K, S);
}
template <typename TO>
cudaError_t launch_b1(const cudaLaunchConfig_t& cfg, const float* ws, TO* out, int64_t E, const float* wsb, TO* db,
                      int64_t K, int32_t S) {
  if (S <= 5) return cudaLaunchKernelEx(&cfg, fold_kernel<TO, 1, 4>, ws, out, E, wsb, db, K, S);
  if (S <= 9) return cudaLaunchKernelEx(&cfg, fold_kernel<TO, 1, 8>, ws, out, E, wsb, db, K, S);
  if (S <= 17) return cudaLaunchKernelEx(&cfg, fold_kernel<TO, 1, 16>, ws, out, E, wsb, db, K, S);
  return cudaLaunchKernelEx(&cfg, fold_kernel<TO, 1, 32>, ws, out, E, wsb, db, K, S);
}

template <typename TO>
cudaError_t launch_typed(const Plan& p, const Args& a) {
  const int64_t E = p.out_elems;
  const int sms = current_sm_count() > 0 ? current_sm_count() : 148;
  TO* out = static_cast<TO*>(a.out);
  TO* db = p.with_bias ? static_cast<TO*>(a.db) : nullptr;
  const int64_t bias_units = p.with_bias ? p.sh.k : 0;
  // 16-byte units (4 elements) when E allows and still gives every SM two
  // CTAs of them, else single floats (more threads, more loads in flight);
  // one thread per unit, up to 8 CTAs per SM resident, a grid-stride loop
  // beyond that.
  const bool vec4 = (E % 4) == 0 && E / 4 >= (int64_t)sms * 2 * kThreads;
  const int grid = launch_grid_cap((vec4 ? E / 4 : E) + bias_units, kThreads, sms, 8);
  // Programmatic dependent launch: the fold may be scheduled as soon as the
  // stage-1 CTAs signal (griddepcontrol.launch_dependents) and then waits in
  // griddepcontrol.wait for stage 1 to finish, hiding its launch latency.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = a.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (vec4) return launch_b4<TO>(cfg, a.ws, out, E, a.ws_bias, db, p.sh.k, p.split);
  return launch_b1<TO>(cfg, a.ws, out, E, a.ws_bias, db, p.sh.k, p.split);
}

}  // namespace

cudaError_t launch_fold(const Plan& p, const Args& a) {
  if (p.sh.out_dt == CONV_F32) return launch_typed<float>(p, a);
  if (p.sh.out_dt == CONV_BF16) return launch_typed<__nv_bfloat16>(p, a);
  return launch_typed<__half>(p, a);
}

}  // namespace cig
