// Stage 2 of split-K: the fold. out[e] = round(sum_{sigma=0..S-1} slab[sigma][e])
// with the slabs added one after another in slice order, then one
// round-to-nearest-even into the output type ("feat(rocke): split-K forward
// implicit-GEMM convolution on gfx1250", "Two-stage split-K": the reduce
// kernel folds the slabs and casts into D). The bias slabs fold the same way
// in the same launch.
//
// Bandwidth- and latency-bound: the slabs were just written by stage 1 and
// usually sit in L2. Each thread owns 1 or 4 consecutive elements and issues
// the loads of a batch of slabs (32 or 16) before it adds any of them, so a
// warp keeps a batch of independent 4- or 16-byte loads in flight; the adds
// still happen strictly in slice order.
#include "common.cuh"

namespace cig {
namespace {

constexpr int kThreads = 256;

template <int V>
struct Vec;
template <>
struct Vec<1> {
  using T = float;
  static constexpr int kBatch = 32;  // slabs whose loads are in flight together
  static __device__ __forceinline__ T load(const float* p) { return __ldcs(p); }
  static __device__ __forceinline__ void add(T& a, const T& b) { a += b; }
};
template <>
struct Vec<4> {
  using T = float4;
  static constexpr int kBatch = 16;
  static __device__ __forceinline__ T load(const float* p) { return __ldcs(reinterpret_cast<const float4*>(p)); }
  static __device__ __forceinline__ void add(T& a, const T& b) {
    a.x += b.x; a.y += b.y; a.z += b.z; a.w += b.w;
  }
};

// Sum of S slabs (stride E floats) at element e, in slice order. Each batch
// issues all of its (predicated) loads before its first add, the last,
// partial batch included, so no slab load waits on the previous add.
template <int V>
__device__ __forceinline__ typename Vec<V>::T fold_at(const float* ws, int64_t E, int32_t S, int64_t e) {
  using T = typename Vec<V>::T;
  constexpr int B = Vec<V>::kBatch;
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
template <typename TO>
__device__ __forceinline__ void store_vec(TO* out, int64_t e, float4 v) {
  store_out(out + e + 0, v.x);
  store_out(out + e + 1, v.y);
  store_out(out + e + 2, v.z);
  store_out(out + e + 3, v.w);
}
__device__ __forceinline__ void store_vec(float* out, int64_t e, float4 v) {
  *reinterpret_cast<float4*>(out + e) = v;
}

// Units [0, E / V) cover the main slabs, then [0, K) the bias slabs (if any).
template <typename TO, int V>
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
      store_vec(out, u * V, fold_at<V>(ws, E, S, u * V));
    } else {
      const int64_t k = u - main_units;
      store_out(db + k, fold_at<1>(wsb, K, S, k));
    }
  }
}

template <typename TO>
cudaError_t launch_typed(const Plan& p, const Args& a) {
  const int64_t E = p.out_elems;
  const int sms = current_sm_count();
  const int cap = (sms > 0 ? sms : 148) * 16;
  TO* out = static_cast<TO*>(a.out);
  TO* db = p.with_bias ? static_cast<TO*>(a.db) : nullptr;
  const int64_t bias_units = p.with_bias ? p.sh.k : 0;
  // 16-byte units when they still give every SM several CTAs; else one float
  // per thread for more loads in flight.
  const bool vec4 = (E % 4) == 0 && (E / 4) >= (int64_t)(sms > 0 ? sms : 148) * kThreads * 4;
  const int grid = launch_grid_cap((vec4 ? E / 4 : E) + bias_units, kThreads, cap / 8 > 0 ? cap / 8 : 1, 8);
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
  const float* ws = a.ws;
  const float* wsb = a.ws_bias;
  const int64_t K = p.sh.k;
  const int32_t S = p.split;
  if (vec4) return cudaLaunchKernelEx(&cfg, fold_kernel<TO, 4>, ws, out, E, wsb, db, K, S);
  return cudaLaunchKernelEx(&cfg, fold_kernel<TO, 1>, ws, out, E, wsb, db, K, S);
}

}  // namespace

cudaError_t launch_fold(const Plan& p, const Args& a) {
  if (p.sh.out_dt == CONV_F32) return launch_typed<float>(p, a);
  if (p.sh.out_dt == CONV_BF16) return launch_typed<__nv_bfloat16>(p, a);
  return launch_typed<__half>(p, a);
}

}  // namespace cig
