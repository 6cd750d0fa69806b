// Stage 2 of split-K: the fold. out[e] = round(sum_{sigma=0..S-1} slab[sigma][e])
// with the slabs added one after another in slice order, then one
// round-to-nearest-even into the output type ("feat(rocke): split-K forward
// implicit-GEMM convolution on gfx1250", "Two-stage split-K": the reduce
// kernel folds the slabs and casts into D). The bias slabs fold the same way
// in the same launch. Bandwidth-bound: every slab byte is read once with
// 16-byte streaming loads, four slabs in flight per step.
#include "common.cuh"

namespace cig {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ float4 ldcs4(const float* p) { return __ldcs(reinterpret_cast<const float4*>(p)); }

template <typename TO>
__device__ __forceinline__ void store4(TO* out, int64_t e, float4 v) {
  store_out(out + e + 0, v.x);
  store_out(out + e + 1, v.y);
  store_out(out + e + 2, v.z);
  store_out(out + e + 3, v.w);
}
template <>
__device__ __forceinline__ void store4<float>(float* out, int64_t e, float4 v) {
  *reinterpret_cast<float4*>(out + e) = v;
}

// Sum of S slabs at element e (vector of 4), in slice order.
__device__ __forceinline__ float4 fold4(const float* ws, int64_t E, int32_t S, int64_t e) {
  float4 acc = ldcs4(ws + e);
  int32_t s = 1;
  for (; s + 4 <= S; s += 4) {
    const float4 a = ldcs4(ws + (int64_t)(s + 0) * E + e);
    const float4 b = ldcs4(ws + (int64_t)(s + 1) * E + e);
    const float4 c = ldcs4(ws + (int64_t)(s + 2) * E + e);
    const float4 d = ldcs4(ws + (int64_t)(s + 3) * E + e);
    acc.x += a.x; acc.y += a.y; acc.z += a.z; acc.w += a.w;
    acc.x += b.x; acc.y += b.y; acc.z += b.z; acc.w += b.w;
    acc.x += c.x; acc.y += c.y; acc.z += c.z; acc.w += c.w;
    acc.x += d.x; acc.y += d.y; acc.z += d.z; acc.w += d.w;
  }
  for (; s < S; ++s) {
    const float4 a = ldcs4(ws + (int64_t)s * E + e);
    acc.x += a.x; acc.y += a.y; acc.z += a.z; acc.w += a.w;
  }
  return acc;
}

__device__ __forceinline__ float fold1(const float* ws, int64_t E, int32_t S, int64_t e) {
  float acc = __ldcs(ws + e);
  for (int32_t s = 1; s < S; ++s) acc += __ldcs(ws + (int64_t)s * E + e);
  return acc;
}

// Elements [0, E) of the main slabs, then [0, K) of the bias slabs (if any).
// vec4: E is a multiple of 4 (the main region runs 4 elements per unit).
template <typename TO, bool kVec4>
__global__ void __launch_bounds__(kThreads) fold_kernel(const float* __restrict__ ws, TO* out, int64_t E,
                                                        const float* __restrict__ wsb, TO* db, int64_t K,
                                                        int32_t S) {
  const int64_t main_units = kVec4 ? E / 4 : E;
  const int64_t units = main_units + (db ? K : 0);
  const int64_t stride = (int64_t)gridDim.x * kThreads;
  for (int64_t u = (int64_t)blockIdx.x * kThreads + threadIdx.x; u < units; u += stride) {
    if (u < main_units) {
      if (kVec4) {
        store4(out, u * 4, fold4(ws, E, S, u * 4));
      } else {
        store_out(out + u, fold1(ws, E, S, u));
      }
    } else {
      const int64_t k = u - main_units;
      store_out(db + k, fold1(wsb, K, S, k));
    }
  }
}

template <typename TO>
cudaError_t launch_typed(const Plan& p, const Args& a) {
  const int64_t E = p.out_elems;
  const bool vec4 = (E % 4) == 0;
  const int64_t units = (vec4 ? E / 4 : E) + (p.with_bias ? p.sh.k : 0);
  const int sms = current_sm_count();
  const int grid = launch_grid_cap(units, kThreads, sms > 0 ? sms : 148, 8);
  TO* out = static_cast<TO*>(a.out);
  TO* db = p.with_bias ? static_cast<TO*>(a.db) : nullptr;
  if (vec4)
    fold_kernel<TO, true><<<grid, kThreads, 0, a.stream>>>(a.ws, out, E, a.ws_bias, db, p.sh.k, p.split);
  else
    fold_kernel<TO, false><<<grid, kThreads, 0, a.stream>>>(a.ws, out, E, a.ws_bias, db, p.sh.k, p.split);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fold(const Plan& p, const Args& a) {
  if (p.sh.out_dt == CONV_F32) return launch_typed<float>(p, a);
  if (p.sh.out_dt == CONV_BF16) return launch_typed<__nv_bfloat16>(p, a);
  return launch_typed<__half>(p, a);
}

}  // namespace cig
