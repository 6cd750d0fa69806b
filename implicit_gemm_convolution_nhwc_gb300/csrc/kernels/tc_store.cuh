// Epilogue of the tensor-core kernels: a 128-row fp32 accumulator in tensor
// memory goes out through shared memory and TMA tensor stores, optionally
// with a bias added to the fp32 values and the result clamped.
#pragma once

#include <cstring>

#include "tc_common.cuh"

namespace cig {

// 16 bytes of TE from 4 (fp32) or 8 (16-bit) values, rounded to nearest even.
template <typename TE>
__device__ __forceinline__ uint4 pack16(const float* v);
template <>
__device__ __forceinline__ uint4 pack16<float>(const float* v) {
  return make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]), __float_as_uint(v[2]), __float_as_uint(v[3]));
}
template <>
__device__ __forceinline__ uint4 pack16<__nv_bfloat16>(const float* v) {
  uint4 r;
  __nv_bfloat162 h[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
  memcpy(&r, h, 16);
  return r;
}
template <>
__device__ __forceinline__ uint4 pack16<__half>(const float* v) {
  uint4 r;
  __half2 h[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) h[i] = __floats2half2_rn(v[2 * i], v[2 * i + 1]);
  memcpy(&r, h, 16);
  return r;
}

// Packed 16-bit values clamped to [lo, hi] (packed the same way); a NaN
// becomes lo, as with fminf(fmaxf(x, lo), hi).
template <typename TE>
__device__ __forceinline__ uint4 clamp16(uint4 x, uint4 lo, uint4 hi);
template <>
__device__ __forceinline__ uint4 clamp16<__nv_bfloat16>(uint4 x, uint4 lo, uint4 hi) {
  __nv_bfloat162 v[4], l[4], h[4];
  memcpy(v, &x, 16);
  memcpy(l, &lo, 16);
  memcpy(h, &hi, 16);
#pragma unroll
  for (int i = 0; i < 4; ++i) v[i] = __hmin2(__hmax2(v[i], l[i]), h[i]);
  memcpy(&x, v, 16);
  return x;
}
template <>
__device__ __forceinline__ uint4 clamp16<__half>(uint4 x, uint4 lo, uint4 hi) {
  __half2 v[4], l[4], h[4];
  memcpy(v, &x, 16);
  memcpy(l, &lo, 16);
  memcpy(h, &hi, 16);
#pragma unroll
  for (int i = 0; i < 4; ++i) v[i] = __hmin2(__hmax2(v[i], l[i]), h[i]);
  memcpy(&x, v, 16);
  return x;
}
template <>
__device__ __forceinline__ uint4 clamp16<float>(uint4 x, uint4, uint4) { return x; }

// The 128 epilogue threads (named barrier 1) store the accumulator columns
// [0, ncols) of their rows: thread m owns tensor-memory lane m (trow already
// carries the warp's lane offset). For each 128-byte column chunk (32 fp32 or
// 64 16-bit values) the thread writes its 128 bytes into a 128B-swizzled
// staging buffer (8 conflict-free 16-byte stores; NBUF 16 KB buffers at
// `stage`, in turn), and the leader thread stores the chunk as one TMA
// box through store(buf, x), where x = x0 + chunk * (values per chunk) is the
// innermost coordinate; the tensor map clips the box at the tensor's bounds.
// Only chunks that start below x_end are stored (each then commits exactly
// one bulk group, which the buffer-reuse wait counts on). With ep, the bias
// (fp32 in shared memory, one per column) is added and the value clamped to
// [ep_lo, ep_hi] (fp32 outputs before the rounding, 16-bit ones after it).
// Few instructions per thread: with one
// CTA per SM these four warps issue every one of them. With two buffers a
// chunk waited for the store of the chunk before last to finish reading its
// buffer (the 128 KB fp32 partial tile of a split-K CTA took ~2.5 us); more
// buffers keep more stores in flight. Several groups of four warps may share
// the columns: group g takes chunks g, g + c_step, ... through its own
// buffers, leader and named barrier bar_id. With tmem_release, the leader
// arrives on that barrier once every thread of the group has read its last
// accumulator column (the accumulator may then be overwritten while the
// stores still run); with wait_global false the call returns once the
// stores have read the staging buffers, not once they reached global memory.
template <typename TE, int NBUF = 2, typename StoreFn>
__device__ __forceinline__ void store_rows_tma(uint32_t trow, uint8_t* stage, int ncols, int32_t x0, int32_t x_end,
                                               int m, bool have_acc, bool leader, bool do_store, StoreFn store,
                                               const float* ep_bias = nullptr, float ep_lo = 0.f, float ep_hi = 0.f,
                                               bool ep = false, int c_first = 0, int c_step = 1,
                                               uint32_t bar_id = 1, uint64_t* tmem_release = nullptr,
                                               bool wait_global = true) {
  constexpr int CW = 128 / (int)sizeof(TE);  // values per 128-byte chunk
  constexpr int VPU = 16 / (int)sizeof(TE);  // values per 16-byte unit
  const int nch = min(ncols / CW, (x_end - x0 + CW - 1) / CW);
  // 16-bit outputs are clamped after the rounding, with packed min/max
  // against the rounded bounds: the same values, as rounding to nearest is
  // monotone (and a NaN still becomes ep_lo).
  constexpr bool k16 = sizeof(TE) == 2;
  uint4 lo16 = {}, hi16 = {};
  if (k16 && ep) {
    const float lo8[8] = {ep_lo, ep_lo, ep_lo, ep_lo, ep_lo, ep_lo, ep_lo, ep_lo};
    const float hi8[8] = {ep_hi, ep_hi, ep_hi, ep_hi, ep_hi, ep_hi, ep_hi, ep_hi};
    lo16 = pack16<TE>(lo8);
    hi16 = pack16<TE>(hi8);
  }
  int i = 0;  // this group's chunk count
  if (tmem_release && c_first >= nch && leader) mbar_arrive(tmem_release);  // no chunk for this group
#pragma unroll 1
  for (int c = c_first; c < nch; c += c_step, ++i) {
    uint8_t* buf = stage + (i % NBUF) * (128 * 128);
    if (i >= NBUF) {  // the store that last read this buffer (this group's chunk i - NBUF) must be done reading
      if (leader) bulk_wait_read<NBUF - 1>();
      named_bar_sync(bar_id, 128);
    }
    float v[CW];
#pragma unroll
    for (int h = 0; h < CW / 32; ++h) {
      if (have_acc) {
        tmem_ld32(trow + (uint32_t)(c * CW + 32 * h), v + 32 * h);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[32 * h + i] = 0.f;
      }
    }
    if (ep) {
      const float4* b4 = reinterpret_cast<const float4*>(ep_bias + c * CW);
#pragma unroll
      for (int i = 0; i < CW; i += 4) {
        const float4 b = b4[i / 4];
        const float2 lo = __fadd2_rn(make_float2(v[i], v[i + 1]), make_float2(b.x, b.y));
        const float2 hi = __fadd2_rn(make_float2(v[i + 2], v[i + 3]), make_float2(b.z, b.w));
        v[i] = lo.x;
        v[i + 1] = lo.y;
        v[i + 2] = hi.x;
        v[i + 3] = hi.y;
        if (!k16) {
          v[i] = fminf(fmaxf(v[i], ep_lo), ep_hi);
          v[i + 1] = fminf(fmaxf(v[i + 1], ep_lo), ep_hi);
          v[i + 2] = fminf(fmaxf(v[i + 2], ep_lo), ep_hi);
          v[i + 3] = fminf(fmaxf(v[i + 3], ep_lo), ep_hi);
        }
      }
    }
    uint8_t* row = buf + m * 128;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      uint4 pk = pack16<TE>(v + u * VPU);
      if (k16 && ep) pk = clamp16<TE>(pk, lo16, hi16);
      st_shared_v4(row + ((u ^ (m & 7)) << 4), pk.x, pk.y, pk.z, pk.w);
    }
    fence_proxy_async_smem();
    const bool last = c + c_step >= nch;
    if (tmem_release && last) tc_fence_before();
    named_bar_sync(bar_id, 128);
    if (leader && tmem_release && last) mbar_arrive(tmem_release);
    if (leader && do_store) {
      store(buf, x0 + c * CW);
      bulk_commit();
    }
  }
  if (leader) {
    if (wait_global) bulk_wait<0>();
    else bulk_wait_read<0>();
  }
  named_bar_sync(bar_id, 128);  // the staging buffers are free again for a next call
}

// TMA tensor store of a 4-D box from shared memory (clipped at the tensor's
// bounds), tracked by the issuing thread's bulk groups.
__device__ __forceinline__ void tma_store_4d(const CUtensorMap* map, const void* src, int32_t c0, int32_t c1,
                                             int32_t c2, int32_t c3) {
  asm volatile("cp.async.bulk.tensor.4d.global.shared::cta.bulk_group [%0, {%2, %3, %4, %5}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(smem_u32(src)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
               : "memory");
}

}  // namespace cig
