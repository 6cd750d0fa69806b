// Epilogue of the tensor-core kernels: a 128-row fp32 accumulator in tensor
// memory goes out through shared memory and TMA tensor stores, optionally
// with a bias + clamp applied to the fp32 values before the one rounding.
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
// [ep_lo, ep_hi] before the rounding. Few instructions per thread: with one
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
        v[i] = fminf(fmaxf(v[i] + b.x, ep_lo), ep_hi);
        v[i + 1] = fminf(fmaxf(v[i + 1] + b.y, ep_lo), ep_hi);
        v[i + 2] = fminf(fmaxf(v[i + 2] + b.z, ep_lo), ep_hi);
        v[i + 3] = fminf(fmaxf(v[i + 3] + b.w, ep_lo), ep_hi);
      }
    }
    uint8_t* row = buf + m * 128;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const uint4 pk = pack16<TE>(v + u * VPU);
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
