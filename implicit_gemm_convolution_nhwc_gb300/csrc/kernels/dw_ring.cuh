// Pieces shared by the depthwise kernels that stream input rows through a
// shared-memory ring (dw_wgrad_ring.cu, dw_fwd_ring.cu).
//
// A CTA walks a run of consecutive (n, ho) output rows. Output row (n, ho)
// reads input rows ho - ph .. ho - ph + F - 1 of image n (unit H stride and
// dilation); consecutive rows of one image share F - 1 of them, so the run's
// input rows form one sequence (a new image starts F fresh rows), and input
// row k of the sequence lives in ring slot k mod RX.
#pragma once

#include "tc_common.cuh"

namespace cig {
namespace dwring {

// Ring depth d = ahead + slack, in steps of tr output rows. The steps from
// S - slack to S + ahead cover m = (d + 1) tr - 1 row advances, each +1 input
// row or +F at an image start (at most ceil(m / Ho) of those); an input-row
// ring of this many slots holds what they read, so loading step S + ahead
// only reuses slots of rows that steps before S - slack read.
inline int64_t ring_rows(int64_t F, int64_t Ho, int64_t d, int64_t tr) {
  const int64_t m = (d + 1) * tr - 1;
  return m + F + (F - 1) * ((m + Ho - 1) / Ho);
}

// An output row's place: the ring slot of the first input row it reads, and
// its (image, output row). Advanced one row at a time, so no loop divides.
// P has fields Ho (output rows an image) and RX (input-row slots).
struct RowPos {
  int32_t xs;
  int32_t ho, n;
  bool first;  // the run's first row: all F input rows are new
  __device__ __forceinline__ int fresh(int F) const { return first || ho == 0 ? F : 1; }
  template <typename P>
  __device__ __forceinline__ int32_t slot(int r, const P& p) const {
    return xs + r >= p.RX ? xs + r - p.RX : xs + r;
  }
  template <typename P>
  __device__ __forceinline__ void advance(int F, const P& p) {
    const bool cross = ++ho == p.Ho;
    if (cross) {
      ho = 0;
      ++n;
    }
    xs += cross ? F : 1;
    if (xs >= p.RX) xs -= p.RX;
    first = false;
  }
};

// A step's slot in the step ring and its wrap count (the slot's mbarrier
// phase parity is the wrap count & 1). P has field RS (step slots).
struct StepPos {
  int32_t ss;
  uint32_t sw;
  template <typename P>
  __device__ __forceinline__ void advance(const P& p) {
    if (++ss == p.RS) {
      ss = 0;
      ++sw;
    }
  }
};

// A 16-bit pair from shared memory (32-bit shared address), widened to fp32.
template <typename T>
__device__ __forceinline__ float2 lds2(uint32_t a);
template <>
__device__ __forceinline__ float2 lds2<__nv_bfloat16>(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(a));
  return make_float2(__uint_as_float(__byte_perm(v, 0u, 0x1044u)), __uint_as_float(v & 0xffff0000u));
}
template <>
__device__ __forceinline__ float2 lds2<__half>(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(a));
  __half2 h;
  memcpy(&h, &v, sizeof(h));
  return __half22float2(h);
}

}  // namespace dwring
}  // namespace cig
