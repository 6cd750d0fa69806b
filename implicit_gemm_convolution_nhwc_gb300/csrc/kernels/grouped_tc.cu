// Grouped 16-bit forward on the tensor cores, as block-diagonal dense blocks.
//
// With Cg = Kg input and output channels per group and 128 a multiple of Cg,
// output channels [k0, k0 + 128) read exactly input channels [k0, k0 + 128).
// So each 128-channel block is a dense forward convolution of that channel
// slice of X with the filter W_bd[k][r][s][c'] = W[k][r][s][c' mod Cg] when
// c' and k mod 128 fall in the same group, else 0 (written into the first
// bytes of the workspace). The forward tensor-core kernel runs it with the X
// channel coordinate offset by the tile's first output channel, 128-wide
// tiles and the reduction (r, s, 128 channels); split-K, fold and the fused
// epilogue are the forward's. The MMAs do 128 / Cg times the useful work
// (16 for 8 channels per group), which the tensor pipe still does faster than
// the FP32 pipe does the useful part.
#include "common.cuh"
#include "../kernel_entry.h"

namespace cig {
namespace {

constexpr int kBlock = 128;  // channels of a dense block

// W [K][R][S][Cg] -> W_bd [K][R][S][128]; one thread writes 8 consecutive
// channels c' of one (k, tap) with a 16-byte store.
template <typename T>
__global__ void __launch_bounds__(256) expand_filter_kernel(const T* __restrict__ w, T* __restrict__ wbd, int64_t K,
                                                            int64_t taps, int64_t Cg) {
  const int64_t u = (int64_t)blockIdx.x * 256 + threadIdx.x;  // unit of 8 channels
  const int64_t units = K * taps * (kBlock / 8);
  if (u >= units) return;
  const int64_t c8 = (u % (kBlock / 8)) * 8;
  const int64_t kt = u / (kBlock / 8);  // k * taps + tap
  const int64_t k = kt / taps;
  const int64_t g_lo = ((k % kBlock) / Cg) * Cg;  // first c' of k's group within the block
  __align__(16) T v[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int64_t c = c8 + j;
    v[j] = c >= g_lo && c < g_lo + Cg ? w[kt * Cg + (c - g_lo)] : T(0.f);
  }
  *reinterpret_cast<uint4*>(wbd + kt * kBlock + c8) = *reinterpret_cast<const uint4*>(v);
}

// The data gradient's block-diagonal filter (see launch_dgrad_grouped_tc):
// W [C][R][S][Cg] (k rows) -> W'_bd [C][R][S][128] with
// W'_bd[c][t'][k'] = W[kb + k'][taps - 1 - t'][c mod Cg] when k' and c mod 128
// fall in the same group (kb = the block's first channel), else 0; one thread
// writes 8 consecutive k' of one (c, t').
template <typename T>
__global__ void __launch_bounds__(256) expand_filter_dgrad_kernel(const T* __restrict__ w, T* __restrict__ wbd,
                                                                  int64_t C, int64_t taps, int64_t Cg) {
  const int64_t u = (int64_t)blockIdx.x * 256 + threadIdx.x;  // unit of 8 channels
  const int64_t units = C * taps * (kBlock / 8);
  if (u >= units) return;
  const int64_t k8 = (u % (kBlock / 8)) * 8;
  const int64_t ct = u / (kBlock / 8);  // c * taps + t'
  const int64_t c = ct / taps, tp = ct % taps;
  const int64_t kb = (c / kBlock) * kBlock;
  const int64_t g_lo = ((c % kBlock) / Cg) * Cg;  // first k' of c's group within the block
  __align__(16) T v[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int64_t kk = k8 + j;
    v[j] = kk >= g_lo && kk < g_lo + Cg ? w[((kb + kk) * taps + (taps - 1 - tp)) * Cg + (c % Cg)] : T(0.f);
  }
  *reinterpret_cast<uint4*>(wbd + ct * kBlock + k8) = *reinterpret_cast<const uint4*>(v);
}

// The dense channel-block problem the forward kernel runs.
Shape block_shape(const Shape& s) {
  Shape b = s;
  b.groups = 1;
  b.cg = kBlock;
  b.kg = s.k;
  return b;
}

}  // namespace

Geometry geometry_fwd_grouped_tc(const Shape& s) {
  if (s.in_dt == CONV_F32 || s.groups < 2 || s.cg != s.kg) return Geometry{};
  if (s.cg < 2 || kBlock % s.cg != 0 || s.c % kBlock != 0) return Geometry{};  // whole groups per block
  return geometry_fwd_tc_block(block_shape(s));
}

cudaError_t launch_fwd_grouped_tc(const Plan& p, const Args& a) {
  const Shape& s = p.sh;
  if (!a.aux) return cudaErrorInvalidValue;
  const int64_t units = s.k * s.r * s.s * (kBlock / 8);
  const int64_t grid = (units + 255) / 256;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  if (s.in_dt == CONV_BF16)
    expand_filter_kernel<__nv_bfloat16><<<(unsigned)grid, 256, 0, a.stream>>>(
        static_cast<const __nv_bfloat16*>(a.b), static_cast<__nv_bfloat16*>(a.aux), s.k, s.r * s.s, s.cg);
  else
    expand_filter_kernel<__half><<<(unsigned)grid, 256, 0, a.stream>>>(
        static_cast<const __half*>(a.b), static_cast<__half*>(a.aux), s.k, s.r * s.s, s.cg);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  Plan bp = p;
  bp.sh = block_shape(s);
  bp.kernel = CONV_KERNEL_FWD_TC;
  bp.geo = geometry_fwd_tc_block(bp.sh);
  Args ba = a;
  ba.b = a.aux;  // W_bd
  ba.aux = nullptr;
  return launch_fwd_tc_block(bp, ba);
}

}  // namespace cig

namespace cig {

// Grouped 16-bit data gradient at stride 1 (Cg = Kg dividing 128, C % 128 =
// 0): the forward problem of dgrad_as_forward_grouped (dY as the input,
// padding dil * (f - 1) - pad) is grouped the same way, so it runs as the
// block-diagonal grouped forward above with the turned filter
// W'_bd[c][r'][s'][k'] = W[kb + k'][R-1-r'][S-1-s'][c mod Cg] in the group
// blocks (written into the workspace), the dY channel coordinate offset by
// the tile's first output channel.
Geometry geometry_dgrad_grouped_tc(const Shape& s) {
  if (s.sh != 1 || s.sw != 1 || s.groups < 2) return Geometry{};
  if (s.ph > s.dh * (s.r - 1) || s.pw > s.dw * (s.s - 1)) return Geometry{};
  return geometry_fwd_grouped_tc(dgrad_as_forward_grouped(s));
}

cudaError_t launch_dgrad_grouped_tc(const Plan& p, const Args& a) {
  const Shape t = dgrad_as_forward_grouped(p.sh);
  if (!a.aux) return cudaErrorInvalidValue;
  const int64_t units = t.k * t.r * t.s * (kBlock / 8);
  const int64_t grid = (units + 255) / 256;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  if (t.in_dt == CONV_BF16)
    expand_filter_dgrad_kernel<__nv_bfloat16><<<(unsigned)grid, 256, 0, a.stream>>>(
        static_cast<const __nv_bfloat16*>(a.b), static_cast<__nv_bfloat16*>(a.aux), t.k, t.r * t.s, t.cg);
  else
    expand_filter_dgrad_kernel<__half><<<(unsigned)grid, 256, 0, a.stream>>>(
        static_cast<const __half*>(a.b), static_cast<__half*>(a.aux), t.k, t.r * t.s, t.cg);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  Plan bp = p;
  bp.sh = block_shape(t);
  bp.dir = CONV_DIR_FWD;
  bp.kernel = CONV_KERNEL_FWD_TC;
  bp.geo = geometry_fwd_tc_block(bp.sh);
  Args ba = a;
  ba.b = a.aux;  // W'_bd
  ba.aux = nullptr;
  return launch_fwd_tc_block(bp, ba);
}

}  // namespace cig
