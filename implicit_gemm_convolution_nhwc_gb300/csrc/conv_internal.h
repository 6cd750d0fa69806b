// Internal host/device declarations shared by the C-ABI layer and the kernels.
#pragma once

#include <cstdint>

#include <cuda_runtime.h>

#include "conv_igemm.h"

namespace cig {

// A validated problem with its derived extents.
struct Shape {
  int64_t n, h, w, c, k, r, s;
  int64_t sh, sw, ph, pw, dh, dw, groups;
  int64_t ho, wo, cg, kg;
  int in_dt, out_dt;
  __host__ __device__ int64_t P() const { return n * ho * wo; }  // wgrad reduction rows
  __host__ __device__ int64_t D() const { return r * s * cg; }  // forward reduction depth
  __host__ __device__ int64_t x_elems() const { return n * h * w * c; }
  __host__ __device__ int64_t w_elems() const { return k * r * s * cg; }
  __host__ __device__ int64_t y_elems() const { return n * ho * wo * k; }
};

// What a kernel needs the planner to know about it.
struct Geometry {
  bool ok = false;           // the kernel takes this problem
  int64_t tiles = 0;         // output tiles (CTAs per slice)
  int64_t blocks = 0;        // reduction blocks a slice is made of
  int ctas_per_sm = 1;       // resident CTAs per SM (sets the auto target)
  int32_t max_split = 0;     // largest degree the kernel takes (0: any up to `blocks`)
};

// Largest thread-block cluster (non-portable size) the single-launch
// split-K forward forms from the S slices of a tile.
constexpr int kMaxClusterSplit = 16;

struct Plan {
  Shape sh;
  conv_dir dir;
  conv_kernel kernel;
  Geometry geo;
  int32_t split;             // S
  bool with_bias;
  int64_t out_elems;         // E: elements of Y or dW
  uint64_t slab_bytes;       // S*E*4 rounded to 256 (0 when S == 1)
  uint64_t bias_slab_bytes;  // S*K*4 rounded to 256 (0 when S == 1 or no bias)
  bool fold;                 // stage 2 runs (S > 1 and the slices do not fold in-launch)
  bool epilogue;             // a non-identity fused forward epilogue (then S == 1)
  uint64_t aux_bytes;        // kernel-private bytes at the start of ws (the data gradient's filter)
  uint64_t ws_bytes() const { return aux_bytes + slab_bytes + bias_slab_bytes; }
};

struct Args {
  const void* x;   // X, or dY (data gradient)
  const void* b;   // W (forward, data gradient) or dY (weight gradient)
  void* out;       // Y, dW or dX
  void* aux;       // the first aux_bytes of ws (nullptr when none)
  void* db;        // bias gradient or nullptr
  float* ws;       // slabs [S][E] (nullptr when S == 1)
  float* ws_bias;  // bias slabs [S][K] (nullptr when S == 1 or no bias)
  // Fused forward epilogue (S == 1 only): out = min(max(acc + ep_bias[k], ep_lo), ep_hi).
  const void* ep_bias = nullptr;  // [K] in the output type, or nullptr
  float ep_lo = 0.f, ep_hi = 0.f;
  bool ep = false;
  // Depthwise forward kernels: read filter tap R*S - 1 - t for tap t (the
  // filter turned by 180 degrees; the data gradient as a forward).
  bool rev_taps = false;
  cudaStream_t stream;
};

// Reduction slice sigma of S over `blocks` blocks: [begin, end), balanced,
// never empty when S <= blocks.
__host__ __device__ inline int64_t slice_begin(int64_t blocks, int64_t S, int64_t sigma) {
  return (blocks * sigma) / S;
}

// The kernels' geometries and launchers are declared in kernel_entry.h.

// SM count of the current device (cached per device), or -1.
int current_sm_count();

}  // namespace cig
