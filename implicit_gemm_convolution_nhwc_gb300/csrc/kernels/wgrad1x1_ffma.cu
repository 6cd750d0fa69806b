// fp32 1x1 weight gradient (+ bias gradient) on FFMA tiles.
//
// A 1x1, stride-1, unpadded weight gradient is the GEMM dW = dY^T X over the
// [N*H*W, C] / [N*H*W, K] views (the F.linear form of "ROCm/rocm-libraries
// PR #11188", "Motivation" and "Test Plan"); db = column sums of dY. The
// reduction (rows p = N*H*W) is cut into S slices; each CTA reduces one
// slice of one 64 x BC output tile and writes an fp32 partial slab
// ("feat(rocke): split-K forward implicit-GEMM convolution on gfx1250",
// "Two-stage split-K").
//
// CTA: 256 threads as 16 (k) x 16 (c) threads, each owning 4 k x BC/16 c
// accumulators. Rows stream global -> shared in 32-row stages through a
// 4-deep cp.async ring (16-byte copies, zero-filled past the slice end or the
// channel edge). A thread's c columns are 2*tc + 32*j (j < BC/32) so each
// warp's shared loads of a row are contiguous. The bias is summed from the
// dY stage already in shared memory (k = tid % 64, 8 rows per thread).
#include "common.cuh"
#include "../kernel_entry.h"

namespace cig {
namespace {

constexpr int kThreads = 256;
constexpr int kBK = 64;       // k rows of a tile
constexpr int kBP = 32;       // reduction rows per stage (= one reduction block)
constexpr int kStages = 4;

template <int BC>
struct Smem {
  float dy[kStages][kBP][kBK];
  float x[kStages][kBP][BC];
  float bias[4][kBK];
};

template <int BC>
__global__ void __launch_bounds__(kThreads, 2)
    wgrad1x1_ffma_kernel(const float* __restrict__ x, const float* __restrict__ dy, float* __restrict__ out,
                         float* __restrict__ ws, float* __restrict__ db, float* __restrict__ ws_bias, int64_t P,
                         int64_t K, int64_t C, int64_t tiles_c, int64_t tiles, int32_t S, int64_t blocks) {
  constexpr int NJ = BC / 32;  // float2 column pairs per thread
  extern __shared__ __align__(16) unsigned char smem_raw[];
  Smem<BC>& sm = *reinterpret_cast<Smem<BC>*>(smem_raw);

  const int tid = threadIdx.x;
  const int64_t tile = blockIdx.x % tiles;
  const int32_t sigma = (int32_t)(blockIdx.x / tiles);
  const int64_t k0 = (tile / tiles_c) * kBK;
  const int64_t c0 = (tile % tiles_c) * BC;
  const int64_t b0 = slice_begin(blocks, S, sigma), b1 = slice_begin(blocks, S, sigma + 1);
  const int64_t p_begin = b0 * kBP;
  int64_t p_end = b1 * kBP;
  if (p_end > P) p_end = P;
  const int nblk = (int)(b1 - b0);

  // Loader: stage `it` = rows p_begin + it*32 .. +31.
  auto load_stage = [&](int it) {
    const int slot = it % kStages;
    const int64_t pr = p_begin + (int64_t)it * kBP;
    // dY: 32 rows x 16 chunks of 4 floats
#pragma unroll
    for (int i = 0; i < (kBP * kBK / 4) / kThreads; ++i) {
      const int chunk = tid + i * kThreads;
      const int row = chunk / (kBK / 4), col = (chunk % (kBK / 4)) * 4;
      const int64_t p = pr + row, k = k0 + col;
      const bool ok = p < p_end && k < K;
      cp_async16(&sm.dy[slot][row][col], ok ? (const void*)(dy + p * K + k) : (const void*)dy, ok ? 16u : 0u);
    }
    // X: 32 rows x BC/4 chunks
#pragma unroll
    for (int i = 0; i < (kBP * BC / 4 + kThreads - 1) / kThreads; ++i) {
      const int chunk = tid + i * kThreads;
      if (chunk < kBP * BC / 4) {
        const int row = chunk / (BC / 4), col = (chunk % (BC / 4)) * 4;
        const int64_t p = pr + row, c = c0 + col;
        const bool ok = p < p_end && c < C;
        cp_async16(&sm.x[slot][row][col], ok ? (const void*)(x + p * C + c) : (const void*)x, ok ? 16u : 0u);
      }
    }
  };

  const int tk = tid / 16, tc = tid % 16;
  float acc[4][2 * NJ];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 2 * NJ; ++j) acc[i][j] = 0.f;
  float bacc = 0.f;
  const int bk = tid % kBK, brow = (tid / kBK) * 8;

#pragma unroll
  for (int it = 0; it < kStages - 1; ++it) {
    if (it < nblk) load_stage(it);
    cp_async_commit();
  }
  for (int it = 0; it < nblk; ++it) {
    cp_async_wait<kStages - 2>();
    __syncthreads();
    if (it + kStages - 1 < nblk) load_stage(it + kStages - 1);
    cp_async_commit();
    const int slot = it % kStages;
    const float* dys = &sm.dy[slot][0][tk * 4];
    const float* xs = &sm.x[slot][0][2 * tc];
#pragma unroll 8
    for (int row = 0; row < kBP; ++row) {
      const float4 a = *reinterpret_cast<const float4*>(dys + row * kBK);
      float2 b[NJ];
#pragma unroll
      for (int j = 0; j < NJ; ++j) b[j] = *reinterpret_cast<const float2*>(xs + row * BC + 32 * j);
      const float av[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
          acc[i][2 * j] = fmaf(av[i], b[j].x, acc[i][2 * j]);
          acc[i][2 * j + 1] = fmaf(av[i], b[j].y, acc[i][2 * j + 1]);
        }
    }
    if (db) {
#pragma unroll
      for (int q = 0; q < 8; ++q) bacc += sm.dy[slot][brow + q][bk];
    }
  }
  cp_async_wait<0>();
  signal_dependents();

  // Epilogue: this CTA's partial tile (or the final values when S == 1).
  const int64_t E = K * C;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t k = k0 + tk * 4 + i;
    if (k >= K) continue;
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      const int64_t c = c0 + 2 * tc + 32 * j;
      if (c >= C) continue;  // C % 4 == 0, so c + 1 < C as well
      float* dst = ws ? ws + (int64_t)sigma * E + k * C + c : out + k * C + c;
      *reinterpret_cast<float2*>(dst) = make_float2(acc[i][2 * j], acc[i][2 * j + 1]);
    }
  }
  if (db && (tile % tiles_c) == 0) {
    sm.bias[tid / kBK][bk] = bacc;
    __syncthreads();
    if (tid < kBK && k0 + tid < K) {
      // rows 0-7, 8-15, 16-23, 24-31 of every stage, added in that order
      const float v = ((sm.bias[0][tid] + sm.bias[1][tid]) + sm.bias[2][tid]) + sm.bias[3][tid];
      if (ws_bias) ws_bias[(int64_t)sigma * K + k0 + tid] = v;
      else db[k0 + tid] = v;
    }
  }
}

int pick_bc(int64_t C) {
  if (C <= 32) return 32;
  if (C <= 64) return 64;
  if (C <= 96) return 96;
  return 128;
}

template <int BC>
cudaError_t launch_bc(const Plan& p, const Args& a, int64_t tiles_c) {
  const size_t smem = sizeof(Smem<BC>);
  cudaError_t err = cudaFuncSetAttribute(wgrad1x1_ffma_kernel<BC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
  if (err != cudaSuccess) return err;
  const int64_t ctas = p.geo.tiles * p.split;
  if (ctas > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  wgrad1x1_ffma_kernel<BC><<<(unsigned)ctas, kThreads, smem, a.stream>>>(
      static_cast<const float*>(a.x), static_cast<const float*>(a.b), static_cast<float*>(a.out), a.ws,
      p.with_bias ? static_cast<float*>(a.db) : nullptr, a.ws_bias, p.sh.P(), p.sh.k, p.sh.c, tiles_c,
      p.geo.tiles, p.split, p.geo.blocks);
  return cudaGetLastError();
}

}  // namespace

Geometry geometry_wgrad1x1_ffma(const Shape& s) {
  Geometry g;
  const bool pointwise = s.r == 1 && s.s == 1 && s.sh == 1 && s.sw == 1 && s.ph == 0 && s.pw == 0;
  if (!pointwise || s.groups != 1 || s.in_dt != CONV_F32 || s.out_dt != CONV_F32) return g;
  if (s.c % 4 != 0 || s.k % 4 != 0) return g;
  const int bc = pick_bc(s.c);
  g.ok = true;
  g.ctas_per_sm = 2;
  g.tiles = ((s.k + kBK - 1) / kBK) * ((s.c + bc - 1) / bc);
  g.blocks = (s.P() + kBP - 1) / kBP;
  return g;
}

cudaError_t launch_wgrad1x1_ffma(const Plan& p, const Args& a) {
  const int bc = pick_bc(p.sh.c);
  const int64_t tiles_c = (p.sh.c + bc - 1) / bc;
  switch (bc) {
    case 32: return launch_bc<32>(p, a, tiles_c);
    case 64: return launch_bc<64>(p, a, tiles_c);
    case 96: return launch_bc<96>(p, a, tiles_c);
    default: return launch_bc<128>(p, a, tiles_c);
  }
}

}  // namespace cig
