// Depthwise forward convolution on the CUDA cores (groups = C = K):
//   Y[n,ho,wo,c] = sum over r, s of X[n, ho*sh + r*dh - ph, wo*sw + s - pw, c] * W[c,r,s]
// (the forward twin of the depthwise weight gradient of "perf(rocke):
// depthwise 7x7 and grouped cpg4/8 wgrad on batched mfma 4x4x4"; that page's
// commit notes also list depthwise and grouped forward kernels). The filter
// width and the W stride are compile-time (3/5/7 and 1/2), so the sliding
// window lives in registers.
//
// A CTA owns 64 channels (each lane two adjacent ones, computed as packed
// fp32 pairs with __ffma2_rn) of 8 or 16 output rows (one or two per warp)
// of one image.
// A warp walks its row in chunks of 8 output columns: per filter row r it
// loads the (8 - 1) * sw + S input positions the chunk reads (each a 128-byte
// coalesced warp load, reused from L1/L2 by the neighbouring rows and
// chunks), then does S x 8 packed FMAs against the row's weights, which the
// CTA staged once in shared memory as lane pairs (conflict-free float2 reads).
// Reduction depth R*S is small, so there is no split-K: one launch, and the
// fused forward epilogue (bias + clamp) applies in the store.
#include "common.cuh"
#include "../kernel_entry.h"

namespace cig {
namespace {

constexpr int kThreads = 256;  // 8 warps
constexpr int kCB = 64;        // channels per CTA (2 per lane)
constexpr int kQ = 8;          // output columns per chunk

// Output rows per warp: 2 when the H stride and dilation are 1 (the two rows
// then read R + 1 input rows between them, each loaded once), else 1.
__host__ __device__ constexpr int rows_per_warp(bool pair) { return pair ? 2 : 1; }

__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }

template <typename T>
__device__ __forceinline__ float2 load2(const T* p);
template <>
__device__ __forceinline__ float2 load2<float>(const float* p) {
  return *reinterpret_cast<const float2*>(p);
}
template <>
__device__ __forceinline__ float2 load2<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(p));
}
template <>
__device__ __forceinline__ float2 load2<__half>(const __half* p) {
  return __half22float2(*reinterpret_cast<const __half2*>(p));
}

template <typename T>
__device__ __forceinline__ void store2(T* p, float2 v);
template <>
__device__ __forceinline__ void store2<float>(float* p, float2 v) {
  *reinterpret_cast<float2*>(p) = v;
}
template <>
__device__ __forceinline__ void store2<__nv_bfloat16>(__nv_bfloat16* p, float2 v) {
  *reinterpret_cast<__nv_bfloat162*>(p) = __floats2bfloat162_rn(v.x, v.y);
}
template <>
__device__ __forceinline__ void store2<__half>(__half* p, float2 v) {
  *reinterpret_cast<__half2*>(p) = __floats2half2_rn(v.x, v.y);
}

struct DwParams {
  int64_t H, W, C, Ho, Wo;
  int64_t row_blocks, cblocks;  // ceil(Ho / rows per CTA), ceil(C / 64)
  int32_t R, ph, pw, sh, dh;
  // fused epilogue: y = min(max(acc + bias[c], lo), hi)
  const void* ep_bias;
  float ep_lo, ep_hi;
  int32_t ep;
  int32_t rev;  // 1: tap t reads filter tap R*S - 1 - t (the data gradient's turned filter)
};

// Stores the kQ outputs of a chunk (ragged tail), with the fused epilogue.
template <typename TO>
__device__ __forceinline__ void store_chunk(TO* yrow, int64_t wo0, int64_t Wo, int64_t C, const float2* acc,
                                            const DwParams& p, float2 bias) {
#pragma unroll
  for (int q = 0; q < kQ; ++q) {
    if (wo0 + q >= Wo) break;
    float2 v = acc[q];
    if (p.ep) {
      v.x = fminf(fmaxf(v.x + bias.x, p.ep_lo), p.ep_hi);
      v.y = fminf(fmaxf(v.y + bias.y, p.ep_lo), p.ep_hi);
    }
    store2(yrow + (wo0 + q) * C, v);
  }
}

template <typename TI, int kSpan>
__device__ __forceinline__ void load_span(float2* xv, const TI* xr, int64_t wi0, int64_t W, int64_t C,
                                          bool interior) {
  if (interior) {  // the whole span inside the row: walk a pointer, no tests
    const TI* q = xr + wi0 * C;
#pragma unroll
    for (int j = 0; j < kSpan; ++j, q += C) xv[j] = load2(q);
  } else {
#pragma unroll
    for (int j = 0; j < kSpan; ++j) {
      const int64_t wi = wi0 + j;
      xv[j] = wi >= 0 && wi < W ? load2(xr + wi * C) : make_float2(0.f, 0.f);
    }
  }
}

template <typename TI, typename TO, int S, int SW, bool PAIR>
__global__ void __launch_bounds__(kThreads, 2) dwconv_fwd_kernel(const TI* __restrict__ x, const TI* __restrict__ w,
                                                              TO* __restrict__ y, DwParams p) {
  extern __shared__ float2 swt[];  // [R*S taps][32 lanes]: this CTA's weights as channel pairs
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t cb = blockIdx.x % p.cblocks;
  const int64_t t = blockIdx.x / p.cblocks;
  const int64_t rb = t % p.row_blocks, n = t / p.row_blocks;
  const int taps = p.R * S;
  for (int i = threadIdx.x; i < taps * 32; i += kThreads) {
    const int tap = i >> 5;
    const int64_t cc = cb * kCB + 2 * (i & 31);
    float2 v = make_float2(0.f, 0.f);
    const int wt = p.rev ? taps - 1 - tap : tap;
    if (cc < p.C) v = make_float2(to_f32(w[cc * taps + wt]), to_f32(w[(cc + 1) * taps + wt]));
    swt[i] = v;
  }
  __syncthreads();  // the last barrier: warps may leave below

  const int64_t c = cb * kCB + 2 * lane;  // this lane's channels c, c + 1 (C is even)
  constexpr int RW = rows_per_warp(PAIR);
  const int64_t ho = (rb * 8 + warp) * RW;  // this warp's first output row
  if (ho >= p.Ho || c >= p.C) return;
  float2 bias = make_float2(0.f, 0.f);
  if (p.ep && p.ep_bias) {  // element loads: the bias is only element-aligned
    const TO* b = static_cast<const TO*>(p.ep_bias);
    bias = make_float2(to_f32(b[c]), to_f32(b[c + 1]));
  }
  const TI* xn = x + n * p.H * p.W * p.C + c;
  TO* yrow = y + (n * p.Ho + ho) * p.Wo * p.C + c;
  const bool second = PAIR && ho + 1 < p.Ho;  // the pair's second row exists
  constexpr int kSpan = (kQ - 1) * SW + S;  // input columns a chunk reads per filter row
#pragma unroll 1
  for (int64_t wo0 = 0; wo0 < p.Wo; wo0 += kQ) {
    float2 acc[kQ], acc2[PAIR ? kQ : 1];
#pragma unroll
    for (int q = 0; q < kQ; ++q) acc[q] = make_float2(0.f, 0.f);
#pragma unroll
    for (int q = 0; q < (PAIR ? kQ : 1); ++q) acc2[q] = make_float2(0.f, 0.f);
    const int64_t wi0 = wo0 * SW - p.pw;
    const bool interior = wi0 >= 0 && wi0 + kSpan <= p.W;
    if (PAIR) {
      // input row i (hi = ho + i - ph) feeds row ho through tap i and row ho + 1 through tap i - 1
#pragma unroll 1
      for (int i = 0; i <= p.R; ++i) {
        const int64_t hi = ho + i - p.ph;
        if (hi < 0 || hi >= p.H) continue;
        float2 xv[kSpan];
        load_span<TI, kSpan>(xv, xn + hi * p.W * p.C, wi0, p.W, p.C, interior);
        if (i < p.R) {
          const float2* wr = swt + i * S * 32 + lane;
#pragma unroll
          for (int s = 0; s < S; ++s) {
            const float2 wv = wr[s * 32];
#pragma unroll
            for (int q = 0; q < kQ; ++q) acc[q] = fma2(xv[q * SW + s], wv, acc[q]);
          }
        }
        if (i >= 1) {
          const float2* wr = swt + (i - 1) * S * 32 + lane;
#pragma unroll
          for (int s = 0; s < S; ++s) {
            const float2 wv = wr[s * 32];
#pragma unroll
            for (int q = 0; q < (PAIR ? kQ : 1); ++q) acc2[q] = fma2(xv[q * SW + s], wv, acc2[q]);
          }
        }
      }
    } else {
#pragma unroll 1
      for (int r = 0; r < p.R; ++r) {
        const int64_t hi = ho * p.sh + r * p.dh - p.ph;
        if (hi < 0 || hi >= p.H) continue;
        float2 xv[kSpan];
        load_span<TI, kSpan>(xv, xn + hi * p.W * p.C, wi0, p.W, p.C, interior);
        const float2* wr = swt + r * S * 32 + lane;
#pragma unroll
        for (int s = 0; s < S; ++s) {
          const float2 wv = wr[s * 32];
#pragma unroll
          for (int q = 0; q < kQ; ++q) acc[q] = fma2(xv[q * SW + s], wv, acc[q]);
        }
      }
    }
    store_chunk(yrow, wo0, p.Wo, p.C, acc, p, bias);
    if (second) store_chunk(yrow + p.Wo * p.C, wo0, p.Wo, p.C, acc2, p, bias);
  }
}

template <typename TI, typename TO, int S, int SW, bool PAIR>
cudaError_t launch_s(const Plan& pl, const Args& a, const DwParams& p) {
  const int64_t ctas = pl.geo.tiles;
  if (ctas > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  const size_t smem = (size_t)p.R * S * 32 * sizeof(float2);
  auto kern = dwconv_fwd_kernel<TI, TO, S, SW, PAIR>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  kern<<<(unsigned)ctas, kThreads, smem, a.stream>>>(static_cast<const TI*>(a.x), static_cast<const TI*>(a.b),
                                                     static_cast<TO*>(a.out), p);
  return cudaGetLastError();
}

// Two output rows per warp: stride and dilation 1 along H, stride 1 along W.
bool pair_rows(const Shape& s) { return s.sh == 1 && s.dh == 1 && s.sw == 1; }

template <typename TI, typename TO>
cudaError_t launch_typed(const Plan& pl, const Args& a) {
  const Shape& s = pl.sh;
  DwParams p;
  p.H = s.h;
  p.W = s.w;
  p.C = s.c;
  p.Ho = s.ho;
  p.Wo = s.wo;
  const bool pair = pair_rows(s);
  const int64_t rows = 8 * rows_per_warp(pair);
  p.row_blocks = (s.ho + rows - 1) / rows;
  p.cblocks = (s.c + kCB - 1) / kCB;
  p.R = (int32_t)s.r;
  p.ph = (int32_t)s.ph;
  p.pw = (int32_t)s.pw;
  p.sh = (int32_t)s.sh;
  p.dh = (int32_t)s.dh;
  p.ep_bias = a.ep_bias;
  p.ep_lo = a.ep_lo;
  p.ep_hi = a.ep_hi;
  p.ep = a.ep ? 1 : 0;
  p.rev = a.rev_taps ? 1 : 0;
  const int key = (int)s.s * 10 + (int)s.sw;
  if (pair) {
    switch (key) {
      case 31: return launch_s<TI, TO, 3, 1, true>(pl, a, p);
      case 51: return launch_s<TI, TO, 5, 1, true>(pl, a, p);
      case 71: return launch_s<TI, TO, 7, 1, true>(pl, a, p);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (key) {
    case 31: return launch_s<TI, TO, 3, 1, false>(pl, a, p);
    case 32: return launch_s<TI, TO, 3, 2, false>(pl, a, p);
    case 51: return launch_s<TI, TO, 5, 1, false>(pl, a, p);
    case 52: return launch_s<TI, TO, 5, 2, false>(pl, a, p);
    case 71: return launch_s<TI, TO, 7, 1, false>(pl, a, p);
    case 72: return launch_s<TI, TO, 7, 2, false>(pl, a, p);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

// The TMA-ring, register-tap form (dw_fwd_ring.cu) the depthwise forward
// takes for 16-bit square 3/5/7 filters at unit stride.
Geometry geometry_fwd_depthwise_ring(const Shape& s);
cudaError_t launch_fwd_depthwise_ring(const Plan& p, const Args& a);

Geometry geometry_fwd_depthwise(const Shape& s) {
  const Geometry ring = geometry_fwd_depthwise_ring(s);
  if (ring.ok) return ring;
  Geometry g;
  const bool depthwise = s.groups == s.c && s.groups == s.k;
  if (!depthwise || s.c % 2 != 0) return g;
  if (!(s.s == 3 || s.s == 5 || s.s == 7) || !(s.sw == 1 || s.sw == 2) || s.dw != 1) return g;
  if (s.r > 64 || s.h > 0x7fffffffLL || s.w > 0x7fffffffLL) return g;
  g.ok = true;
  g.ctas_per_sm = 4;
  const int64_t rows = 8 * rows_per_warp(pair_rows(s));  // output rows per CTA
  g.tiles = s.n * ((s.ho + rows - 1) / rows) * ((s.c + kCB - 1) / kCB);
  if (g.tiles < 1) g.tiles = 1;
  g.blocks = 1;  // no split: the reduction is R*S taps
  return g;
}

cudaError_t launch_fwd_depthwise(const Plan& p, const Args& a) {
  if (p.split != 1 || a.ws) return cudaErrorInvalidValue;
  if (geometry_fwd_depthwise_ring(p.sh).ok) return launch_fwd_depthwise_ring(p, a);
  const int in = p.sh.in_dt, out = p.sh.out_dt;
  if (in == CONV_F32) return launch_typed<float, float>(p, a);
  if (in == CONV_BF16)
    return out == CONV_F32 ? launch_typed<__nv_bfloat16, float>(p, a)
                           : launch_typed<__nv_bfloat16, __nv_bfloat16>(p, a);
  return out == CONV_F32 ? launch_typed<__half, float>(p, a) : launch_typed<__half, __half>(p, a);
}

}  // namespace cig
