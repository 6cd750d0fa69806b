// Depthwise weight gradient (groups = C = K) on CUDA cores.
//
//   dW[c, r, s] = sum over (n, ho, wo) of dY[n, ho, wo, c] * X[n, ho + r - ph, wo + s - pw, c]
//
// ("perf(rocke): depthwise 7x7 and grouped cpg4/8 wgrad on batched mfma
// 4x4x4", "Technical Details"; stride 1, dilation 1). Each channel is an
// independent 2-D correlation, so there is no dense contraction to hand to
// the tensor cores; the work is FP32-FMA bound (about 24 flop per byte at
// 7x7), not HBM bound.
//
// CTA: 64 channels (32 lanes x 2 channels as a 16-bit pair) and one slice of
// the output rows (n, ho) of the batch. Warp w < R owns filter row r = w and
// keeps S fp32x2 accumulators. For every output row it walks wo with a
// register window of the S input values the taps need, one 4-byte load of
// dY and one of X per step and S packed FMAs (fma.rn.f32x2); the loop is
// unrolled by S so the window rotates through registers without moves.
// Rows arrive in a shared-memory ring through 16-byte cp.async copies
// (coalesced NHWC rows: 64 channels = 128 bytes per pixel), zero-filled for
// rows outside the image; the pw padding columns of every ring slot are zero.
// One __syncthreads per output row. Partial sums of the slice go to an fp32
// slab ("feat(rocke): split-K forward implicit-GEMM convolution on gfx1250",
// "Two-stage split-K"), or straight to dW with one slice.
#include "common.cuh"

namespace cig {
namespace {

constexpr int kThreads = 256;
constexpr int kCG = 64;          // channels per CTA
constexpr int kPix = kCG * 2;    // bytes per pixel of one 16-bit channel group
constexpr int kPref = 2;         // rows prefetched ahead
constexpr int kMaxR = 8;         // filter rows (one warp each)
constexpr int kMaxS = 11;        // filter width
constexpr int kMaxW = 256;       // input width the ring is sized for

struct DwParams {
  int64_t N, H, W, C, Ho, Wo;
  int32_t R, Sf, ph, pw;
  int64_t rows;        // N * Ho: the reduction blocks
  int64_t groups;      // C / 64: the tiles
  int32_t split;
  int32_t ring;        // X rows held: R + kPref
  int32_t xrow_bytes;  // (W + 2 pw + Sf) * 128
  int32_t dyrow_bytes; // Wo * 128
};

// acc += a * b on both lanes of a register pair (one packed FP32 FMA).
__device__ __forceinline__ void ffma2(float2& acc, float2 a, float2 b) { acc = __ffma2_rn(a, b, acc); }

template <typename TI>
__device__ __forceinline__ float2 unpack2(uint32_t u);
template <>
__device__ __forceinline__ float2 unpack2<__nv_bfloat16>(uint32_t u) {
  return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xFFFF0000u));
}
template <>
__device__ __forceinline__ float2 unpack2<__half>(uint32_t u) {
  __half2 h = *reinterpret_cast<__half2*>(&u);
  return __half22float2(h);
}

// One output row for one filter row: acc[s] += dy[wo] * x[wo + s] (padded x);
// with BIAS also bsum += dy[wo].
template <typename TI, int S, bool BIAS>
__device__ __forceinline__ void row_pass(const uint8_t* xrow, const uint8_t* dyrow, int Wo, int lane,
                                         float2 (&acc)[kMaxS], float2& bsum) {
  const uint8_t* xp = xrow + lane * 4;
  const uint8_t* dp = dyrow + lane * 4;
  float2 win[S];
#pragma unroll
  for (int j = 0; j < S; ++j) win[j] = unpack2<TI>(*reinterpret_cast<const uint32_t*>(xp + j * kPix));
  int wo = 0;
  for (; wo + S <= Wo; wo += S) {
#pragma unroll
    for (int t = 0; t < S; ++t) {
      const float2 d = unpack2<TI>(*reinterpret_cast<const uint32_t*>(dp + (wo + t) * kPix));
#pragma unroll
      for (int j = 0; j < S; ++j) ffma2(acc[j], d, win[(t + j) % S]);
      if (BIAS) bsum = __fadd2_rn(bsum, d);
      win[t] = unpack2<TI>(*reinterpret_cast<const uint32_t*>(xp + (wo + t + S) * kPix));
    }
  }
  for (; wo < Wo; ++wo) {  // the last Wo % S outputs, straight from shared memory
    const float2 d = unpack2<TI>(*reinterpret_cast<const uint32_t*>(dp + wo * kPix));
    if (BIAS) bsum = __fadd2_rn(bsum, d);
#pragma unroll
    for (int j = 0; j < S; ++j)
      ffma2(acc[j], d, unpack2<TI>(*reinterpret_cast<const uint32_t*>(xp + (wo + j) * kPix)));
  }
}

// db (when requested) is summed by the warp of filter row 0, which reads
// every dY value of the slice exactly once.
template <typename TI, typename TO, int S>
__global__ void __launch_bounds__(kThreads, 2)
    dw_wgrad_kernel(const TI* __restrict__ x, const TI* __restrict__ dy, TO* out, float* ws, TO* db,
                    float* ws_bias, DwParams p) {
  extern __shared__ __align__(16) uint8_t smem[];
  uint8_t* xring = smem;                                       // ring rows of (W + 2 pw + S) pixels
  uint8_t* dyring = smem + (size_t)p.ring * p.xrow_bytes;      // kPref + 1 rows of Wo pixels
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32, tid = threadIdx.x;
  const int64_t g = blockIdx.x % p.groups;
  const int32_t sigma = (int32_t)(blockIdx.x / p.groups);
  const int64_t c0 = g * kCG;
  const int64_t row_b = slice_begin(p.rows, p.split, sigma), row_e = slice_begin(p.rows, p.split, sigma + 1);
  const int Wp = (int)p.W + 2 * p.pw + S;  // padded ring row width in pixels

  // Zero every ring row once: padding columns stay zero, real columns are
  // overwritten by every copy.
  for (int i = tid * 16; i < p.ring * p.xrow_bytes; i += kThreads * 16)
    *reinterpret_cast<uint4*>(xring + i) = make_uint4(0, 0, 0, 0);
  __syncthreads();

  float2 acc[kMaxS];
#pragma unroll
  for (int j = 0; j < kMaxS; ++j) acc[j] = make_float2(0.f, 0.f);
  float2 bsum = make_float2(0.f, 0.f);

  // Copy X row h of image n into ring slot h mod ring (zeros outside the image).
  auto load_x = [&](int64_t n, int64_t h) {
    uint8_t* dst = xring + (size_t)(((h % p.ring) + p.ring) % p.ring) * p.xrow_bytes + p.pw * kPix;
    const bool inside = h >= 0 && h < p.H;
    const TI* src = x + ((n * p.H + (inside ? h : 0)) * p.W) * p.C + c0;
    for (int i = tid; i < p.W * 8; i += kThreads) {
      const int px = i >> 3, ch = (i & 7) * 8;
      cp_async16(dst + px * kPix + ch * 2, inside ? (const void*)(src + px * p.C + ch) : (const void*)x,
                 inside ? 16u : 0u);
    }
  };
  auto load_dy = [&](int64_t n, int64_t ho) {
    uint8_t* dst = dyring + (size_t)(ho % (kPref + 1)) * p.dyrow_bytes;
    const TI* src = dy + ((n * p.Ho + ho) * p.Wo) * p.C + c0;
    for (int i = tid; i < p.Wo * 8; i += kThreads) {
      const int px = i >> 3, ch = (i & 7) * 8;
      cp_async16(dst + px * kPix + ch * 2, src + px * p.C + ch, 16u);
    }
  };

  // Walk the slice image by image: rows [row_b, row_e) of the flattened (n, ho).
  for (int64_t row = row_b; row < row_e;) {
    const int64_t n = row / p.Ho;
    const int64_t ho_a = row % p.Ho;
    const int64_t ho_b = (n + 1) * p.Ho <= row_e ? p.Ho : row_e - n * p.Ho;
    // prologue: the first R - 1 X rows of the window
    __syncthreads();
    for (int r = 0; r + 1 < p.R; ++r) load_x(n, ho_a - p.ph + r);
    for (int d = 0; d < kPref; ++d) {
      const int64_t ho = ho_a + d;
      if (ho < ho_b) {
        load_x(n, ho - p.ph + p.R - 1);
        load_dy(n, ho);
      }
      cp_async_commit();
    }
    for (int64_t ho = ho_a; ho < ho_b; ++ho) {
      cp_async_wait<kPref - 1>();
      __syncthreads();
      const int64_t hn = ho + kPref;
      if (hn < ho_b) {
        load_x(n, hn - p.ph + p.R - 1);
        load_dy(n, hn);
      }
      cp_async_commit();
      if (warp < p.R) {
        const int64_t h = ho - p.ph + warp;
        const uint8_t* xr = xring + (size_t)(((h % p.ring) + p.ring) % p.ring) * p.xrow_bytes;
        const uint8_t* dr = dyring + (size_t)(ho % (kPref + 1)) * p.dyrow_bytes;
        if (warp == 0 && db) row_pass<TI, S, true>(xr, dr, (int)p.Wo, lane, acc, bsum);
        else row_pass<TI, S, false>(xr, dr, (int)p.Wo, lane, acc, bsum);
      }
    }
    cp_async_wait<0>();
    row = n * p.Ho + ho_b;
  }
  (void)Wp;

  if (warp == 0 && db) {
    const int64_t c = c0 + 2 * lane;
    if (ws_bias) {
      ws_bias[(int64_t)sigma * p.C + c] = bsum.x;
      ws_bias[(int64_t)sigma * p.C + c + 1] = bsum.y;
    } else {
      store_out(db + c, bsum.x);
      store_out(db + c + 1, bsum.y);
    }
  }
  if (warp < p.R) {
    const int64_t E = p.C * p.R * S;
    const int64_t c = c0 + 2 * lane;
#pragma unroll
    for (int j = 0; j < S; ++j) {
      const int64_t e0 = (c * p.R + warp) * S + j;     // dW[c][r][s]
      const int64_t e1 = ((c + 1) * p.R + warp) * S + j;
      if (ws) {
        ws[(int64_t)sigma * E + e0] = acc[j].x;
        ws[(int64_t)sigma * E + e1] = acc[j].y;
      } else {
        store_out(out + e0, acc[j].x);
        store_out(out + e1, acc[j].y);
      }
    }
  }
}

DwParams make_params(const Plan& pl) {
  const Shape& s = pl.sh;
  DwParams p;
  p.N = s.n; p.H = s.h; p.W = s.w; p.C = s.c; p.Ho = s.ho; p.Wo = s.wo;
  p.R = (int32_t)s.r; p.Sf = (int32_t)s.s; p.ph = (int32_t)s.ph; p.pw = (int32_t)s.pw;
  p.rows = s.n * s.ho;
  p.groups = s.c / kCG;
  p.split = pl.split;
  p.ring = p.R + kPref;
  p.xrow_bytes = (int32_t)((s.w + 2 * s.pw + s.s) * kPix);
  p.dyrow_bytes = (int32_t)(s.wo * kPix);
  return p;
}

size_t smem_bytes(const DwParams& p) {
  return (size_t)p.ring * p.xrow_bytes + (size_t)(kPref + 1) * p.dyrow_bytes;
}

template <typename TI, typename TO, int S>
cudaError_t launch_s(const Plan& pl, const Args& a) {
  const DwParams p = make_params(pl);
  const size_t smem = smem_bytes(p);
  cudaError_t err = cudaFuncSetAttribute(dw_wgrad_kernel<TI, TO, S>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
  if (err != cudaSuccess) return err;
  const int64_t ctas = p.groups * p.split;
  if (ctas > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  dw_wgrad_kernel<TI, TO, S><<<(unsigned)ctas, kThreads, smem, a.stream>>>(
      static_cast<const TI*>(a.x), static_cast<const TI*>(a.b), static_cast<TO*>(a.out), a.ws,
      pl.with_bias ? static_cast<TO*>(a.db) : nullptr, a.ws_bias, p);
  return cudaGetLastError();
}

template <typename TI, typename TO>
cudaError_t launch_t(const Plan& pl, const Args& a) {
  switch (pl.sh.s) {
    case 3: return launch_s<TI, TO, 3>(pl, a);
    case 5: return launch_s<TI, TO, 5>(pl, a);
    case 7: return launch_s<TI, TO, 7>(pl, a);
    case 9: return launch_s<TI, TO, 9>(pl, a);
    case 11: return launch_s<TI, TO, 11>(pl, a);
    default: return cudaErrorNotSupported;
  }
}

}  // namespace

Geometry geometry_wgrad_depthwise(const Shape& s) {
  Geometry g;
  const bool depthwise = s.groups == s.c && s.groups == s.k;
  if (!depthwise || s.in_dt == CONV_F32 || s.sh != 1 || s.sw != 1 || s.dh != 1 || s.dw != 1) return g;
  if (s.c % kCG != 0 || s.r > kMaxR || s.w > kMaxW || s.n < 1) return g;
  if (!(s.s == 3 || s.s == 5 || s.s == 7 || s.s == 9 || s.s == 11)) return g;
  if (s.pw > s.s || s.ph > s.r) return g;
  DwParams p;
  p.ring = (int32_t)s.r + kPref;
  p.xrow_bytes = (int32_t)((s.w + 2 * s.pw + s.s) * kPix);
  p.dyrow_bytes = (int32_t)(s.wo * kPix);
  if (smem_bytes(p) > 110 * 1024) return g;  // two CTAs per SM
  g.ok = true;
  g.ctas_per_sm = 2;
  g.tiles = s.c / kCG;
  g.blocks = s.n * s.ho;
  return g;
}

cudaError_t launch_wgrad_depthwise(const Plan& p, const Args& a) {
  const int in = p.sh.in_dt, out = p.sh.out_dt;
  if (in == CONV_BF16)
    return out == CONV_F32 ? launch_t<__nv_bfloat16, float>(p, a) : launch_t<__nv_bfloat16, __nv_bfloat16>(p, a);
  return out == CONV_F32 ? launch_t<__half, float>(p, a) : launch_t<__half, __half>(p, a);
}

}  // namespace cig
