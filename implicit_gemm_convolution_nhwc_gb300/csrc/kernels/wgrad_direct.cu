// Depthwise (groups = C = K) and grouped (Cg = Kg = 4 or 8) weight gradients
// on CUDA cores:
//
//   dW[k, r, s, c] = sum over (n, ho, wo) of dY[n, ho, wo, k] * X[n, ho + r - ph, wo + s - pw, g Cg + c]
//   db[k]          = sum over (n, ho, wo) of dY[n, ho, wo, k]
//
// ("perf(rocke): depthwise 7x7 and grouped cpg4/8 wgrad on batched mfma
// 4x4x4", "Technical Details"; stride 1, dilation 1). A depthwise channel is
// an independent 2-D correlation and a 4/8-channel group an 8 x 72 (or 4 x 36)
// contraction: neither is a dense tile for the tensor cores, and both are
// FP32-FMA bound (18-36 flop per byte of input), not HBM bound.
//
// CTA: 64 channels (= 64/Cg whole groups) and one slice of the batch's output
// rows (n, ho); 16 warps. Rows come in with 16-byte global loads issued two
// rows ahead into registers, are widened ONCE to fp32 and stored in a shared
// ring (R + 1 input rows, padded with pw zero columns on each side; 2 dY
// rows), so the inner loop is only shared loads and packed FMAs
// (__ffma2_rn). Warp w < R*WS owns filter row r = w % R and part w / R of
// every output row (WS = 16 / R parts). Lane l owns output channels
// c0 + 2l and c0 + 2l + 1:
//  - depthwise: per pixel one float2 of dY and one float2 of X (the same two
//    channels); S packed FMAs on a register window of S input pixels that
//    rotates without moves (the loop is unrolled by S);
//  - grouped: per pixel the dY pair (broadcast once into two register pairs)
//    and the group's Cg input channels as Cg/2 pairs; S*Cg packed FMAs.
// The filter-row-0 warps also sum db. One __syncthreads per output row.
// The parts of a filter row are added in part order at the end, and the
// slice's partial sums go to an fp32 slab ("feat(rocke): split-K forward
// implicit-GEMM convolution on gfx1250", "Two-stage split-K") or, with one
// slice, straight to dW / db.
#include "common.cuh"

namespace cig {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kCG = 64;            // channels per CTA
constexpr int kPixIn = kCG * 2;    // bytes per pixel in global memory (16-bit)
constexpr int kPix = kCG * 4;      // bytes per pixel in the fp32 ring
constexpr int kMaxItems = 2;       // 16-byte loads per thread per row step
constexpr int kMaxW = 256;
constexpr int kSmemLimit = 200 * 1024;

struct DirParams {
  int64_t N, H, W, C, Ho, Wo;
  int32_t R, ph, pw;
  int32_t WS;          // parts per output row
  int64_t rows;        // N * Ho: the reduction blocks
  int64_t groups;      // C / 64: the tiles
  int32_t split;
  int32_t xrow_bytes;  // (W + 2 pw + S) * 256
  int32_t dyrow_bytes; // Wo * 256
  int32_t items;       // 16-byte global loads per row step: (W + Wo) * 8
};

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

// Accumulators of one lane: depthwise (CPG = 1) v[s][0][0] = (dW[c][r][s], dW[c+1][r][s]);
// grouped v[s][ki][cp] = (dW[k+ki][r][s][2cp], dW[k+ki][r][s][2cp+1]).
template <int S, int CPG>
struct Acc {
  static constexpr int KI = CPG == 1 ? 1 : 2;
  static constexpr int CP = CPG == 1 ? 1 : CPG / 2;
  float2 v[S][KI][CP];
};

// Output pixels [wo_a, wo_b) of one row for one filter row. xrow: the padded
// fp32 input row (pixel i <-> w = i - pw); dyrow: the fp32 dY row.
template <int S, int CPG, bool BIAS>
__device__ __forceinline__ void row_pass(const uint8_t* xrow, const uint8_t* dyrow, int wo_a, int wo_b, int lane,
                                         Acc<S, CPG>& acc, float2& bsum) {
  constexpr int CP = Acc<S, CPG>::CP;
  const uint8_t* dp = dyrow + lane * 8;
  // depthwise: this lane's two channels; grouped: its group's first channel
  const uint8_t* xp = xrow + (CPG == 1 ? lane * 8 : ((2 * lane) / CPG) * CPG * 4);
  float2 win[S][CP];
  auto load_x = [&](int px, float2* v) {
#pragma unroll
    for (int c = 0; c < CP; ++c) v[c] = *reinterpret_cast<const float2*>(xp + px * kPix + c * 8);
  };
#pragma unroll
  for (int j = 0; j < S; ++j) load_x(wo_a + j, win[j]);
  int wo = wo_a;
  for (; wo + S <= wo_b; wo += S) {
#pragma unroll
    for (int t = 0; t < S; ++t) {
      const float2 d = *reinterpret_cast<const float2*>(dp + (wo + t) * kPix);
      if constexpr (CPG == 1) {
#pragma unroll
        for (int j = 0; j < S; ++j) acc.v[j][0][0] = __ffma2_rn(d, win[(t + j) % S][0], acc.v[j][0][0]);
      } else {
        const float2 d0 = make_float2(d.x, d.x), d1 = make_float2(d.y, d.y);
#pragma unroll
        for (int j = 0; j < S; ++j)
#pragma unroll
          for (int c = 0; c < CP; ++c) {
            acc.v[j][0][c] = __ffma2_rn(d0, win[(t + j) % S][c], acc.v[j][0][c]);
            acc.v[j][1][c] = __ffma2_rn(d1, win[(t + j) % S][c], acc.v[j][1][c]);
          }
      }
      if (BIAS) bsum = __fadd2_rn(bsum, d);
      load_x(wo + t + S, win[t]);
    }
  }
  for (; wo < wo_b; ++wo) {  // the last (wo_b - wo_a) % S pixels
    const float2 d = *reinterpret_cast<const float2*>(dp + wo * kPix);
    if (BIAS) bsum = __fadd2_rn(bsum, d);
#pragma unroll
    for (int j = 0; j < S; ++j) {
      float2 v[CP];
      load_x(wo + j, v);
      if constexpr (CPG == 1) {
        acc.v[j][0][0] = __ffma2_rn(d, v[0], acc.v[j][0][0]);
      } else {
        const float2 d0 = make_float2(d.x, d.x), d1 = make_float2(d.y, d.y);
#pragma unroll
        for (int c = 0; c < CP; ++c) {
          acc.v[j][0][c] = __ffma2_rn(d0, v[c], acc.v[j][0][c]);
          acc.v[j][1][c] = __ffma2_rn(d1, v[c], acc.v[j][1][c]);
        }
      }
    }
  }
}

template <typename TI, typename TO, int S, int CPG>
__global__ void __launch_bounds__(kThreads, 1)
    direct_wgrad_kernel(const TI* __restrict__ x, const TI* __restrict__ dy, TO* out, float* ws, TO* db,
                        float* ws_bias, DirParams p) {
  using A = Acc<S, CPG>;
  extern __shared__ __align__(16) uint8_t smem[];
  const int ring = p.R + 1;
  uint8_t* xring = smem;                                   // ring rows of (W + 2 pw + S) pixels, fp32
  uint8_t* dyring = smem + (size_t)ring * p.xrow_bytes;    // 2 rows of Wo pixels, fp32
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32, tid = threadIdx.x;
  const int64_t g = blockIdx.x % p.groups;
  const int32_t sigma = (int32_t)(blockIdx.x / p.groups);
  const int64_t c0 = g * kCG;
  const int64_t row_b = slice_begin(p.rows, p.split, sigma), row_e = slice_begin(p.rows, p.split, sigma + 1);
  const bool compute = warp < p.R * p.WS;
  const int r = warp % p.R, part = warp / p.R;
  const int wo_a = compute ? (int)((p.Wo * part) / p.WS) : 0;
  const int wo_b = compute ? (int)((p.Wo * (part + 1)) / p.WS) : 0;
  const bool bias_warp = compute && r == 0 && db != nullptr;

  for (int i = tid * 16; i < ring * p.xrow_bytes; i += kThreads * 16)
    *reinterpret_cast<uint4*>(xring + i) = make_uint4(0, 0, 0, 0);

  A acc;
#pragma unroll
  for (int j = 0; j < S; ++j)
#pragma unroll
    for (int ki = 0; ki < A::KI; ++ki)
#pragma unroll
      for (int c = 0; c < A::CP; ++c) acc.v[j][ki][c] = make_float2(0.f, 0.f);
  float2 bsum = make_float2(0.f, 0.f);

  // Row-step data of output row ho of image n: X row ho - ph + R - 1 (the row
  // that enters the window) and dY row ho, as 16-byte items per thread.
  uint4 buf[2][kMaxItems];
  auto fetch = [&](int64_t n, int64_t ho, uint4* b) {
    const int64_t h = ho - p.ph + p.R - 1;
    const bool inside = h >= 0 && h < p.H;
#pragma unroll
    for (int m = 0; m < kMaxItems; ++m) {
      const int i = tid + m * kThreads;
      b[m] = make_uint4(0, 0, 0, 0);
      if (i < p.W * 8) {
        if (inside) b[m] = __ldg(reinterpret_cast<const uint4*>(x + ((n * p.H + h) * p.W + (i >> 3)) * p.C + c0 + (i & 7) * 8));
      } else if (i < p.items) {
        const int j = i - (int)p.W * 8;
        b[m] = __ldg(reinterpret_cast<const uint4*>(dy + ((n * p.Ho + ho) * p.Wo + (j >> 3)) * p.C + c0 + (j & 7) * 8));
      }
    }
  };
  auto widen_store = [&](int64_t ho, const uint4* b) {
    const int64_t h = ho - p.ph + p.R - 1;
    uint8_t* xdst = xring + (size_t)(((h % ring) + ring) % ring) * p.xrow_bytes + p.pw * kPix;
    uint8_t* ddst = dyring + (size_t)(ho & 1) * p.dyrow_bytes;
#pragma unroll
    for (int m = 0; m < kMaxItems; ++m) {
      const int i = tid + m * kThreads;
      if (i >= p.items) break;
      const uint4 u = b[m];
      const float2 a = unpack2<TI>(u.x), bb = unpack2<TI>(u.y), c = unpack2<TI>(u.z), d = unpack2<TI>(u.w);
      uint8_t* dst = i < p.W * 8 ? xdst + (i >> 3) * kPix + (i & 7) * 32
                                 : ddst + ((i - (int)p.W * 8) >> 3) * kPix + ((i - (int)p.W * 8) & 7) * 32;
      reinterpret_cast<float4*>(dst)[0] = make_float4(a.x, a.y, bb.x, bb.y);
      reinterpret_cast<float4*>(dst)[1] = make_float4(c.x, c.y, d.x, d.y);
    }
  };
  // The first R - 1 input rows of a window (ho_a - ph .. ho_a - ph + R - 2).
  auto prologue_rows = [&](int64_t n, int64_t ho_a) {
    for (int rr = 0; rr + 1 < p.R; ++rr) {
      uint4 b[kMaxItems];
      const int64_t h = ho_a - p.ph + rr;
      const bool inside = h >= 0 && h < p.H;
      uint8_t* xdst = xring + (size_t)(((h % ring) + ring) % ring) * p.xrow_bytes + p.pw * kPix;
#pragma unroll
      for (int m = 0; m < kMaxItems; ++m) {
        const int i = tid + m * kThreads;
        b[m] = make_uint4(0, 0, 0, 0);
        if (inside && i < p.W * 8)
          b[m] = __ldg(reinterpret_cast<const uint4*>(x + ((n * p.H + h) * p.W + (i >> 3)) * p.C + c0 + (i & 7) * 8));
      }
#pragma unroll
      for (int m = 0; m < kMaxItems; ++m) {
        const int i = tid + m * kThreads;
        if (i >= p.W * 8) break;
        const uint4 u = b[m];
        const float2 a = unpack2<TI>(u.x), bb = unpack2<TI>(u.y), c = unpack2<TI>(u.z), d = unpack2<TI>(u.w);
        uint8_t* dst = xdst + (i >> 3) * kPix + (i & 7) * 32;
        reinterpret_cast<float4*>(dst)[0] = make_float4(a.x, a.y, bb.x, bb.y);
        reinterpret_cast<float4*>(dst)[1] = make_float4(c.x, c.y, d.x, d.y);
      }
    }
  };

  for (int64_t row = row_b; row < row_e;) {
    const int64_t n = row / p.Ho;
    const int64_t ho_a = row % p.Ho;
    const int64_t ho_b = (n + 1) * p.Ho <= row_e ? p.Ho : row_e - n * p.Ho;
    __syncthreads();  // the previous image's rows are no longer read
    prologue_rows(n, ho_a);
    fetch(n, ho_a, buf[0]);
    widen_store(ho_a, buf[0]);
    if (ho_a + 1 < ho_b) fetch(n, ho_a + 1, buf[1]);
    if (ho_a + 2 < ho_b) fetch(n, ho_a + 2, buf[0]);
    // One output row: nxt holds row step ho + 1 on entry and is refilled with
    // step ho + 3 (the other buffer holds step ho + 2).
    auto step = [&](int64_t ho, uint4* nxt) {
      __syncthreads();  // row step ho is in shared memory; step ho - 1 is done
      if (ho + 1 < ho_b) widen_store(ho + 1, nxt);
      if (ho + 3 < ho_b) fetch(n, ho + 3, nxt);
      if (compute) {
        const int64_t h = ho - p.ph + r;
        const uint8_t* xr = xring + (size_t)(((h % ring) + ring) % ring) * p.xrow_bytes;
        const uint8_t* dr = dyring + (size_t)(ho & 1) * p.dyrow_bytes;
        if (bias_warp) row_pass<S, CPG, true>(xr, dr, wo_a, wo_b, lane, acc, bsum);
        else row_pass<S, CPG, false>(xr, dr, wo_a, wo_b, lane, acc, bsum);
      }
    };
    // Unrolled by two so each buffer is named at compile time (kept in registers).
    for (int64_t ho = ho_a; ho < ho_b; ho += 2) {
      step(ho, buf[1]);
      if (ho + 1 < ho_b) step(ho + 1, buf[0]);
    }
    row = n * p.Ho + ho_b;
  }

  // Add the WS parts of each filter row in part order, then store.
  constexpr int PER = S * A::KI * A::CP * 2 + 2;  // dW partials, then the db pair
  __syncthreads();
  float* red = reinterpret_cast<float*>(smem);
  if (compute && part > 0) {
    float* dst = red + ((size_t)warp * 32 + lane) * PER;
    int q = 0;
#pragma unroll
    for (int j = 0; j < S; ++j)
#pragma unroll
      for (int ki = 0; ki < A::KI; ++ki)
#pragma unroll
        for (int c = 0; c < A::CP; ++c) {
          dst[q++] = acc.v[j][ki][c].x;
          dst[q++] = acc.v[j][ki][c].y;
        }
    dst[PER - 2] = bsum.x;
    dst[PER - 1] = bsum.y;
  }
  __syncthreads();
  if (!(compute && part == 0)) return;
  for (int pt = 1; pt < p.WS; ++pt) {
    const float* src = red + ((size_t)(pt * p.R + r) * 32 + lane) * PER;
    int q = 0;
#pragma unroll
    for (int j = 0; j < S; ++j)
#pragma unroll
      for (int ki = 0; ki < A::KI; ++ki)
#pragma unroll
        for (int c = 0; c < A::CP; ++c) {
          acc.v[j][ki][c].x += src[q++];
          acc.v[j][ki][c].y += src[q++];
        }
    bsum.x += src[PER - 2];
    bsum.y += src[PER - 1];
  }
  const int cg = CPG == 1 ? 1 : CPG;
  const int64_t E = p.C * p.R * S * cg;
  auto put = [&](int64_t e, float v) {
    if (ws) ws[(int64_t)sigma * E + e] = v;
    else store_out(out + e, v);
  };
  const int64_t k = c0 + 2 * lane;
#pragma unroll
  for (int j = 0; j < S; ++j) {
    if constexpr (CPG == 1) {
      put((k * p.R + r) * S + j, acc.v[j][0][0].x);        // dW[k][r][s]
      put(((k + 1) * p.R + r) * S + j, acc.v[j][0][0].y);
    } else {
#pragma unroll
      for (int ki = 0; ki < 2; ++ki)
#pragma unroll
        for (int c = 0; c < A::CP; ++c) {
          const int64_t e = (((k + ki) * p.R + r) * S + j) * CPG + 2 * c;  // dW[k][r][s][2c]
          put(e, acc.v[j][ki][c].x);
          put(e + 1, acc.v[j][ki][c].y);
        }
    }
  }
  if (bias_warp) {
    if (ws_bias) {
      ws_bias[(int64_t)sigma * p.C + k] = bsum.x;
      ws_bias[(int64_t)sigma * p.C + k + 1] = bsum.y;
    } else {
      store_out(db + k, bsum.x);
      store_out(db + k + 1, bsum.y);
    }
  }
}

DirParams make_params(const Shape& s, int32_t split) {
  DirParams p;
  p.N = s.n; p.H = s.h; p.W = s.w; p.C = s.c; p.Ho = s.ho; p.Wo = s.wo;
  p.R = (int32_t)s.r; p.ph = (int32_t)s.ph; p.pw = (int32_t)s.pw;
  p.WS = kWarps / p.R;
  p.rows = s.n * s.ho;
  p.groups = s.c / kCG;
  p.split = split;
  p.xrow_bytes = (int32_t)((s.w + 2 * s.pw + s.s) * kPix);
  p.dyrow_bytes = (int32_t)(s.wo * kPix);
  p.items = (int32_t)((s.w + s.wo) * 8);
  return p;
}

size_t smem_bytes(const DirParams& p, int S, int cpg) {
  const size_t ringb = (size_t)(p.R + 1) * p.xrow_bytes + 2 * (size_t)p.dyrow_bytes;
  const int per = S * (cpg == 1 ? 2 : 2 * cpg) + 2;
  const size_t red = (size_t)(p.R * p.WS) * 32 * per * 4;
  return ringb > red ? ringb : red;
}

// Shapes both kernels share: stride 1, dilation 1, 16-bit inputs, whole
// 64-channel CTAs, rows that fit the ring and the per-thread load slots.
bool common_ok(const Shape& s) {
  if (s.in_dt == CONV_F32 || s.sh != 1 || s.sw != 1 || s.dh != 1 || s.dw != 1 || s.n < 1) return false;
  if (s.c % kCG != 0 || s.c != s.k || s.r > kWarps / 2 || s.w > kMaxW) return false;
  if (s.pw > s.s || s.ph > s.r) return false;
  if ((s.w + s.wo) * 8 > (int64_t)kMaxItems * kThreads) return false;
  return true;
}

template <typename TI, typename TO, int S, int CPG>
cudaError_t launch_s(const Plan& pl, const Args& a) {
  const DirParams p = make_params(pl.sh, pl.split);
  const size_t smem = smem_bytes(p, S, CPG);
  cudaError_t err = cudaFuncSetAttribute(direct_wgrad_kernel<TI, TO, S, CPG>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  const int64_t ctas = p.groups * p.split;
  if (ctas > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  direct_wgrad_kernel<TI, TO, S, CPG><<<(unsigned)ctas, kThreads, smem, a.stream>>>(
      static_cast<const TI*>(a.x), static_cast<const TI*>(a.b), static_cast<TO*>(a.out), a.ws,
      pl.with_bias ? static_cast<TO*>(a.db) : nullptr, a.ws_bias, p);
  return cudaGetLastError();
}

template <typename TI, typename TO>
cudaError_t launch_depthwise_t(const Plan& pl, const Args& a) {
  switch (pl.sh.s) {
    case 3: return launch_s<TI, TO, 3, 1>(pl, a);
    case 5: return launch_s<TI, TO, 5, 1>(pl, a);
    case 7: return launch_s<TI, TO, 7, 1>(pl, a);
    case 9: return launch_s<TI, TO, 9, 1>(pl, a);
    case 11: return launch_s<TI, TO, 11, 1>(pl, a);
    default: return cudaErrorNotSupported;
  }
}

template <typename TI, typename TO>
cudaError_t launch_grouped_t(const Plan& pl, const Args& a) {
  switch (pl.sh.s * 16 + pl.sh.cg) {
    case 1 * 16 + 4: return launch_s<TI, TO, 1, 4>(pl, a);
    case 1 * 16 + 8: return launch_s<TI, TO, 1, 8>(pl, a);
    case 3 * 16 + 4: return launch_s<TI, TO, 3, 4>(pl, a);
    case 3 * 16 + 8: return launch_s<TI, TO, 3, 8>(pl, a);
    case 5 * 16 + 4: return launch_s<TI, TO, 5, 4>(pl, a);
    default: return cudaErrorNotSupported;
  }
}

Geometry direct_geometry(const Shape& s, int cpg) {
  Geometry g;
  const DirParams p = make_params(s, 1);
  if (smem_bytes(p, (int)s.s, cpg) > kSmemLimit) return g;
  g.ok = true;
  g.ctas_per_sm = 1;
  g.tiles = s.c / kCG;
  g.blocks = s.n * s.ho;
  return g;
}

}  // namespace

Geometry geometry_wgrad_depthwise(const Shape& s) {
  const bool depthwise = s.groups == s.c && s.groups == s.k;
  if (!depthwise || !common_ok(s)) return Geometry{};
  if (!(s.s == 3 || s.s == 5 || s.s == 7 || s.s == 9 || s.s == 11)) return Geometry{};
  return direct_geometry(s, 1);
}

Geometry geometry_wgrad_grouped(const Shape& s) {
  if (!(s.cg == 4 || s.cg == 8) || s.kg != s.cg || !common_ok(s)) return Geometry{};
  if (!(s.s == 1 || s.s == 3 || (s.s == 5 && s.cg == 4))) return Geometry{};
  return direct_geometry(s, (int)s.cg);
}

cudaError_t launch_wgrad_depthwise(const Plan& p, const Args& a) {
  const int in = p.sh.in_dt, out = p.sh.out_dt;
  if (in == CONV_BF16)
    return out == CONV_F32 ? launch_depthwise_t<__nv_bfloat16, float>(p, a)
                           : launch_depthwise_t<__nv_bfloat16, __nv_bfloat16>(p, a);
  return out == CONV_F32 ? launch_depthwise_t<__half, float>(p, a) : launch_depthwise_t<__half, __half>(p, a);
}

cudaError_t launch_wgrad_grouped(const Plan& p, const Args& a) {
  const int in = p.sh.in_dt, out = p.sh.out_dt;
  if (in == CONV_BF16)
    return out == CONV_F32 ? launch_grouped_t<__nv_bfloat16, float>(p, a)
                           : launch_grouped_t<__nv_bfloat16, __nv_bfloat16>(p, a);
  return out == CONV_F32 ? launch_grouped_t<__half, float>(p, a) : launch_grouped_t<__half, __half>(p, a);
}

}  // namespace cig
