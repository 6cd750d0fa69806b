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
// rows (n, ho); 16 warps. A step covers RB output rows at once. Rows come in
// with 16-byte global loads issued two steps ahead into registers, are
// widened ONCE to fp32 and stored in a shared ring (R + 2 RB - 1 input rows,
// padded with pw zero columns on each side; 2 RB dY rows), so the inner loop
// is only shared loads and packed FMAs (__ffma2_rn). Warp w < R*RB*WS owns
// filter row r = w % R, row q = (w / R) % RB of the step and part w / (R RB)
// of that output row. Lane l owns output channels c0 + 2l and c0 + 2l + 1:
//  - depthwise: per pixel one float2 of dY and one float2 of X (the same two
//    channels); S packed FMAs on a register window of S input pixels that
//    rotates without moves (the loop is unrolled by S);
//  - grouped: per pixel the dY pair (broadcast once into two register pairs)
//    and the group's Cg input channels as Cg/2 pairs; S*Cg packed FMAs.
// The filter-row-0 warps also sum db. One __syncthreads per step. At the end
// the warps of each filter row are added in warp order, and the slice's
// partial sums go to an fp32 slab ("feat(rocke): split-K forward
// implicit-GEMM convolution on gfx1250", "Two-stage split-K") or, with one
// slice, straight to dW / db.
#include "common.cuh"
#include "../kernel_entry.h"

namespace cig {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kCG = 64;            // channels per CTA
constexpr int kPix = kCG * 4;      // bytes per pixel in the fp32 ring
// 16-byte loads per thread per step (prefetch registers): fewer where the
// 8-channel groups need the registers for accumulators.
__host__ __device__ constexpr int load_slots(int cpg) { return cpg == 8 ? 2 : 4; }
constexpr int kMaxW = 256;
constexpr int kSmemLimit = 220 * 1024;

struct DirParams {
  int64_t N, H, W, C, Ho, Wo;
  int32_t R, ph, pw;
  int32_t RB;          // output rows per step
  int32_t WS;          // parts per output row
  int32_t XR;          // input rows in the ring: R + 2 RB - 1
  int64_t rows;        // N * Ho: the reduction blocks
  int64_t groups;      // C / 64: the tiles
  int32_t split;
  int32_t xrow_bytes;  // (W + 2 pw + 1) * 256
  int32_t dyrow_bytes; // Wo * 256
  int32_t row_items;   // 16-byte loads per output row: (W + Wo) * 8
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

// c + a * b on both halves of a register pair (one packed FP32 FMA).
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }

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
        for (int j = 0; j < S; ++j) acc.v[j][0][0] = fma2(d, win[(t + j) % S][0], acc.v[j][0][0]);
      } else {
        const float2 d0 = make_float2(d.x, d.x), d1 = make_float2(d.y, d.y);
#pragma unroll
        for (int j = 0; j < S; ++j)
#pragma unroll
          for (int c = 0; c < CP; ++c) {
            acc.v[j][0][c] = fma2(d0, win[(t + j) % S][c], acc.v[j][0][c]);
            acc.v[j][1][c] = fma2(d1, win[(t + j) % S][c], acc.v[j][1][c]);
          }
      }
      if (BIAS) bsum = __fadd2_rn(bsum, d);
      if (t + 1 < S || wo + S < wo_b) load_x(wo + t + S, win[t]);
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
        acc.v[j][0][0] = fma2(d, v[0], acc.v[j][0][0]);
      } else {
        const float2 d0 = make_float2(d.x, d.x), d1 = make_float2(d.y, d.y);
#pragma unroll
        for (int c = 0; c < CP; ++c) {
          acc.v[j][0][c] = fma2(d0, v[c], acc.v[j][0][c]);
          acc.v[j][1][c] = fma2(d1, v[c], acc.v[j][1][c]);
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
  constexpr int MI = load_slots(CPG);
  extern __shared__ __align__(16) uint8_t smem[];
  uint8_t* xring = smem;                                      // XR rows of (W + 2 pw + 1) pixels, fp32
  uint8_t* dyring = smem + (size_t)p.XR * p.xrow_bytes;       // 2 RB rows of Wo pixels, fp32
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32, tid = threadIdx.x;
  const int64_t g = blockIdx.x % p.groups;
  const int32_t sigma = (int32_t)(blockIdx.x / p.groups);
  const int64_t c0 = g * kCG;
  const int64_t row_b = slice_begin(p.rows, p.split, sigma), row_e = slice_begin(p.rows, p.split, sigma + 1);
  const bool compute = warp < p.R * p.RB * p.WS;
  const int r = warp % p.R, q = (warp / p.R) % p.RB, part = warp / (p.R * p.RB);
  const int wo_a = compute ? (int)((p.Wo * part) / p.WS) : 0;
  const int wo_b = compute ? (int)((p.Wo * (part + 1)) / p.WS) : 0;
  const bool bias_warp = compute && r == 0 && db != nullptr;
  const int x_items = (int)p.W * 8;

  for (int i = tid * 16; i < p.XR * p.xrow_bytes; i += kThreads * 16)
    *reinterpret_cast<uint4*>(xring + i) = make_uint4(0, 0, 0, 0);

  A acc;
#pragma unroll
  for (int j = 0; j < S; ++j)
#pragma unroll
    for (int ki = 0; ki < A::KI; ++ki)
#pragma unroll
      for (int c = 0; c < A::CP; ++c) acc.v[j][ki][c] = make_float2(0.f, 0.f);
  float2 bsum = make_float2(0.f, 0.f);

  auto xslot = [&](int64_t h) -> uint8_t* {
    return xring + (size_t)(((h % p.XR) + p.XR) % p.XR) * p.xrow_bytes + p.pw * kPix;
  };
  auto dyslot = [&](int64_t ho) -> uint8_t* { return dyring + (size_t)(ho % (2 * p.RB)) * p.dyrow_bytes; };
  auto widen_to = [&](uint8_t* dst, uint4 u) {
    const float2 a = unpack2<TI>(u.x), b = unpack2<TI>(u.y), c = unpack2<TI>(u.z), d = unpack2<TI>(u.w);
    reinterpret_cast<float4*>(dst)[0] = make_float4(a.x, a.y, b.x, b.y);
    reinterpret_cast<float4*>(dst)[1] = make_float4(c.x, c.y, d.x, d.y);
  };
  // The data a step brings in: for output rows ho0 .. ho0 + nr - 1, the input
  // rows that enter the window (ho - ph + R - 1) and the dY rows.
  auto fetch = [&](int64_t n, int64_t ho0, int nr, uint4* b) {
#pragma unroll
    for (int m = 0; m < MI; ++m) {
      const int i = tid + m * kThreads;
      b[m] = make_uint4(0, 0, 0, 0);
      const int qq = i / p.row_items, rem = i - qq * p.row_items;
      if (qq >= nr) continue;
      const int64_t ho = ho0 + qq;
      if (rem < x_items) {
        const int64_t h = ho - p.ph + p.R - 1;
        if (h >= 0 && h < p.H)
          b[m] = __ldg(reinterpret_cast<const uint4*>(x + ((n * p.H + h) * p.W + (rem >> 3)) * p.C + c0 + (rem & 7) * 8));
      } else {
        const int j = rem - x_items;
        b[m] = __ldg(reinterpret_cast<const uint4*>(dy + ((n * p.Ho + ho) * p.Wo + (j >> 3)) * p.C + c0 + (j & 7) * 8));
      }
    }
  };
  auto store = [&](int64_t ho0, int nr, const uint4* b) {
#pragma unroll
    for (int m = 0; m < MI; ++m) {
      const int i = tid + m * kThreads;
      const int qq = i / p.row_items, rem = i - qq * p.row_items;
      if (qq >= nr) continue;
      const int64_t ho = ho0 + qq;
      if (rem < x_items) widen_to(xslot(ho - p.ph + p.R - 1) + (rem >> 3) * kPix + (rem & 7) * 32, b[m]);
      else widen_to(dyslot(ho) + ((rem - x_items) >> 3) * kPix + ((rem - x_items) & 7) * 32, b[m]);
    }
  };

  uint4 bufA[MI], bufB[MI];
  for (int64_t row = row_b; row < row_e;) {
    const int64_t n = row / p.Ho;
    const int64_t ho_a = row % p.Ho;
    const int64_t ho_b = (n + 1) * p.Ho <= row_e ? p.Ho : row_e - n * p.Ho;
    auto rows_at = [&](int64_t ho0) -> int { return (int)(ho0 + p.RB <= ho_b ? p.RB : ho_b - ho0); };
    __syncthreads();  // the previous image's rows are no longer read
    // Prologue: the first R - 1 input rows of the window, straight to the ring.
    for (int rr = 0; rr + 1 < p.R; ++rr) {
      const int64_t h = ho_a - p.ph + rr;
      for (int i = tid; i < x_items; i += kThreads) {
        uint4 u = make_uint4(0, 0, 0, 0);
        if (h >= 0 && h < p.H)
          u = __ldg(reinterpret_cast<const uint4*>(x + ((n * p.H + h) * p.W + (i >> 3)) * p.C + c0 + (i & 7) * 8));
        widen_to(xslot(h) + (i >> 3) * kPix + (i & 7) * 32, u);
      }
    }
    fetch(n, ho_a, rows_at(ho_a), bufA);
    store(ho_a, rows_at(ho_a), bufA);
    if (ho_a + p.RB < ho_b) fetch(n, ho_a + p.RB, rows_at(ho_a + p.RB), bufB);
    if (ho_a + 2 * p.RB < ho_b) fetch(n, ho_a + 2 * p.RB, rows_at(ho_a + 2 * p.RB), bufA);
    // One step: rows ho0 .. ho0 + RB - 1. nxt holds step ho0 + RB on entry and is
    // refilled with step ho0 + 3 RB (the other buffer holds step ho0 + 2 RB).
    auto step = [&](int64_t ho0, uint4* nxt) {
      __syncthreads();  // this step's rows are in shared memory; the previous step is done
      const int64_t h1 = ho0 + p.RB, h3 = ho0 + 3 * p.RB;
      if (h1 < ho_b) store(h1, rows_at(h1), nxt);
      if (h3 < ho_b) fetch(n, h3, rows_at(h3), nxt);
      const int64_t ho = ho0 + q;
      if (compute && ho < ho_b) {
        const uint8_t* xr = xslot(ho - p.ph + r) - p.pw * kPix;
        const uint8_t* dr = dyslot(ho);
        if (bias_warp) row_pass<S, CPG, true>(xr, dr, wo_a, wo_b, lane, acc, bsum);
        else row_pass<S, CPG, false>(xr, dr, wo_a, wo_b, lane, acc, bsum);
      }
    };
    // Unrolled by two so each buffer is named at compile time (kept in registers).
    for (int64_t ho0 = ho_a; ho0 < ho_b; ho0 += 2 * p.RB) {
      step(ho0, bufB);
      if (ho0 + p.RB < ho_b) step(ho0 + p.RB, bufA);
    }
    row = n * p.Ho + ho_b;
  }

  signal_dependents();
  // Add the warps of each filter row in warp order, then store.
  constexpr int PER = S * A::KI * A::CP * 2 + 2;  // dW partials, then the db pair
  __syncthreads();
  float* red = reinterpret_cast<float*>(smem);
  const bool leader = compute && warp < p.R;
  if (compute && !leader) {
    float* dst = red + ((size_t)warp * 32 + lane) * PER;
    int o = 0;
#pragma unroll
    for (int j = 0; j < S; ++j)
#pragma unroll
      for (int ki = 0; ki < A::KI; ++ki)
#pragma unroll
        for (int c = 0; c < A::CP; ++c) {
          dst[o++] = acc.v[j][ki][c].x;
          dst[o++] = acc.v[j][ki][c].y;
        }
    dst[PER - 2] = bsum.x;
    dst[PER - 1] = bsum.y;
  }
  __syncthreads();
  if (!leader) return;
  for (int w = warp + p.R; w < p.R * p.RB * p.WS; w += p.R) {
    const float* src = red + ((size_t)w * 32 + lane) * PER;
    int o = 0;
#pragma unroll
    for (int j = 0; j < S; ++j)
#pragma unroll
      for (int ki = 0; ki < A::KI; ++ki)
#pragma unroll
        for (int c = 0; c < A::CP; ++c) {
          acc.v[j][ki][c].x += src[o++];
          acc.v[j][ki][c].y += src[o++];
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
  if (r == 0 && db) {
    if (ws_bias) {
      ws_bias[(int64_t)sigma * p.C + k] = bsum.x;
      ws_bias[(int64_t)sigma * p.C + k + 1] = bsum.y;
    } else {
      store_out(db + k, bsum.x);
      store_out(db + k + 1, bsum.y);
    }
  }
}

size_t smem_bytes(const DirParams& p, int S, int cpg) {
  const size_t ringb = (size_t)p.XR * p.xrow_bytes + 2 * (size_t)p.RB * p.dyrow_bytes;
  const int per = S * (cpg == 1 ? 2 : 2 * cpg) + 2;
  const size_t red = (size_t)(p.R * p.RB * p.WS) * 32 * per * 4;
  return ringb > red ? ringb : red;
}

// Rows per step: as many as the warps, the shared-memory budget and the
// per-thread load slots allow.
DirParams make_params(const Shape& s, int32_t split, int cpg) {
  DirParams p;
  p.N = s.n; p.H = s.h; p.W = s.w; p.C = s.c; p.Ho = s.ho; p.Wo = s.wo;
  p.R = (int32_t)s.r; p.ph = (int32_t)s.ph; p.pw = (int32_t)s.pw;
  p.rows = s.n * s.ho;
  p.groups = s.c / kCG;
  p.split = split;
  p.xrow_bytes = (int32_t)((s.w + 2 * s.pw + 1) * kPix);
  p.dyrow_bytes = (int32_t)(s.wo * kPix);
  p.row_items = (int32_t)((s.w + s.wo) * 8);
  p.RB = 1;
  for (int rb = kWarps / p.R; rb >= 1; --rb) {
    DirParams t = p;
    t.RB = rb;
    t.WS = kWarps / (p.R * rb);
    t.XR = p.R + 2 * rb - 1;
    if ((int64_t)rb * p.row_items <= (int64_t)load_slots(cpg) * kThreads && smem_bytes(t, (int)s.s, cpg) <= kSmemLimit) {
      p.RB = rb;
      break;
    }
  }
  p.WS = kWarps / (p.R * p.RB);
  p.XR = p.R + 2 * p.RB - 1;
  return p;
}

// Shapes both kernels share: stride 1, dilation 1, 16-bit inputs, whole
// 64-channel CTAs, rows that fit the ring and the per-thread load slots.
bool common_ok(const Shape& s, int cpg) {
  if (s.in_dt == CONV_F32 || s.sh != 1 || s.sw != 1 || s.dh != 1 || s.dw != 1 || s.n < 1) return false;
  if (s.c % kCG != 0 || s.c != s.k || s.r > kWarps || s.w > kMaxW) return false;
  if (s.pw > s.s || s.ph > s.r) return false;
  if ((s.w + s.wo) * 8 > (int64_t)load_slots(cpg) * kThreads) return false;
  const DirParams p = make_params(s, 1, cpg);
  return smem_bytes(p, (int)s.s, cpg) <= kSmemLimit;
}

template <typename TI, typename TO, int S, int CPG>
cudaError_t launch_s(const Plan& pl, const Args& a) {
  const DirParams p = make_params(pl.sh, pl.split, CPG);
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

Geometry direct_geometry(const Shape& s) {
  Geometry g;
  g.ok = true;
  g.ctas_per_sm = 1;
  g.tiles = s.c / kCG;
  g.blocks = s.n * s.ho;
  return g;
}

}  // namespace

// The TMA-ring, register-tap form (dw_wgrad_ring.cu) the depthwise kernel
// takes for square 3/5/7 filters.
Geometry geometry_wgrad_depthwise_ring(const Shape& s);
cudaError_t launch_wgrad_depthwise_ring(const Plan& p, const Args& a);

Geometry geometry_wgrad_depthwise(const Shape& s) {
  const Geometry reg = geometry_wgrad_depthwise_ring(s);  // square 3/5/7 filters: TMA row rings, taps in registers
  if (reg.ok) return reg;
  const bool depthwise = s.groups == s.c && s.groups == s.k;
  if (!depthwise || !common_ok(s, 1)) return Geometry{};
  if (!(s.s == 3 || s.s == 5 || s.s == 7 || s.s == 9 || s.s == 11)) return Geometry{};
  return direct_geometry(s);
}

Geometry geometry_wgrad_grouped(const Shape& s) {
  if (!(s.cg == 4 || s.cg == 8) || s.kg != s.cg || !common_ok(s, (int)s.cg)) return Geometry{};
  if (!(s.s == 1 || s.s == 3 || (s.s == 5 && s.cg == 4))) return Geometry{};
  return direct_geometry(s);
}

cudaError_t launch_wgrad_depthwise(const Plan& p, const Args& a) {
  if (geometry_wgrad_depthwise_ring(p.sh).ok) return launch_wgrad_depthwise_ring(p, a);
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
