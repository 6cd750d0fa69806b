// Grouped weight gradient with 4 or 8 channels per group (Cg = Kg) on CUDA
// cores:
//
//   dW[k, r, s, c] = sum over (n, ho, wo) of dY[n, ho, wo, k] * X[n, ho + r - ph, wo + s - pw, g Cg + c],
//   g = k / Kg,   db[k] = sum of dY[n, ho, wo, k]
//
// ("perf(rocke): depthwise 7x7 and grouped cpg4/8 wgrad on batched mfma
// 4x4x4", "Technical Details"; stride 1, dilation 1). Each group is an
// 8 x 72 (or 4 x 36) contraction over N*Ho*Wo: too narrow for a tensor-core
// tile, FP32-FMA bound at 18-36 flop per byte.
//
// CTA: 64 channels (= 64/Cg whole groups, since Cg = Kg and C = K here) and
// one slice of the output rows (n, ho). Lane l owns output channels
// c0 + 2l, c0 + 2l + 1 (one group); warp w < R*WS owns filter row r = w % R
// and part w / R of each output row (WS = 8 / R parts). Per output pixel a
// lane loads its dY pair (broadcast once into two register pairs) and, per
// filter tap, its group's Cg input channels as Cg/2 register pairs (one 8- or
// 16-byte load shared by the group's lanes), then does S*Cg packed FMAs
// (__ffma2_rn). Rows stream into a shared-memory ring by cp.async exactly as
// in the depthwise kernel. db is summed by the filter-row-0 warps. Partial
// sums per slice go to an fp32 slab ("feat(rocke): split-K forward
// implicit-GEMM convolution on gfx1250", "Two-stage split-K").
#include "common.cuh"

namespace cig {
namespace {

constexpr int kThreads = 256;
constexpr int kCG = 64;          // channels per CTA
constexpr int kPix = kCG * 2;    // bytes per pixel of one 16-bit channel group
constexpr int kPref = 2;
constexpr int kMaxW = 256;

struct GrpParams {
  int64_t N, H, W, C, Ho, Wo;
  int32_t R, ph, pw;
  int32_t WS;          // wo parts per filter row
  int64_t rows;        // N * Ho: the reduction blocks
  int64_t groups;      // C / 64: the tiles
  int32_t split;
  int32_t ring;
  int32_t xrow_bytes;
  int32_t dyrow_bytes;
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

// CPG 16-bit values at p (8 or 16 bytes) -> CPG/2 float pairs.
template <typename TI, int CPG>
__device__ __forceinline__ void load_group(const uint8_t* p, float2* v) {
  if constexpr (CPG == 8) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    v[0] = unpack2<TI>(u.x); v[1] = unpack2<TI>(u.y); v[2] = unpack2<TI>(u.z); v[3] = unpack2<TI>(u.w);
  } else {
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    v[0] = unpack2<TI>(u.x); v[1] = unpack2<TI>(u.y);
  }
}

// acc[j][ki][cp] : (dW[k0+ki][r][j][2cp], dW[k0+ki][r][j][2cp+1]) partial sums.
template <int S, int CPG>
struct Acc {
  float2 v[S][2][CPG / 2];
};

// Output pixels [wo_a, wo_b) of one row for one filter row.
template <typename TI, int S, int CPG, bool BIAS>
__device__ __forceinline__ void row_pass(const uint8_t* xrow, const uint8_t* dyrow, int wo_a, int wo_b, int lane,
                                         Acc<S, CPG>& acc, float2& bsum) {
  constexpr int CP = CPG / 2;
  const int gb = ((2 * lane) / CPG) * CPG;  // first channel of this lane's group within the CTA's 64
  const uint8_t* xp = xrow + gb * 2;
  const uint8_t* dp = dyrow + lane * 4;
  float2 win[S][CP];
#pragma unroll
  for (int j = 0; j < S; ++j) load_group<TI, CPG>(xp + (wo_a + j) * kPix, win[j]);
  int wo = wo_a;
  for (; wo + S <= wo_b; wo += S) {
#pragma unroll
    for (int t = 0; t < S; ++t) {
      const float2 d = unpack2<TI>(*reinterpret_cast<const uint32_t*>(dp + (wo + t) * kPix));
      const float2 d0 = make_float2(d.x, d.x), d1 = make_float2(d.y, d.y);
#pragma unroll
      for (int j = 0; j < S; ++j)
#pragma unroll
        for (int c = 0; c < CP; ++c) {
          acc.v[j][0][c] = __ffma2_rn(d0, win[(t + j) % S][c], acc.v[j][0][c]);
          acc.v[j][1][c] = __ffma2_rn(d1, win[(t + j) % S][c], acc.v[j][1][c]);
        }
      if (BIAS) bsum = __fadd2_rn(bsum, d);
      load_group<TI, CPG>(xp + (wo + t + S) * kPix, win[t]);
    }
  }
  for (; wo < wo_b; ++wo) {
    const float2 d = unpack2<TI>(*reinterpret_cast<const uint32_t*>(dp + wo * kPix));
    const float2 d0 = make_float2(d.x, d.x), d1 = make_float2(d.y, d.y);
    if (BIAS) bsum = __fadd2_rn(bsum, d);
#pragma unroll
    for (int j = 0; j < S; ++j) {
      float2 v[CP];
      load_group<TI, CPG>(xp + (wo + j) * kPix, v);
#pragma unroll
      for (int c = 0; c < CP; ++c) {
        acc.v[j][0][c] = __ffma2_rn(d0, v[c], acc.v[j][0][c]);
        acc.v[j][1][c] = __ffma2_rn(d1, v[c], acc.v[j][1][c]);
      }
    }
  }
}

template <typename TI, typename TO, int S, int CPG>
__global__ void __launch_bounds__(kThreads, 2)
    grp_wgrad_kernel(const TI* __restrict__ x, const TI* __restrict__ dy, TO* out, float* ws, TO* db,
                     float* ws_bias, GrpParams p) {
  constexpr int CP = CPG / 2;
  extern __shared__ __align__(16) uint8_t smem[];
  uint8_t* xring = smem;
  uint8_t* dyring = smem + (size_t)p.ring * p.xrow_bytes;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32, tid = threadIdx.x;
  const int64_t g = blockIdx.x % p.groups;
  const int32_t sigma = (int32_t)(blockIdx.x / p.groups);
  const int64_t c0 = g * kCG;
  const int64_t row_b = slice_begin(p.rows, p.split, sigma), row_e = slice_begin(p.rows, p.split, sigma + 1);
  const bool compute = warp < p.R * p.WS;
  const int r = warp % p.R, part = warp / p.R;
  const int wo_a = (int)((p.Wo * part) / p.WS), wo_b = (int)((p.Wo * (part + 1)) / p.WS);
  const bool bias_warp = compute && r == 0 && db != nullptr;

  for (int i = tid * 16; i < p.ring * p.xrow_bytes; i += kThreads * 16)
    *reinterpret_cast<uint4*>(xring + i) = make_uint4(0, 0, 0, 0);
  __syncthreads();

  Acc<S, CPG> acc;
#pragma unroll
  for (int j = 0; j < S; ++j)
#pragma unroll
    for (int c = 0; c < CP; ++c) acc.v[j][0][c] = acc.v[j][1][c] = make_float2(0.f, 0.f);
  float2 bsum = make_float2(0.f, 0.f);

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

  for (int64_t row = row_b; row < row_e;) {
    const int64_t n = row / p.Ho;
    const int64_t ho_a = row % p.Ho;
    const int64_t ho_b = (n + 1) * p.Ho <= row_e ? p.Ho : row_e - n * p.Ho;
    __syncthreads();
    for (int rr = 0; rr + 1 < p.R; ++rr) load_x(n, ho_a - p.ph + rr);
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
      if (compute) {
        const int64_t h = ho - p.ph + r;
        const uint8_t* xr = xring + (size_t)(((h % p.ring) + p.ring) % p.ring) * p.xrow_bytes;
        const uint8_t* dr = dyring + (size_t)(ho % (kPref + 1)) * p.dyrow_bytes;
        if (bias_warp) row_pass<TI, S, CPG, true>(xr, dr, wo_a, wo_b, lane, acc, bsum);
        else row_pass<TI, S, CPG, false>(xr, dr, wo_a, wo_b, lane, acc, bsum);
      }
    }
    cp_async_wait<0>();
    row = n * p.Ho + ho_b;
  }

  // Combine the WS parts of each filter row in part order, then store.
  __syncthreads();
  float* red = reinterpret_cast<float*>(smem);  // [R*WS warps][32 lanes][PER]
  constexpr int PER = S * CPG * 2 + 2;           // dW partials, then the db pair
  if (compute && part > 0) {
    float* dst = red + ((size_t)warp * 32 + lane) * PER;
#pragma unroll
    for (int j = 0; j < S; ++j)
#pragma unroll
      for (int ki = 0; ki < 2; ++ki)
#pragma unroll
        for (int c = 0; c < CP; ++c) {
          dst[((j * 2 + ki) * CP + c) * 2] = acc.v[j][ki][c].x;
          dst[((j * 2 + ki) * CP + c) * 2 + 1] = acc.v[j][ki][c].y;
        }
    dst[PER - 2] = bsum.x;
    dst[PER - 1] = bsum.y;
  }
  __syncthreads();
  if (compute && part == 0) {
    for (int q = 1; q < p.WS; ++q) {
      const float* src = red + ((size_t)(q * p.R + r) * 32 + lane) * PER;
#pragma unroll
      for (int j = 0; j < S; ++j)
#pragma unroll
        for (int ki = 0; ki < 2; ++ki)
#pragma unroll
          for (int c = 0; c < CP; ++c) {
            acc.v[j][ki][c].x += src[((j * 2 + ki) * CP + c) * 2];
            acc.v[j][ki][c].y += src[((j * 2 + ki) * CP + c) * 2 + 1];
          }
      bsum.x += src[PER - 2];
      bsum.y += src[PER - 1];
    }
    const int64_t E = p.C * p.R * S * CPG;
#pragma unroll
    for (int ki = 0; ki < 2; ++ki) {
      const int64_t k = c0 + 2 * lane + ki;
#pragma unroll
      for (int j = 0; j < S; ++j)
#pragma unroll
        for (int c = 0; c < CP; ++c) {
          const int64_t e = ((k * p.R + r) * S + j) * CPG + 2 * c;  // dW[k][r][s][2c], then 2c+1
          if (ws) {
            ws[(int64_t)sigma * E + e] = acc.v[j][ki][c].x;
            ws[(int64_t)sigma * E + e + 1] = acc.v[j][ki][c].y;
          } else {
            store_out(out + e, acc.v[j][ki][c].x);
            store_out(out + e + 1, acc.v[j][ki][c].y);
          }
        }
    }
    if (bias_warp) {
      const int64_t k = c0 + 2 * lane;
      if (ws_bias) {
        ws_bias[(int64_t)sigma * p.C + k] = bsum.x;
        ws_bias[(int64_t)sigma * p.C + k + 1] = bsum.y;
      } else {
        store_out(db + k, bsum.x);
        store_out(db + k + 1, bsum.y);
      }
    }
  }
}

GrpParams make_params(const Plan& pl) {
  const Shape& s = pl.sh;
  GrpParams p;
  p.N = s.n; p.H = s.h; p.W = s.w; p.C = s.c; p.Ho = s.ho; p.Wo = s.wo;
  p.R = (int32_t)s.r; p.ph = (int32_t)s.ph; p.pw = (int32_t)s.pw;
  p.WS = 8 / p.R;
  p.rows = s.n * s.ho;
  p.groups = s.c / kCG;
  p.split = pl.split;
  p.ring = p.R + kPref;
  p.xrow_bytes = (int32_t)((s.w + 2 * s.pw + s.s) * kPix);
  p.dyrow_bytes = (int32_t)(s.wo * kPix);
  return p;
}

size_t smem_bytes(const GrpParams& p, int S, int cpg) {
  const size_t ring = (size_t)p.ring * p.xrow_bytes + (size_t)(kPref + 1) * p.dyrow_bytes;
  const size_t red = (size_t)(p.R * p.WS) * 32 * (S * cpg * 2 + 2) * 4;
  return ring > red ? ring : red;
}

template <typename TI, typename TO, int S, int CPG>
cudaError_t launch_s(const Plan& pl, const Args& a) {
  const GrpParams p = make_params(pl);
  const size_t smem = smem_bytes(p, S, CPG);
  cudaError_t err = cudaFuncSetAttribute(grp_wgrad_kernel<TI, TO, S, CPG>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  const int64_t ctas = p.groups * p.split;
  if (ctas > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  grp_wgrad_kernel<TI, TO, S, CPG><<<(unsigned)ctas, kThreads, smem, a.stream>>>(
      static_cast<const TI*>(a.x), static_cast<const TI*>(a.b), static_cast<TO*>(a.out), a.ws,
      pl.with_bias ? static_cast<TO*>(a.db) : nullptr, a.ws_bias, p);
  return cudaGetLastError();
}

template <typename TI, typename TO>
cudaError_t launch_t(const Plan& pl, const Args& a) {
  const int cpg = (int)pl.sh.cg;
  switch (pl.sh.s * 16 + cpg) {
    case 1 * 16 + 4: return launch_s<TI, TO, 1, 4>(pl, a);
    case 1 * 16 + 8: return launch_s<TI, TO, 1, 8>(pl, a);
    case 3 * 16 + 4: return launch_s<TI, TO, 3, 4>(pl, a);
    case 3 * 16 + 8: return launch_s<TI, TO, 3, 8>(pl, a);
    case 5 * 16 + 4: return launch_s<TI, TO, 5, 4>(pl, a);
    default: return cudaErrorNotSupported;
  }
}

}  // namespace

Geometry geometry_wgrad_grouped(const Shape& s) {
  Geometry g;
  if (s.in_dt == CONV_F32 || s.sh != 1 || s.sw != 1 || s.dh != 1 || s.dw != 1 || s.n < 1) return g;
  if (!(s.cg == 4 || s.cg == 8) || s.kg != s.cg || s.c != s.k) return g;
  if (s.c % kCG != 0 || s.r > 8 || s.w > kMaxW) return g;
  if (!(s.s == 1 || s.s == 3 || (s.s == 5 && s.cg == 4)) || s.pw > s.s || s.ph > s.r) return g;
  GrpParams p;
  p.R = (int32_t)s.r;
  p.WS = 8 / p.R;
  p.ring = p.R + kPref;
  p.xrow_bytes = (int32_t)((s.w + 2 * s.pw + s.s) * kPix);
  p.dyrow_bytes = (int32_t)(s.wo * kPix);
  if (smem_bytes(p, (int)s.s, (int)s.cg) > 110 * 1024) return g;
  g.ok = true;
  g.ctas_per_sm = 2;
  g.tiles = s.c / kCG;
  g.blocks = s.n * s.ho;
  return g;
}

cudaError_t launch_wgrad_grouped(const Plan& p, const Args& a) {
  const int in = p.sh.in_dt, out = p.sh.out_dt;
  if (in == CONV_BF16)
    return out == CONV_F32 ? launch_t<__nv_bfloat16, float>(p, a) : launch_t<__nv_bfloat16, __nv_bfloat16>(p, a);
  return out == CONV_F32 ? launch_t<__half, float>(p, a) : launch_t<__half, __half>(p, a);
}

}  // namespace cig
