// fp32 convolutions as implicit GEMMs on the CUDA cores (FFMA tiles), for
// every direction: the forward, the data gradient at stride 1 (the forward on
// the turned problem, the filter read in place), and the weight gradient
// (+ bias gradient), each with deterministic two-stage split-K. Every product
// is one fp32 FMA, so the result carries only fp32 accumulation rounding.
//
// GEMM views (one group; C, K multiples of 4):
//   forward   Y[p][k]        = sum over (r, s, c) of X[p shifted by (r, s)][c] * W[k][r][s][c]
//   data grad dX[p][c]       = sum over (r', s', k) of dY[p shifted][k] * W[k][R-1-r'][S-1-s'][c]
//   weight    dW[k][r][s][c] = sum over p of dY[p][k] * X[p shifted by (r, s)][c]
// ("ROCm/rocm-libraries PR #11188", "Motivation": the NHWC implicit-GEMM
// convolution; "feat(rocke): split-K forward implicit-GEMM convolution on
// gfx1250", "Two-stage split-K".) A CTA computes a 128 x 128 tile (the weight
// gradient: of one tap) over a split-K slice of 16-deep reduction steps;
// both operands are staged in shared memory as [reduction][128] rows (the
// im2col gather and the zero padding done by the loads), double-buffered
// through registers, and each thread accumulates an 8 x 8 block with
// float4 shared loads (16 FMAs per load).
#include "common.cuh"
#include "../kernel_entry.h"

namespace cig {
namespace {

constexpr int kThreads = 256;
constexpr int kT = 128;      // tile rows and columns
constexpr int kBK = 16;      // reduction elements a step
constexpr int kLD = kT + 4;  // shared row stride (floats)
constexpr int kCtasPerSm = 2;  // 2 x 256 threads x 128 registers fill the register file

enum { kFwd = 0, kDgrad = 1, kWgrad = 2 };

// Division of n < 2^31 by a divisor d in [1, 2^31] fixed at launch, as a
// multiply-high and a shift (Granlund and Montgomery, "Division by Invariant
// Integers using Multiplication", 1994, section 4): with l = ceil(log2 d) and
// m = floor(2^32 (2^l - d) / d) + 1, floor(n / d) = (mulhi(m, n) + n) >> l;
// n < 2^31 keeps the sum inside 32 bits.
struct DivU32 {
  uint32_t d = 1, m = 1, l = 0;
  DivU32() = default;
  explicit DivU32(uint32_t dv) : d(dv) {
    while ((1ull << l) < dv) ++l;
    m = (uint32_t)((((1ull << 32) * ((1ull << l) - dv)) / dv) + 1);
  }
  __host__ __device__ __forceinline__ uint32_t div(uint32_t n) const {
#ifdef __CUDA_ARCH__
    return (__umulhi(m, n) + n) >> l;
#else
    return (uint32_t)((((uint64_t)m * n) >> 32) + n) >> l;
#endif
  }
};

struct FfParams {
  const float* a;  // forward: X; data gradient: dY; weight gradient: dY
  const float* b;  // forward and data gradient: W; weight gradient: X
  float* out;
  float* ws;
  float* db;
  float* ws_bias;
  int64_t M, N;        // GEMM extents (weight gradient: M = K output channels, N = C input channels)
  int64_t tiles_m, tiles_n;
  int64_t blocks;      // reduction steps
  int64_t E;           // output elements (the slab stride)
  int64_t P;           // weight gradient: output pixels
  // the forward-form problem: input [N][H][W][C], output [N][Ho][Wo][K], filter R x S
  int64_t H, W, C, Ho, Wo, K;
  int32_t R, S, sh, sw, ph, pw, dh, dw;
  DivU32 div_wo, div_ho;  // weight gradient: pixel -> (n, ho, wo)
  int32_t cblocks;     // ceil(C / 16) (forward, data gradient)
  int32_t split;
  // fused forward epilogue (unsplit only): y = min(max(acc + bias[k], ep_lo), ep_hi)
  const float* ep_bias;
  float ep_lo, ep_hi;
  int32_t ep;
};

// One operand tile's loads for a step: 2 float4 a thread, staged in registers.
struct Stage {
  float4 v[2];
};

template <int DIR>
__global__ void __launch_bounds__(kThreads, kCtasPerSm) ffma_igemm_kernel(FfParams fp) {
  __shared__ __align__(16) float As[2][kBK][kLD];
  __shared__ __align__(16) float Bs[2][kBK][kLD];
  const int t = threadIdx.x;
  const int taps = fp.R * fp.S;
  // CTA -> (tile, slice); the weight gradient's tiles also run over the taps
  int64_t tile = blockIdx.x;
  const int64_t ntiles = fp.tiles_m * fp.tiles_n * (DIR == kWgrad ? taps : 1);
  const int32_t sigma = (int32_t)(tile / ntiles);
  tile %= ntiles;
  const int32_t tap = DIR == kWgrad ? (int32_t)(tile % taps) : 0;
  if (DIR == kWgrad) tile /= taps;
  const int64_t m0 = (tile / fp.tiles_n) * kT, n0 = (tile % fp.tiles_n) * kT;
  const int64_t b0 = slice_begin(fp.blocks, fp.split, sigma), b1 = slice_begin(fp.blocks, fp.split, sigma + 1);
  const int32_t tr = tap / fp.S, ts = tap % fp.S;

  // Loads. Forward / data gradient A: pixel rows m0 + t / 4 (+ 64), 4 channels at 4 (t % 4) of the
  // step (transposed into As). B: forward W rows n0 + t / 4 (+ 64), 4 channels (transposed); data
  // gradient: W[k][tap'][c] for step row t / 32 (+ 8), columns n0 + 4 (t % 32) (straight).
  // Weight gradient A: dY pixel t / 32 (+ 8) of the step, channels m0 + 4 (t % 32) (straight); B: X at
  // that pixel shifted by the tap, channels n0 + 4 (t % 32) (straight).
  // Spatial index arithmetic runs in 32 bits (the host admits only shapes where it cannot overflow).
  int32_t pn[2], pho[2], pwo[2];  // forward / data gradient: the forward-form pixels of this thread's A rows
  bool pok[2];
  if (DIR != kWgrad) {
    for (int i = 0; i < 2; ++i) {
      const int64_t m = m0 + t / 4 + 64 * i;
      pok[i] = m < fp.M;
      const int64_t mm = pok[i] ? m : 0;
      pwo[i] = (int32_t)(mm % fp.Wo);
      pho[i] = (int32_t)((mm / fp.Wo) % fp.Ho);
      pn[i] = (int32_t)(mm / (fp.Wo * fp.Ho));
    }
  }
  const float4 zero4 = make_float4(0.f, 0.f, 0.f, 0.f);

  auto load_step = [&](int64_t blk, Stage& sa, Stage& sb) {
    if (DIR != kWgrad) {
      const int32_t rs = (int32_t)(blk / fp.cblocks);
      const int64_t c0 = (blk % fp.cblocks) * kBK;
      const int32_t r = rs / fp.S, s = rs % fp.S;
      const int64_t c = c0 + 4 * (t % 4);
      for (int i = 0; i < 2; ++i) {
        const int32_t hi = pho[i] * fp.sh + r * fp.dh - fp.ph, wi = pwo[i] * fp.sw + s * fp.dw - fp.pw;
        const bool in = pok[i] && c < fp.C && hi >= 0 && hi < fp.H && wi >= 0 && wi < fp.W;
        sa.v[i] = in ? *reinterpret_cast<const float4*>(fp.a + ((pn[i] * fp.H + hi) * fp.W + wi) * fp.C + c) : zero4;
      }
      if (DIR == kFwd) {
        for (int i = 0; i < 2; ++i) {
          const int64_t k = n0 + t / 4 + 64 * i;
          sb.v[i] = k < fp.N && c < fp.C ? *reinterpret_cast<const float4*>(fp.b + (k * taps + rs) * fp.C + c) : zero4;
        }
      } else {  // W'[c][tap'][k] = W[k][taps - 1 - tap'][c]: row k = c0 + t / 32 (+ 8), columns c
        const int64_t cc = n0 + 4 * (t % 32);
        for (int i = 0; i < 2; ++i) {
          const int64_t k = c0 + t / 32 + 8 * i;
          sb.v[i] = k < fp.C && cc < fp.N
                        ? *reinterpret_cast<const float4*>(fp.b + (k * taps + (taps - 1 - rs)) * fp.N + cc)
                        : zero4;
        }
      }
    } else {
      const int64_t k = m0 + 4 * (t % 32), c = n0 + 4 * (t % 32);
      for (int i = 0; i < 2; ++i) {
        // pixel p of the step -> (n, ho, wo), no state kept across steps
        const uint32_t p = (uint32_t)blk * kBK + t / 32 + 8 * i;
        const bool pin = p < (uint32_t)fp.P;
        sa.v[i] = pin && k < fp.M ? *reinterpret_cast<const float4*>(fp.a + (int64_t)p * fp.K + k) : zero4;
        const uint32_t q = fp.div_wo.div(p), n = fp.div_ho.div(q);
        const int32_t wo = (int32_t)(p - q * fp.div_wo.d), ho = (int32_t)(q - n * fp.div_ho.d);
        const int32_t hi = ho * fp.sh + tr * fp.dh - fp.ph, wi = wo * fp.sw + ts * fp.dw - fp.pw;
        const bool in = pin && c < fp.N && hi >= 0 && hi < fp.H && wi >= 0 && wi < fp.W;
        sb.v[i] = in ? *reinterpret_cast<const float4*>(fp.b + (((int64_t)n * fp.H + hi) * fp.W + wi) * fp.C + c)
                     : zero4;
      }
    }
  };
  auto store_step = [&](int buf, const Stage& sa, const Stage& sb) {
    if (DIR != kWgrad) {  // A transposed: As[reduction][pixel]
      for (int i = 0; i < 2; ++i) {
        const int m = t / 4 + 64 * i, k = 4 * (t % 4);
        As[buf][k][m] = sa.v[i].x;
        As[buf][k + 1][m] = sa.v[i].y;
        As[buf][k + 2][m] = sa.v[i].z;
        As[buf][k + 3][m] = sa.v[i].w;
      }
    } else {
      for (int i = 0; i < 2; ++i) *reinterpret_cast<float4*>(&As[buf][t / 32 + 8 * i][4 * (t % 32)]) = sa.v[i];
    }
    if (DIR == kFwd) {  // B transposed: Bs[reduction][output channel]
      for (int i = 0; i < 2; ++i) {
        const int n = t / 4 + 64 * i, k = 4 * (t % 4);
        Bs[buf][k][n] = sb.v[i].x;
        Bs[buf][k + 1][n] = sb.v[i].y;
        Bs[buf][k + 2][n] = sb.v[i].z;
        Bs[buf][k + 3][n] = sb.v[i].w;
      }
    } else {
      for (int i = 0; i < 2; ++i) *reinterpret_cast<float4*>(&Bs[buf][t / 32 + 8 * i][4 * (t % 32)]) = sb.v[i];
    }
  };

  // this thread's 8 x 8 block: rows ty*4 + (0..3) and 64 + ty*4 + (0..3), columns likewise with tx
  const int ty = t / 16, tx = t % 16;
  float acc[8][8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
  // bias gradient (weight gradient, the CTAs of tap 0 and input-channel tile 0): thread t < 128 sums
  // output channel m0 + t over the steps' pixels, in step order
  const bool do_bias = DIR == kWgrad && (fp.db || fp.ws_bias) && tap == 0 && n0 == 0;
  float bsum = 0.f;

  Stage sa, sb;
  if (b0 < b1) {
    load_step(b0, sa, sb);
    store_step(0, sa, sb);
  }
  __syncthreads();
  int buf = 0;
  for (int64_t blk = b0; blk < b1; ++blk) {
    const bool more = blk + 1 < b1;
    if (more) load_step(blk + 1, sa, sb);  // in flight while this step computes
#pragma unroll
    for (int kk = 0; kk < kBK; ++kk) {
      const float4 a0 = *reinterpret_cast<const float4*>(&As[buf][kk][ty * 4]);
      const float4 a1 = *reinterpret_cast<const float4*>(&As[buf][kk][64 + ty * 4]);
      const float4 bb0 = *reinterpret_cast<const float4*>(&Bs[buf][kk][tx * 4]);
      const float4 bb1 = *reinterpret_cast<const float4*>(&Bs[buf][kk][64 + tx * 4]);
      const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      const float bv[8] = {bb0.x, bb0.y, bb0.z, bb0.w, bb1.x, bb1.y, bb1.z, bb1.w};
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    if (do_bias && t < kT) {
#pragma unroll
      for (int kk = 0; kk < kBK; ++kk) bsum += As[buf][kk][t];
    }
    if (more) store_step(buf ^ 1, sa, sb);
    __syncthreads();
    buf ^= 1;
  }
  signal_dependents();

  // Store: row m, four columns n at a time (N % 4 == 0), into the output or slab sigma.
  float* dst = fp.ws ? fp.ws + (int64_t)sigma * fp.E : fp.out;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int64_t m = m0 + (i < 4 ? ty * 4 + i : 64 + ty * 4 + (i - 4));
    if (m >= fp.M) continue;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int64_t n = n0 + h * 64 + tx * 4;
      if (n >= fp.N) continue;
      const int64_t row = DIR == kWgrad ? (m * taps + tap) * fp.N : m * fp.N;
      float4 v = make_float4(acc[i][4 * h], acc[i][4 * h + 1], acc[i][4 * h + 2], acc[i][4 * h + 3]);
      if (DIR == kFwd && fp.ep) {  // bias + clamp on the fp32 sum (the forward runs unsplit then)
        const float4 b = fp.ep_bias ? make_float4(fp.ep_bias[n], fp.ep_bias[n + 1], fp.ep_bias[n + 2], fp.ep_bias[n + 3])
                                    : make_float4(0.f, 0.f, 0.f, 0.f);
        v.x = fminf(fmaxf(v.x + b.x, fp.ep_lo), fp.ep_hi);
        v.y = fminf(fmaxf(v.y + b.y, fp.ep_lo), fp.ep_hi);
        v.z = fminf(fmaxf(v.z + b.z, fp.ep_lo), fp.ep_hi);
        v.w = fminf(fmaxf(v.w + b.w, fp.ep_lo), fp.ep_hi);
      }
      *reinterpret_cast<float4*>(dst + row + n) = v;
    }
  }
  if (do_bias && t < kT && m0 + t < fp.M) {
    if (fp.ws_bias) fp.ws_bias[(int64_t)sigma * fp.M + m0 + t] = bsum;
    else fp.db[m0 + t] = bsum;
  }
}

bool admissible(const Shape& s, conv_dir dir) {
  if (s.in_dt != CONV_F32 || s.out_dt != CONV_F32 || s.groups != 1 || s.n < 1) return false;
  if (s.c % 4 != 0 || s.k % 4 != 0) return false;  // 16-byte channel groups
  if (dir == CONV_DIR_DGRAD && (s.sh != 1 || s.sw != 1 || s.ph > s.dh * (s.r - 1) || s.pw > s.dw * (s.s - 1)))
    return false;
  if (s.r * s.s > 0x7fffffffLL || (s.c + kBK - 1) / kBK * s.r * s.s > 0x7fffffffLL) return false;
  // The kernel's spatial index arithmetic is 32-bit: in the forward form, hi = ho*sh + r*dh - ph
  // lies in [-ph, H + ph), so H + 2 ph (and likewise W + 2 pw) and the image count must stay below
  // 2^31; the weight gradient's pixel index (up to P + 15) too.
  const Shape f = dir == CONV_DIR_DGRAD ? dgrad_as_forward(s) : s;
  const int64_t lim = 0x7fffffffLL;
  if (f.n >= lim || f.h + 2 * f.ph >= lim || f.w + 2 * f.pw >= lim) return false;
  if (dir == CONV_DIR_WGRAD && s.n * s.ho * s.wo + kBK >= lim) return false;
  return true;
}

// The GEMM extents and reduction steps of a direction.
void extents(const Shape& s, conv_dir dir, int64_t* M, int64_t* N, int64_t* blocks, int64_t* tiles) {
  if (dir == CONV_DIR_FWD) {
    *M = s.n * s.ho * s.wo;
    *N = s.k;
    *blocks = s.r * s.s * ((s.c + kBK - 1) / kBK);
  } else if (dir == CONV_DIR_DGRAD) {
    *M = s.n * s.h * s.w;
    *N = s.c;
    *blocks = s.r * s.s * ((s.k + kBK - 1) / kBK);
  } else {
    *M = s.k;
    *N = s.c;
    *blocks = (s.n * s.ho * s.wo + kBK - 1) / kBK;
  }
  *tiles = ((*M + kT - 1) / kT) * ((*N + kT - 1) / kT) * (dir == CONV_DIR_WGRAD ? s.r * s.s : 1);
}

}  // namespace

Geometry geometry_ffma(const Shape& s, conv_dir dir) {
  Geometry g;
  if (!admissible(s, dir)) return g;
  int64_t M, N, blocks, tiles;
  extents(s, dir, &M, &N, &blocks, &tiles);
  g.ok = true;
  g.ctas_per_sm = kCtasPerSm;
  g.tiles = tiles;
  g.blocks = blocks;
  return g;
}

cudaError_t launch_ffma(const Plan& p, const Args& a) {
  const Shape& s = p.sh;
  FfParams fp{};
  int64_t tiles;
  extents(s, p.dir, &fp.M, &fp.N, &fp.blocks, &tiles);
  fp.tiles_m = (fp.M + kT - 1) / kT;
  fp.tiles_n = (fp.N + kT - 1) / kT;
  fp.split = p.split;
  fp.out = static_cast<float*>(a.out);
  fp.ws = a.ws;
  fp.E = p.out_elems;
  fp.R = (int32_t)s.r;
  fp.S = (int32_t)s.s;
  fp.dh = (int32_t)s.dh;
  fp.dw = (int32_t)s.dw;
  if (p.dir == CONV_DIR_DGRAD) {  // the forward form: input dY (Ho x Wo, K channels), output dX, turned filter
    const Shape t = dgrad_as_forward(s);
    fp.H = t.h; fp.W = t.w; fp.C = t.c; fp.Ho = t.ho; fp.Wo = t.wo; fp.K = t.k;
    fp.sh = 1; fp.sw = 1; fp.ph = (int32_t)t.ph; fp.pw = (int32_t)t.pw;
  } else {
    fp.H = s.h; fp.W = s.w; fp.C = s.c; fp.Ho = s.ho; fp.Wo = s.wo; fp.K = s.k;
    fp.sh = (int32_t)s.sh; fp.sw = (int32_t)s.sw; fp.ph = (int32_t)s.ph; fp.pw = (int32_t)s.pw;
  }
  fp.cblocks = (int32_t)((fp.C + kBK - 1) / kBK);
  fp.P = s.n * s.ho * s.wo;
  if (p.dir == CONV_DIR_WGRAD) {
    fp.div_wo = DivU32((uint32_t)s.wo);
    fp.div_ho = DivU32((uint32_t)s.ho);
  }
  const int64_t ctas = tiles * p.split;
  if (ctas > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  if (p.dir == CONV_DIR_FWD) {
    fp.a = static_cast<const float*>(a.x);
    fp.b = static_cast<const float*>(a.b);
    if (a.ep && a.ws) return cudaErrorInvalidValue;  // the epilogue runs unsplit only
    fp.ep = a.ep ? 1 : 0;
    fp.ep_bias = static_cast<const float*>(a.ep_bias);
    fp.ep_lo = a.ep_lo;
    fp.ep_hi = a.ep_hi;
    ffma_igemm_kernel<kFwd><<<(unsigned)ctas, kThreads, 0, a.stream>>>(fp);
  } else if (p.dir == CONV_DIR_DGRAD) {
    fp.a = static_cast<const float*>(a.x);  // dY
    fp.b = static_cast<const float*>(a.b);  // W
    ffma_igemm_kernel<kDgrad><<<(unsigned)ctas, kThreads, 0, a.stream>>>(fp);
  } else {
    fp.a = static_cast<const float*>(a.b);  // dY
    fp.b = static_cast<const float*>(a.x);  // X
    fp.db = p.with_bias && !a.ws_bias ? static_cast<float*>(a.db) : nullptr;
    fp.ws_bias = p.with_bias ? a.ws_bias : nullptr;
    ffma_igemm_kernel<kWgrad><<<(unsigned)ctas, kThreads, 0, a.stream>>>(fp);
  }
  return cudaGetLastError();
}

}  // namespace cig
