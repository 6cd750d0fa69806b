// Generic direct kernels (CUDA cores) for the forward, weight gradient and
// data gradient: every shape, stride, dilation, padding,
// group count and storage type the ABI accepts. One thread owns one output
// element of one reduction slice and walks the slice in order, so the result
// of a slice is deterministic. These are the correctness floor under the fast
// kernels, not a fast path.
#include "common.cuh"
#include "../kernel_entry.h"

namespace cig {
namespace {

constexpr int kThreads = 256;
constexpr int64_t kRowsPerBlock = 64;   // weight-gradient reduction block (rows of N*Ho*Wo)
constexpr int64_t kDepthPerBlock = 32;  // forward / data-gradient reduction block (of R*S*Cg / R*S*Kg)

// dW[k,r,s,c] over the rows of slice sigma:
//   sum dY[n,ho,wo,k] * X[n, ho*sh + r*dh - ph, wo*sw + s*dw - pw, g*Cg + c].
template <typename TI, typename TO>
__global__ void __launch_bounds__(kThreads) generic_wgrad_kernel(Shape sh, const TI* __restrict__ x,
                                                                 const TI* __restrict__ dy, TO* out,
                                                                 float* ws, int32_t S, int64_t tiles,
                                                                 int64_t blocks) {
  const int64_t tile = blockIdx.x % tiles;
  const int32_t sigma = (int32_t)(blockIdx.x / tiles);
  const int64_t E = sh.w_elems();
  const int64_t e = tile * kThreads + threadIdx.x;
  if (e >= E) return;
  const int64_t c = e % sh.cg;
  int64_t t = e / sh.cg;
  const int64_t s = t % sh.s;
  t /= sh.s;
  const int64_t r = t % sh.r;
  const int64_t k = t / sh.r;
  const int64_t cin = (k / sh.kg) * sh.cg + c;
  const int64_t P = sh.P();
  int64_t p = slice_begin(blocks, S, sigma) * kRowsPerBlock;
  int64_t p_end = slice_begin(blocks, S, sigma + 1) * kRowsPerBlock;
  if (p_end > P) p_end = P;
  float acc = 0.f;
  if (p < p_end) {
    int64_t wo = p % sh.wo;
    int64_t ho = (p / sh.wo) % sh.ho;
    int64_t n = p / (sh.wo * sh.ho);
    const int64_t dr = r * sh.dh - sh.ph, ds = s * sh.dw - sh.pw;
    for (; p < p_end; ++p) {
      const int64_t h = ho * sh.sh + dr, w = wo * sh.sw + ds;
      if (h >= 0 && h < sh.h && w >= 0 && w < sh.w)
        acc = fmaf(to_f32(dy[p * sh.k + k]), to_f32(x[((n * sh.h + h) * sh.w + w) * sh.c + cin]), acc);
      if (++wo == sh.wo) {
        wo = 0;
        if (++ho == sh.ho) {
          ho = 0;
          ++n;
        }
      }
    }
  }
  store_result(out, ws, E, sigma, e, acc);
}

// db[k] over the rows of slice sigma.
template <typename TI, typename TO>
__global__ void __launch_bounds__(kThreads) generic_bias_kernel(Shape sh, const TI* __restrict__ dy, TO* db,
                                                                float* ws_bias, int32_t S, int64_t ktiles,
                                                                int64_t blocks) {
  const int64_t k = (int64_t)(blockIdx.x % ktiles) * kThreads + threadIdx.x;
  const int32_t sigma = (int32_t)(blockIdx.x / ktiles);
  if (k >= sh.k) return;
  const int64_t P = sh.P();
  int64_t p = slice_begin(blocks, S, sigma) * kRowsPerBlock;
  int64_t p_end = slice_begin(blocks, S, sigma + 1) * kRowsPerBlock;
  if (p_end > P) p_end = P;
  float acc = 0.f;
  for (; p < p_end; ++p) acc += to_f32(dy[p * sh.k + k]);
  store_result(db, ws_bias, sh.k, sigma, k, acc);
}

// Y[n,ho,wo,k] over the reduction depth (r, s, c) of slice sigma; unsplit,
// with the fused epilogue min(max(acc + bias[k], lo), hi) when ep is set.
template <typename TI, typename TO>
__global__ void __launch_bounds__(kThreads) generic_fwd_kernel(Shape sh, const TI* __restrict__ x,
                                                               const TI* __restrict__ wt, TO* out, float* ws,
                                                               int32_t S, int64_t tiles, int64_t blocks,
                                                               const TO* ep_bias, float ep_lo, float ep_hi,
                                                               bool ep) {
  const int64_t tile = blockIdx.x % tiles;
  const int32_t sigma = (int32_t)(blockIdx.x / tiles);
  const int64_t E = sh.y_elems();
  const int64_t e = tile * kThreads + threadIdx.x;
  if (e >= E) return;
  const int64_t k = e % sh.k;
  int64_t t = e / sh.k;
  const int64_t wo = t % sh.wo;
  t /= sh.wo;
  const int64_t ho = t % sh.ho;
  const int64_t n = t / sh.ho;
  const int64_t cbase = (k / sh.kg) * sh.cg;
  const int64_t D = sh.D();
  int64_t d = slice_begin(blocks, S, sigma) * kDepthPerBlock;
  int64_t d_end = slice_begin(blocks, S, sigma + 1) * kDepthPerBlock;
  if (d_end > D) d_end = D;
  float acc = 0.f;
  if (d < d_end) {
    int64_t c = d % sh.cg;
    int64_t s = (d / sh.cg) % sh.s;
    int64_t r = d / (sh.cg * sh.s);
    const TI* wk = wt + k * D;
    for (; d < d_end; ++d) {
      const int64_t h = ho * sh.sh + r * sh.dh - sh.ph, w = wo * sh.sw + s * sh.dw - sh.pw;
      if (h >= 0 && h < sh.h && w >= 0 && w < sh.w)
        acc = fmaf(to_f32(x[((n * sh.h + h) * sh.w + w) * sh.c + cbase + c]), to_f32(wk[d]), acc);
      if (++c == sh.cg) {
        c = 0;
        if (++s == sh.s) {
          s = 0;
          ++r;
        }
      }
    }
  }
  if (ep) acc = fminf(fmaxf(acc + (ep_bias ? to_f32(ep_bias[k]) : 0.f), ep_lo), ep_hi);
  store_result(out, ws, E, sigma, e, acc);
}

// dX[n,h,w,g*Cg + c] over the reduction (r, s, k in group g) of slice sigma:
//   sum dY[n,ho,wo,k] * W[k,r,s,c] for ho*sh + r*dh - ph = h, wo*sw + s*dw - pw = w.
template <typename TI, typename TO>
__global__ void __launch_bounds__(kThreads) generic_dgrad_kernel(Shape sh, const TI* __restrict__ dy,
                                                                 const TI* __restrict__ wt, TO* out, float* ws,
                                                                 int32_t S, int64_t tiles, int64_t blocks) {
  const int64_t tile = blockIdx.x % tiles;
  const int32_t sigma = (int32_t)(blockIdx.x / tiles);
  const int64_t E = sh.x_elems();
  const int64_t e = tile * kThreads + threadIdx.x;
  if (e >= E) return;
  const int64_t ci = e % sh.c;
  int64_t t = e / sh.c;
  const int64_t w = t % sh.w;
  t /= sh.w;
  const int64_t h = t % sh.h;
  const int64_t n = t / sh.h;
  const int64_t g = ci / sh.cg, c = ci % sh.cg;
  const int64_t D = sh.r * sh.s * sh.kg;
  int64_t d = slice_begin(blocks, S, sigma) * kDepthPerBlock;
  int64_t d_end = slice_begin(blocks, S, sigma + 1) * kDepthPerBlock;
  if (d_end > D) d_end = D;
  float acc = 0.f;
  while (d < d_end) {
    // one (r, s) tap: its k range within the slice
    const int64_t rs = d / sh.kg, k_lo = d % sh.kg;
    const int64_t r = rs / sh.s, s = rs % sh.s;
    const int64_t k_hi = (rs + 1) * sh.kg <= d_end ? sh.kg : d_end - rs * sh.kg;
    d += k_hi - k_lo;
    const int64_t hn = h + sh.ph - r * sh.dh, wn = w + sh.pw - s * sh.dw;
    if (hn < 0 || wn < 0 || hn % sh.sh != 0 || wn % sh.sw != 0) continue;
    const int64_t ho = hn / sh.sh, wo = wn / sh.sw;
    if (ho >= sh.ho || wo >= sh.wo) continue;
    const TI* dyp = dy + ((n * sh.ho + ho) * sh.wo + wo) * sh.k + g * sh.kg;
    const TI* wp = wt + ((g * sh.kg * sh.r + r) * sh.s + s) * sh.cg + c;
    const int64_t wstride = sh.r * sh.s * sh.cg;
    for (int64_t kk = k_lo; kk < k_hi; ++kk) acc = fmaf(to_f32(dyp[kk]), to_f32(wp[kk * wstride]), acc);
  }
  store_result(out, ws, E, sigma, e, acc);
}

template <typename TI, typename TO>
cudaError_t launch_typed(const Plan& p, const Args& a) {
  const int64_t ctas = p.geo.tiles * p.split;
  const int64_t ktiles = (p.sh.k + kThreads - 1) / kThreads;
  if (ctas > 0x7fffffffLL || ktiles * p.split > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  const TI* x = static_cast<const TI*>(a.x);
  const TI* b = static_cast<const TI*>(a.b);
  TO* out = static_cast<TO*>(a.out);
  if (p.dir == CONV_DIR_WGRAD) {
    generic_wgrad_kernel<TI, TO><<<(unsigned)ctas, kThreads, 0, a.stream>>>(p.sh, x, b, out, a.ws, p.split,
                                                                             p.geo.tiles, p.geo.blocks);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess || !p.with_bias) return err;
    generic_bias_kernel<TI, TO><<<(unsigned)(ktiles * p.split), kThreads, 0, a.stream>>>(
        p.sh, b, static_cast<TO*>(a.db), a.ws_bias, p.split, ktiles, p.geo.blocks);
    return cudaGetLastError();
  }
  if (p.dir == CONV_DIR_DGRAD) {
    generic_dgrad_kernel<TI, TO><<<(unsigned)ctas, kThreads, 0, a.stream>>>(p.sh, x, b, out, a.ws, p.split,
                                                                             p.geo.tiles, p.geo.blocks);
    return cudaGetLastError();
  }
  generic_fwd_kernel<TI, TO><<<(unsigned)ctas, kThreads, 0, a.stream>>>(
      p.sh, x, b, out, a.ws, p.split, p.geo.tiles, p.geo.blocks, static_cast<const TO*>(a.ep_bias), a.ep_lo, a.ep_hi,
      a.ep);
  return cudaGetLastError();
}

}  // namespace

Geometry geometry_generic(const Shape& s, conv_dir dir) {
  Geometry g;
  g.ok = true;
  g.ctas_per_sm = 8;
  const int64_t E = dir == CONV_DIR_FWD ? s.y_elems() : dir == CONV_DIR_WGRAD ? s.w_elems() : s.x_elems();
  g.tiles = (E + kThreads - 1) / kThreads;
  if (g.tiles < 1) g.tiles = 1;
  if (dir == CONV_DIR_FWD) g.blocks = (s.D() + kDepthPerBlock - 1) / kDepthPerBlock;
  else if (dir == CONV_DIR_WGRAD) g.blocks = (s.P() + kRowsPerBlock - 1) / kRowsPerBlock;
  else g.blocks = (s.r * s.s * s.kg + kDepthPerBlock - 1) / kDepthPerBlock;
  return g;
}

cudaError_t launch_generic(const Plan& p, const Args& a) {
  const int in = p.sh.in_dt, out = p.sh.out_dt;
  if (in == CONV_F32) return launch_typed<float, float>(p, a);
  if (in == CONV_BF16)
    return out == CONV_F32 ? launch_typed<__nv_bfloat16, float>(p, a) : launch_typed<__nv_bfloat16, __nv_bfloat16>(p, a);
  return out == CONV_F32 ? launch_typed<__half, float>(p, a) : launch_typed<__half, __half>(p, a);
}

}  // namespace cig
