// 16-bit depthwise forward convolution (groups = C = K) for square F x F
// filters (3, 5, 7), unit stride and dilation, with the filter taps in
// registers and the input rows streamed by TMA:
//
//   Y[n, ho, wo, c] = epilogue(sum over r, s of X[n, ho + r - ph, wo + s - pw, c] * W[c, r, s])
//
// (the forward twin of the depthwise weight gradient of "perf(rocke):
// depthwise 7x7 and grouped cpg4/8 wgrad on batched mfma 4x4x4"; that page's
// commit notes also list depthwise and grouped forward kernels), with the
// fused epilogue min(max(acc + bias[c], lo), hi) applied before the one
// rounding.
//
// A CTA owns 64 channels and a run of consecutive (n, ho) output rows, and
// walks it 8 rows (a step) at a time, one row per warp. The run's input rows
// stream through a shared-memory ring of row buffers (box {64 channels, W
// columns}, zero fill outside the image and past C; see dw_ring.cuh). A step
// slot has one full mbarrier, on which the input rows the step is the first
// to read all land, and one empty mbarrier, on which every warp arrives when
// done with the step; the loads of step S + 1 are issued at step S by warp
// S mod 8, one lane a box, and every wait is bounded.
//
// A lane holds all F*F taps of its two adjacent channels as packed fp32 pairs
// and walks its row's input columns u left to right: column u meets output
// column wo = u + pw - s through tap column s, so the lane keeps the F
// outputs u + pw - F + 1 .. u + pw in a register window, adds F*F packed FMAs
// (__ffma2_rn) per column from F four-byte shared-memory loads widened to
// fp32, and after each column writes out the output that column completes
// (the warp writes 128 contiguous bytes).
#include <type_traits>

#include "dw_ring.cuh"
#include "../kernel_entry.h"

namespace cig {
namespace {

using dwring::lds2;
using dwring::ring_rows;
using dwring::RowPos;
using dwring::StepPos;

constexpr int kThreads = 256;  // 8 warps, up to 255 registers a thread
constexpr int kWarps = kThreads / 32;
constexpr int kTR = kWarps;    // output rows a step: one a warp
constexpr int kCB = 64;        // channels per CTA (2 per lane)
constexpr int kSms = 152;      // the grid is sized for this many SMs (fewer run it in more waves)
constexpr size_t kSmemLimit = 227 * 1024;

struct FwdRingParams {
  int64_t C, Ho, Wo;
  int64_t rows;        // N * Ho
  int64_t cblocks;     // ceil(C / 64)
  int64_t cta_rows;    // output rows a CTA (a multiple of 8)
  int32_t W, ph, pw;
  int32_t RX, RS;      // ring slots: input rows, steps
  const void* ep_bias;  // fused epilogue, when ep
  float ep_lo, ep_hi;
  int32_t ep;
  int32_t rev;          // 1: tap t reads filter tap F*F - 1 - t (the data gradient's turned filter)
};

// The ring is one step deep plus the step in use (ahead 1, no slack).
constexpr int kDepth = 1;

size_t ring_smem(const Shape& s) {
  const int64_t rx = ring_rows(s.s, s.ho, kDepth, kTR), rs = 1 + kDepth;
  return (size_t)(rx * s.w * 128 + 2 * rs * 8 + rs * 4 + 16);
}

// Output rows a CTA: enough CTAs for one per SM over all channel blocks.
int64_t cta_rows(const Shape& s) {
  const int64_t rows = s.n * s.ho, cblocks = (s.c + kCB - 1) / kCB;
  int64_t r = (rows * cblocks + kSms - 1) / kSms;
  r = (r + kTR - 1) / kTR * kTR;
  return r < kTR ? kTR : r;
}

template <typename T>
__device__ __forceinline__ float ldf(const T* p);
template <>
__device__ __forceinline__ float ldf<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __bfloat162float(*p);
}
template <>
__device__ __forceinline__ float ldf<__half>(const __half* p) {
  return __half2float(*p);
}
template <>
__device__ __forceinline__ float ldf<float>(const float* p) {
  return *p;
}

template <typename T>
__device__ __forceinline__ void st2(T* p, float2 v);
template <>
__device__ __forceinline__ void st2<float>(float* p, float2 v) {
  *reinterpret_cast<float2*>(p) = v;
}
template <>
__device__ __forceinline__ void st2<__nv_bfloat16>(__nv_bfloat16* p, float2 v) {
  *reinterpret_cast<__nv_bfloat162*>(p) = __floats2bfloat162_rn(v.x, v.y);
}
template <>
__device__ __forceinline__ void st2<__half>(__half* p, float2 v) {
  *reinterpret_cast<__half2*>(p) = __floats2half2_rn(v.x, v.y);
}

struct FwdRing {
  const CUtensorMap* tm_x;
  uint8_t* xring;
  uint64_t* full;
  uint64_t* empty;
  int32_t* siss;  // wrap count of the last step loaded into each step slot (-1: none)
  volatile uint32_t* abort_flag;
  unsigned* err;
  uint32_t rowX;
  int32_t c0;
};

// Loads the input rows that the `rows` output rows of a step (the first at
// row position a) are the first to read, all landing on the step slot's full
// mbarrier, once every warp is done with the slot's previous step. False: the
// wait gave up.
template <int F>
__device__ bool issue_step(const FwdRing& g, const FwdRingParams& p, RowPos a, StepPos st, int32_t rows) {
  if (st.sw > 0 && !mbar_wait(&g.empty[st.ss], (st.sw - 1u) & 1u, g.abort_flag, g.err)) return false;
  uint32_t nrows = 0;
  {
    RowPos b = a;
    for (int32_t j = 0; j < rows; ++j, b.advance(F, p)) nrows += (uint32_t)b.fresh(F);
  }
  uint64_t* bar = &g.full[st.ss];
  mbar_arrive_expect_tx(bar, nrows * g.rowX);
  for (int32_t j = 0; j < rows; ++j, a.advance(F, p))
    for (int r = F - a.fresh(F); r < F; ++r)
      tma_load_4d(g.xring + (size_t)a.slot(r, p) * g.rowX, g.tm_x, g.c0, 0, a.ho - p.ph + r, a.n, bar);
  g.siss[st.ss] = (int32_t)st.sw;
  return true;
}

// issue_step by a whole warp: lane 0 waits for the slot and arms its full
// barrier, then lane b issues box b (the rows' new input rows in order), so
// the issuing warp pays for one copy instruction rather than one per row.
// Every lane must call it, with the same arguments. False: the wait gave up.
template <int F>
__device__ bool issue_step_warp(const FwdRing& g, const FwdRingParams& p, RowPos a, StepPos st, int32_t rows) {
  const int lane = threadIdx.x & 31;
  uint32_t nrows = 0;
  {
    RowPos b = a;
    for (int32_t j = 0; j < rows; ++j, b.advance(F, p)) nrows += (uint32_t)b.fresh(F);
  }
  uint64_t* bar = &g.full[st.ss];
  bool ok = true;
  if (lane == 0) {
    if (st.sw > 0) ok = mbar_wait(&g.empty[st.ss], (st.sw - 1u) & 1u, g.abort_flag, g.err);
    if (ok) mbar_arrive_expect_tx(bar, nrows * g.rowX);
  }
  if (!__shfl_sync(0xffffffffu, ok, 0)) return false;
  int box = 0;
  for (int32_t j = 0; j < rows; ++j, a.advance(F, p))
    for (int r = F - a.fresh(F); r < F; ++r)
      if ((box++ & 31) == lane)
        tma_load_4d(g.xring + (size_t)a.slot(r, p) * g.rowX, g.tm_x, g.c0, 0, a.ho - p.ph + r, a.n, bar);
  if (lane == 0) g.siss[st.ss] = (int32_t)st.sw;
  __syncwarp();
  return true;
}

// One output row: input row r at xs[r] (column u at xs[r] + u * 128), outputs
// to yrow[wo * C]. Column u adds tap (r, s) into output u + pw - s; output
// slot (wo - pw + F - 1) mod F, so at column u0 + t (u0 a multiple of F)
// tap column s goes to slot (t + F - 1 - s) mod F and slot t holds the output
// the column completes. Columns past W add nothing and only complete outputs.
template <typename TI, typename TO, int F>
__device__ __forceinline__ void sweep_row(const float2 (&tap)[F * F], const uint32_t (&xs)[F], TO* yrow,
                                          const FwdRingParams& p, float2 bias, bool cok) {
  const float2 zero = make_float2(0.f, 0.f);
  float2 ow[F];
#pragma unroll
  for (int k = 0; k < F; ++k) ow[k] = zero;  // outputs pw - F + 1 .. pw - 1 start empty
  auto emit = [&](int32_t wo, float2 v) {
    if (wo >= 0 && wo < p.Wo && cok) {
      if (p.ep) {
        v.x = fminf(fmaxf(v.x + bias.x, p.ep_lo), p.ep_hi);
        v.y = fminf(fmaxf(v.y + bias.y, p.ep_lo), p.ep_hi);
      }
      st2<TO>(yrow + (int64_t)wo * p.C, v);
    }
  };
  // T columns from u0 (u0 a multiple of F); columns u >= W only complete outputs
  auto columns = [&](int32_t u0, auto tcount, bool guard) {
    constexpr int T = decltype(tcount)::value;
#pragma unroll
    for (int t = 0; t < T; ++t) {
      const int32_t u = u0 + t;
      if (!guard || u < p.W) {
        float2 xv[F];
#pragma unroll
        for (int r = 0; r < F; ++r) xv[r] = lds2<TI>(xs[r] + (uint32_t)(u * 128));
#pragma unroll
        for (int s = 0; s < F; ++s) {
          const int k = (t + F - 1 - s) % F;
#pragma unroll
          for (int r = 0; r < F; ++r)
            ow[k] = s == 0 && r == 0 ? __fmul2_rn(xv[0], tap[s]) : __ffma2_rn(xv[r], tap[r * F + s], ow[k]);
        }
      } else {
        ow[(t + F - 1) % F] = zero;  // the output this column would have started
      }
      emit(u + p.pw - F + 1, ow[t % F]);
    }
  };
  int32_t u0 = 0;
#pragma unroll 1
  for (; u0 + F <= p.W; u0 += F) columns(u0, std::integral_constant<int, F>{}, false);
  // the last W mod F columns and F - 1 columns that only complete outputs
  columns(u0, std::integral_constant<int, 2 * F - 1>{}, true);
}

template <typename TI, typename TO, int F>
__global__ void __launch_bounds__(kThreads, 1)
    dw_fwd_ring_kernel(const __grid_constant__ CUtensorMap tm_x, const TI* __restrict__ w, TO* y,
                       FwdRingParams p, unsigned* err) {
  constexpr int FF = F * F;
  extern __shared__ __align__(128) uint8_t smem[];
  FwdRing g;
  g.tm_x = &tm_x;
  g.rowX = (uint32_t)p.W * 128u;
  g.xring = smem;
  g.full = reinterpret_cast<uint64_t*>(smem + (size_t)p.RX * g.rowX);
  g.empty = g.full + p.RS;
  g.siss = reinterpret_cast<int32_t*>(g.empty + p.RS);
  g.abort_flag = reinterpret_cast<volatile uint32_t*>(g.siss + p.RS);
  g.err = err;

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t cb = blockIdx.x % p.cblocks;
  const int64_t q_b = (blockIdx.x / p.cblocks) * p.cta_rows;
  const int64_t q_e = q_b + p.cta_rows < p.rows ? q_b + p.cta_rows : p.rows;
  g.c0 = (int32_t)(cb * kCB);
  const RowPos start{0, (int32_t)(q_b % p.Ho), (int32_t)(q_b / p.Ho), true};

  if (threadIdx.x == 0) {
    for (int i = 0; i < p.RS; ++i) {
      mbar_init(&g.full[i], 1);
      mbar_init(&g.empty[i], kWarps);
      g.siss[i] = -1;
    }
    *g.abort_flag = 0u;
    mbar_fence_init();
    tma_prefetch(&tm_x);
    // Step 0 loads into fresh slots.
    if (q_b < q_e) issue_step<F>(g, p, start, StepPos{0, 0u}, q_e - q_b < kTR ? (int32_t)(q_e - q_b) : kTR);
  }

  // The lane's taps and bias (zero for channels past C, whose outputs are not written).
  const int64_t c = cb * kCB + 2 * lane;
  const bool cok = c < p.C;
  float2 tap[FF];
#pragma unroll
  for (int i = 0; i < FF; ++i)
    tap[i] = cok ? make_float2(ldf<TI>(w + c * FF + (p.rev ? FF - 1 - i : i)),
                               ldf<TI>(w + (c + 1) * FF + (p.rev ? FF - 1 - i : i)))
                 : make_float2(0.f, 0.f);
  float2 bias = make_float2(0.f, 0.f);
  if (p.ep && p.ep_bias && cok) {
    const TO* b = static_cast<const TO*>(p.ep_bias);
    bias = make_float2(ldf<TO>(b + c), ldf<TO>(b + c + 1));
  }
  __syncthreads();

  RowPos mine = start;  // this warp's row of the step
  for (int i = 0; i < warp; ++i) mine.advance(F, p);
  RowPos la = start;  // first row of the next step
  for (int i = 0; i < kTR; ++i) la.advance(F, p);
  StepPos sc{0, 0u};
  int32_t issuer = 0;  // warp that loads at step S: S mod 8

  for (int64_t q = q_b; q < q_e; q += kTR) {
    const int64_t qa = q + kTR;  // first row of step S + 1
    if (warp == issuer && qa < q_e) {
      StepPos sl = sc;
      sl.advance(p);
      issue_step_warp<F>(g, p, la, sl, q_e - qa < kTR ? (int32_t)(q_e - qa) : kTR);
    }
    for (int i = 0; i < kTR; ++i) la.advance(F, p);
    issuer = (issuer + 1) & (kWarps - 1);

    if (!__all_sync(0xffffffffu, mbar_wait(&g.full[sc.ss], sc.sw & 1u, g.abort_flag, g.err))) break;

    if (q + warp < q_e) {
      uint32_t xs[F];
#pragma unroll
      for (int r = 0; r < F; ++r) xs[r] = smem_u32(g.xring + (size_t)mine.slot(r, p) * g.rowX + lane * 4);
      TO* yrow = y + (((int64_t)mine.n * p.Ho + mine.ho) * p.Wo) * p.C + c;
      sweep_row<TI, TO, F>(tap, xs, yrow, p, bias, cok);
    }

    __syncwarp();
    if (lane == 0) mbar_arrive(&g.empty[sc.ss]);
    __syncwarp();
    for (int i = 0; i < kTR; ++i) mine.advance(F, p);
    sc.advance(p);
  }

  // No copy may still be landing in shared memory when the CTA exits: wait
  // for the last step loaded into each step slot (bounded, no early exit).
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int i = 0; i < p.RS; ++i)
      if (g.siss[i] >= 0) mbar_wait(&g.full[i], (uint32_t)g.siss[i] & 1u, nullptr, err);
  }
}

template <typename TI, typename TO, int F>
cudaError_t launch_f(const Plan& pl, const Args& a, const FwdRingParams& p, CUtensorMapDataType dt) {
  const Shape& s = pl.sh;
  CUtensorMap tm_x;
  const uint64_t x_dims[4] = {(uint64_t)s.c, (uint64_t)s.w, (uint64_t)s.h, (uint64_t)s.n};
  const uint64_t x_strides[3] = {(uint64_t)s.c * 2u, (uint64_t)(s.w * s.c) * 2u, (uint64_t)(s.h * s.w * s.c) * 2u};
  const uint32_t x_box[4] = {(uint32_t)kCB, (uint32_t)s.w, 1u, 1u};
  if (!encode_tmap(&tm_x, dt, 4, a.x, x_dims, x_strides, x_box, CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  const size_t smem = ring_smem(s);
  auto kern = dw_fwd_ring_kernel<TI, TO, F>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  const int64_t ctas = pl.geo.tiles;
  if (ctas > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  kern<<<(unsigned)ctas, kThreads, smem, a.stream>>>(tm_x, static_cast<const TI*>(a.b), static_cast<TO*>(a.out), p,
                                                     device_error_word());
  return cudaGetLastError();
}

template <typename TI, typename TO>
cudaError_t launch_typed(const Plan& pl, const Args& a, CUtensorMapDataType dt) {
  const Shape& s = pl.sh;
  FwdRingParams p;
  p.C = s.c;
  p.Ho = s.ho;
  p.Wo = s.wo;
  p.rows = s.n * s.ho;
  p.cblocks = (s.c + kCB - 1) / kCB;
  p.cta_rows = cta_rows(s);
  p.W = (int32_t)s.w;
  p.ph = (int32_t)s.ph;
  p.pw = (int32_t)s.pw;
  p.RX = (int32_t)ring_rows(s.s, s.ho, kDepth, kTR);
  p.RS = 1 + kDepth;
  p.ep_bias = a.ep_bias;
  p.ep_lo = a.ep_lo;
  p.ep_hi = a.ep_hi;
  p.ep = a.ep ? 1 : 0;
  p.rev = a.rev_taps ? 1 : 0;
  switch (s.s) {
    case 3: return launch_f<TI, TO, 3>(pl, a, p, dt);
    case 5: return launch_f<TI, TO, 5>(pl, a, p, dt);
    case 7: return launch_f<TI, TO, 7>(pl, a, p, dt);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

Geometry geometry_fwd_depthwise_ring(const Shape& s) {
  Geometry g;
  const bool depthwise = s.groups == s.c && s.groups == s.k;
  if (!depthwise || s.in_dt == CONV_F32 || s.n < 1) return g;
  if (s.r != s.s || !(s.s == 3 || s.s == 5 || s.s == 7)) return g;
  if (s.sh != 1 || s.sw != 1 || s.dh != 1 || s.dw != 1) return g;
  if (s.pw > s.s - 1 || s.ph > s.r - 1) return g;
  // TMA: 16-byte row strides, a 64-channel box inside the channel extent,
  // whole rows of at most 256 columns; coordinates in 32 bits.
  if (s.c % 8 != 0 || s.c < kCB || s.w > 256) return g;
  if (s.n > 0x7fffffffLL || s.h + s.r > 0x7fffffffLL) return g;
  if (ring_smem(s) > kSmemLimit) return g;
  g.ok = true;
  g.ctas_per_sm = 1;
  g.tiles = ((s.c + kCB - 1) / kCB) * ((s.n * s.ho + cta_rows(s) - 1) / cta_rows(s));
  g.blocks = 1;  // no split: the reduction is F*F taps
  return g;
}

cudaError_t launch_fwd_depthwise_ring(const Plan& p, const Args& a) {
  if (p.split != 1 || a.ws) return cudaErrorInvalidValue;
  const int in = p.sh.in_dt, out = p.sh.out_dt;
  if (in == CONV_BF16)
    return out == CONV_F32 ? launch_typed<__nv_bfloat16, float>(p, a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16)
                           : launch_typed<__nv_bfloat16, __nv_bfloat16>(p, a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16);
  return out == CONV_F32 ? launch_typed<__half, float>(p, a, CU_TENSOR_MAP_DATA_TYPE_FLOAT16)
                         : launch_typed<__half, __half>(p, a, CU_TENSOR_MAP_DATA_TYPE_FLOAT16);
}

}  // namespace cig
