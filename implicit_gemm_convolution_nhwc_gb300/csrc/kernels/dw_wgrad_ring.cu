// 16-bit depthwise weight gradient (+ bias gradient) for square F x F filters
// (3, 5, 7), unit stride and dilation, with the filter taps in registers and
// the input rows streamed by TMA:
//
//   dW[c, r, s] = sum over (n, ho, wo) of dY[n, ho, wo, c] * X[n, ho + r - ph, wo + s - pw, c]
//   db[c]       = sum over (n, ho, wo) of dY[n, ho, wo, c]
//
// ("perf(rocke): depthwise 7x7 and grouped cpg4/8 wgrad on batched mfma
// 4x4x4", "Technical Details".)
//
// A CTA owns 64 channels and a split-K slice [q_b, q_e) of the (n, ho) output
// rows, and walks it TR output rows (one step) at a time. Output row (n, ho)
// reads input rows ho - ph .. ho - ph + F - 1 of image n; consecutive rows of
// one image share F - 1 of them, so the slice's input rows form one sequence
// (a new image starts F fresh rows) streamed through a ring of shared-memory
// row buffers, each the box {64 channels, W columns} of one row (TMA fills
// rows outside the image, and channels past C, with zeros). A step's dY rows
// sit in its step slot, each padded with zero columns on both sides so that
// the inner loop reads dY column j in [-(F - 1), pw + W) unguarded. A step
// slot has one full mbarrier, on which the step's dY rows and the input rows
// it is the first to read all land, and one empty mbarrier, on which every
// warp arrives when done with the step. The loads of step S + ahead are
// issued at step S by warp S mod 8, one lane a box, so the issuing work
// rotates over the warps; every wait is bounded. The rings hold `slack` steps more
// than the loads in flight need, so an issue at step S only reuses slots that
// steps before S - slack used: the warps may drift apart by that many steps
// before an issuing warp waits for the slowest one.
//
// Each of the 8 warps takes a range of input columns, and a lane all F*F
// taps of its two adjacent channels as packed fp32 pairs. Walking its input
// columns wi left to right, column wi meets output pixel wo = wi + pw - s
// through tap column s, so the lane keeps the last F dY pairs of each output
// row in a register window and does F*F packed FMAs (__ffma2_rn) per row per
// column, from four-byte shared-memory loads widened to fp32; the rows of a
// step within one image share one sweep (each adds one input row). At the end,
// once every load has landed, the warps' sums are added in warp order, one
// filter row at a time (deterministic), in shared memory over the rings'
// bytes, and the tile goes out as contiguous fp32 to slab sigma of the
// workspace or, unsplit, rounded into dW / db.
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
constexpr int kCB = 64;              // channels per CTA (2 per lane)
constexpr int kMaxDepth = 5;         // ahead + slack, at most
constexpr size_t kSmemLimit = 227 * 1024;

struct RingParams {
  int64_t C, Ho;
  int64_t rows;     // N * Ho: the reduction blocks
  int64_t cblocks;  // ceil(C / 64): the tiles
  int32_t W, Wo, ph, pw;
  int32_t CW;       // input columns of a warp
  int32_t RX, RS;   // ring slots: input rows, steps
  int32_t TR;       // output rows a step
  int32_t ahead;    // steps between a load's issue and its use
  int32_t red_off;  // byte offset of the reduction's buffers in shared memory
  int32_t split;
};

// Shared memory of the warp-order reduction (red, res, resb), which reuses
// the rings' bytes once every load has landed.
constexpr size_t reduce_smem(int F) {
  return (size_t)kWarps * F * 2 * 32 * 4 + (size_t)kCB * F * F * 4 + kCB * 4;
}

// Columns of a dY ring slot: F - 1 zero columns, then dY columns 0 .. Wo - 1,
// then zero columns up to column pw + W - 1.
int64_t dy_slot_cols(int64_t W, int64_t pw, int64_t F) { return F - 1 + pw + W; }

// Ring depth d = ahead + slack (in steps of TR rows): d + 1 step slots.
int ahead_of_depth(int d) { return d >= 3 ? 2 : 1; }

size_t ring_smem(const Shape& s, int d, int tr) {
  const int64_t rx = ring_rows(s.s, s.ho, d, tr), rs = 1 + d;
  return (size_t)(rx * s.w * 128 + rs * tr * dy_slot_cols(s.w, s.pw, s.s) * 128 + 2 * rs * 8 + rs * 4 + 16);
}

struct RingShape {
  int d = 0, tr = 0;
};

// Where the reduction goes: over the ring rows and dY rows when they are large
// enough (the mbarriers after them are never overwritten), else after
// everything.
size_t ring_data_bytes(const Shape& s, const RingShape& rs) {
  return (size_t)(ring_rows(s.s, s.ho, rs.d, rs.tr) * s.w * 128 +
                  (1 + rs.d) * rs.tr * dy_slot_cols(s.w, s.pw, s.s) * 128);
}
size_t reduce_offset(const Shape& s, const RingShape& rs) {
  return ring_data_bytes(s, rs) >= reduce_smem((int)s.s) ? 0 : (ring_smem(s, rs.d, rs.tr) + 127) / 128 * 128;
}
size_t kernel_smem(const Shape& s, const RingShape& rs) {
  const size_t off = reduce_offset(s, rs);
  return off == 0 ? ring_smem(s, rs.d, rs.tr) : off + reduce_smem((int)s.s);
}

// Three, else two rows a step with the deepest ring that fits (up to
// kMaxDepth, at least one step of slack), else one row a step ({0, 0}: none
// fits).
RingShape ring_shape(const Shape& s) {
  for (int tr = 3; tr >= 1; --tr)
    for (int d = kMaxDepth; d >= 2; --d)
      if (kernel_smem(s, RingShape{d, tr}) <= kSmemLimit) return RingShape{d, tr};
  if (kernel_smem(s, RingShape{1, 1}) <= kSmemLimit) return RingShape{1, 1};
  return RingShape{};
}

struct Ring {
  const CUtensorMap* tm_x;
  const CUtensorMap* tm_dy;
  uint8_t* xring;
  uint8_t* dring;
  uint64_t* full;
  uint64_t* empty;
  int32_t* siss;  // wrap count of the last step loaded into each step slot (-1: none)
  volatile uint32_t* abort_flag;
  unsigned* err;
  uint32_t rowX, rowD, txD;
  int32_t c0;
};

// Loads a step: the dY rows of its `rows` output rows (the first at row
// position a) and the input rows they are the first to read, all landing on
// the step slot's full mbarrier, once every warp is done with the slot's
// previous step. False: the wait gave up.
template <int F>
__device__ bool issue_step(const Ring& g, const RingParams& p, RowPos a, StepPos st, int32_t rows) {
  if (st.sw > 0 && !mbar_wait(&g.empty[st.ss], (st.sw - 1u) & 1u, g.abort_flag, g.err)) return false;
  uint32_t bytes = 0;
  {
    RowPos b = a;
    for (int32_t j = 0; j < rows; ++j, b.advance(F, p)) bytes += g.txD + (uint32_t)b.fresh(F) * g.rowX;
  }
  uint64_t* bar = &g.full[st.ss];
  mbar_arrive_expect_tx(bar, bytes);
  for (int32_t j = 0; j < rows; ++j, a.advance(F, p)) {
    tma_load_4d(g.dring + ((size_t)st.ss * p.TR + j) * g.rowD + (size_t)(F - 1) * 128, g.tm_dy, g.c0, 0, a.ho, a.n,
                bar);
    for (int r = F - a.fresh(F); r < F; ++r)
      tma_load_4d(g.xring + (size_t)a.slot(r, p) * g.rowX, g.tm_x, g.c0, 0, a.ho - p.ph + r, a.n, bar);
  }
  g.siss[st.ss] = (int32_t)st.sw;
  return true;
}

// issue_step by a whole warp: lane 0 waits for the slot and arms its full
// barrier, then lane b issues box b of the step (its rows in order, each dY
// row followed by the input rows it is the first to read), so the issuing
// warp pays for one copy instruction rather than one per box. Every lane
// must call it, with the same arguments. False: the wait gave up.
template <int F>
__device__ bool issue_step_warp(const Ring& g, const RingParams& p, RowPos a, StepPos st, int32_t rows) {
  const int lane = threadIdx.x & 31;
  uint32_t bytes = 0;
  {
    RowPos b = a;
    for (int32_t j = 0; j < rows; ++j, b.advance(F, p)) bytes += g.txD + (uint32_t)b.fresh(F) * g.rowX;
  }
  uint64_t* bar = &g.full[st.ss];
  bool ok = true;
  if (lane == 0) {
    if (st.sw > 0) ok = mbar_wait(&g.empty[st.ss], (st.sw - 1u) & 1u, g.abort_flag, g.err);
    if (ok) mbar_arrive_expect_tx(bar, bytes);
  }
  if (!__shfl_sync(0xffffffffu, ok, 0)) return false;
  int box = 0;
  for (int32_t j = 0; j < rows; ++j, a.advance(F, p)) {
    if ((box++ & 31) == lane)
      tma_load_4d(g.dring + ((size_t)st.ss * p.TR + j) * g.rowD + (size_t)(F - 1) * 128, g.tm_dy, g.c0, 0, a.ho, a.n,
                  bar);
    for (int r = F - a.fresh(F); r < F; ++r)
      if ((box++ & 31) == lane)
        tma_load_4d(g.xring + (size_t)a.slot(r, p) * g.rowX, g.tm_x, g.c0, 0, a.ho - p.ph + r, a.n, bar);
  }
  if (lane == 0) g.siss[st.ss] = (int32_t)st.sw;
  __syncwarp();
  return true;
}

// One column sweep of a warp over NROWS output rows of one image (NROWS = 2:
// rows ho and ho + 1, which share all but one of their input rows): dY row j
// at dy0[j] (column c at dy0[j] + c * 128), input row i of the first row at
// xs[i] (32-bit shared addresses). For each input column u in [u_beg, u_end)
// the lane loads the dY pair of every row and the input pair of every row in
// reach, then adds tap (r, s) of row j as x[r + j][u] * dY_j[u + pw - s], in a
// fixed order.
template <typename TI, int F, int NROWS>
__device__ __forceinline__ void sweep(float2 (&acc)[F * F], float2& bsum, const uint32_t (&dy0)[NROWS],
                                      const uint32_t (&xs)[F + NROWS - 1], int32_t u_beg, int32_t u_end, int32_t pw,
                                      bool warp0) {
  constexpr int NX = F + NROWS - 1;
  const float2 zero = make_float2(0.f, 0.f);
  // Window slot ((u - u_beg) mod F) of row j holds its dY column pw + u;
  // before u = u_beg it holds columns pw + u_beg - F + 1 .. pw + u_beg - 1.
  // Warp 0's window covers the columns below pw, which no warp's columns
  // reach, so it adds those to the bias sum.
  float2 dwin[NROWS][F];
#pragma unroll
  for (int j = 0; j < NROWS; ++j) {
    dwin[j][0] = zero;
#pragma unroll
    for (int k = 1; k < F; ++k) {
      dwin[j][F - k] = lds2<TI>(dy0[j] + (uint32_t)((pw + u_beg - k) * 128));
      if (warp0) bsum = __fadd2_rn(bsum, dwin[j][F - k]);
    }
  }
  // F columns from u0 (cnt < F: only the first cnt, at the end of the range)
  auto columns = [&](int32_t u0, int32_t cnt) {
#pragma unroll
    for (int t = 0; t < F; ++t) {
      if (t < cnt) {
        const int32_t u = u0 + t;  // input column wi
#pragma unroll
        for (int j = 0; j < NROWS; ++j) {
          dwin[j][t] = lds2<TI>(dy0[j] + (uint32_t)((pw + u) * 128));
          bsum = __fadd2_rn(bsum, dwin[j][t]);
        }
        float2 xv[NX];
#pragma unroll
        for (int i = 0; i < NX; ++i) xv[i] = lds2<TI>(xs[i] + (uint32_t)(u * 128));
#pragma unroll
        for (int j = 0; j < NROWS; ++j)
#pragma unroll
          for (int i = 0; i < F * F; ++i) {
            const int r = i / F, s = i % F;
            acc[i] = __ffma2_rn(xv[r + j], dwin[j][(t - s + F) % F], acc[i]);
          }
      }
    }
  };
  int32_t u0 = u_beg;
#pragma unroll 1
  for (; u0 + F <= u_end; u0 += F) columns(u0, F);
  if (u0 < u_end) columns(u0, u_end - u0);
}

// A warp's part of the kernel: the step loop, then its share of the
// warp-order reduction into res / resb.
template <typename TI, int F>
__device__ __forceinline__ void run_warp(const Ring& g, const RingParams& p, int64_t q_b, int64_t q_e,
                                         float (*red)[F][2][32], float* res, float* resb) {
  constexpr int FF = F * F;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const float2 zero = make_float2(0.f, 0.f);
  float2 acc[FF];
#pragma unroll
  for (int i = 0; i < FF; ++i) acc[i] = zero;
  float2 bsum = zero;
  const int32_t u_beg = warp * p.CW;
  const int32_t u_end = u_beg + p.CW < p.W ? u_beg + p.CW : p.W;

  RowPos cur{0, (int32_t)(q_b % p.Ho), (int32_t)(q_b / p.Ho), true};
  StepPos sc{0, 0u};
  RowPos la = cur;  // first row of the step loaded for at step S: S + ahead
  StepPos sl{0, 0u};
  for (int i = 0; i < p.ahead * p.TR && q_b + i < q_e; ++i) la.advance(F, p);
  for (int i = 0; i < p.ahead; ++i) sl.advance(p);
  int32_t issuer = 0;  // warp that loads at step S: S mod 8
  int64_t qa = q_b + (int64_t)p.ahead * p.TR;  // first row of step S + ahead

  for (int64_t q = q_b; q < q_e; q += p.TR) {
    const int32_t rows = q_e - q < p.TR ? (int32_t)(q_e - q) : p.TR;
    if (warp == issuer && qa < q_e)
      issue_step_warp<F>(g, p, la, sl, q_e - qa < p.TR ? (int32_t)(q_e - qa) : p.TR);
    for (int32_t j = 0; j < p.TR && qa < q_e; ++j, ++qa) la.advance(F, p);
    sl.advance(p);
    issuer = (issuer + 1) & (kWarps - 1);

    if (!__all_sync(0xffffffffu, mbar_wait(&g.full[sc.ss], sc.sw & 1u, g.abort_flag, g.err))) break;

    // dY row j of the step: column c at dy_row(j) + c * 128 (zero for c < 0 and c >= Wo)
    auto dy_row = [&](int32_t j) {
      return smem_u32(g.dring + ((size_t)sc.ss * p.TR + j) * g.rowD + (size_t)(F - 1) * 128 + lane * 4);
    };
    auto x_row = [&](int r) { return smem_u32(g.xring + (size_t)cur.slot(r, p) * g.rowX + lane * 4); };
    // The step's rows in runs within one image; a run of L rows shares one
    // sweep (and all but L - 1 of its input rows).
#pragma unroll 1
    for (int32_t j = 0; j < rows;) {
      const int32_t left = p.Ho - cur.ho;  // rows of this image from cur on
      const int32_t run = rows - j < left ? rows - j : left;
      if (run >= 3) {
        if (u_beg < u_end) {
          const uint32_t dy0[3] = {dy_row(j), dy_row(j + 1), dy_row(j + 2)};
          uint32_t xs[F + 2];
#pragma unroll
          for (int i = 0; i < F + 2; ++i) xs[i] = x_row(i);
          sweep<TI, F, 3>(acc, bsum, dy0, xs, u_beg, u_end, p.pw, warp == 0);
        }
        j += 3;
        cur.advance(F, p);
        cur.advance(F, p);
        cur.advance(F, p);
      } else if (run == 2) {
        if (u_beg < u_end) {
          const uint32_t dy0[2] = {dy_row(j), dy_row(j + 1)};
          uint32_t xs[F + 1];
#pragma unroll
          for (int i = 0; i <= F; ++i) xs[i] = x_row(i);
          sweep<TI, F, 2>(acc, bsum, dy0, xs, u_beg, u_end, p.pw, warp == 0);
        }
        j += 2;
        cur.advance(F, p);
        cur.advance(F, p);
      } else {
        if (u_beg < u_end) {
          const uint32_t dy0[1] = {dy_row(j)};
          uint32_t xs[F];
#pragma unroll
          for (int i = 0; i < F; ++i) xs[i] = x_row(i);
          sweep<TI, F, 1>(acc, bsum, dy0, xs, u_beg, u_end, p.pw, warp == 0);
        }
        j += 1;
        cur.advance(F, p);
      }
    }

    __syncwarp();
    if (lane == 0) mbar_arrive(&g.empty[sc.ss]);
    __syncwarp();
    sc.advance(p);
  }
  signal_dependents();

  // The reduction below reuses the rings' shared memory: first every load
  // must have landed (wait for the last step loaded into each step slot;
  // bounded, no early exit).
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int i = 0; i < p.RS; ++i)
      if (g.siss[i] >= 0) mbar_wait(&g.full[i], (uint32_t)g.siss[i] & 1u, nullptr, g.err);
  }
  __syncthreads();

  // Warp-order sums, one filter row at a time: in round r every warp puts
  // its taps (r, s) into red[warp][s], then thread i adds value
  // (s, component, lane) = (i / 64, (i / 32) % 2, i % 32) over warps 0..7.
#pragma unroll
  for (int r = 0; r < F; ++r) {
#pragma unroll
    for (int s = 0; s < F; ++s) {
      red[warp][s][0][lane] = acc[r * F + s].x;
      red[warp][s][1][lane] = acc[r * F + s].y;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < F * 64; i += kThreads) {
      const int s = i >> 6, comp = (i >> 5) & 1, l = i & 31;
      float sum = red[0][s][comp][l];
#pragma unroll
      for (int w = 1; w < kWarps; ++w) sum += red[w][s][comp][l];
      res[(2 * l + comp) * FF + r * F + s] = sum;
    }
    __syncthreads();
  }
  red[warp][0][0][lane] = bsum.x;
  red[warp][0][1][lane] = bsum.y;
  __syncthreads();
  if (threadIdx.x < 64) {
    const int comp = threadIdx.x >> 5, l = threadIdx.x & 31;
    float sum = red[0][0][comp][l];
#pragma unroll
    for (int w = 1; w < kWarps; ++w) sum += red[w][0][comp][l];
    resb[2 * l + comp] = sum;
  }
}

template <typename TI, typename TO, int F>
__global__ void __launch_bounds__(kThreads, 1)
    dw_wgrad_ring_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_dy,
                         TO* out, float* ws, TO* db, float* ws_bias, RingParams p, unsigned* err) {
  constexpr int FF = F * F;
  extern __shared__ __align__(128) uint8_t smem[];
  // After the step loop: one filter row of every warp's sums (lane-minor), the
  // tile [64 channels][F][F] and the bias sums, over the rings' bytes.
  auto red = reinterpret_cast<float (*)[F][2][32]>(smem + p.red_off);
  float* res = reinterpret_cast<float*>(smem + p.red_off + (size_t)kWarps * F * 2 * 32 * 4);
  float* resb = res + kCB * FF;
  const int32_t dcols = F - 1 + p.pw + p.W;  // columns of a dY slot

  Ring g;
  g.tm_x = &tm_x;
  g.tm_dy = &tm_dy;
  g.rowX = (uint32_t)p.W * 128u;
  g.rowD = (uint32_t)dcols * 128u;
  g.txD = (uint32_t)p.Wo * 128u;
  g.xring = smem;
  g.dring = smem + (size_t)p.RX * g.rowX;
  g.full = reinterpret_cast<uint64_t*>(g.dring + (size_t)p.RS * p.TR * g.rowD);
  g.empty = g.full + p.RS;
  g.siss = reinterpret_cast<int32_t*>(g.empty + p.RS);
  g.abort_flag = reinterpret_cast<volatile uint32_t*>(g.siss + p.RS);
  g.err = err;

  const int64_t cb = blockIdx.x % p.cblocks;
  const int32_t sigma = (int32_t)(blockIdx.x / p.cblocks);
  g.c0 = (int32_t)(cb * kCB);
  const int64_t q_b = slice_begin(p.rows, p.split, sigma), q_e = slice_begin(p.rows, p.split, sigma + 1);

  if (threadIdx.x == 0) {
    for (int i = 0; i < p.RS; ++i) {
      mbar_init(&g.full[i], 1);
      mbar_init(&g.empty[i], kWarps);
      g.siss[i] = -1;
    }
    *g.abort_flag = 0u;
    mbar_fence_init();
    tma_prefetch(&tm_x);
    tma_prefetch(&tm_dy);
    // The first `ahead` steps load into fresh slots.
    RowPos a{0, (int32_t)(q_b % p.Ho), (int32_t)(q_b / p.Ho), true};
    StepPos st{0, 0u};
    for (int64_t q = q_b; q < q_e && st.ss < p.ahead; st.advance(p)) {
      const int32_t rows = q_e - q < p.TR ? (int32_t)(q_e - q) : p.TR;
      issue_step<F>(g, p, a, st, rows);
      for (int32_t j = 0; j < rows; ++j, ++q) a.advance(F, p);
    }
  }
  {  // the zero columns of the dY rows (TMA writes only columns F - 1 .. F - 2 + Wo)
    const int32_t pads = dcols - p.Wo, words = p.RS * p.TR * pads * 32;
    for (int32_t i = threadIdx.x; i < words; i += kThreads) {
      const int32_t slot = i / (pads * 32), col = (i / 32) % pads, word = i % 32;
      const int32_t pos = col < F - 1 ? col : col + p.Wo;
      reinterpret_cast<uint32_t*>(g.dring + (size_t)slot * g.rowD + (size_t)pos * 128)[word] = 0u;
    }
  }
  __syncthreads();

  run_warp<TI, F>(g, p, q_b, q_e, red, res, resb);
  __syncthreads();

  const int64_t nc = p.C - cb * kCB < kCB ? p.C - cb * kCB : kCB;
  const int64_t E = p.C * FF, base = cb * kCB * FF;  // dW [C][F][F][1]: the tile is contiguous
  for (int64_t i = threadIdx.x; i < nc * FF; i += kThreads) {
    if (ws) ws[(int64_t)sigma * E + base + i] = res[i];
    else store_out(out + base + i, res[i]);
  }
  if (db) {
    for (int64_t i = threadIdx.x; i < nc; i += kThreads) {
      if (ws_bias) ws_bias[(int64_t)sigma * p.C + cb * kCB + i] = resb[i];
      else store_out(db + cb * kCB + i, resb[i]);
    }
  }
}

template <typename TI, typename TO, int F>
cudaError_t launch_f(const Plan& pl, const Args& a, const RingParams& p, CUtensorMapDataType dt) {
  const Shape& s = pl.sh;
  CUtensorMap tm_x, tm_dy;
  const uint64_t x_dims[4] = {(uint64_t)s.c, (uint64_t)s.w, (uint64_t)s.h, (uint64_t)s.n};
  const uint64_t x_strides[3] = {(uint64_t)s.c * 2u, (uint64_t)(s.w * s.c) * 2u, (uint64_t)(s.h * s.w * s.c) * 2u};
  const uint32_t x_box[4] = {(uint32_t)kCB, (uint32_t)s.w, 1u, 1u};
  const uint64_t y_dims[4] = {(uint64_t)s.c, (uint64_t)s.wo, (uint64_t)s.ho, (uint64_t)s.n};
  const uint64_t y_strides[3] = {(uint64_t)s.c * 2u, (uint64_t)(s.wo * s.c) * 2u, (uint64_t)(s.ho * s.wo * s.c) * 2u};
  const uint32_t y_box[4] = {(uint32_t)kCB, (uint32_t)s.wo, 1u, 1u};
  if (!encode_tmap(&tm_x, dt, 4, a.x, x_dims, x_strides, x_box, CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !encode_tmap(&tm_dy, dt, 4, a.b, y_dims, y_strides, y_box, CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  const size_t smem = kernel_smem(s, RingShape{p.RS - 1, p.TR});
  auto kern = dw_wgrad_ring_kernel<TI, TO, F>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  const int64_t ctas = pl.geo.tiles * pl.split;
  if (ctas > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  kern<<<(unsigned)ctas, kThreads, smem, a.stream>>>(tm_x, tm_dy, static_cast<TO*>(a.out), a.ws,
                                                     pl.with_bias ? static_cast<TO*>(a.db) : nullptr, a.ws_bias, p,
                                                     device_error_word());
  return cudaGetLastError();
}

template <typename TI, typename TO>
cudaError_t launch_typed(const Plan& pl, const Args& a, CUtensorMapDataType dt) {
  const Shape& s = pl.sh;
  RingParams p;
  p.C = s.c;
  p.Ho = s.ho;
  p.rows = s.n * s.ho;
  p.cblocks = (s.c + kCB - 1) / kCB;
  p.W = (int32_t)s.w;
  p.Wo = (int32_t)s.wo;
  p.ph = (int32_t)s.ph;
  p.pw = (int32_t)s.pw;
  p.CW = (int32_t)((s.w + kWarps - 1) / kWarps);
  const RingShape rs = ring_shape(s);
  if (rs.d < 1) return cudaErrorInvalidValue;
  p.ahead = ahead_of_depth(rs.d);
  p.TR = rs.tr;
  p.RX = (int32_t)ring_rows(s.s, s.ho, rs.d, rs.tr);
  p.RS = 1 + rs.d;
  p.red_off = (int32_t)reduce_offset(s, rs);
  p.split = pl.split;
  switch (s.s) {
    case 3: return launch_f<TI, TO, 3>(pl, a, p, dt);
    case 5: return launch_f<TI, TO, 5>(pl, a, p, dt);
    case 7: return launch_f<TI, TO, 7>(pl, a, p, dt);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

Geometry geometry_wgrad_depthwise_ring(const Shape& s) {
  Geometry g;
  const bool depthwise = s.groups == s.c && s.groups == s.k;
  if (!depthwise || s.in_dt == CONV_F32 || s.n < 1) return g;
  if (s.r != s.s || !(s.s == 3 || s.s == 5 || s.s == 7)) return g;
  if (s.sh != 1 || s.sw != 1 || s.dh != 1 || s.dw != 1) return g;
  if (s.pw > s.s - 1 || s.ph > s.r - 1) return g;
  // TMA: 16-byte row strides, a 64-channel box inside the channel extent,
  // whole rows of at most 256 columns; coordinates in 32 bits.
  if (s.c % 8 != 0 || s.c < kCB || s.w > 256 || s.wo > 256) return g;
  if (s.n > 0x7fffffffLL || s.h + s.r > 0x7fffffffLL) return g;
  if (ring_shape(s).d < 1) return g;
  g.ok = true;
  g.ctas_per_sm = 1;
  g.tiles = (s.c + kCB - 1) / kCB;
  g.blocks = s.n * s.ho;
  return g;
}

cudaError_t launch_wgrad_depthwise_ring(const Plan& p, const Args& a) {
  const int in = p.sh.in_dt, out = p.sh.out_dt;
  if (in == CONV_BF16)
    return out == CONV_F32 ? launch_typed<__nv_bfloat16, float>(p, a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16)
                           : launch_typed<__nv_bfloat16, __nv_bfloat16>(p, a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16);
  return out == CONV_F32 ? launch_typed<__half, float>(p, a, CU_TENSOR_MAP_DATA_TYPE_FLOAT16)
                         : launch_typed<__half, __half>(p, a, CU_TENSOR_MAP_DATA_TYPE_FLOAT16);
}

}  // namespace cig
