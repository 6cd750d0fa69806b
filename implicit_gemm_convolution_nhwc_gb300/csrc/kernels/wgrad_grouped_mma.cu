// Grouped 16-bit weight gradient (+ bias gradient) on warp-level tensor-core
// MMAs ("perf(rocke): depthwise 7x7 and grouped cpg4/8 wgrad on batched mfma
// 4x4x4", "Technical Details": the grouped wgrad), for Cg = Kg in
// {2, 4, 8, 16, 32}, C % 64 = 0, unit stride and dilation.
//
//   dW[k, r, s, c] = sum over (n, ho, u) of dY[n, ho, u - s + pw, k] * X[n, ho + r - ph, u, c]
//
// (u = wo + s - pw runs over the input columns; dY is zero outside
// [0, Wo) and X outside the image.) For one group, input row ho + r - ph and
// a run of 16 input columns u this is an MMA m16n8k16 with the reduction
// over u: B[u][c] = X[row][u][c] (8 input channels, N) and
// A[(s, k)][u] = dY[ho][u - s + pw][k] (8 output channels for each of two
// filter columns s, M = 16): the filter column shifts dY, not X, so both
// halves of M are useful (with the shift on X instead, one MMA would hold a
// single tap and half of M would idle). Every product of the 16 x 8 result is
// a weight-gradient element: nothing is thrown away for 8 or more channels
// per group. Both fragments come from ldmatrix.trans of the NHWC rows as TMA
// lands them (128B swizzle, so the eight pixels of a matrix hit eight
// different bank groups), the per-lane row addresses doing the shift.
//
// Rows stream as in the depthwise weight gradient's ring (dw_ring.cuh): a CTA
// owns 64 channels and a split-K slice of (n, ho) output rows, walked TR rows
// (a step) at a time; input rows ho - ph .. ho - ph + R - 1 form one
// sequence through a ring of row slots (box {64 channels, 16-column multiple
// of W columns}, zero past the image), and a step's dY rows sit in its step
// slot, each loaded from column pw - S + 1 so every shifted read is in the
// slot (TMA zero-fills dY outside [0, Wo)). Warp w owns the (k chunk, c
// chunk) pairs w, w + 8, ... of the CTA's 8 channel chunks of 8 (for fewer
// than 8 channels per group a chunk holds several groups, and only its
// diagonal blocks are kept) and the bias sum of chunk w. Each output element
// belongs to one warp and one lane: no reduction across warps, and the sums
// run in a fixed order (deterministic).
#include <type_traits>

#include "dw_ring.cuh"
#include "../kernel_entry.h"

namespace cig {
namespace {

using dwring::ring_rows;
using dwring::RowPos;
using dwring::StepPos;

constexpr int kCB = 64;        // channels per CTA: 8 chunks of 8
constexpr int kMaxDepth = 6;   // ahead + slack, at most
constexpr int kMaxTR = 8;      // output rows a step, at most
constexpr size_t kSmemLimit = 227 * 1024;

struct GmParams {
  int64_t C, Ho;
  int64_t rows;     // N * Ho: the reduction blocks
  int64_t cblocks;  // C / 64: the tiles
  int32_t W, Wo, ph, pw, S, Cg;
  int32_t US;       // steps of 16 input columns: ceil(W / 16)
  int32_t XP, DP;   // pixels of an input-row slot and of a dY-row slot (multiples of 8)
  int32_t RX, RS;   // ring slots: input rows, steps
  int32_t TR;       // output rows a step
  int32_t ahead;    // steps between a load's issue and its use
  int32_t split;
};

// Pixels of the slots: input columns 0 .. 16 US - 1; dY columns
// pw - S + 1 .. pw + 16 US - 1; rounded up to 8 pixels (1024 bytes, the
// 128B-swizzle atom a TMA destination starts on).
int64_t x_slot_pixels(const Shape& s) { return (s.w + 15) / 16 * 16; }
int64_t dy_slot_pixels(const Shape& s) { return ((s.w + 15) / 16 * 16 + s.s - 1 + 7) / 8 * 8; }

size_t ring_smem(const Shape& s, int d, int tr) {
  const int64_t rx = ring_rows(s.r, s.ho, d, tr), rs = 1 + d;
  return 1024 + (size_t)(rx * x_slot_pixels(s) * 128 + rs * tr * dy_slot_pixels(s) * 128) + 2 * rs * 8 + rs * 4 + 16 +
         (size_t)rs * tr * 4;
}

struct RingShape {
  int d = 0, tr = 0;
};

int warp_groups(const Shape& s);

// The most rows a step (up to 8: the per-step bookkeeping is paid once per
// step) that still lets the loads run two steps ahead with two of slack, a
// multiple of the warp groups (which split a step's rows evenly); else the
// most rows with the deepest ring that fits, at least one step ahead and one
// of slack. With one step of 7 rows ahead the warps waited for their rows for
// a quarter of the loop.
RingShape ring_shape(const Shape& s) {
  const int ng = warp_groups(s);
  for (int tr = kMaxTR; tr >= ng; --tr) {
    if (tr % ng != 0) continue;
    for (int d = kMaxDepth; d >= 4; --d)
      if (ring_smem(s, d, tr) <= kSmemLimit) return RingShape{d, tr};
  }
  for (int tr = kMaxTR; tr >= 1; --tr)
    for (int d = kMaxDepth; d >= 2; --d)
      if (ring_smem(s, d, tr) <= kSmemLimit) return RingShape{d, tr};
  return RingShape{};
}

int ahead_of_depth(int d) { return d >= 4 ? d - 1 : 1; }

struct Ring {
  const CUtensorMap* tm_x;
  const CUtensorMap* tm_dy;
  const CUtensorMap* tm_xt;   // boxes of TR input rows (TR consecutive ring slots)
  const CUtensorMap* tm_dyt;  // boxes of TR dY rows (a whole step slot)
  uint8_t* xring;
  uint8_t* dring;
  uint64_t* full;
  uint64_t* empty;
  int32_t* siss;  // wrap count of the last step loaded into each step slot (-1: none)
  volatile uint32_t* abort_flag;
  // per step slot and row: the shared address of the ring slot of the row's last input row, + 1
  // when the row starts a new input-row sequence (the run's first row or an image's first row)
  int32_t* rowinfo;
  unsigned* err;
  uint32_t rowX, rowD, txX, txD, txXT, txDT;
  int32_t c0;
};

// Loads a step: the dY rows of its `rows` output rows (the first at row
// position a) and the input rows they are the first to read, all landing on
// the step slot's full mbarrier, once every warp is done with the slot's
// previous step. False: the wait gave up. A full step within one image loads
// its dY rows as one box of TR rows, and, when each row adds one input row
// and their ring slots do not wrap, its input rows as one more: two copies a
// step instead of 2 TR (issuing each copy costs the issuing warp a few
// hundred cycles).
template <int R>
__device__ bool issue_step(const Ring& g, const GmParams& p, RowPos a, StepPos st, int32_t rows) {
  if (st.sw > 0 && !mbar_wait(&g.empty[st.ss], (st.sw - 1u) & 1u, g.abort_flag, g.err)) return false;
  const bool dblk = rows == p.TR && a.ho + p.TR <= p.Ho;
  const int32_t s0 = a.slot(R - 1, p);
  const bool xblk = dblk && !a.first && a.ho != 0 && s0 + p.TR <= p.RX;
  uint32_t bytes = (dblk ? g.txDT : 0u) + (xblk ? g.txXT : 0u);
  // the rows' input slots, published by the arrive below (release) to the warps that wait on it
  const uint32_t xbase = smem_u32(g.xring);
  if (xblk) {  // consecutive slots, none starting a window
    for (int32_t j = 0; j < rows; ++j) g.rowinfo[st.ss * p.TR + j] = (int32_t)(xbase + (uint32_t)(s0 + j) * g.rowX);
  } else {
    RowPos b = a;
    for (int32_t j = 0; j < rows; ++j, b.advance(R, p)) {
      if (!dblk) bytes += g.txD;
      bytes += (uint32_t)b.fresh(R) * g.txX;
      g.rowinfo[st.ss * p.TR + j] =
          (int32_t)(xbase + (uint32_t)b.slot(R - 1, p) * g.rowX + (b.fresh(R) == R ? 1u : 0u));
    }
  }
  uint64_t* bar = &g.full[st.ss];
  mbar_arrive_expect_tx(bar, bytes);
  if (dblk)
    tma_load_4d(g.dring + (size_t)st.ss * p.TR * g.rowD, g.tm_dyt, g.c0, p.pw - p.S + 1, a.ho, a.n, bar);
  if (xblk) tma_load_4d(g.xring + (size_t)s0 * g.rowX, g.tm_xt, g.c0, 0, a.ho - p.ph + R - 1, a.n, bar);
  if (!dblk || !xblk) {
    for (int32_t j = 0; j < rows; ++j, a.advance(R, p)) {
      if (!dblk)
        tma_load_4d(g.dring + ((size_t)st.ss * p.TR + j) * g.rowD, g.tm_dy, g.c0, p.pw - p.S + 1, a.ho, a.n, bar);
      if (!xblk)
        for (int r = R - a.fresh(R); r < R; ++r)
          tma_load_4d(g.xring + (size_t)a.slot(r, p) * g.rowX, g.tm_x, g.c0, 0, a.ho - p.ph + r, a.n, bar);
    }
  }
  g.siss[st.ss] = (int32_t)st.sw;
  return true;
}

// 16-byte chunk `ch` of pixel `pix` in a 128B-swizzled slot at shared address base.
__device__ __forceinline__ uint32_t chunk_addr(uint32_t base, int32_t pix, int32_t ch) {
  return base + (uint32_t)(pix * 128) + ((uint32_t)(ch ^ (pix & 7)) << 4);
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&v)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2_t(uint32_t addr, uint32_t (&v)[2]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0, %1}, [%2];" : "=r"(v[0]), "=r"(v[1]) : "r"(addr));
}

template <typename TI>
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]);
template <>
__device__ __forceinline__ void mma16816<__nv_bfloat16>(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
  asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
               : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
               : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}
template <>
__device__ __forceinline__ void mma16816<__half>(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
  asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
               : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
               : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// The c chunk of pair i of the warp that owns k chunk w (every pair of a warp
// shares its k chunk, so the A fragments are loaded once for all of them):
// for Cg >= 8 the i-th of the Cg / 8 chunks of w's group, for Cg < 8 chunk w
// itself (which holds several whole groups).
__device__ __forceinline__ int c_chunk_of(int w, int i, int cg) {
  if (cg < 8) return w;
  const int g8 = cg / 8;
  return (w / g8) * g8 + i;
}

// The fragments of one 16-column step: A for each pair of filter columns, B
// for each filter row.
template <int R, int SP, int CPW>
struct Frags {
  uint32_t a[SP][4];
  uint32_t b[CPW][R][2];
};

// SP = ceil(S / 2) pairs of filter columns; CPW chunk pairs a warp; NG warp
// groups of 8 (a group takes every NG-th row of a step; their sums are added
// in group order at the end).
template <typename TI, typename TO, int R, int SP, int CPW, int NG>
__global__ void __launch_bounds__(256 * NG, 1)
    wgrad_grouped_mma_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_dy,
                             const __grid_constant__ CUtensorMap tm_xt, const __grid_constant__ CUtensorMap tm_dyt,
                             TO* out, float* ws, TO* db, float* ws_bias, GmParams p, unsigned* err) {
  constexpr int kT = 256 * NG;          // threads
  constexpr int kW = kT / 32;           // warps
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  Ring g;
  g.tm_x = &tm_x;
  g.tm_dy = &tm_dy;
  g.tm_xt = &tm_xt;
  g.tm_dyt = &tm_dyt;
  g.rowX = (uint32_t)p.XP * 128u;
  g.rowD = (uint32_t)p.DP * 128u;
  g.txX = (uint32_t)(p.US * 16) * 128u;
  g.txD = (uint32_t)(p.US * 16 + p.S - 1) * 128u;
  g.txXT = (uint32_t)p.TR * g.txX;  // the TR-row boxes: input rows US * 16 pixels, dY rows the slot's DP
  g.txDT = (uint32_t)p.TR * g.rowD;
  g.xring = smem;
  g.dring = smem + (size_t)p.RX * g.rowX;
  g.full = reinterpret_cast<uint64_t*>(g.dring + (size_t)p.RS * p.TR * g.rowD);
  g.empty = g.full + p.RS;
  g.siss = reinterpret_cast<int32_t*>(g.empty + p.RS);
  g.abort_flag = reinterpret_cast<volatile uint32_t*>(g.siss + p.RS);
  g.rowinfo = reinterpret_cast<int32_t*>(g.siss + p.RS + 4);
  g.err = err;

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int wl = warp & 7, grp = warp >> 3;  // warp within its group, group
  const int64_t cb = blockIdx.x % p.cblocks;
  const int32_t sigma = (int32_t)(blockIdx.x / p.cblocks);
  g.c0 = (int32_t)(cb * kCB);
  const int64_t q_b = slice_begin(p.rows, p.split, sigma), q_e = slice_begin(p.rows, p.split, sigma + 1);

  if (threadIdx.x == 0) {
    for (int i = 0; i < p.RS; ++i) {
      mbar_init(&g.full[i], 1);
      mbar_init(&g.empty[i], kW);
      g.siss[i] = -1;
    }
    *g.abort_flag = 0u;
    mbar_fence_init();
    tma_prefetch(&tm_x);
    tma_prefetch(&tm_dy);
    tma_prefetch(&tm_xt);
    tma_prefetch(&tm_dyt);
    // The first `ahead` steps load into fresh slots.
    RowPos a{0, (int32_t)(q_b % p.Ho), (int32_t)(q_b / p.Ho), true};
    StepPos st{0, 0u};
    for (int64_t q = q_b; q < q_e && st.ss < p.ahead; st.advance(p)) {
      const int32_t rows = q_e - q < p.TR ? (int32_t)(q_e - q) : p.TR;
      issue_step<R>(g, p, a, st, rows);
      for (int32_t j = 0; j < rows; ++j, ++q) a.advance(R, p);
    }
  }
  __syncthreads();

  // This warp's chunk pairs and the lane's ldmatrix rows: for A (x4) matrix
  // mi = lane / 8 holds filter column s0 (mi even) or s1 (mi odd) and input
  // columns u0 + 8 (mi / 2) + lane % 8; for B (x2) lanes 0..15 give input
  // columns u0 + lane (lanes 16..31 repeat them; their addresses are unused).
  // u0 is a multiple of 16, so the swizzled offset of a lane's row within a
  // slot is u0 * 128 plus a per-lane constant.
  const int kch = wl;
  int cch[CPW];
#pragma unroll
  for (int i = 0; i < CPW; ++i) cch[i] = c_chunk_of(wl, i, p.Cg);
  const int mi = lane >> 3, arow = (mi >> 1) * 8 + (lane & 7), brow = lane & 15;
  // aoff: the x4 load of a pair (a single last column, S odd, fills both halves)
  uint32_t aoff[SP], boff[CPW];
#pragma unroll
  for (int sp = 0; sp < SP; ++sp) {
    const int s = 2 * sp + (mi & 1);
    const int pix = arow + p.S - 1 - (s < p.S ? s : p.S - 1);  // dY slot pixel = input column + S - 1 - s
    aoff[sp] = chunk_addr(0u, pix, kch);
  }
#pragma unroll
  for (int i = 0; i < CPW; ++i) boff[i] = chunk_addr(0u, brow, cch[i]);
  // The bias of chunk wl comes from the A fragments of filter column pw (a
  // real tap), whose window is dY columns 0 .. 16 US - 1, each once, zero past
  // Wo: one more MMA a row with a B of ones sums them over the 16 columns
  // (every column of the result is that sum). Thread (g = lane / 4) holds
  // row g (filter column 2 bsp, output channel g) in register 0 and row g + 8
  // (column 2 bsp + 1) in register 2.
  const int bsp = p.pw / 2, bh = p.pw % 2;
  const uint32_t one2 = std::is_same<TI, __half>::value ? 0x3C003C00u : 0x3F803F80u;  // two 1.0s
  const uint32_t ones[2] = {one2, one2};
  float acc[CPW][R][SP][4];
#pragma unroll
  for (int i = 0; i < CPW; ++i)
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int sp = 0; sp < SP; ++sp)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[i][r][sp][e] = 0.f;
  float bacc[4] = {0.f, 0.f, 0.f, 0.f};
  const uint32_t dring_u32 = smem_u32(g.dring), xring_u32 = smem_u32(g.xring);

  StepPos sc{0, 0u};
  StepPos sl{0, 0u};  // the step slot of step S + ahead
  for (int i = 0; i < p.ahead; ++i) sl.advance(p);
  int32_t issuer = 0;  // warp that loads at step S: S mod kW
  int64_t qa = q_b + (int64_t)p.ahead * p.TR;  // first row of step S + ahead
  // The issuing lane places row qa in closed form (only it pays the divisions):
  // its image and row, and its first input row's index in the slice's input-row
  // sequence (R rows for the slice's first row and for each image start, one
  // more for every other row), which modulo RX is its ring slot.
  // (32-bit arithmetic: N * Ho < 2^31 is a condition of the kernel.)
  const uint32_t ho_u = (uint32_t)p.Ho, n_b = (uint32_t)q_b / ho_u;
  auto row_pos = [&](int64_t qq) {
    const uint32_t n = (uint32_t)qq / ho_u, ho = (uint32_t)qq - n * ho_u;
    const uint32_t seq = (uint32_t)(qq - q_b) + (uint32_t)(R - 1) * (n - n_b);
    return RowPos{(int32_t)(seq % (uint32_t)p.RX), (int32_t)ho, (int32_t)n, qq == q_b};
  };

  for (int64_t q = q_b; q < q_e; q += p.TR) {
    const int32_t rows = q_e - q < p.TR ? (int32_t)(q_e - q) : p.TR;
    if (warp == issuer && lane == 0 && qa < q_e)
      issue_step<R>(g, p, row_pos(qa), sl, q_e - qa < p.TR ? (int32_t)(q_e - qa) : p.TR);
    // Lanes that spin on an mbarrier can hold up a divergent lane of the same
    // warp; reconverge before any of them waits.
    __syncwarp();
    qa += p.TR;
    sl.advance(p);
    issuer = issuer + 1 == kW ? 0 : issuer + 1;

    if (!__all_sync(0xffffffffu, mbar_wait(&g.full[sc.ss], sc.sw & 1u, g.abort_flag, g.err))) break;

    {
      // This group's rows of the step: a contiguous run [j0, j1), walked for
      // each 16-column step with the B fragments of the R input rows in a
      // window that slides by one row within an image (one new input row a row).
      const int32_t j0 = (rows * grp) / NG, j1 = (rows * (grp + 1)) / NG;
      const int32_t* info = g.rowinfo + sc.ss * p.TR + j0;
#pragma unroll 1
      for (int32_t us = 0; us < p.US; ++us) {
        const uint32_t uo = (uint32_t)us * 2048u;
        uint32_t bw[CPW][R][2];
#pragma unroll
        for (int32_t jj = 0; jj < kMaxTR; ++jj) {
          if (j0 + jj >= j1) break;
          const int32_t j = j0 + jj;
          const int32_t inf = info[jj];
          const uint32_t xlast = (uint32_t)inf & ~1u;  // the window's last input row
          if (jj == 0 || (inf & 1) != 0) {  // a fresh window: rows R - 1 - r before the last, in the ring
#pragma unroll
            for (int r = 0; r < R; ++r) {
              int32_t xa = (int32_t)xlast - (R - 1 - r) * (int32_t)g.rowX;
              if (xa < (int32_t)xring_u32) xa += p.RX * (int32_t)g.rowX;
#pragma unroll
              for (int i = 0; i < CPW; ++i) ldsm_x2_t((uint32_t)xa + uo + boff[i], bw[i][r]);
            }
          } else {  // slide by one input row
            const uint32_t xa = xlast + uo;
#pragma unroll
            for (int i = 0; i < CPW; ++i) {
#pragma unroll
              for (int r = 0; r + 1 < R; ++r) {
                bw[i][r][0] = bw[i][r + 1][0];
                bw[i][r][1] = bw[i][r + 1][1];
              }
              ldsm_x2_t(xa + boff[i], bw[i][R - 1]);
            }
          }
          const uint32_t dslot = dring_u32 + (uint32_t)((sc.ss * p.TR + j) * g.rowD) + uo;
          uint32_t af[SP][4];
#pragma unroll
          for (int sp = 0; sp < SP; ++sp) ldsm_x4_t(dslot + aoff[sp], af[sp]);
#pragma unroll
          for (int i = 0; i < CPW; ++i)
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
              for (int sp = 0; sp < SP; ++sp) mma16816<TI>(acc[i][r][sp], af[sp], bw[i][r]);
#pragma unroll
          for (int sp = 0; sp < SP; ++sp)  // the pair holding filter column pw (a select, no local memory)
            if (sp == bsp) mma16816<TI>(bacc, af[sp], ones);
        }
      }
    }

    __syncwarp();
    if (lane == 0) mbar_arrive(&g.empty[sc.ss]);
    sc.advance(p);
  }
  signal_dependents();

  // No copy may still be landing in shared memory when the CTA exits, nor
  // when the groups' sums reuse it below (wait for the last step loaded into
  // each step slot; bounded, no early exit).
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int i = 0; i < p.RS; ++i)
      if (g.siss[i] >= 0) mbar_wait(&g.full[i], (uint32_t)g.siss[i] & 1u, nullptr, err);
  }
  __syncthreads();
  const bool ok = *g.abort_flag == 0u;

  // the bias partial sum of output channel lane / 4 of chunk wl (every lane of the channel holds it)
  float bsum = bh ? bacc[2] : bacc[0];
  if (NG > 1) {
    // groups 1.. hand their sums to group 0 through shared memory (over the
    // ring), which adds them in group order
    constexpr int NV = CPW * R * SP * 4;
    float* red = reinterpret_cast<float*>(smem);  // [group - 1][8 warps][NV + 1][32 lanes]
    if (grp > 0) {
      float* mine = red + (((size_t)(grp - 1) * 8 + wl) * (NV + 1)) * 32 + lane;
      int v = 0;
#pragma unroll
      for (int i = 0; i < CPW; ++i)
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
          for (int sp = 0; sp < SP; ++sp)
#pragma unroll
            for (int e = 0; e < 4; ++e) mine[(v++) * 32] = acc[i][r][sp][e];
      mine[NV * 32] = bsum;
    }
    __syncthreads();
    if (grp > 0) return;
#pragma unroll 1
    for (int gg = 1; gg < NG; ++gg) {
      const float* theirs = red + (((size_t)(gg - 1) * 8 + wl) * (NV + 1)) * 32 + lane;
      int v = 0;
#pragma unroll
      for (int i = 0; i < CPW; ++i)
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
          for (int sp = 0; sp < SP; ++sp)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[i][r][sp][e] += theirs[(v++) * 32];
      bsum += theirs[NV * 32];
    }
  }

  // The results: fragment element e of pair i, filter row r and column pair
  // sp is row m = lane / 4 + 8 (e / 2) (filter column 2 sp + m / 8, output
  // channel m % 8 of the k chunk) and column n = 2 (lane % 4) + e % 2 (input
  // channel n of the c chunk).
  // Cg divides 64 (a power of two), so the CTA's first channel is a group
  // boundary: group membership and the channel within the group follow from
  // the channel indices within the CTA by masks (no 64-bit divisions).
  const int32_t cgm = p.Cg - 1;
  const int64_t E = p.C * R * p.S * (int64_t)p.Cg;  // dW elements (C = K)
  float* slab = ws ? ws + (int64_t)sigma * E : nullptr;
#pragma unroll
  for (int i = 0; i < CPW; ++i)
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int sp = 0; sp < SP; ++sp)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int m = (lane >> 2) + 8 * (e >> 1), n = 2 * (lane & 3) + (e & 1);
          const int s = 2 * sp + (m >> 3);
          const int32_t kl = kch * 8 + (m & 7), cl = cch[i] * 8 + n;  // within the CTA's 64 channels
          if (!ok || s >= p.S || ((kl ^ cl) & ~cgm) != 0) continue;
          const int64_t k = cb * kCB + kl;
          const int64_t dst = ((k * R + r) * p.S + s) * p.Cg + (cl & cgm);
          if (ws) slab[dst] = acc[i][r][sp][e];
          else store_out(out + dst, acc[i][r][sp][e]);
        }
  if ((db || ws_bias) && (lane & 3) == 0 && ok) {
    const int64_t k = cb * kCB + wl * 8 + (lane >> 2);
    if (ws_bias) ws_bias[(int64_t)sigma * p.C + k] = bsum;
    else store_out(db + k, bsum);
  }
}

// Chunk pairs a warp: 8 pairs a CTA for Cg <= 8, Cg for more.
int pairs_per_warp(const Shape& s) { return s.cg <= 8 ? 1 : (int)(s.cg / 8); }

// Warp groups: 2 (512 threads) when a warp's accumulator tiles (R x SP x pairs) are at most 8, so its
// registers stay within the 128 a thread that 512 threads allow; else 1.
constexpr int groups_of(int tiles) { return tiles <= 8 ? 2 : 1; }
// The filter columns' pairs the kernel is instantiated with for R filter rows.
int sp_of(int64_t r) { return r == 1 ? 1 : r == 3 ? 2 : 3; }
int warp_groups(const Shape& s) { return groups_of((int)(s.r * sp_of(s.r) * pairs_per_warp(s))); }

template <typename TI, typename TO, int R, int SP, int CPW, int NG>
cudaError_t launch_k(const Plan& pl, const Args& a, const GmParams& p, CUtensorMapDataType dt, size_t smem) {
  const Shape& s = pl.sh;
  CUtensorMap tm_x, tm_dy, tm_xt, tm_dyt;
  const uint64_t x_dims[4] = {(uint64_t)s.c, (uint64_t)s.w, (uint64_t)s.h, (uint64_t)s.n};
  const uint64_t x_strides[3] = {(uint64_t)s.c * 2u, (uint64_t)(s.w * s.c) * 2u, (uint64_t)(s.h * s.w * s.c) * 2u};
  const uint32_t x_box[4] = {(uint32_t)kCB, (uint32_t)(p.US * 16), 1u, 1u};
  const uint64_t y_dims[4] = {(uint64_t)s.k, (uint64_t)s.wo, (uint64_t)s.ho, (uint64_t)s.n};
  const uint64_t y_strides[3] = {(uint64_t)s.k * 2u, (uint64_t)(s.wo * s.k) * 2u, (uint64_t)(s.ho * s.wo * s.k) * 2u};
  const uint32_t y_box[4] = {(uint32_t)kCB, (uint32_t)(p.US * 16 + s.s - 1), 1u, 1u};
  // the same tensors in boxes of TR rows: TR ring slots of input rows, a whole dY step slot (DP pixels a row)
  const uint32_t xt_box[4] = {(uint32_t)kCB, (uint32_t)(p.US * 16), (uint32_t)p.TR, 1u};
  const uint32_t yt_box[4] = {(uint32_t)kCB, (uint32_t)p.DP, (uint32_t)p.TR, 1u};
  if (!encode_tmap(&tm_x, dt, 4, a.x, x_dims, x_strides, x_box, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tmap(&tm_dy, dt, 4, a.b, y_dims, y_strides, y_box, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tmap(&tm_xt, dt, 4, a.x, x_dims, x_strides, xt_box, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tmap(&tm_dyt, dt, 4, a.b, y_dims, y_strides, yt_box, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  auto kern = wgrad_grouped_mma_kernel<TI, TO, R, SP, CPW, NG>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  const int64_t ctas = pl.geo.tiles * pl.split;
  if (ctas > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  kern<<<(unsigned)ctas, 256 * NG, smem, a.stream>>>(tm_x, tm_dy, tm_xt, tm_dyt, static_cast<TO*>(a.out), a.ws,
                                                     pl.with_bias ? static_cast<TO*>(a.db) : nullptr,
                                                     pl.with_bias ? a.ws_bias : nullptr, p, device_error_word());
  return cudaGetLastError();
}

// Chunk pairs a warp: 1, 2 or 4, as many as keep R x SP x pairs <= 24 accumulator tiles.
template <typename TI, typename TO, int R, int SP>
cudaError_t launch_rs(const Plan& pl, const Args& a, const GmParams& p, CUtensorMapDataType dt, size_t smem) {
  // two groups of 8 warps (16 warps an SM) while the accumulators stay small enough
  switch (pairs_per_warp(pl.sh)) {
    case 1: return launch_k<TI, TO, R, SP, 1, groups_of(R * SP)>(pl, a, p, dt, smem);
    case 2: return R * SP * 2 <= 24
                       ? launch_k<TI, TO, R, SP, (R * SP * 2 <= 24 ? 2 : 1), groups_of(R * SP * 2)>(pl, a, p, dt, smem)
                       : cudaErrorInvalidValue;
    case 4: return R * SP * 4 <= 24
                       ? launch_k<TI, TO, R, SP, (R * SP * 4 <= 24 ? 4 : 1), groups_of(R * SP * 4)>(pl, a, p, dt, smem)
                       : cudaErrorInvalidValue;
    default: return cudaErrorInvalidValue;
  }
}

template <typename TI, typename TO>
cudaError_t launch_typed(const Plan& pl, const Args& a, CUtensorMapDataType dt) {
  const Shape& s = pl.sh;
  GmParams p;
  p.C = s.c;
  p.Ho = s.ho;
  p.rows = s.n * s.ho;
  p.cblocks = s.c / kCB;
  p.W = (int32_t)s.w;
  p.Wo = (int32_t)s.wo;
  p.ph = (int32_t)s.ph;
  p.pw = (int32_t)s.pw;
  p.S = (int32_t)s.s;
  p.Cg = (int32_t)s.cg;
  p.US = (int32_t)((s.w + 15) / 16);
  p.XP = (int32_t)x_slot_pixels(s);
  p.DP = (int32_t)dy_slot_pixels(s);
  const RingShape rs = ring_shape(s);
  if (rs.d < 1) return cudaErrorInvalidValue;
  p.ahead = ahead_of_depth(rs.d);
  p.TR = rs.tr;
  p.RX = (int32_t)ring_rows(s.r, s.ho, rs.d, rs.tr);
  p.RS = 1 + rs.d;
  p.split = pl.split;
  const size_t smem = ring_smem(s, rs.d, rs.tr);
  // filter rows -> the instantiated column pairs (3 rows: up to 4 columns, 5 rows: up to 6)
  switch (s.r) {
    case 1: return launch_rs<TI, TO, 1, 1>(pl, a, p, dt, smem);
    case 3: return launch_rs<TI, TO, 3, 2>(pl, a, p, dt, smem);
    case 5: return launch_rs<TI, TO, 5, 3>(pl, a, p, dt, smem);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

Geometry geometry_wgrad_grouped_mma(const Shape& s) {
  Geometry g;
  if (s.in_dt == CONV_F32 || s.groups < 2 || s.cg != s.kg || s.n < 1) return g;
  if (!(s.cg == 2 || s.cg == 4 || s.cg == 8 || s.cg == 16 || s.cg == 32)) return g;
  if (s.c % kCB != 0) return g;
  if (s.sh != 1 || s.sw != 1 || s.dh != 1 || s.dw != 1) return g;
  // filters: 1x1, 3 rows of up to 4 columns, 5 rows of up to 6 columns; the accumulators of a
  // warp's chunk pairs (R x ceil(S/2) x 4 floats each) at most 96 registers
  const int64_t sp = (s.s + 1) / 2;
  if (!((s.r == 1 && s.s == 1) || (s.r == 3 && sp <= 2 && s.s >= 1) || (s.r == 5 && sp <= 3))) return g;
  const int64_t spk = sp_of(s.r);  // the instantiated column pairs
  if (s.r * spk * pairs_per_warp(s) > 24) return g;
  if (s.ph > s.r - 1 || s.pw > s.s - 1) return g;
  // TMA: rows of at most 256 columns (the dY box adds S - 1), 32-bit coordinates
  if ((s.w + 15) / 16 * 16 + s.s - 1 > 256 || s.wo > s.w + 2 * s.pw) return g;
  if (s.n > 0x7fffffffLL || s.h + s.r > 0x7fffffffLL) return g;
  if (s.n * s.ho > 0x7fffffffLL) return g;  // the issuing lane places rows in 32-bit arithmetic
  const RingShape rs = ring_shape(s);
  if (rs.d < 1) return g;
  // two warp groups add their sums through shared memory over the ring's rows
  const int64_t tiles = s.r * spk * pairs_per_warp(s);
  const size_t ring_bytes = ring_smem(s, rs.d, rs.tr) - 1024;
  if (tiles <= 8 && (size_t)(tiles * 4 + 1) * 8 * 32 * 4 > ring_bytes) return g;
  g.ok = true;
  g.ctas_per_sm = 1;
  g.tiles = s.c / kCB;
  g.blocks = s.n * s.ho;
  return g;
}

cudaError_t launch_wgrad_grouped_mma(const Plan& p, const Args& a) {
  const int in = p.sh.in_dt, out = p.sh.out_dt;
  if (in == CONV_BF16)
    return out == CONV_F32 ? launch_typed<__nv_bfloat16, float>(p, a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16)
                           : launch_typed<__nv_bfloat16, __nv_bfloat16>(p, a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16);
  return out == CONV_F32 ? launch_typed<__half, float>(p, a, CU_TENSOR_MAP_DATA_TYPE_FLOAT16)
                         : launch_typed<__half, __half>(p, a, CU_TENSOR_MAP_DATA_TYPE_FLOAT16);
}

}  // namespace cig
