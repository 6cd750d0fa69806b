// 16-bit grouped forward convolution on warp-level tensor-core MMAs, and with
// the filter turned the stride-1 grouped data gradient, for 4 or 8 channels
// per group (Cg = Kg), unit stride and dilation, 1x1, 3x3 and 5x5 filters,
// rows of at most 64 output columns:
//
//   Y[n, ho, wo, k] = sum over (r, s, c in k's group) of X[n, ho + r - ph, wo + s - pw, c] * W[k, r, s, c]
//
// ("perf(rocke): depthwise 7x7 and grouped cpg4/8 wgrad on batched mfma
// 4x4x4", "Technical Details": small per-group matrix products instead of
// block-diagonal dense ones.) For one output row and 16 output columns this is
// an MMA m16n8k16 per pair of filter taps (t0, t1):
//   A[px][(t, c)] = X[row ho + r_t - ph][px + s_t - pw][c]   (M: 16 output pixels;
//                                                              K: two taps x 8 input channels)
//   B[(t, c)][k]  = W[k][t][c]                                (N: 8 output channels)
// The tap shifts the pixel of A's rows, so every product belongs to an output
// (for 8 channels per group; with 4, a warp's 8 channels hold two groups and B
// is zero off their diagonal blocks). A comes from ldmatrix of the input rows
// as TMA lands them (128B swizzle: the 8 pixels of a matrix hit 8 bank groups),
// each lane's row address doing the tap's shift; B is the same for every row
// and sits in registers. The reduction is the R S taps of one group, so a CTA
// writes finished outputs: no split-K, no fold, and the fused bias + clamp
// epilogue applies directly.
//
// Rows stream as in the grouped weight gradient's ring: a CTA owns 64
// channels and a run of (n, ho) output rows, walked TR rows (a step) at a
// time; input rows ho - ph .. ho - ph + R - 1 form one sequence through a ring
// of row slots (box {64 channels, XP columns} from column -pw, zero outside
// the image), loaded by lane 0 of a rotating warp `ahead` steps early (a step
// whose new rows fill consecutive slots in one image loads them as one box).
// Warp w owns channels 8w .. 8w + 7 of the block, in and out.
//
// The data gradient at stride 1 is this forward over dY with padding
// dil (f - 1) - pad and the turned filter W'[c][r'][s'][k] = W[k][R-1-r'][S-1-s'][c]
// within each group, read in place from W (only B's loads differ).
#include "dw_ring.cuh"
#include "../kernel_entry.h"

namespace cig {
namespace {

using dwring::ring_rows;
using dwring::RowPos;
using dwring::StepPos;

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kCB = 64;        // channels a CTA (in and out): 8 a warp
constexpr int kMaxDepth = 6;   // ahead + slack, at most
constexpr int kMaxTR = 8;      // output rows a step, at most
constexpr int kMaxMT = 4;      // 16-pixel output tiles a row, at most (Wo <= 64)
constexpr int kCtasPerSm = 2;  // two CTAs (16 warps) an SM: 8 warps left the MMAs latency-bound
constexpr size_t kSmemLimit = 227 * 1024 / kCtasPerSm - 1024;
constexpr int kSms = 152;      // the grid is sized for this many SMs (fewer run it in more waves)

struct FgParams {
  const void* w;       // the filter as given, [K][R][S][Cg] (turned: the data gradient's, read in place)
  void* y;
  int64_t Ho, Wo, K;
  int64_t rows;        // N * Ho
  int64_t cblocks;     // C / 64
  int64_t cta_rows;    // output rows a CTA
  int32_t ph, pw, Cg, taps, MT;
  int32_t XP;          // pixels of an input-row slot (a multiple of 8)
  int32_t RX, RS, TR, ahead;
  int32_t turned;
  const void* ep_bias;  // fused epilogue, when ep
  float ep_lo, ep_hi;
  int32_t ep;
};

struct Ring {
  const CUtensorMap* tm_x;
  const CUtensorMap* tm_xt;  // boxes of TR input rows (TR consecutive ring slots)
  uint8_t* xring;
  uint64_t* full;
  uint64_t* empty;
  int32_t* siss;   // wrap count of the last step loaded into each step slot (-1: none)
  volatile uint32_t* abort_flag;
  int32_t* rowinfo;  // per step slot and row: the ring slot of the row's first input row
  unsigned* err;
  uint32_t rowX, txX, txXT;
  int32_t c0;
};

// Loads a step: the input rows its `rows` output rows (the first at row
// position a) are the first to read, landing on the step slot's full
// mbarrier, once every warp is done with the slot's previous step. False: the
// wait gave up.
template <int R>
__device__ bool issue_step(const Ring& g, const FgParams& p, RowPos a, StepPos st, int32_t rows) {
  if (st.sw > 0 && !mbar_wait(&g.empty[st.ss], (st.sw - 1u) & 1u, g.abort_flag, g.err)) return false;
  const int32_t s0 = a.slot(R - 1, p);
  const bool xblk = rows == p.TR && !a.first && a.ho != 0 && a.ho + p.TR <= p.Ho && s0 + p.TR <= p.RX;
  uint32_t bytes = xblk ? g.txXT : 0u;
  {  // the rows' first slots, published by the arrive below (release) to the warps that wait on it
    RowPos b = a;
    for (int32_t j = 0; j < rows; ++j, b.advance(R, p)) {
      if (!xblk) bytes += (uint32_t)b.fresh(R) * g.txX;
      g.rowinfo[st.ss * p.TR + j] = b.xs;
    }
  }
  uint64_t* bar = &g.full[st.ss];
  mbar_arrive_expect_tx(bar, bytes);
  if (xblk) {
    tma_load_4d(g.xring + (size_t)s0 * g.rowX, g.tm_xt, g.c0, -p.pw, a.ho - p.ph + R - 1, a.n, bar);
  } else {
    for (int32_t j = 0; j < rows; ++j, a.advance(R, p))
      for (int r = R - a.fresh(R); r < R; ++r)
        tma_load_4d(g.xring + (size_t)a.slot(r, p) * g.rowX, g.tm_x, g.c0, -p.pw, a.ho - p.ph + r, a.n, bar);
  }
  g.siss[st.ss] = (int32_t)st.sw;
  return true;
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&v)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3])
               : "r"(addr));
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

// Two outputs (channels k, k + 1 of one pixel) rounded into Y.
template <typename TO>
__device__ __forceinline__ void store2(TO* dst, float a, float b);
template <>
__device__ __forceinline__ void store2<float>(float* dst, float a, float b) {
  *reinterpret_cast<float2*>(dst) = make_float2(a, b);
}
template <>
__device__ __forceinline__ void store2<__nv_bfloat16>(__nv_bfloat16* dst, float a, float b) {
  *reinterpret_cast<__nv_bfloat162*>(dst) = __floats2bfloat162_rn(a, b);
}
template <>
__device__ __forceinline__ void store2<__half>(__half* dst, float a, float b) {
  *reinterpret_cast<__half2*>(dst) = __floats2half2_rn(a, b);
}

// B's pair for lane (output channel kout; input channels cin, cin + 1) at tap
// `tap`: zero past the filter or when the channels are in different groups
// (Cg = 4 or 8 divides the 64-channel block, so a mask compares the groups).
template <typename TI>
__device__ __forceinline__ uint32_t b_pair(const FgParams& p, int64_t kout, int64_t cin, int tap) {
  if (tap >= p.taps || ((kout ^ cin) & ~(int64_t)(p.Cg - 1)) != 0) return 0u;
  const TI* w = static_cast<const TI*>(p.w);
  const int64_t cm = p.Cg - 1;
  if (!p.turned) {  // W[kout][tap][c]: c and c + 1 adjacent
    return *reinterpret_cast<const uint32_t*>(w + (kout * p.taps + tap) * p.Cg + (cin & cm));
  }
  // the turned filter: W'[kout][tap][cin] = W[cin][taps - 1 - tap][kout mod Cg]
  const int64_t i0 = (cin * p.taps + (p.taps - 1 - tap)) * p.Cg + (kout & cm);
  uint16_t lo, hi;
  memcpy(&lo, w + i0, 2);
  memcpy(&hi, w + i0 + (int64_t)p.taps * p.Cg, 2);
  return (uint32_t)lo | ((uint32_t)hi << 16);
}

// MTC: a compile-time bound on the 16-pixel tiles of a row (2 or 4; the
// tiles past p.MT are skipped). Every tile of a row accumulates in two sets
// (even and odd tap pairs), so a warp keeps 2 MTC independent MMA chains in
// flight.
template <typename TI, typename TO, int R, int S, int MTC>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
    fwd_grouped_mma_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_xt,
                           FgParams p, unsigned* err) {
  constexpr int TAPS = R * S, TP = (TAPS + 1) / 2;
  constexpr int NSET = 2;  // accumulator sets a tile (even / odd tap pairs)
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  Ring g;
  g.tm_x = &tm_x;
  g.tm_xt = &tm_xt;
  g.rowX = (uint32_t)p.XP * 128u;
  g.txX = g.rowX;
  g.txXT = (uint32_t)p.TR * g.rowX;
  g.xring = smem;
  g.full = reinterpret_cast<uint64_t*>(smem + (size_t)p.RX * g.rowX);
  g.empty = g.full + p.RS;
  g.siss = reinterpret_cast<int32_t*>(g.empty + p.RS);
  g.abort_flag = reinterpret_cast<volatile uint32_t*>(g.siss + p.RS);
  g.rowinfo = reinterpret_cast<int32_t*>(g.siss + p.RS + 4);
  g.err = err;

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t cb = blockIdx.x % p.cblocks;
  const int64_t q_b = (blockIdx.x / p.cblocks) * p.cta_rows;
  const int64_t q_e = q_b + p.cta_rows < p.rows ? q_b + p.cta_rows : p.rows;
  if (q_b >= q_e) return;  // uniform over the CTA, before any barrier
  g.c0 = (int32_t)(cb * kCB);

  if (threadIdx.x == 0) {
    for (int i = 0; i < p.RS; ++i) {
      mbar_init(&g.full[i], 1);
      mbar_init(&g.empty[i], kWarps);
      g.siss[i] = -1;
    }
    *g.abort_flag = 0u;
    mbar_fence_init();
    tma_prefetch(&tm_x);
    tma_prefetch(&tm_xt);
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

  // B: lane (gq, tq) holds output channel gq and input channels 2 tq, 2 tq + 1 of the warp's 8, for
  // both taps of every pair.
  const int gq = lane >> 2, tq = lane & 3;
  const int64_t kw = cb * kCB + 8 * warp;  // the warp's first channel
  uint32_t bf[TP][2];
#pragma unroll
  for (int tp = 0; tp < TP; ++tp) {
    bf[tp][0] = b_pair<TI>(p, kw + gq, kw + 2 * tq, 2 * tp);
    bf[tp][1] = b_pair<TI>(p, kw + gq, kw + 2 * tq, 2 * tp + 1);
  }
  // A: lane l supplies pixel prow of the 16-pixel tile at tap 2 tp + half of each pair (the pad tap
  // of an odd count repeats tap 2 tp: finite data times B's zeros); col = its 16-byte row's offset
  // within a slot (128B swizzle; a tile of 16 pixels is 2048 bytes and keeps the pattern).
  const int half = lane >> 4, prow = 8 * ((lane >> 3) & 1) + (lane & 7);
  uint32_t col[TP];
#pragma unroll
  for (int tp = 0; tp < TP; ++tp) {
    const int t = 2 * tp + half < TAPS ? 2 * tp + half : 2 * tp;
    const int px = prow + t % S;
    col[tp] = (uint32_t)(px * 128) + ((uint32_t)(warp ^ (px & 7)) << 4);
  }
  const uint32_t xring_u32 = smem_u32(g.xring);
  TO* y = static_cast<TO*>(p.y);
  const TO* ep_bias = static_cast<const TO*>(p.ep_bias);
  float2 bias = make_float2(0.f, 0.f);
  if (p.ep && ep_bias) bias = make_float2(to_f32(ep_bias[kw + 2 * tq]), to_f32(ep_bias[kw + 2 * tq + 1]));

  StepPos sc{0, 0u};
  StepPos sl{0, 0u};  // the step slot of step S + ahead
  for (int i = 0; i < p.ahead; ++i) sl.advance(p);
  int32_t issuer = 0;  // warp that loads at step S: S mod 8
  int64_t qa = q_b + (int64_t)p.ahead * p.TR;  // first row of step S + ahead
  // The issuing lane places row qa in closed form (32-bit: N * Ho < 2^31 is a condition of the
  // kernel): its image and row, and its first input row's index in the run's input-row sequence
  // (R rows for the run's first row and each image start, one more for every other row).
  const uint32_t ho_u = (uint32_t)p.Ho, n_b = (uint32_t)q_b / ho_u;
  auto row_pos = [&](int64_t qq) {
    const uint32_t n = (uint32_t)qq / ho_u, ho = (uint32_t)qq - n * ho_u;
    const uint32_t seq = (uint32_t)(qq - q_b) + (uint32_t)(R - 1) * (n - n_b);
    return RowPos{(int32_t)(seq % (uint32_t)p.RX), (int32_t)ho, (int32_t)n, qq == q_b};
  };
  int32_t on = (int32_t)(q_b / p.Ho), oho = (int32_t)(q_b % p.Ho);  // the next output row

  for (int64_t q = q_b; q < q_e; q += p.TR) {
    const int32_t rows = q_e - q < p.TR ? (int32_t)(q_e - q) : p.TR;
    if (warp == issuer && lane == 0 && qa < q_e)
      issue_step<R>(g, p, row_pos(qa), sl, q_e - qa < p.TR ? (int32_t)(q_e - qa) : p.TR);
    // Lanes that spin on an mbarrier can hold up a divergent lane of the same
    // warp; reconverge before any of them waits.
    __syncwarp();
    qa += p.TR;
    sl.advance(p);
    issuer = issuer + 1 == kWarps ? 0 : issuer + 1;

    if (!__all_sync(0xffffffffu, mbar_wait(&g.full[sc.ss], sc.sw & 1u, g.abort_flag, g.err))) break;

    // Row j's MMAs into acc, then the outputs of an accumulator into Y.
    auto row_mmas = [&](int32_t j, float (&acc)[NSET][MTC][4]) {
      const int32_t xs = g.rowinfo[sc.ss * p.TR + j];
      uint32_t slot[R];
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const int32_t s_ = xs + r >= p.RX ? xs + r - p.RX : xs + r;
        slot[r] = xring_u32 + (uint32_t)s_ * g.rowX;
      }
#pragma unroll
      for (int e = 0; e < NSET * MTC * 4; ++e) (&acc[0][0][0])[e] = 0.f;
      // The fragments of tap pair tp + 1 are loaded before the MMAs of pair tp
      // (loads and MMAs are issued in program order), so the ldmatrix latency
      // overlaps the MMAs.
      uint32_t af[2][MTC][4];
      auto load_pair = [&](int tp, uint32_t (&f)[MTC][4]) {
        const int r0 = (2 * tp) / S, r1 = (2 * tp + 1 < TAPS ? 2 * tp + 1 : 2 * tp) / S;
        const uint32_t base = (half ? slot[r1] : slot[r0]) + col[tp];
#pragma unroll
        for (int mt = 0; mt < MTC; ++mt)
          if (mt < p.MT) ldsm_x4(base + (uint32_t)mt * 2048u, f[mt]);
      };
      load_pair(0, af[0]);
#pragma unroll
      for (int tp = 0; tp < TP; ++tp) {
        if (tp + 1 < TP) load_pair(tp + 1, af[(tp + 1) & 1]);
#pragma unroll
        for (int mt = 0; mt < MTC; ++mt)
          if (mt < p.MT) mma16816<TI>(acc[tp % NSET][mt], af[tp & 1][mt], bf[tp]);
      }
    };
    auto row_store = [&](const float (&acc)[NSET][MTC][4], TO* yrow) {
#pragma unroll
      for (int mt = 0; mt < MTC; ++mt) {
        if (mt >= p.MT) break;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int64_t wo = (int64_t)mt * 16 + gq + 8 * hh;
          if (wo < p.Wo) {
            float v0 = acc[0][mt][2 * hh], v1 = acc[0][mt][2 * hh + 1];
            if (NSET > 1) {
              v0 += acc[NSET - 1][mt][2 * hh];
              v1 += acc[NSET - 1][mt][2 * hh + 1];
            }
            if (p.ep) {
              v0 = fminf(fmaxf(v0 + bias.x, p.ep_lo), p.ep_hi);
              v1 = fminf(fmaxf(v1 + bias.y, p.ep_lo), p.ep_hi);
            }
            store2<TO>(yrow + wo * p.K, v0, v1);
          }
        }
      }
    };
    auto next_row = [&]() {  // Y row of the next output row, then advance
      TO* yrow = y + ((int64_t)on * p.Ho + oho) * p.Wo * p.K + kw + 2 * tq;
      if (++oho == p.Ho) {
        oho = 0;
        ++on;
      }
      return yrow;
    };
    float acc_a[NSET][MTC][4];
    if (kCtasPerSm > 1) {  // 16 warps an SM hide the latency; the registers allow one row at a time
#pragma unroll 1
      for (int32_t j = 0; j < rows; ++j) {
        row_mmas(j, acc_a);
        row_store(acc_a, next_row());
      }
    } else {  // one CTA an SM: rows in pairs, each row's outputs stored after the next row's MMAs
      float acc_b[NSET][MTC][4];
      TO* y_b = nullptr;
#pragma unroll 1
      for (int32_t j = 0; j < rows; j += 2) {
        row_mmas(j, acc_a);
        TO* y_a = next_row();
        if (y_b) row_store(acc_b, y_b);
        if (j + 1 < rows) {
          row_mmas(j + 1, acc_b);
          y_b = next_row();
          row_store(acc_a, y_a);
        } else {
          row_store(acc_a, y_a);
          y_b = nullptr;
        }
      }
      if (y_b) row_store(acc_b, y_b);
    }

    __syncwarp();
    if (lane == 0) mbar_arrive(&g.empty[sc.ss]);
    sc.advance(p);
  }

  // No copy may still be landing in shared memory when the CTA exits (wait
  // for the last step loaded into each step slot; bounded, no early exit).
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int i = 0; i < p.RS; ++i)
      if (g.siss[i] >= 0) mbar_wait(&g.full[i], (uint32_t)g.siss[i] & 1u, nullptr, err);
  }
}

int64_t tiles_of_row(const Shape& s) { return (s.wo + 15) / 16; }
int64_t slot_pixels(const Shape& s) { return (tiles_of_row(s) * 16 + s.s - 1 + 7) / 8 * 8; }

size_t ring_smem(const Shape& s, int d, int tr) {
  const int64_t rx = ring_rows(s.r, s.ho, d, tr), rs = 1 + d;
  return 1024 + (size_t)(rx * slot_pixels(s) * 128) + 2 * rs * 8 + rs * 4 + 16 + (size_t)rs * tr * 4;
}

struct RingShape {
  int d = 0, tr = 0;
};

// The most rows a step (up to 8) that still lets the loads run three steps
// ahead with one of slack, else the deepest ring that fits.
RingShape ring_shape(const Shape& s) {
  for (int tr = kMaxTR; tr >= 1; --tr)
    for (int d = kMaxDepth; d >= 4; --d)
      if (ring_smem(s, d, tr) <= kSmemLimit) return RingShape{d, tr};
  for (int tr = kMaxTR; tr >= 1; --tr)
    for (int d = kMaxDepth; d >= 2; --d)
      if (ring_smem(s, d, tr) <= kSmemLimit) return RingShape{d, tr};
  return RingShape{};
}

int ahead_of_depth(int d) { return d >= 4 ? d - 1 : 1; }

// Output rows a CTA: about kCtasPerSm CTAs per SM over all channel blocks, a multiple of the step.
int64_t cta_rows(const Shape& s, int tr) {
  const int64_t rows = s.n * s.ho, cblocks = s.c / kCB;
  int64_t r = (rows * cblocks + kSms * kCtasPerSm - 1) / (kSms * kCtasPerSm);
  r = (r + tr - 1) / tr * tr;
  return r < tr ? tr : r;
}

// The forward problem this kernel runs (the data gradient's turned problem
// included): 16-bit, grouped with Cg = Kg in {4, 8}, 64-channel blocks, unit
// stride and dilation, 1x1 / 3x3 / 5x5 filters, rows of at most 128 output
// columns.
Geometry geometry_problem(const Shape& s) {
  Geometry g;
  if (s.in_dt == CONV_F32 || s.groups < 2 || s.cg != s.kg || !(s.cg == 4 || s.cg == 8)) return g;
  if (s.c % kCB != 0 || s.c != s.k || s.n < 1) return g;
  if (s.sh != 1 || s.sw != 1 || s.dh != 1 || s.dw != 1) return g;
  if (!((s.r == 1 && s.s == 1) || (s.r == 3 && s.s == 3) || (s.r == 5 && s.s == 5))) return g;
  if (s.ph > s.r - 1 || s.pw > s.s - 1 || s.ph < 0 || s.pw < 0) return g;
  if (s.wo < 1 || s.wo > kMaxMT * 16 || slot_pixels(s) > 256) return g;
  if (s.n * s.ho > 0x7fffffffLL || s.h + s.r > 0x7fffffffLL) return g;
  const RingShape rs = ring_shape(s);
  if (rs.d < 1) return g;
  g.ok = true;
  g.ctas_per_sm = kCtasPerSm;
  g.tiles = (s.c / kCB) * ((s.n * s.ho + cta_rows(s, rs.tr) - 1) / cta_rows(s, rs.tr));
  g.blocks = 1;  // no split: the reduction is the R S taps of a group
  return g;
}

template <typename TI, typename TO, int R, int S, int MTC>
cudaError_t launch_rs(const Plan& pl, const Args& a, const FgParams& p, const Shape& s, CUtensorMapDataType dt,
                      size_t smem) {
  CUtensorMap tm_x, tm_xt;
  const uint64_t x_dims[4] = {(uint64_t)s.c, (uint64_t)s.w, (uint64_t)s.h, (uint64_t)s.n};
  const uint64_t x_strides[3] = {(uint64_t)s.c * 2u, (uint64_t)(s.w * s.c) * 2u, (uint64_t)(s.h * s.w * s.c) * 2u};
  const uint32_t x_box[4] = {(uint32_t)kCB, (uint32_t)p.XP, 1u, 1u};
  const uint32_t xt_box[4] = {(uint32_t)kCB, (uint32_t)p.XP, (uint32_t)p.TR, 1u};
  if (!encode_tmap(&tm_x, dt, 4, a.x, x_dims, x_strides, x_box, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tmap(&tm_xt, dt, 4, a.x, x_dims, x_strides, xt_box, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  auto kern = fwd_grouped_mma_kernel<TI, TO, R, S, MTC>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  const int64_t ctas = pl.geo.tiles;
  if (ctas > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  kern<<<(unsigned)ctas, kThreads, smem, a.stream>>>(tm_x, tm_xt, p, device_error_word());
  return cudaGetLastError();
}

template <typename TI, typename TO, int R, int S>
cudaError_t launch_mtc(const Plan& pl, const Args& a, const FgParams& p, const Shape& s, CUtensorMapDataType dt,
                       size_t smem) {
  if (p.MT <= 2) return launch_rs<TI, TO, R, S, 2>(pl, a, p, s, dt, smem);
  if (p.MT <= 4) return launch_rs<TI, TO, R, S, 4>(pl, a, p, s, dt, smem);
  return cudaErrorInvalidValue;
}

// s: the forward problem run (for the data gradient, the turned one).
template <typename TI, typename TO>
cudaError_t launch_typed(const Plan& pl, const Args& a, const Shape& s, bool turned, CUtensorMapDataType dt) {
  const RingShape rs = ring_shape(s);
  if (rs.d < 1) return cudaErrorInvalidValue;
  FgParams p;
  p.w = a.b;
  p.y = a.out;
  p.Ho = s.ho;
  p.Wo = s.wo;
  p.K = s.k;
  p.rows = s.n * s.ho;
  p.cblocks = s.c / kCB;
  p.cta_rows = cta_rows(s, rs.tr);
  p.ph = (int32_t)s.ph;
  p.pw = (int32_t)s.pw;
  p.Cg = (int32_t)s.cg;
  p.taps = (int32_t)(s.r * s.s);
  p.MT = (int32_t)tiles_of_row(s);
  p.XP = (int32_t)slot_pixels(s);
  p.RX = (int32_t)ring_rows(s.r, s.ho, rs.d, rs.tr);
  p.RS = 1 + rs.d;
  p.TR = rs.tr;
  p.ahead = ahead_of_depth(rs.d);
  p.turned = turned ? 1 : 0;
  p.ep_bias = a.ep_bias;
  p.ep_lo = a.ep_lo;
  p.ep_hi = a.ep_hi;
  p.ep = a.ep ? 1 : 0;
  const size_t smem = ring_smem(s, rs.d, rs.tr);
  switch (s.r) {
    case 1: return launch_mtc<TI, TO, 1, 1>(pl, a, p, s, dt, smem);
    case 3: return launch_mtc<TI, TO, 3, 3>(pl, a, p, s, dt, smem);
    case 5: return launch_mtc<TI, TO, 5, 5>(pl, a, p, s, dt, smem);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_any(const Plan& pl, const Args& a, const Shape& s, bool turned) {
  if (pl.split != 1 || a.ws) return cudaErrorInvalidValue;
  const int in = s.in_dt, out = s.out_dt;
  if (in == CONV_BF16)
    return out == CONV_F32
               ? launch_typed<__nv_bfloat16, float>(pl, a, s, turned, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16)
               : launch_typed<__nv_bfloat16, __nv_bfloat16>(pl, a, s, turned, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16);
  return out == CONV_F32 ? launch_typed<__half, float>(pl, a, s, turned, CU_TENSOR_MAP_DATA_TYPE_FLOAT16)
                         : launch_typed<__half, __half>(pl, a, s, turned, CU_TENSOR_MAP_DATA_TYPE_FLOAT16);
}

}  // namespace

Geometry geometry_fwd_grouped_mma(const Shape& s) { return geometry_problem(s); }

cudaError_t launch_fwd_grouped_mma(const Plan& p, const Args& a) { return launch_any(p, a, p.sh, false); }

// The stride-1 grouped data gradient as the forward over dY with the turned
// filter (padding dil (f - 1) - pad >= 0).
Geometry geometry_dgrad_grouped_mma(const Shape& s) {
  if (s.sh != 1 || s.sw != 1 || s.groups < 2) return Geometry{};
  if (s.ph > s.dh * (s.r - 1) || s.pw > s.dw * (s.s - 1)) return Geometry{};
  return geometry_problem(dgrad_as_forward_grouped(s));
}

cudaError_t launch_dgrad_grouped_mma(const Plan& p, const Args& a) {
  return launch_any(p, a, dgrad_as_forward_grouped(p.sh), true);
}

}  // namespace cig
