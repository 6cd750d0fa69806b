// 16-bit depthwise weight gradient (+ bias gradient) on warp-level tensor-core
// MMAs, for filters of up to 7 x 7, unit stride and dilation, rows of at most
// 64 input and output columns:
//
//   dW[c, r, s] = sum over (n, ho, j) of X[n, ho + r - ph, j, c] * dY[n, ho, j - s + pw, c]
//   db[c]       = sum over (n, ho, wo) of dY[n, ho, wo, c]
//
// ("perf(rocke): depthwise 7x7 and grouped cpg4/8 wgrad on batched mfma
// 4x4x4", "Technical Details": the depthwise weight gradient as small matrix
// products on the matrix cores.) For one channel and one output row this is
// an MMA m16n8k16 per 16 input columns j0 .. j0 + 15, the reduction over j:
//   A[r][k] = X[ho + r - ph][j0 + k]      (M: the filter rows, 7 of 16 used)
//   B[k][s] = dY[ho][j0 + k - s + pw]     (N: the filter columns, a Toeplitz
//                                          operand: column s is dY shifted by s)
// so one MMA yields all 49 taps of a 7 x 7 filter. A's rows 8 .. 15 repeat
// rows 0 .. 7 (one x2 ldmatrix: shared-memory bandwidth, not the MMA rate,
// bounds this kernel, and A is read afresh for every MMA). The bias gradient
// is summed in fp32 from the dY row's words while it is transposed.
//
// NHWC keeps the channels of a pixel together, while these operands want the
// pixels of one channel together, so each row is transposed in shared memory
// on its way in (ldmatrix.trans / stmatrix, 8 x 8 blocks). Every warp owns 8
// of the CTA's 64 channels and works alone: it stages its own 16-byte column
// of each row with cp.async (a ring of rows per warp, the loads running
// kLead output rows ahead), transposes it into its channels' rows, and
// accumulates its channels' 16 x 8 tiles in registers over the CTA's slice of
// output rows. No CTA barrier, no cross-warp reduction: the sums run in a
// fixed order (deterministic). Transposed layouts:
//   Xt [channel][7 slots][72 pixels]: input rows of the current output row in
//      a ring of 7 slots; the 8 pixels of padding a row put the rows of an
//      8 x 8 block (and the channels) in distinct bank groups;
//   dYt [2 copies][channel][88 pixels]: the dY row at pixel offset 8, zero
//      around it; copy 1 is shifted by one pixel, so the pair a lane reads for
//      B (pixels p, p + 1, p of either parity) is one aligned 32-bit word, and
//      starts 64 bytes further on, so the lanes reading copy 0 and copy 1 hit
//      disjoint banks.
#include "tc_common.cuh"
#include "../kernel_entry.h"

namespace cig {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kCB = 64;                        // channels a CTA, 8 a warp
constexpr int kBW = 64;                        // staged pixels a row (16 bytes each: a warp's 8 channels)
constexpr int kRowB = kBW * 16;                // staged row bytes
constexpr int kMaxF = 7;                       // filter rows and columns, at most
constexpr int kLead = 4;                       // output rows the loads run ahead
constexpr int kQd = kLead + 1;                 // staged dY rows a warp
constexpr int kQx = kLead + kMaxF;             // staged input rows a warp (a run start brings R)
constexpr int kXtSlot = (kBW + 8) * 2;         // 144 bytes
constexpr int kXtChan = 7 * kXtSlot;           // 1008 bytes (112 mod 128: channel rows in distinct banks)
constexpr int kDtRow = (kBW + 24) * 2;         // 176 bytes: pixels -8 .. 79
constexpr int kDtOff = 8 * 2;                  // byte offset of pixel 0 in a dY row
constexpr int kDtCopy1 = 8 * kDtRow + 64;      // byte offset of copy 1
constexpr int kWarpSmem = (kQd + kQx) * kRowB + 8 * kXtChan + kDtCopy1 + 8 * kDtRow;
constexpr size_t kSmem = (size_t)kWarps * kWarpSmem;
static_assert(kSmem <= 227 * 1024, "shared memory");
static_assert(kWarpSmem % 16 == 0, "16-byte aligned warp regions");

struct DmParams {
  const void* x;
  const void* dy;
  int64_t C, H, W, Ho, Wo;
  int64_t rows;     // N * Ho: the reduction blocks
  int64_t cblocks;  // ceil(C / 64): the tiles
  int32_t R, S, ph, pw;
  int32_t split;
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
// Waits until at most `pending` (0 .. kLead) of this thread's commit groups are in flight.
__device__ __forceinline__ void cp_async_wait_pending(int pending);

// ldmatrix results feed only MMAs, so these are not volatile: the compiler may
// issue a load early (the "memory" clobber keeps it after the stores and
// barriers that produced its data).
__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t (&v)[2]) {
  asm("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];" : "=r"(v[0]), "=r"(v[1]) : "r"(addr) : "memory");
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&v)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3])
               : "r"(addr)
               : "memory");
}
__device__ __forceinline__ void stsm_x4(uint32_t addr, const uint32_t (&v)[4]) {
  asm volatile("stmatrix.sync.aligned.m8n8.x4.shared.b16 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v[0]), "r"(v[1]),
               "r"(v[2]), "r"(v[3])
               : "memory");
}
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ void sts32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// A pair of 16-bit values widened to fp32.
template <typename T>
__device__ __forceinline__ float2 widen2(uint32_t v);
template <>
__device__ __forceinline__ float2 widen2<__nv_bfloat16>(uint32_t v) {
  return make_float2(__uint_as_float(v << 16), __uint_as_float(v & 0xffff0000u));
}
template <>
__device__ __forceinline__ float2 widen2<__half>(uint32_t v) {
  __half2 h;
  memcpy(&h, &v, sizeof(h));
  return __half22float2(h);
}

template <typename TI>
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1);
template <>
__device__ __forceinline__ void mma16816<__nv_bfloat16>(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                                        uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
template <>
__device__ __forceinline__ void mma16816<__half>(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// An output row's place in the slice: (image, row), and whether it starts a
// new run of input rows (the slice's first row or an image's first row: R
// fresh input rows, else one). Advanced one row at a time.
struct Cursor {
  int32_t n, ho;
  bool first;
  __device__ __forceinline__ bool starts() const { return first || ho == 0; }
  __device__ __forceinline__ void advance(int64_t Ho) {
    first = false;
    if (++ho == Ho) {
      ho = 0;
      ++n;
    }
  }
};

__device__ __forceinline__ void cp_async_wait_pending(int pending) {
  switch (pending) {
    case 0: cp_async_wait<0>(); break;
    case 1: cp_async_wait<1>(); break;
    case 2: cp_async_wait<2>(); break;
    case 3: cp_async_wait<3>(); break;
    default: cp_async_wait<4>(); break;
  }
}
static_assert(kLead == 4, "cp_async_wait_pending covers 0 .. kLead");

// One staged row (the warp's 16-byte column of kBW pixels) into dst: pixel px
// from row + px * C, zeros past `width` pixels or for a row outside the image
// (cp.async with no source bytes writes zeros). Lane l copies pixels l and
// l + 32.
template <typename TI>
__device__ __forceinline__ void stage_row(uint32_t dst, const TI* row, int64_t C, int64_t width, bool valid,
                                          const TI* any) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int px = (int)(threadIdx.x & 31) + 32 * h;
    const bool ok = valid && px < width;
    cp_async16(dst + (uint32_t)px * 16u, ok ? row + px * C : any, ok ? 16u : 0u);
  }
}

// A staged row -> its transposed rows: 8 x 8 blocks (8 pixels x the warp's 8
// channels) read transposed, written as rows of one channel. dst: row of the
// warp's channel 0, channel rows `pitch` bytes apart. NB4 groups of 4 blocks.
template <int NB4>
__device__ __forceinline__ void transpose_row(uint32_t src, uint32_t dst, uint32_t pitch, uint32_t (&v)[8]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    uint32_t w[4] = {0u, 0u, 0u, 0u};
    if (q < NB4) {
      const int blk = 4 * q + (lane >> 3);
      ldsm_x4_t(src + (uint32_t)((blk * 8 + (lane & 7)) * 16), w);
      stsm_x4(dst + (uint32_t)(lane & 7) * pitch + (uint32_t)blk * 16u, w);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) v[4 * q + i] = w[i];
  }
}

// SP: the filter's (R, S) with R, S <= 7; NCH chunks of 16 input columns.
template <typename TI, typename TO, int NCH>
__global__ void __launch_bounds__(kThreads, 1)
    dw_wgrad_mma_kernel(TO* out, float* ws, TO* db, float* ws_bias, DmParams p) {
  constexpr int NB4 = (2 * NCH + 3) / 4;  // groups of 4 pixel blocks covering 16 NCH pixels
  extern __shared__ __align__(128) uint8_t smem[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t cb = blockIdx.x % p.cblocks;
  const int32_t sigma = (int32_t)(blockIdx.x / p.cblocks);
  const int64_t c0 = cb * kCB + warp * 8;  // the warp's first channel
  if (c0 >= p.C) return;                   // C % 8 = 0: a warp's channels are all in or all out
  const int64_t q_b = slice_begin(p.rows, p.split, sigma), q_e = slice_begin(p.rows, p.split, sigma + 1);

  const uint32_t base = smem_u32(smem) + (uint32_t)(warp * kWarpSmem);
  const uint32_t dstg = base;                           // kQd staged dY rows
  const uint32_t xstg = dstg + kQd * kRowB;             // kQx staged input rows
  const uint32_t xt = xstg + kQx * kRowB;               // [8 channels][7 slots][72 pixels]
  const uint32_t dyt = xt + 8 * kXtChan;                // [2 copies][8 channels][88 pixels]
  const uint32_t dyo = dyt + kDtCopy1;                  // copy 1: pixel q holds dY[q + 1]

  // The dY rows' zero surround (both copies; rows are rewritten only at
  // pixels 0 .. 32 NB4 - 1 and copy 1's pixels -2, -1).
  for (int i = lane; i < (kDtCopy1 + 8 * kDtRow) / 4; i += 32) sts32(dyt + 4u * (uint32_t)i, 0u);

  const TI* xg = static_cast<const TI*>(p.x);
  const TI* dyg = static_cast<const TI*>(p.dy);
  const Cursor start{(int32_t)(q_b / p.Ho), (int32_t)(q_b % p.Ho), true};

  // The loads of one output row: its dY row, and its fresh input rows (R at
  // the start of a run, else the one below the window).
  int dsl_i = 0, xsl_i = 0;
  auto issue = [&](const Cursor& cu) {
    stage_row<TI>(dstg + (uint32_t)(dsl_i * kRowB), dyg + (((int64_t)cu.n * p.Ho + cu.ho) * p.Wo) * p.C + c0, p.C,
                  p.Wo, true, dyg);
    if (++dsl_i == kQd) dsl_i = 0;
    const int nx = cu.starts() ? p.R : 1;
    for (int i = 0; i < nx; ++i) {
      const int64_t h = (int64_t)cu.ho - p.ph + (p.R - nx) + i;
      const bool v = h >= 0 && h < p.H;
      stage_row<TI>(xstg + (uint32_t)(xsl_i * kRowB), v ? xg + (((int64_t)cu.n * p.H + h) * p.W) * p.C + c0 : xg,
                    p.C, p.W, v, xg);
      if (++xsl_i == kQx) xsl_i = 0;
    }
  };

  // One commit group a row, issued up to kLead rows ahead while the staged
  // input rows fit (a run start brings R of them; near image starts the lead
  // shrinks rather than overwrite rows not yet transposed). `issued` and
  // `x_fly` (staged input rows not yet transposed) are the same in every lane.
  Cursor iss = start;
  const int64_t nsteps = q_e - q_b;
  int64_t issued = 0;
  int x_fly = 0;
  auto issue_upto = [&](int64_t limit) {
    while (issued < limit && issued < nsteps) {
      const int nx = iss.starts() ? p.R : 1;
      if (x_fly + nx > kQx) break;
      issue(iss);
      cp_async_commit();
      iss.advance(p.Ho);
      ++issued;
      x_fly += nx;
    }
  };
  issue_upto(kLead);

  // B: lane (g, t) reads dY pixels p, p + 1 with p = j0 + 2t + pw - g, from
  // the copy where that pair is one aligned word.
  const int g = lane >> 2, t = lane & 3;
  const int p0 = 2 * t + p.pw - g;
  const uint32_t b_lane = (p0 & 1) ? dyo + (uint32_t)(kDtOff + (p0 - 1) * 2) : dyt + (uint32_t)(kDtOff + p0 * 2);
  // A (x2): lane l < 16 supplies row m = l % 8 of the K half l / 8: filter
  // row m (m < R), else any valid row (its products are dropped).
  const int m = lane & 7, khalf = (lane >> 3) & 1;
  float2 bsum = make_float2(0.f, 0.f);  // the bias: channel g, this lane's pixels

  float acc[8][4];
#pragma unroll
  for (int ci = 0; ci < 8; ++ci)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[ci][e] = 0.f;

  Cursor con = start;
  int dsl_c = 0, xsl_c = 0, xt_new = 6;  // Xt slot of the newest input row
  for (int64_t q = q_b; q < q_e; ++q) {
    const int64_t step = q - q_b;
    issue_upto(step + 1 + kLead);  // step `step` itself always fits: nothing older is staged
    cp_async_wait_pending((int)(issued - step - 1));  // this row's group has landed (this lane's copies)
    __syncwarp();                                     // ... and every lane's

    uint32_t v[8];
    const int nx = con.starts() ? p.R : 1;
    for (int i = 0; i < nx; ++i) {
      if (++xt_new == 7) xt_new = 0;
      transpose_row<NB4>(xstg + (uint32_t)(xsl_c * kRowB), xt + (uint32_t)(xt_new * kXtSlot), kXtChan, v);
      if (++xsl_c == kQx) xsl_c = 0;
    }
    x_fly -= nx;
    transpose_row<NB4>(dstg + (uint32_t)(dsl_c * kRowB), dyt + kDtOff, kDtRow, v);
    if (++dsl_c == kQd) dsl_c = 0;
#pragma unroll
    for (int b = 0; b < 4 * NB4; ++b) bsum = __fadd2_rn(bsum, widen2<TI>(v[b]));
    {  // copy 1, word (q, q + 1) = dY pixels q + 1, q + 2 (q = 8 b + 2 t): the high half of this lane's
       // word and the low half of the next pair's, from lane t + 1 or (t = 3) the next block's lane 0
      const int partner = (lane & ~3) | ((lane + 1) & 3);
      uint32_t o[8];
#pragma unroll
      for (int b = 0; b < 8; ++b) {
        const uint32_t send = t == 0 ? (b + 1 < 8 ? v[b + 1] : 0u) : v[b];
        const uint32_t recv = __shfl_sync(0xffffffffu, send, partner);
        o[b] = __byte_perm(v[b], recv, 0x5432);
      }
#pragma unroll
      for (int qq = 0; qq < NB4; ++qq) {
        const uint32_t w[4] = {o[4 * qq], o[4 * qq + 1], o[4 * qq + 2], o[4 * qq + 3]};
        stsm_x4(dyo + kDtOff + (uint32_t)(lane & 7) * kDtRow + (uint32_t)(4 * qq + (lane >> 3)) * 16u, w);
      }
      if (t == 0) sts32(dyo + kDtOff - 4 + (uint32_t)g * kDtRow, v[0] << 16);  // pixels -2, -1: 0, dY[0]
    }
    __syncwarp();

    int slot = xt_new - (p.R - 1 - (m < p.R ? m : 0));
    if (slot < 0) slot += 7;
    const uint32_t a_lane = xt + (uint32_t)(slot * kXtSlot + khalf * 16);
#pragma unroll
    for (int jc = 0; jc < NCH; ++jc)
#pragma unroll
      for (int ci = 0; ci < 8; ++ci) {
        uint32_t a2[2];
        ldsm_x2(a_lane + (uint32_t)(ci * kXtChan + jc * 32), a2);
        const uint32_t a[4] = {a2[0], a2[0], a2[1], a2[1]};
        const uint32_t bb = b_lane + (uint32_t)(ci * kDtRow + jc * 32);
        mma16816<TI>(acc[ci], a, lds32(bb), lds32(bb + 16u));
      }
    __syncwarp();  // the next row's transposes overwrite what these read
    con.advance(p.Ho);
  }
  cp_async_wait<0>();  // nothing may land after the warp exits

  // Lane (g, t) holds D[g][2t + e] (e = 0, 1) of each channel: tap (r, s) =
  // (g, 2t + e). The bias of channel g: this lane's pixels, then the channel's
  // four lanes in a fixed order.
  float bias = bsum.x + bsum.y;
  bias += __shfl_xor_sync(0xffffffffu, bias, 1);
  bias += __shfl_xor_sync(0xffffffffu, bias, 2);
  if (t == 0) {
    if (ws_bias) ws_bias[(int64_t)sigma * p.C + c0 + g] = bias;
    else if (db) store_out(db + c0 + g, bias);
  }
  const int64_t E = p.C * p.R * p.S;
  float* slab = ws ? ws + (int64_t)sigma * E : nullptr;
#pragma unroll
  for (int ci = 0; ci < 8; ++ci) {
    const int64_t c = c0 + ci;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int s = 2 * t + e;
      if (g < p.R && s < p.S) {
        const int64_t dst = (c * p.R + g) * p.S + s;
        if (slab) slab[dst] = acc[ci][e];
        else store_out(out + dst, acc[ci][e]);
      }
    }
  }
}

// 16-input-column chunks: the reduction covers input columns [0, W) and the
// bias dY columns [0, Wo), so 16 NCH >= max(W, Wo).
int64_t chunks_of(const Shape& s) { return ((s.w > s.wo ? s.w : s.wo) + 15) / 16; }

template <typename TI, typename TO, int NCH>
cudaError_t launch_n(const Plan& pl, const Args& a, const DmParams& p) {
  auto kern = dw_wgrad_mma_kernel<TI, TO, NCH>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
  if (err != cudaSuccess) return err;
  const int64_t ctas = pl.geo.tiles * pl.split;
  if (ctas > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  kern<<<(unsigned)ctas, kThreads, kSmem, a.stream>>>(static_cast<TO*>(a.out), a.ws,
                                                      pl.with_bias ? static_cast<TO*>(a.db) : nullptr,
                                                      pl.with_bias ? a.ws_bias : nullptr, p);
  return cudaGetLastError();
}

template <typename TI, typename TO>
cudaError_t launch_typed(const Plan& pl, const Args& a) {
  const Shape& s = pl.sh;
  DmParams p;
  p.x = a.x;
  p.dy = a.b;
  p.C = s.c;
  p.H = s.h;
  p.W = s.w;
  p.Ho = s.ho;
  p.Wo = s.wo;
  p.rows = s.n * s.ho;
  p.cblocks = (s.c + kCB - 1) / kCB;
  p.R = (int32_t)s.r;
  p.S = (int32_t)s.s;
  p.ph = (int32_t)s.ph;
  p.pw = (int32_t)s.pw;
  p.split = pl.split;
  switch (chunks_of(s)) {
    case 1: return launch_n<TI, TO, 1>(pl, a, p);
    case 2: return launch_n<TI, TO, 2>(pl, a, p);
    case 3: return launch_n<TI, TO, 3>(pl, a, p);
    case 4: return launch_n<TI, TO, 4>(pl, a, p);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

Geometry geometry_wgrad_depthwise_mma(const Shape& s) {
  Geometry g;
  const bool depthwise = s.groups == s.c && s.groups == s.k;
  if (!depthwise || s.in_dt == CONV_F32 || s.n < 1) return g;
  if (s.r > kMaxF || s.s > kMaxF || s.r < 1 || s.s < 1) return g;
  if (s.sh != 1 || s.sw != 1 || s.dh != 1 || s.dw != 1) return g;
  if (s.ph > s.r - 1 || s.pw > s.s - 1) return g;
  // rows of at most kBW input and output columns; 16-byte channel groups
  if (s.w > kBW || s.wo > kBW || s.c % 8 != 0) return g;
  if (s.n * s.ho > 0x7fffffffLL || s.h + s.r > 0x7fffffffLL) return g;
  g.ok = true;
  g.ctas_per_sm = 1;
  g.tiles = (s.c + kCB - 1) / kCB;
  g.blocks = s.n * s.ho;
  return g;
}

cudaError_t launch_wgrad_depthwise_mma(const Plan& p, const Args& a) {
  const int in = p.sh.in_dt, out = p.sh.out_dt;
  if (in == CONV_BF16)
    return out == CONV_F32 ? launch_typed<__nv_bfloat16, float>(p, a) : launch_typed<__nv_bfloat16, __nv_bfloat16>(p, a);
  return out == CONV_F32 ? launch_typed<__half, float>(p, a) : launch_typed<__half, __half>(p, a);
}

}  // namespace cig
