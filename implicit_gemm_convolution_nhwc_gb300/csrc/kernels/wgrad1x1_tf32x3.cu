// fp32 1x1 weight gradient (+ bias gradient) on the tcgen05 tensor cores,
// with fp32 accuracy from a 3xTF32-style operand split.
//
// Operation: dW[k,c] = sum_p dY[p,k] X[p,c] and db[k] = sum_p dY[p,k] over the
// [N*H*W, K] and [N*H*W, C] views of a 1x1, stride-1, unpadded convolution
// (the F.linear form of "ROCm/rocm-libraries PR #11188", "Motivation" and
// "Test Plan"). The reduction (rows p) is split into S slices, each CTA
// writes one fp32 partial slab ("feat(rocke): split-K forward implicit-GEMM
// convolution on gfx1250", "Two-stage split-K"), and the fold sums them.
//
// Precision: a tf32 operand keeps 10 explicit mantissa bits. Every fp32 input
// v is split as hi = v with its low 13 mantissa bits cleared (exact in tf32)
// and lo = v - hi (exact in fp32, rounded to tf32 by the unit). One
// M=128 x N=2*BC MMA per 8 rows computes [dY_hi; dY_lo]^T x [X_hi | X_lo]:
// accumulator rows 0..63 are hi(dY) times (hi|lo)(X), rows 64..127 lo(dY)
// times (hi|lo)(X), so
//   dW[k,c] = (D[k,c] + D[k,BC+c]) + (D[64+k,c] + D[64+k,BC+c]),
// every product of the split. The tensor core's fp32 accumulation is not an
// IEEE round-to-nearest sum and its error grows with the number of rows added
// into one accumulator, so the accumulator is double-buffered in TMEM and
// drained every kPeriod blocks (512 rows) into fp32 registers with ordinary
// round-to-nearest adds.
//
// Layouts: the tf32 MMA takes K-major operands only (the reduction index
// contiguous), while NHWC rows hold channels contiguously. So:
//  - A = the dY split lives in TMEM (lane = row m, one column per row p),
//    written with tcgen05.st: a warp reads one 128-byte swizzled row of the
//    raw dY chunk per load (conflict-free) and each lane keeps its channel;
//  - B = the X split is transposed into a K-major 128B-swizzled shared tile
//    (row = channel, 32 rows p per 128 bytes): each lane owns one row p, and
//    every store writes one full 128-byte row (conflict-free).
// Data path: TMA (3-D maps over [N][H*W][ch], 32 channels x 32 rows per box,
// 128B swizzle) -> raw ring -> 8 converter warps (split, transpose, db) ->
// operand ring (B in smem, A in TMEM) -> one thread issues the MMAs ->
// tcgen05.commit frees the operand stage. Warp roles: 0 TMA producer, 1 MMA
// issuer, 2 TMEM owner, 4-11 converters, which also drain the accumulators
// and run the epilogue.
#include "tc_common.cuh"
#include "../kernel_entry.h"

namespace cig {
namespace {

constexpr int kThreads = 384;
constexpr int kConv = 256;                // converter threads (warps 4..11)
constexpr int kBP = 32;                   // rows per stage = one reduction block
constexpr int kChunk = kBP * 128;         // bytes of one 32-channel x kBP-row raw chunk
constexpr int kBK = 64;                   // k rows of an output tile (M = 2 x 64 with the split)
constexpr int kSmemBudget = 200 * 1024;
constexpr int kPeriod = 16;               // blocks accumulated in TMEM before a drain
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kDcol = 192;           // accumulator buffer b at column kDcol * b
constexpr uint32_t kAcol = 384;           // operand A ring at columns 384 + 32 * stage
constexpr int kMaxRaw = 12;               // raw stages at most (barrier area)

// BC: output channels c of a tile; Q: operand stages (the raw ring gets the
// rest of the shared-memory budget).
template <int BC, int Q>
struct Cfg {
  static constexpr int QS = Q;
  static constexpr int NC = BC / 32;                      // raw X chunks per stage
  static constexpr int RAW = (2 + NC) * kChunk;           // raw dY (2 chunks) + raw X
  static constexpr int OPB = 2 * BC * 128;                // K-major B: 2*BC rows x 128 B
  static constexpr int R0 = (kSmemBudget - QS * OPB) / RAW;
  static constexpr int R = R0 > kMaxRaw ? kMaxRaw : R0;   // raw stages
  static constexpr int N = 2 * BC;
  static constexpr int HALF = BC / 2;                     // output columns per converter thread
  static constexpr uint32_t TX = (uint32_t)RAW;
  static constexpr int BAR_BYTES = 512;
  static constexpr size_t SMEM = 1024 + (size_t)R * RAW + (size_t)QS * OPB + BAR_BYTES;
  static constexpr uint32_t IDESC = mma_idesc(2u, 0u, 0u, (uint32_t)N, 128u);
  static_assert(R >= 2, "raw pipeline too shallow");
  static_assert((2 * R + 2 * QS + 4) * 8 + 8 <= BAR_BYTES, "barrier area too small");
  static_assert(N % 16 == 0 && N >= 16 && N <= (int)kDcol, "invalid MMA N for M=128");
  static_assert(kAcol + 32 * QS <= kTmemCols && kDcol * 2 <= kAcol, "TMEM overflow");
  static_assert(QS < kPeriod, "a drain must come before its buffer is reused");
};

__device__ __forceinline__ float tf32_hi(float v) { return __uint_as_float(__float_as_uint(v) & 0xFFFFE000u); }

template <int BC, int Q>
__global__ void __launch_bounds__(kThreads, 1)
    wgrad1x1_tf32x3_kernel(const __grid_constant__ CUtensorMap tm_dy, const __grid_constant__ CUtensorMap tm_x,
                           float* __restrict__ out, float* __restrict__ ws, float* __restrict__ db,
                           float* __restrict__ ws_bias, int64_t K, int64_t C, int64_t blocks_per_sample,
                           int64_t tiles_c, int64_t tiles, int32_t S, int64_t blocks, unsigned* err) {
  using G = Cfg<BC, Q>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* raw = smem;                                   // R raw stages
  uint8_t* opb = smem + (size_t)G::R * G::RAW;           // G::QS operand (B) stages
  uint64_t* raw_full = reinterpret_cast<uint64_t*>(opb + (size_t)G::QS * G::OPB);
  uint64_t* raw_empty = raw_full + G::R;
  uint64_t* op_full = raw_empty + G::R;
  uint64_t* op_empty = op_full + G::QS;
  uint64_t* acc_full = op_empty + G::QS;                    // [2]
  uint64_t* acc_empty = acc_full + 2;                    // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + 2);
  volatile uint32_t* abort_flag = tmem_slot + 1;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int64_t tile = blockIdx.x % tiles;
  const int32_t sigma = (int32_t)(blockIdx.x / tiles);
  const int64_t k0 = (tile / tiles_c) * kBK;
  const int64_t c0 = (tile % tiles_c) * BC;
  const int64_t b0 = slice_begin(blocks, S, sigma);
  const int64_t nblk = slice_begin(blocks, S, sigma + 1) - b0;
  const int64_t nper = (nblk + kPeriod - 1) / kPeriod;   // accumulation periods

  if (threadIdx.x == 0) {
    for (int i = 0; i < G::R; ++i) {
      mbar_init(&raw_full[i], 1);
      mbar_init(&raw_empty[i], kConv);
    }
    for (int i = 0; i < G::QS; ++i) {
      mbar_init(&op_full[i], kConv);
      mbar_init(&op_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], kConv);
    }
    *abort_flag = 0u;
    mbar_fence_init();
    tma_prefetch(&tm_dy);
    tma_prefetch(&tm_x);
  }
  if (warp == 2) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---------------------------------------------------- TMA producer
    if (lane == 0) {
      // Ring stage s and the parity ph of its current round advance by
      // increments (no divisions in the loop); so do the sample and row.
      int s = 0;
      uint32_t ph = 0;
      int32_t n = (int32_t)(b0 / blocks_per_sample);
      int32_t row = (int32_t)((b0 % blocks_per_sample) * kBP);
      const int32_t row_end = (int32_t)(blocks_per_sample * kBP);
      int64_t it = 0;
      for (; it < nblk; ++it) {
        if (it >= G::R && !mbar_wait(&raw_empty[s], ph ^ 1u, abort_flag, err)) break;
        uint8_t* st = raw + (size_t)s * G::RAW;
        mbar_arrive_expect_tx(&raw_full[s], G::TX);
        tma_load_3d(st, &tm_dy, (int32_t)k0, row, n, &raw_full[s]);
        tma_load_3d(st + kChunk, &tm_dy, (int32_t)k0 + 32, row, n, &raw_full[s]);
#pragma unroll
        for (int j = 0; j < G::NC; ++j)
          tma_load_3d(st + (2 + j) * kChunk, &tm_x, (int32_t)(c0 + 32 * j), row, n, &raw_full[s]);
        if ((row += kBP) == row_end) {
          row = 0;
          ++n;
        }
        if (++s == G::R) {
          s = 0;
          ph ^= 1u;
        }
      }
      // Before the CTA can exit, every copy it started must have landed.
      for (int64_t q = it > G::R ? it - G::R : 0; q < it; ++q)
        mbar_wait(&raw_full[q % G::R], (uint32_t)(q / G::R) & 1u, nullptr, err);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t bbase = smem_u32(opb);
      int s = 0;
      uint32_t ph = 0;
      for (int64_t it = 0; it < nblk; ++it) {
        const int64_t per = it / kPeriod;
        const int within = (int)(it % kPeriod);
        const uint32_t d = tmem + kDcol * (uint32_t)(per & 1);
        if (within == 0 && per >= 2 && !mbar_wait(&acc_empty[per & 1], (uint32_t)((per >> 1) - 1) & 1u, abort_flag, err))
          break;
        if (!mbar_wait(&op_full[s], ph, abort_flag, err)) break;
        tc_fence_after();
        const uint32_t b = bbase + (uint32_t)(s * G::OPB);
        const uint32_t a = tmem + kAcol + 32u * (uint32_t)s;
#pragma unroll
        for (int kk = 0; kk < kBP / 8; ++kk) {
          // K-major SW128 B: 8-row groups 1024 B apart; the k step of 8 rows p
          // is a 32-byte advance inside the swizzled 128-byte row.
          const uint64_t bd = smem_desc_sw128(b + 32u * kk, 16, 1024);
          mma_tf32_ts(d, a + 8u * kk, bd, G::IDESC, (within > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&op_empty[s]);
        if (within == kPeriod - 1 || it == nblk - 1) mma_commit(&acc_full[per & 1]);
        if (++s == G::QS) {
          s = 0;
          ph ^= 1u;
        }
      }
    }
  } else if (warp >= 4) {
    // ---------------------------------------------------- converters
    const int cw = warp - 4;          // 0..7
    const int q = cw & 3;             // TMEM lane quarter (= warp % 4)
    const int hh = cw >> 2;           // rows p 16 hh .. 16 hh + 15 of a stage go to TMEM from this warp;
                                      // output columns hh * BC/2 .. of the tile are drained by it
    const int jdy = q & 1;            // raw dY chunk (channels 32 jdy ..) of this warp's lanes
    const bool lo_rows = q >= 2;      // lanes 64..127 hold lo(dY)
    // dY loads: row p = 16 hh + i, element = lane (channel), 128B swizzle
    int dsw[8];
#pragma unroll
    for (int t = 0; t < 8; ++t) dsw[t] = ((((lane >> 2) ^ t) << 4) | ((lane & 3) << 2)) + (16 * hh + t) * 128;
    const int dbase = jdy * kChunk;
    // X loads: row p = lane, unit (4 channels) cw of each 32-channel chunk
    const int xoff = 2 * kChunk + lane * 128 + ((cw ^ (lane & 7)) << 4);
    // B stores: channel c = 32 j + 4 cw + i -> K-major row c, column p = lane
    int sofs[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      sofs[i] = (4 * cw + i) * 128 + ((((lane >> 2) ^ (((cw & 1) << 2) + i)) << 4) | ((lane & 3) << 2));

    float acc[G::HALF];
#pragma unroll
    for (int i = 0; i < G::HALF; ++i) acc[i] = 0.f;
    float bsum = 0.f;  // db partial of channel k0 + 32 jdy + lane (hi warps only)
    int64_t drained = 0;
    bool alive = true;

    // Adds accumulator period `pd` (buffer pd & 1) into the registers.
    auto drain = [&](int64_t pd) -> bool {
      if (!mbar_wait(&acc_full[pd & 1], (uint32_t)(pd >> 1) & 1u, abort_flag, err)) return false;
      tc_fence_after();
      const uint32_t t = tmem + ((uint32_t)(32 * q) << 16) + kDcol * (uint32_t)(pd & 1) + (uint32_t)(hh * G::HALF);
#pragma unroll
      for (int j = 0; j < G::HALF / 16; ++j) {
        float part[16];
        tmem_ld16(t + 16u * j, part);  // products with X_hi
#pragma unroll
        for (int i = 0; i < 16; ++i) acc[16 * j + i] += part[i];
        tmem_ld16(t + BC + 16u * j, part);  // products with X_lo
#pragma unroll
        for (int i = 0; i < 16; ++i) acc[16 * j + i] += part[i];
      }
      tc_fence_before();
      mbar_arrive(&acc_empty[pd & 1]);
      return true;
    };

    int rs = 0, qs = 0;          // raw and operand ring stages
    uint32_t rph = 0, qph = 0;   // parities of their current rounds
    for (int64_t it = 0; it < nblk; ++it) {
      if (it >= kPeriod + G::QS && (it - G::QS) % kPeriod == 0) {
        if (!drain(drained)) { alive = false; break; }
        ++drained;
      }
      if (!mbar_wait(&raw_full[rs], rph, abort_flag, err)) { alive = false; break; }
      if (it >= G::QS && !mbar_wait(&op_empty[qs], qph ^ 1u, abort_flag, err)) {
        alive = false;
        break;
      }
      tc_fence_after();
      const uint8_t* st = raw + (size_t)rs * G::RAW;
      // dY -> TMEM A: lane = channel, 16 rows p per warp.
      {
        const uint8_t* cd = st + dbase;
        float v[16];
        if (lo_rows) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float f = *reinterpret_cast<const float*>(cd + dsw[i & 7] + (i >> 3) * 1024);
            v[i] = f - tf32_hi(f);
          }
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float f = *reinterpret_cast<const float*>(cd + dsw[i & 7] + (i >> 3) * 1024);
            v[i] = tf32_hi(f);
            bsum += f;
          }
        }
        tmem_st16(tmem + ((uint32_t)(32 * q) << 16) + kAcol + 32u * (uint32_t)qs + 16u * (uint32_t)hh, v);
      }
      // X -> K-major B: lane = row p, 4 channels per chunk, hi and lo rows.
      uint8_t* ob = opb + (size_t)qs * G::OPB;
#pragma unroll
      for (int j = 0; j < G::NC; ++j) {
        const float4 f = *reinterpret_cast<const float4*>(st + xoff + j * kChunk);
        const float fv[4] = {f.x, f.y, f.z, f.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float h = tf32_hi(fv[i]);
          *reinterpret_cast<float*>(ob + j * 4096 + sofs[i]) = h;
          *reinterpret_cast<float*>(ob + BC * 128 + j * 4096 + sofs[i]) = fv[i] - h;
        }
      }
      tmem_wait_st();
      tc_fence_before();
      fence_proxy_async_smem();  // B writes -> visible to the tensor core
      mbar_arrive(&raw_empty[rs]);
      mbar_arrive(&op_full[qs]);
      if (++rs == G::R) {
        rs = 0;
        rph ^= 1u;
      }
      if (++qs == G::QS) {
        qs = 0;
        qph ^= 1u;
      }
    }
    while (alive && drained < nper) {
      if (!drain(drained)) alive = false;
      ++drained;
    }

    // ---------------------------------------------------- epilogue
    signal_dependents();
    const bool ok = alive && *abort_flag == 0u;
    constexpr int LD = BC + 4;
    float* comb = reinterpret_cast<float*>(raw);                      // [64][LD]
    float* bred = reinterpret_cast<float*>(raw + 64 * LD * 4);        // [2][64]
    const int kl = 32 * jdy + lane;
    if (!lo_rows) bred[hh * 64 + kl] = bsum;
    if (lo_rows) {
      float* dst = comb + kl * LD + hh * G::HALF;
#pragma unroll
      for (int i = 0; i < G::HALF; i += 4) *reinterpret_cast<float4*>(dst + i) = make_float4(acc[i], acc[i + 1], acc[i + 2], acc[i + 3]);
    }
    asm volatile("bar.sync 1, 256;" ::: "memory");
    const int64_t E = K * C;
    const int64_t k = k0 + kl;
    if (!lo_rows && ok && k < K) {
      const float* cb = comb + kl * LD + hh * G::HALF;
      const int64_t cc = c0 + hh * G::HALF;
      float* dst = ws ? ws + (int64_t)sigma * E + k * C + cc : out + k * C + cc;
#pragma unroll
      for (int i = 0; i < G::HALF; i += 4) {
        if (cc + i < C) {  // C % 4 == 0: a 4-wide group is all in or all out
          const float4 o = *reinterpret_cast<const float4*>(cb + i);
          *reinterpret_cast<float4*>(dst + i) =
              make_float4(acc[i] + o.x, acc[i + 1] + o.y, acc[i + 2] + o.z, acc[i + 3] + o.w);
        }
      }
      if (hh == 0 && db && (tile % tiles_c) == 0) {
        const float v = bred[kl] + bred[64 + kl];  // rows 0-15 then 16-31 of every stage
        if (ws_bias) ws_bias[(int64_t)sigma * K + k] = v;
        else db[k] = v;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

int pick_bc(int64_t C) {
  if (C <= 32) return 32;
  if (C <= 64) return 64;
  return 96;
}

template <int BC, int Q>
cudaError_t launch_bc(const Plan& p, const Args& a) {
  using G = Cfg<BC, Q>;
  const Shape& s = p.sh;
  const int64_t hw = s.h * s.w;
  CUtensorMap tm_dy, tm_x;
  const uint64_t dy_dims[3] = {(uint64_t)s.k, (uint64_t)hw, (uint64_t)s.n};
  const uint64_t dy_strides[2] = {(uint64_t)s.k * 4u, (uint64_t)(hw * s.k) * 4u};
  const uint64_t x_dims[3] = {(uint64_t)s.c, (uint64_t)hw, (uint64_t)s.n};
  const uint64_t x_strides[2] = {(uint64_t)s.c * 4u, (uint64_t)(hw * s.c) * 4u};
  const uint32_t box[3] = {32u, (uint32_t)kBP, 1u};
  if (!encode_tmap(&tm_dy, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, a.b, dy_dims, dy_strides, box,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tmap(&tm_x, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, a.x, x_dims, x_strides, box,
                   CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  cudaError_t err = cudaFuncSetAttribute(wgrad1x1_tf32x3_kernel<BC, Q>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)G::SMEM);
  if (err != cudaSuccess) return err;
  const int64_t ctas = p.geo.tiles * p.split;
  if (ctas > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  const int64_t tiles_c = (s.c + BC - 1) / BC;
  const int64_t bps = (hw + kBP - 1) / kBP;
  wgrad1x1_tf32x3_kernel<BC, Q><<<(unsigned)ctas, kThreads, G::SMEM, a.stream>>>(
      tm_dy, tm_x, static_cast<float*>(a.out), a.ws, p.with_bias ? static_cast<float*>(a.db) : nullptr, a.ws_bias,
      s.k, s.c, bps, tiles_c, p.geo.tiles, p.split, p.geo.blocks, device_error_word());
  return cudaGetLastError();
}

}  // namespace

Geometry geometry_wgrad1x1_tf32x3(const Shape& s) {
  Geometry g;
  const bool pointwise = s.r == 1 && s.s == 1 && s.sh == 1 && s.sw == 1 && s.ph == 0 && s.pw == 0;
  if (!pointwise || s.groups != 1 || s.in_dt != CONV_F32 || s.out_dt != CONV_F32) return g;
  if (s.c % 4 != 0 || s.k % 4 != 0) return g;              // 16-byte row strides for TMA
  if (s.n < 1) return g;                                    // an empty batch takes the other kernels
  if (s.k < 32 || s.c < 32 || s.h * s.w < kBP) return g;    // no TMA box larger than its tensor
  if (s.h * s.w > 0x7fffffffLL || s.n > 0x7fffffffLL) return g;  // 32-bit TMA coordinates
  const int bc = pick_bc(s.c);
  g.ok = true;
  g.ctas_per_sm = 1;
  g.tiles = ((s.k + kBK - 1) / kBK) * ((s.c + bc - 1) / bc);
  g.blocks = s.n * ((s.h * s.w + kBP - 1) / kBP);
  return g;
}

cudaError_t launch_wgrad1x1_tf32x3(const Plan& p, const Args& a) {
  // Three operand stages (the rest of shared memory feeds the raw ring):
  // measured best of 2, 3 and 4 on the N=64 512x512 C=96 K=64 problem.
  switch (pick_bc(p.sh.c)) {
    case 32: return launch_bc<32, 3>(p, a);
    case 64: return launch_bc<64, 3>(p, a);
    default: return launch_bc<96, 3>(p, a);
  }
}

}  // namespace cig
