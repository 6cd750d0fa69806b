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
// and lo = v - hi (exact in fp32, then rounded to tf32 by the unit). The tile
// computes [dY_hi; dY_lo]^T x [X_hi | X_lo] as ONE M=128 x N=2*BC MMA per 8
// rows: rows 0..63 of the accumulator are hi(dY) times (hi|lo)(X), rows
// 64..127 are lo(dY) times (hi|lo)(X), so
//   dW[k,c] = (D[k,c] + D[k,BC+c]) + (D[64+k,c] + D[64+k,BC+c]),
// all four products of the split, with fp32 accumulation in TMEM.
//
// Data path (per CTA, one 64 x BC output tile, one slice of rows):
//   TMA (3-D maps over [N][H*W][ch], 128-byte swizzle, 32 channels x 32 rows
//   per box) lands raw dY and X rows in shared memory in exactly the
//   MN-major SW128 layout the MMA reads -> 4 converter warps split each value
//   into hi (in place) and lo (a parallel chunk), summing db from the raw dY on
//   the way -> one thread issues the MMAs -> tcgen05.commit frees the stage.
//   Warp roles: 0 TMA producer, 1 MMA issuer, 2 TMEM owner, 4-7 converters
//   and epilogue (TMEM lane quarters 0-3).
#include "tc_common.cuh"

namespace cig {
namespace {

constexpr int kThreads = 256;
constexpr int kBP = 32;                   // rows per stage = one reduction block
constexpr int kChunk = kBP * 128;         // bytes of one 32-channel x kBP-row swizzled chunk
constexpr int kBK = 64;                   // k rows of an output tile (M = 2 x 64 with the split)
constexpr int kSmemBudget = 200 * 1024;

template <int BC>
struct Cfg {
  static constexpr int NC = BC / 32;                     // raw X chunks per stage
  static constexpr int A_BYTES = 4 * kChunk;             // dY: hi k0-31, hi k32-63, lo, lo
  static constexpr int B_BYTES = 2 * NC * kChunk;        // X: hi chunks then lo chunks
  static constexpr int STAGE = A_BYTES + B_BYTES;
  static constexpr int STAGES = kSmemBudget / STAGE < 6 ? kSmemBudget / STAGE : 6;
  static constexpr int N = 2 * BC;                       // MMA N
  static constexpr int TMEM_COLS = N <= 64 ? 64 : (N <= 128 ? 128 : 256);
  static constexpr uint32_t TX = (2 + NC) * kChunk;      // raw bytes TMA lands per stage
  static constexpr int BAR_BYTES = 256;
  static constexpr size_t SMEM = 1024 + (size_t)STAGES * STAGE + BAR_BYTES;
  static constexpr uint32_t IDESC = mma_idesc(2u, 1u, 1u, (uint32_t)N, 128u);
  static_assert(STAGES >= 2, "pipeline too shallow");
  static_assert(N % 16 == 0 && N >= 16 && N <= 256, "invalid MMA N for M=128");
};

__device__ __forceinline__ float tf32_hi(float v) { return __uint_as_float(__float_as_uint(v) & 0xFFFFE000u); }

// Split one 16-byte unit (4 values) in place: hi stays, lo goes to `lo_dst`.
__device__ __forceinline__ float4 split_unit(float4* unit, float4* lo_dst) {
  const float4 v = *unit;
  float4 hi, lo;
  hi.x = tf32_hi(v.x); lo.x = v.x - hi.x;
  hi.y = tf32_hi(v.y); lo.y = v.y - hi.y;
  hi.z = tf32_hi(v.z); lo.z = v.z - hi.z;
  hi.w = tf32_hi(v.w); lo.w = v.w - hi.w;
  *unit = hi;
  *lo_dst = lo;
  return v;
}

template <int BC>
__global__ void __launch_bounds__(kThreads, 1)
    wgrad1x1_tf32x3_kernel(const __grid_constant__ CUtensorMap tm_dy, const __grid_constant__ CUtensorMap tm_x,
                           float* __restrict__ out, float* __restrict__ ws, float* __restrict__ db,
                           float* __restrict__ ws_bias, int64_t K, int64_t C, int64_t blocks_per_sample,
                           int64_t tiles_c, int64_t tiles, int32_t S, int64_t blocks, unsigned* err) {
  using G = Cfg<BC>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)G::STAGES * G::STAGE);
  uint64_t* conv = full + G::STAGES;
  uint64_t* empty = conv + G::STAGES;
  uint64_t* tmem_full = empty + G::STAGES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tmem_full + 1);
  volatile uint32_t* abort_flag = tmem_slot + 1;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int64_t tile = blockIdx.x % tiles;
  const int32_t sigma = (int32_t)(blockIdx.x / tiles);
  const int64_t k0 = (tile / tiles_c) * kBK;
  const int64_t c0 = (tile % tiles_c) * BC;
  const int64_t b0 = slice_begin(blocks, S, sigma);
  const int64_t nblk = slice_begin(blocks, S, sigma + 1) - b0;

  if (threadIdx.x == 0) {
    for (int i = 0; i < G::STAGES; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&conv[i], 128);
      mbar_init(&empty[i], 1);
    }
    mbar_init(tmem_full, 1);
    *abort_flag = 0u;
    mbar_fence_init();
    tma_prefetch(&tm_dy);
    tma_prefetch(&tm_x);
  }
  if (warp == 2) {
    tmem_alloc(tmem_slot, G::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---------------------------------------------------- TMA producer
    if (lane == 0) {
      int64_t it = 0;
      for (; it < nblk; ++it) {
        const int s = (int)(it % G::STAGES);
        const uint32_t round = (uint32_t)(it / G::STAGES);
        if (it >= G::STAGES && !mbar_wait(&empty[s], (round - 1) & 1u, abort_flag, err)) break;
        const int64_t b = b0 + it;
        const int32_t n = (int32_t)(b / blocks_per_sample);
        const int32_t row = (int32_t)((b % blocks_per_sample) * kBP);
        uint8_t* st = smem + (size_t)s * G::STAGE;
        mbar_arrive_expect_tx(&full[s], G::TX);
        tma_load_3d(st, &tm_dy, (int32_t)k0, row, n, &full[s]);
        tma_load_3d(st + kChunk, &tm_dy, (int32_t)k0 + 32, row, n, &full[s]);
#pragma unroll
        for (int j = 0; j < G::NC; ++j)
          tma_load_3d(st + G::A_BYTES + j * kChunk, &tm_x, (int32_t)(c0 + 32 * j), row, n, &full[s]);
      }
      // Before the CTA can exit, every copy it started must have landed.
      for (int64_t q = it > G::STAGES ? it - G::STAGES : 0; q < it; ++q)
        mbar_wait(&full[q % G::STAGES], (uint32_t)(q / G::STAGES) & 1u, nullptr, err);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t sbase = smem_u32(smem);
      for (int64_t it = 0; it < nblk; ++it) {
        const int s = (int)(it % G::STAGES);
        if (!mbar_wait(&conv[s], (uint32_t)(it / G::STAGES) & 1u, abort_flag, err)) break;
        tc_fence_after();
        const uint32_t a = sbase + (uint32_t)(s * G::STAGE);
        const uint32_t bb = a + G::A_BYTES;
#pragma unroll
        for (int kk = 0; kk < kBP / 8; ++kk) {
          // MN-major, 128B swizzle: 32-channel chunks kChunk bytes apart (LBO),
          // 8-row groups 1024 bytes apart (SBO); one MMA consumes one group.
          const uint64_t da = smem_desc_sw128(a + kk * 1024, kChunk, 1024);
          const uint64_t db_ = smem_desc_sw128(bb + kk * 1024, kChunk, 1024);
          mma_tf32(tmem, da, db_, G::IDESC, (it > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&empty[s]);
      }
      // Arrives once every MMA issued above has completed (or at once if none).
      if (nblk > 0) mma_commit(tmem_full);
      else mbar_arrive(tmem_full);
    }
  } else if (warp >= 4) {
    // ---------------------------------------------------- converters + epilogue
    const int ct = threadIdx.x - 128;  // 0..127
    const int u = ct % 8;              // logical 16-byte unit (4 channels) this thread owns
    const int r0 = ct / 8;             // first row (0..15); rows r0 and r0 + 16
    float bsum[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    for (int64_t it = 0; it < nblk; ++it) {
      const int s = (int)(it % G::STAGES);
      if (!mbar_wait(&full[s], (uint32_t)(it / G::STAGES) & 1u, abort_flag, err)) break;
      uint8_t* st = smem + (size_t)s * G::STAGE;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int row = r0 + 16 * h;
          const int off = row * 128 + ((u ^ (row & 7)) << 4);
          float4* unit = reinterpret_cast<float4*>(st + j * kChunk + off);
          const float4 v = split_unit(unit, reinterpret_cast<float4*>(st + (2 + j) * kChunk + off));
          bsum[j][0] += v.x; bsum[j][1] += v.y; bsum[j][2] += v.z; bsum[j][3] += v.w;
        }
      }
#pragma unroll
      for (int j = 0; j < G::NC; ++j) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int row = r0 + 16 * h;
          const int off = row * 128 + ((u ^ (row & 7)) << 4);
          uint8_t* xb = st + G::A_BYTES;
          split_unit(reinterpret_cast<float4*>(xb + j * kChunk + off),
                     reinterpret_cast<float4*>(xb + (G::NC + j) * kChunk + off));
        }
      }
      fence_proxy_async_smem();  // these writes -> visible to the tensor core
      mbar_arrive(&conv[s]);
    }

    // All MMAs done: the stage buffers are free for the epilogue's scratch.
    const bool ok = mbar_wait(tmem_full, 0u, nullptr, err) && *abort_flag == 0u;
    tc_fence_after();
    float* comb = reinterpret_cast<float*>(smem);                      // [64][BC + 4]
    float* bred = reinterpret_cast<float*>(smem + 64 * (BC + 4) * 4);  // [16][64]
    constexpr int LD = BC + 4;
    const int q = warp - 4;  // TMEM lane quarter
    const int m = 32 * q + lane;
    const uint32_t trow = tmem + ((uint32_t)(32 * q) << 16);
    if (q >= 2) {
#pragma unroll 1
      for (int j = 0; j < G::NC; ++j) {
        float hi[32], lo[32];
        if (nblk > 0) {
          tmem_ld32(trow + 32 * j, hi);
          tmem_ld32(trow + BC + 32 * j, lo);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) hi[i] = lo[i] = 0.f;
        }
        float* dst = comb + (m - 64) * LD + 32 * j;
#pragma unroll
        for (int i = 0; i < 32; i += 4)
          *reinterpret_cast<float4*>(dst + i) =
              make_float4(hi[i] + lo[i], hi[i + 1] + lo[i + 1], hi[i + 2] + lo[i + 2], hi[i + 3] + lo[i + 3]);
      }
    }
    // db partials of this thread: k = 32 j + 4 u + i
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int i = 0; i < 4; ++i) bred[r0 * 64 + 32 * j + 4 * u + i] = bsum[j][i];
    asm volatile("bar.sync 1, 128;" ::: "memory");
    const int64_t E = K * C;
    if (q < 2) {
      const int64_t k = k0 + m;
#pragma unroll 1
      for (int j = 0; j < G::NC; ++j) {
        float hi[32], lo[32];
        if (nblk > 0) {
          tmem_ld32(trow + 32 * j, hi);
          tmem_ld32(trow + BC + 32 * j, lo);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) hi[i] = lo[i] = 0.f;
        }
        const float* cb = comb + m * LD + 32 * j;
        const int64_t cc = c0 + 32 * j;
        if (ok && k < K) {
          float* dst = ws ? ws + (int64_t)sigma * E + k * C + cc : out + k * C + cc;
#pragma unroll
          for (int i = 0; i < 32; i += 4) {
            if (cc + i < C) {  // C % 4 == 0: a 4-wide group is all in or all out
              const float4 o = *reinterpret_cast<const float4*>(cb + i);
              *reinterpret_cast<float4*>(dst + i) =
                  make_float4((hi[i] + lo[i]) + o.x, (hi[i + 1] + lo[i + 1]) + o.y,
                              (hi[i + 2] + lo[i + 2]) + o.z, (hi[i + 3] + lo[i + 3]) + o.w);
            }
          }
        }
      }
    }
    if (db && (tile % tiles_c) == 0 && ct < 64 && ok) {
      float v = 0.f;
#pragma unroll
      for (int g = 0; g < 16; ++g) v += bred[g * 64 + ct];
      const int64_t k = k0 + ct;
      if (k < K) {
        if (ws_bias) ws_bias[(int64_t)sigma * K + k] = v;
        else db[k] = v;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, G::TMEM_COLS);
  }
}

int pick_bc(int64_t C) {
  if (C <= 32) return 32;
  if (C <= 64) return 64;
  if (C <= 96) return 96;
  return 128;
}

template <int BC>
cudaError_t launch_bc(const Plan& p, const Args& a) {
  using G = Cfg<BC>;
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
  cudaError_t err = cudaFuncSetAttribute(wgrad1x1_tf32x3_kernel<BC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)G::SMEM);
  if (err != cudaSuccess) return err;
  const int64_t ctas = p.geo.tiles * p.split;
  if (ctas > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  const int64_t tiles_c = (s.c + BC - 1) / BC;
  const int64_t bps = (hw + kBP - 1) / kBP;
  wgrad1x1_tf32x3_kernel<BC><<<(unsigned)ctas, kThreads, G::SMEM, a.stream>>>(
      tm_dy, tm_x, static_cast<float*>(a.out), a.ws, p.with_bias ? static_cast<float*>(a.db) : nullptr, a.ws_bias,
      s.k, s.c, bps, tiles_c, p.geo.tiles, p.split, p.geo.blocks, device_error_word());
  return cudaGetLastError();
}

}  // namespace

Geometry geometry_wgrad1x1_tf32x3(const Shape& s) {
  Geometry g;
  const bool pointwise = s.r == 1 && s.s == 1 && s.sh == 1 && s.sw == 1 && s.ph == 0 && s.pw == 0;
  if (!pointwise || s.groups != 1 || s.in_dt != CONV_F32 || s.out_dt != CONV_F32) return g;
  if (s.c % 4 != 0 || s.k % 4 != 0) return g;         // 16-byte row strides for TMA
  if (s.n < 1) return g;                               // an empty batch takes the other kernels
  if (s.k < 32 || s.c < 32 || s.h * s.w < kBP) return g;  // no TMA box larger than its tensor
  if (s.h * s.w > 0x7fffffffLL || s.n > 0x7fffffffLL) return g;  // 32-bit TMA coordinates
  const int bc = pick_bc(s.c);
  g.ok = true;
  g.ctas_per_sm = 1;
  g.tiles = ((s.k + kBK - 1) / kBK) * ((s.c + bc - 1) / bc);
  g.blocks = s.n * ((s.h * s.w + kBP - 1) / kBP);
  return g;
}

cudaError_t launch_wgrad1x1_tf32x3(const Plan& p, const Args& a) {
  switch (pick_bc(p.sh.c)) {
    case 32: return launch_bc<32>(p, a);
    case 64: return launch_bc<64>(p, a);
    case 96: return launch_bc<96>(p, a);
    default: return launch_bc<128>(p, a);
  }
}

}  // namespace cig
