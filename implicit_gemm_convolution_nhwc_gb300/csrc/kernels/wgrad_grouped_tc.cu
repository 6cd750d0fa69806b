// Grouped 16-bit weight gradient (+ bias gradient) on the tensor cores, as
// block-diagonal dense blocks ("perf(rocke): depthwise 7x7 and grouped
// cpg4/8 wgrad on batched mfma 4x4x4": the grouped wgrad; here for Cg = Kg
// in {2, 4, 8, 16, 32} and C a multiple of 128).
//
// Output channels [k0, k0 + 128) read input channels [k0, k0 + 128), so per
// filter tap (r, s) the block's gradient is the dense 128 x 128 product
//   D[k][c'] = sum over pixels p of dY[p][k0 + k] * X[p shifted by (r, s)][k0 + c'],
// of which dW keeps the diagonal Cg x Cg blocks (c' in k's group). The MMA
// runs with both operands MN-major (channels contiguous, the pixel
// reduction across 128-byte rows), exactly as TMA boxes {64 channels, rows}
// with 128B swizzle land: no transposition. A CTA owns one channel block,
// the S taps of one filter row (S <= 4: one 128-column TMEM accumulator
// each) and a split-K slice of pixel blocks; a pixel block is TR whole output
// rows, padded to a multiple of 16 rows with zeros that TMA never overwrites.
// Per block it loads the dY tile once and one shifted X tile per tap (TMA
// traversal strides give the convolution stride). The bias gradient (db = sum
// of dY) is summed from the dY tiles in shared memory by the epilogue warps,
// which are idle during the main loop, on the CTAs of filter row 0.
//
// Warp roles: 0 TMA producer, 1 MMA issuer, 2 TMEM owner, 4-7 bias sums and
// epilogue.
#include <type_traits>

#include "tc_common.cuh"
#include "../kernel_entry.h"

namespace cig {
namespace {

constexpr int kThreads = 256;
constexpr int kCB = 128;             // channels of a block (M and N of the MMA)
constexpr int kStages = 3;
constexpr int kMaxTaps = 4;          // taps per CTA (TMEM: 4 x 128 columns)
constexpr uint32_t kTmemCols = 512;
constexpr int kMaxRows = 128;        // pixel rows of a block (the box height limit keeps TR*Wo <= 128)

struct GwParams {
  int64_t N, H, W, C, K, Ho, Wo;
  int32_t R, S, ph, pw, sh, sw, dh, dw, Cg;
  int32_t TR;            // output rows per pixel block
  int32_t BP;            // pixel rows padded to 16
  int64_t tiles_per_img;  // ceil(Ho / TR)
  int64_t blocks;         // N * tiles_per_img (the split-K reduction blocks)
  int64_t kblocks;        // K / 128
  int32_t split;
  int64_t E;              // dW elements (one slab)
};

template <typename TI, typename TO>
__global__ void __launch_bounds__(kThreads, 1)
    wgrad_grouped_tc_kernel(const __grid_constant__ CUtensorMap tm_dy, const __grid_constant__ CUtensorMap tm_x,
                            TO* out, float* ws, TO* db, float* ws_bias, GwParams gp, unsigned* err) {
  const int AS = gp.BP * 128;              // one 64-channel atom of a tile
  const int T = gp.S;                      // taps per CTA (one filter row)
  const int stage_bytes = (2 + 2 * T) * AS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)kStages * stage_bytes);
  uint64_t* empty = full + kStages;
  uint64_t* tmem_full = empty + kStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tmem_full + 1);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  constexpr uint32_t FMT = std::is_same<TI, __nv_bfloat16>::value ? 1u : 0u;
  constexpr uint32_t IDESC = mma_idesc(FMT, 1u, 1u, (uint32_t)kCB, (uint32_t)kCB);
  constexpr uint32_t IDESC2 = mma_idesc(FMT, 1u, 1u, (uint32_t)(2 * kCB), (uint32_t)kCB);  // two taps at once

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int64_t tiles = gp.kblocks * gp.R;
  const int64_t tile = blockIdx.x % tiles;
  const int32_t sigma = (int32_t)(blockIdx.x / tiles);
  const int64_t kb = tile % gp.kblocks;
  const int32_t rrow = (int32_t)(tile / gp.kblocks);  // the filter row of this CTA's taps
  const int32_t k0 = (int32_t)(kb * kCB);
  const int64_t b0 = slice_begin(gp.blocks, gp.split, sigma);
  const int64_t nblk = slice_begin(gp.blocks, gp.split, sigma + 1) - b0;
  const bool do_bias = db != nullptr && rrow == 0;
  const uint32_t box_bytes = (uint32_t)(gp.TR * gp.Wo * 128);
  const uint32_t tx = (uint32_t)(2 + 2 * T) * box_bytes;

  // Zero the ring once: the pad rows of every tile stay zero (TMA writes only
  // the first TR*Wo rows of each atom).
  for (int i = threadIdx.x; i < kStages * stage_bytes / 16; i += kThreads)
    reinterpret_cast<uint4*>(smem)[i] = make_uint4(0u, 0u, 0u, 0u);
  fence_proxy_async_smem();
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1 + (do_bias ? 128 : 0));
    }
    mbar_init(tmem_full, 1);
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
      int s = 0;
      uint32_t ph = 0;
      int64_t n = b0 / gp.tiles_per_img;
      int64_t tr = b0 % gp.tiles_per_img;
      int64_t it = 0;
      for (; it < nblk; ++it) {
        if (it >= kStages && !mbar_wait(&empty[s], ph ^ 1u, abort_flag, err)) break;
        uint8_t* st = smem + (size_t)s * stage_bytes;
        const int32_t ho0 = (int32_t)(tr * gp.TR);
        mbar_arrive_expect_tx(&full[s], tx);
        for (int h = 0; h < 2; ++h)  // dY: the block's pixels x channels k0 + 64 h ..
          tma_load_4d(st + h * AS, &tm_dy, k0 + 64 * h, 0, ho0, (int32_t)n, &full[s]);
        for (int t = 0; t < T; ++t)  // X shifted by tap (rrow, t), channels k0 + 64 h ..
          for (int h = 0; h < 2; ++h)
            tma_load_4d(st + (2 + 2 * t + h) * AS, &tm_x, k0 + 64 * h, t * gp.dw - gp.pw,
                        ho0 * gp.sh + rrow * gp.dh - gp.ph, (int32_t)n, &full[s]);
        if (++tr == gp.tiles_per_img) {
          tr = 0;
          ++n;
        }
        if (++s == kStages) {
          s = 0;
          ph ^= 1u;
        }
      }
      for (int64_t q = it > kStages ? it - kStages : 0; q < it; ++q)
        mbar_wait(&full[q % kStages], (uint32_t)(q / kStages) & 1u, nullptr, err);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t base = smem_u32(smem);
      int s = 0;
      uint32_t ph = 0;
      for (int64_t j = 0; j < nblk; ++j) {
        if (!mbar_wait(&full[s], ph, abort_flag, err)) break;
        tc_fence_after();
        const uint32_t a = base + (uint32_t)(s * stage_bytes);
        // Taps t and t + 1 have adjacent B tiles (4 atoms AS apart) and adjacent
        // accumulators, so one N = 256 MMA covers both (measured ~1.4x the
        // multiply-add rate of two N = 128 MMAs here); an odd last tap uses N = 128.
        for (int t = 0; t < T; t += 2) {
          const uint32_t b = a + (uint32_t)((2 + 2 * t) * AS);
          const uint32_t idesc = t + 1 < T ? IDESC2 : IDESC;
          for (int kk = 0; kk < gp.BP / 16; ++kk) {
            // MN-major SW128: 64-channel atoms AS bytes apart (LBO), 8-row groups
            // 1024 bytes apart (SBO); 16 pixel rows = 2048 bytes further.
            mma_f16(tmem + (uint32_t)(t * kCB), smem_desc_sw128(a + 2048u * kk, (uint32_t)AS, 1024),
                    smem_desc_sw128(b + 2048u * kk, (uint32_t)AS, 1024), idesc, (j > 0 || kk > 0) ? 1u : 0u);
          }
        }
        mma_commit(&empty[s]);
        if (++s == kStages) {
          s = 0;
          ph ^= 1u;
        }
      }
      if (nblk > 0) mma_commit(tmem_full);
      else mbar_arrive(tmem_full);
    }
  } else if (warp >= 4) {
    const int q = warp - 4;
    const int m = 32 * q + lane;  // block channel k0 + m (TMEM lane m)
    // ---------------------------------------------------- bias sums (filter row 0)
    float bsum = 0.f;
    if (do_bias) {
      const int rows = gp.TR * gp.Wo;
      const int hofs = (m / 64) * AS, unit = (m % 64) / 8, el = (m % 8) * 2;
      int s = 0;
      uint32_t ph = 0;
      for (int64_t j = 0; j < nblk; ++j) {
        if (!mbar_wait(&full[s], ph, abort_flag, err)) break;
        const uint8_t* at = smem + (size_t)s * stage_bytes + hofs;
        float part = 0.f;
        for (int p = 0; p < rows; ++p)
          part += to_f32(*reinterpret_cast<const TI*>(at + p * 128 + ((unit ^ (p & 7)) << 4) + el));
        bsum += part;
        mbar_arrive(&empty[s]);
        if (++s == kStages) {
          s = 0;
          ph ^= 1u;
        }
      }
    }
    // ---------------------------------------------------- epilogue
    const bool ok = mbar_wait(tmem_full, 0u, nullptr, err) && *abort_flag == 0u;
    signal_dependents();
    tc_fence_after();
    const int Cg = gp.Cg;
    const int gl = (lane / Cg) * Cg;  // first column (within the warp's 32) of this row's group
    const int64_t k = k0 + m;
    for (int t = 0; t < T; ++t) {
      float v[32];
      if (nblk > 0) {
        tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(t * kCB + 32 * q), v);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = 0.f;
      }
      if (!ok || k >= gp.K) continue;
      const int64_t tap = (int64_t)rrow * gp.S + t;
      const int64_t dst = (k * gp.R * gp.S + tap) * Cg;  // dW[k][r][s][0..Cg)
      // row m's group columns gl .. gl + Cg - 1 of the warp's 32 (static selects)
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        if (c >= Cg) break;
        float val = 0.f;
#pragma unroll
        for (int g = 0; g < 32; ++g)
          if (g == gl + c) val = v[g];
        if (ws) ws[(int64_t)sigma * gp.E + dst + c] = val;
        else store_out(out + dst + c, val);
      }
    }
    if (do_bias && ok && k < gp.K) {
      if (ws_bias) ws_bias[(int64_t)sigma * gp.K + k] = bsum;
      else store_out(db + k, bsum);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// Output rows of a pixel block: about 64 pixels, whole output rows.
int64_t block_rows(const Shape& s) {
  const int64_t tr = 64 / s.wo;
  return tr < 1 ? 1 : (tr > s.ho ? s.ho : tr);
}

bool admissible(const Shape& s) {
  if (s.in_dt == CONV_F32 || s.groups < 2 || s.cg != s.kg) return false;
  if (!(s.cg == 2 || s.cg == 4 || s.cg == 8 || s.cg == 16 || s.cg == 32)) return false;
  if (s.c % kCB != 0 || s.s > kMaxTaps || s.sh > 8 || s.sw > 8) return false;
  if (s.wo > kMaxRows || s.wo * s.sw > 256 || s.wo * s.sw > s.w) return false;  // boxes span whole rows
  const int64_t tr = block_rows(s);
  if (tr * s.wo > kMaxRows || tr * s.sh > 256 || tr * s.sh > s.h) return false;
  if (s.n < 1 || s.n > 0x7fffffffLL || s.h > 0x7fffffffLL || s.w > 0x7fffffffLL) return false;
  const int64_t bp = (tr * s.wo + 15) / 16 * 16;
  const int64_t smem = 1024 + kStages * (2 + 2 * s.s) * bp * 128 + 256;
  return smem <= 227 * 1024;
}

template <typename TI, typename TO>
cudaError_t launch_typed(const Plan& p, const Args& a, CUtensorMapDataType dt) {
  const Shape& s = p.sh;
  GwParams gp;
  gp.N = s.n; gp.H = s.h; gp.W = s.w; gp.C = s.c; gp.K = s.k; gp.Ho = s.ho; gp.Wo = s.wo;
  gp.R = (int32_t)s.r; gp.S = (int32_t)s.s;
  gp.ph = (int32_t)s.ph; gp.pw = (int32_t)s.pw; gp.sh = (int32_t)s.sh; gp.sw = (int32_t)s.sw;
  gp.dh = (int32_t)s.dh; gp.dw = (int32_t)s.dw; gp.Cg = (int32_t)s.cg;
  gp.TR = (int32_t)block_rows(s);
  gp.BP = (int32_t)((gp.TR * s.wo + 15) / 16 * 16);
  gp.tiles_per_img = (s.ho + gp.TR - 1) / gp.TR;
  gp.blocks = s.n * gp.tiles_per_img;
  gp.kblocks = s.k / kCB;
  gp.split = p.split;
  gp.E = s.w_elems();
  CUtensorMap tm_dy, tm_x;
  const uint64_t y_dims[4] = {(uint64_t)s.k, (uint64_t)s.wo, (uint64_t)s.ho, (uint64_t)s.n};
  const uint64_t y_strides[3] = {(uint64_t)s.k * 2u, (uint64_t)(s.wo * s.k) * 2u, (uint64_t)(s.ho * s.wo * s.k) * 2u};
  const uint32_t y_box[4] = {64u, (uint32_t)s.wo, (uint32_t)gp.TR, 1u};
  const uint64_t x_dims[4] = {(uint64_t)s.c, (uint64_t)s.w, (uint64_t)s.h, (uint64_t)s.n};
  const uint64_t x_strides[3] = {(uint64_t)s.c * 2u, (uint64_t)(s.w * s.c) * 2u, (uint64_t)(s.h * s.w * s.c) * 2u};
  const uint32_t x_box[4] = {64u, (uint32_t)(s.wo * s.sw), (uint32_t)(gp.TR * s.sh), 1u};
  const uint32_t x_estr[4] = {1u, (uint32_t)s.sw, (uint32_t)s.sh, 1u};
  if (!encode_tmap(&tm_dy, dt, 4, a.b, y_dims, y_strides, y_box, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tmap(&tm_x, dt, 4, a.x, x_dims, x_strides, x_box, CU_TENSOR_MAP_SWIZZLE_128B, x_estr))
    return cudaErrorInvalidValue;
  const size_t smem = 1024 + (size_t)kStages * (2 + 2 * s.s) * gp.BP * 128 + 256;
  auto kern = wgrad_grouped_tc_kernel<TI, TO>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  const int64_t ctas = p.geo.tiles * p.split;
  if (ctas > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  kern<<<(unsigned)ctas, kThreads, smem, a.stream>>>(tm_dy, tm_x, static_cast<TO*>(a.out), a.ws,
                                                     p.with_bias ? static_cast<TO*>(a.db) : nullptr, a.ws_bias, gp,
                                                     device_error_word());
  return cudaGetLastError();
}

}  // namespace

Geometry geometry_wgrad_grouped_tc(const Shape& s) {
  Geometry g;
  if (!admissible(s)) return g;
  g.ok = true;
  g.ctas_per_sm = 1;
  g.tiles = (s.k / kCB) * s.r;
  g.blocks = s.n * ((s.ho + block_rows(s) - 1) / block_rows(s));
  return g;
}

cudaError_t launch_wgrad_grouped_tc(const Plan& p, const Args& a) {
  if (p.sh.in_dt == CONV_BF16) {
    if (p.sh.out_dt == CONV_F32) return launch_typed<__nv_bfloat16, float>(p, a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16);
    return launch_typed<__nv_bfloat16, __nv_bfloat16>(p, a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16);
  }
  if (p.sh.out_dt == CONV_F32) return launch_typed<__half, float>(p, a, CU_TENSOR_MAP_DATA_TYPE_FLOAT16);
  return launch_typed<__half, __half>(p, a, CU_TENSOR_MAP_DATA_TYPE_FLOAT16);
}

}  // namespace cig
