// 16-bit forward convolution on the tcgen05 tensor cores, im2col gathered on
// the fly by TMA, deterministic split-K over the reduction (r, s, c).
//
// GEMM view: M = output pixels, N = output channels k, reduction (r, s, c)
// with c innermost:
//   A[m][(r,s,c)] = X[n, ho + r*dh - ph, wo + s*dw - pw, c],  B[k][(r,s,c)] = W[k,r,s,c].
// Both are K-major in NHWC / channels-last memory, as the bf16/fp16 MMA wants.
// An M tile is TR whole output rows (TR*Wo <= 128 pixels). For a reduction
// block (r, s, 64 channels) its A tile is ONE 4-D TMA box {64 ch, Wo, TR, 1}
// of X starting at (c0, s*dw - pw, ho0 + r*dh - ph, n): coordinates outside
// the image read zeros, which is exactly the zero padding, and the box lands
// as TR*Wo rows of 128 bytes in the 128B-swizzled K-major layout the MMA
// reads. B is a 2-D box {64, 128} of W viewed as [K][R*S*C].
//
// Split-K ("feat(rocke): split-K forward implicit-GEMM convolution on
// gfx1250", "Two-stage split-K"): CTA (tile, sigma) reduces the blocks of
// slice sigma and stores its fp32 partial tile into slab sigma of the
// workspace, every element written once; the fold kernel sums the slabs in
// slice order and rounds into Y. With one slice the epilogue rounds straight
// into Y. No fused epilogue is applied under split-K ("Review follow-ups":
// a bias or activation cannot be applied per slice).
//
// Warp roles: 0 TMA producer, 1 MMA issuer, 2 TMEM owner, 4-7 epilogue.
#include "tc_common.cuh"

namespace cig {
namespace {

constexpr int kThreads = 256;
constexpr int kBM = 128;
constexpr int kBN = 128;
constexpr int kBK = 64;                     // channels per reduction block (128 bytes of 16-bit)
constexpr int kStages = 3;
constexpr int kA = kBM * 128;               // A tile bytes (128 rows x 128 B)
constexpr int kB = kBN * 128;
constexpr int kStage = kA + kB;
constexpr size_t kSmem = 1024 + (size_t)kStages * kStage + 256;
constexpr uint32_t kTmemCols = 128;

struct FwdParams {
  int64_t K, Ho, Wo, Cg, S_f;   // S_f: filter width
  int64_t E;                    // output elements N*Ho*Wo*K (one slab)
  int64_t cblocks;              // Cg / 64
  int64_t tiles_m_per_img;      // ceil(Ho / TR)
  int64_t tiles_n;              // ceil(K / 128)
  int64_t tiles;                // N * tiles_m_per_img * tiles_n
  int64_t blocks;               // R * S * cblocks
  int32_t TR;                   // output rows per M tile
  int32_t ph, pw, dh, dw;
  int32_t split;
};

template <typename TO>
__device__ __forceinline__ void store8(TO* dst, const float* v);
template <>
__device__ __forceinline__ void store8<float>(float* dst, const float* v) {
  reinterpret_cast<float4*>(dst)[0] = make_float4(v[0], v[1], v[2], v[3]);
  reinterpret_cast<float4*>(dst)[1] = make_float4(v[4], v[5], v[6], v[7]);
}
template <>
__device__ __forceinline__ void store8<__nv_bfloat16>(__nv_bfloat16* dst, const float* v) {
  __nv_bfloat162 h[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
  *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<uint4*>(h);
}
template <>
__device__ __forceinline__ void store8<__half>(__half* dst, const float* v) {
  __half2 h[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) h[i] = __floats2half2_rn(v[2 * i], v[2 * i + 1]);
  *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<uint4*>(h);
}

template <typename TO, uint32_t FMT>
__global__ void __launch_bounds__(kThreads, 2)
    fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w, TO* out,
                  float* ws, FwdParams fp, unsigned* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)kStages * kStage);
  uint64_t* empty = full + kStages;
  uint64_t* tmem_full = empty + kStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tmem_full + 1);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  constexpr uint32_t IDESC = mma_idesc(FMT, 0u, 0u, (uint32_t)kBN, (uint32_t)kBM);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int64_t tile = blockIdx.x % fp.tiles;
  const int32_t sigma = (int32_t)(blockIdx.x / fp.tiles);
  const int64_t tn = tile % fp.tiles_n;
  const int64_t tm = tile / fp.tiles_n;
  const int64_t img = tm / fp.tiles_m_per_img;
  const int64_t ho0 = (tm % fp.tiles_m_per_img) * fp.TR;
  const int64_t k0 = tn * kBN;
  const int64_t b0 = slice_begin(fp.blocks, fp.split, sigma);
  const int64_t nblk = slice_begin(fp.blocks, fp.split, sigma + 1) - b0;
  const uint32_t tx = (uint32_t)(fp.TR * fp.Wo * 128 + kB);

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_init(tmem_full, 1);
    *abort_flag = 0u;
    mbar_fence_init();
    tma_prefetch(&tm_x);
    tma_prefetch(&tm_w);
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
    if (lane == 0) {
      int64_t it = 0;
      for (; it < nblk; ++it) {
        const int s = (int)(it % kStages);
        const uint32_t round = (uint32_t)(it / kStages);
        if (it >= kStages && !mbar_wait(&empty[s], (round - 1) & 1u, abort_flag, err)) break;
        const int64_t b = b0 + it;
        const int64_t cb = b % fp.cblocks;
        const int64_t rs = b / fp.cblocks;
        const int32_t r = (int32_t)(rs / fp.S_f), sx = (int32_t)(rs % fp.S_f);
        uint8_t* st = smem + (size_t)s * kStage;
        mbar_arrive_expect_tx(&full[s], tx);
        tma_load_4d(st, &tm_x, (int32_t)(cb * kBK), sx * fp.dw - fp.pw, (int32_t)ho0 + r * fp.dh - fp.ph,
                    (int32_t)img, &full[s]);
        tma_load_2d(st + kA, &tm_w, (int32_t)(rs * fp.Cg + cb * kBK), (int32_t)k0, &full[s]);
      }
      for (int64_t q = it > kStages ? it - kStages : 0; q < it; ++q)
        mbar_wait(&full[q % kStages], (uint32_t)(q / kStages) & 1u, nullptr, err);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t base = smem_u32(smem);
      for (int64_t it = 0; it < nblk; ++it) {
        const int s = (int)(it % kStages);
        if (!mbar_wait(&full[s], (uint32_t)(it / kStages) & 1u, abort_flag, err)) break;
        tc_fence_after();
        const uint32_t a = base + (uint32_t)(s * kStage), b = a + kA;
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk) {
          // K-major SW128: 8-row groups 1024 B apart; a K step of 16 elements is
          // a 32-byte advance inside the swizzled 128-byte row.
          mma_f16(tmem, smem_desc_sw128(a + 32u * kk, 16, 1024), smem_desc_sw128(b + 32u * kk, 16, 1024), IDESC,
                  (it > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&empty[s]);
      }
      if (nblk > 0) mma_commit(tmem_full);
      else mbar_arrive(tmem_full);
    }
  } else if (warp >= 4) {
    const bool ok = mbar_wait(tmem_full, 0u, nullptr, err) && *abort_flag == 0u;
    signal_dependents();
    tc_fence_after();
    const int q = warp - 4;
    const int m = 32 * q + lane;  // tile row = output pixel within the tile
    const int64_t ho = ho0 + m / fp.Wo, wo = m % fp.Wo;
    const bool row_ok = ok && m < fp.TR * fp.Wo && ho < fp.Ho;
    const int64_t pix = (img * fp.Ho + ho) * fp.Wo + wo;
    float* slab = ws ? ws + (int64_t)sigma * fp.E : nullptr;
#pragma unroll 1
    for (int j = 0; j < kBN / 32; ++j) {
      float v[32];
      if (nblk > 0) {
        tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + 32u * j, v);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = 0.f;
      }
      if (!row_ok) continue;
#pragma unroll
      for (int i = 0; i < 32; i += 8) {
        const int64_t k = k0 + 32 * j + i;
        if (k >= fp.K) continue;  // K % 8 == 0: an 8-wide group is all in or all out
        if (slab) {
          store8<float>(slab + pix * fp.K + k, v + i);
        } else {
          store8<TO>(out + pix * fp.K + k, v + i);
        }
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

bool fwd_tc_admissible(const Shape& s) {
  if (s.in_dt == CONV_F32 || s.groups != 1 || s.sh != 1 || s.sw != 1) return false;
  if (s.cg % kBK != 0 || s.k % 8 != 0 || s.k < kBN) return false;
  if (s.wo > kBM || s.wo > s.w) return false;    // one TMA box spans a whole output row
  if (s.n < 1 || s.n > 0x7fffffffLL || s.h > 0x7fffffffLL || s.w > 0x7fffffffLL) return false;
  const int64_t tr = kBM / s.wo;
  if ((tr < s.ho ? tr : s.ho) > s.h) return false;  // no box taller than the image
  if (s.r * s.s * s.cg > 0x7fffffffLL) return false;
  return true;
}

FwdParams make_params(const Plan& p) {
  const Shape& s = p.sh;
  FwdParams fp;
  fp.K = s.k;
  fp.E = s.y_elems();
  fp.Ho = s.ho;
  fp.Wo = s.wo;
  fp.Cg = s.cg;
  fp.S_f = s.s;
  fp.cblocks = s.cg / kBK;
  fp.TR = (int32_t)(kBM / s.wo < s.ho ? kBM / s.wo : s.ho);
  fp.tiles_m_per_img = (s.ho + fp.TR - 1) / fp.TR;
  fp.tiles_n = (s.k + kBN - 1) / kBN;
  fp.tiles = s.n * fp.tiles_m_per_img * fp.tiles_n;
  fp.blocks = s.r * s.s * fp.cblocks;
  fp.ph = (int32_t)s.ph;
  fp.pw = (int32_t)s.pw;
  fp.dh = (int32_t)s.dh;
  fp.dw = (int32_t)s.dw;
  fp.split = p.split;
  return fp;
}

template <typename TO, uint32_t FMT>
cudaError_t launch_typed(const Plan& p, const Args& a, CUtensorMapDataType dt) {
  const Shape& s = p.sh;
  FwdParams fp = make_params(p);
  CUtensorMap tm_x, tm_w;
  const uint64_t x_dims[4] = {(uint64_t)s.c, (uint64_t)s.w, (uint64_t)s.h, (uint64_t)s.n};
  const uint64_t x_strides[3] = {(uint64_t)s.c * 2u, (uint64_t)(s.w * s.c) * 2u, (uint64_t)(s.h * s.w * s.c) * 2u};
  const uint32_t x_box[4] = {(uint32_t)kBK, (uint32_t)s.wo, (uint32_t)fp.TR, 1u};
  const uint64_t w_dims[2] = {(uint64_t)(s.r * s.s * s.cg), (uint64_t)s.k};
  const uint64_t w_strides[1] = {(uint64_t)(s.r * s.s * s.cg) * 2u};
  const uint32_t w_box[2] = {(uint32_t)kBK, (uint32_t)kBN};
  if (!encode_tmap(&tm_x, dt, 4, a.x, x_dims, x_strides, x_box, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tmap(&tm_w, dt, 2, a.b, w_dims, w_strides, w_box, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  cudaError_t err =
      cudaFuncSetAttribute(fwd_tc_kernel<TO, FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
  if (err != cudaSuccess) return err;
  const int64_t ctas = fp.tiles * p.split;
  if (ctas > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  // Slab sigma starts at ws + sigma * E; the kernel indexes pixels within it.
  fwd_tc_kernel<TO, FMT><<<(unsigned)ctas, kThreads, kSmem, a.stream>>>(tm_x, tm_w, static_cast<TO*>(a.out), a.ws,
                                                                        fp, device_error_word());
  return cudaGetLastError();
}

}  // namespace

Geometry geometry_fwd_tc(const Shape& s) {
  Geometry g;
  if (!fwd_tc_admissible(s)) return g;
  const int64_t tr = kBM / s.wo < s.ho ? kBM / s.wo : s.ho;
  g.ok = true;
  g.ctas_per_sm = 2;
  g.tiles = s.n * ((s.ho + tr - 1) / tr) * ((s.k + kBN - 1) / kBN);
  g.blocks = s.r * s.s * (s.cg / kBK);
  return g;
}

cudaError_t launch_fwd_tc(const Plan& p, const Args& a) {
  if (p.sh.in_dt == CONV_BF16) {
    if (p.sh.out_dt == CONV_F32) return launch_typed<float, 1u>(p, a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16);
    return launch_typed<__nv_bfloat16, 1u>(p, a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16);
  }
  if (p.sh.out_dt == CONV_F32) return launch_typed<float, 0u>(p, a, CU_TENSOR_MAP_DATA_TYPE_FLOAT16);
  return launch_typed<__half, 0u>(p, a, CU_TENSOR_MAP_DATA_TYPE_FLOAT16);
}

}  // namespace cig
