// Dense 16-bit weight gradient (+ bias gradient) on the tcgen05 tensor cores,
// deterministic split-K over the output pixels.
//
// Per filter tap (r, s) the weight gradient is a GEMM over the output pixels
// p = (n, ho, wo) ("ROCm/rocm-libraries PR #11188", "Motivation": the NHWC
// implicit-GEMM weight gradient; a 1x1 one is dY^T X on the reshaped tensors):
//   dW[k][r][s][c] = sum_p dY[p][k] * X[n, ho*sh + r*dh - ph, wo*sw + s*dw - pw][c],
// with M = output channels k, N = input channels c and the pixels as the
// MMA's reduction dimension. In NHWC memory both operands have their channels
// contiguous and consecutive pixels 128 bytes apart once a TMA box of 64
// channels lands: they are MN-major, exactly as TMA boxes {64 channels, BW
// columns, TR rows, 1 image} with 128B swizzle write them, so nothing is
// transposed. The shifted X box of a tap reads the convolution stride through
// TMA traversal strides and the zero padding through out-of-image coordinates
// (zero fill).
//
// A CTA owns MS x 128 output channels (M sub-tiles sharing the X tile), BN
// input channels (64..256) and one tap, and a split-K slice of pixel blocks; a
// pixel block is TR x BW output positions of one image, its rows padded to a
// multiple of 16 with zeros that TMA never overwrites. Split-K ("feat(rocke):
// split-K forward implicit-GEMM convolution on gfx1250", "Two-stage split-K",
// applied to this reduction): CTA (tile, sigma) stores its fp32 partial tile
// into slab sigma, every element once; the fold sums the slabs in slice order.
// The CTAs of one slice are consecutive, so the tiles that read the same
// pixels run together and share them through L2. The bias gradient (db = sum
// of dY) is summed from the dY tiles in shared memory by the epilogue warps,
// idle during the main loop, each output channel's sum in one of the CTAs that
// read its dY (spread over the taps and input-channel tiles).
//
// Warp roles: 0 TMA producer, 1 MMA issuer, 2 TMEM owner, 4-7 bias sums and
// epilogue (TMA-store through shared memory).
#include <type_traits>

#include "tc_store.cuh"
#include "../kernel_entry.h"

namespace cig {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxStages = 8;
constexpr int kStageBudget = 64 * 1024;  // bytes of one ring stage at most
constexpr int kEpiBufs = 4;               // epilogue staging buffers of 16 KB (the ring is at least 118 KB)
constexpr size_t kSmemMax = 232448;      // dynamic shared memory a CTA may use (227 KB)

// A pair of 16-bit values (one 32-bit word, the lower one first) widened to fp32.
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

struct WtParams {
  int64_t K, Ho, Wo;        // output channels (all groups), output extent
  int32_t Cg, Kg;           // channels per group
  int32_t R, S, ph, pw, sh, sw, dh, dw;
  int32_t TR, BW, BP;       // output rows and columns of a pixel block; its rows padded to 16
  int64_t hblocks, wblocks;  // ceil(Ho / TR), ceil(Wo / BW)
  int64_t blocks;           // N * hblocks * wblocks (the split-K reduction blocks)
  int32_t MS, BN;           // M sub-tiles of 128 output channels; input channels of a tile
  int64_t ktiles, ctiles;   // ceil(Kg / (128 MS)), ceil(Cg / BN)
  int64_t tiles;            // groups * ktiles * ctiles * R * S
  int32_t split, stages;
  uint32_t tmem_cols;
};

// The MMAs of one pixel block: KK steps of 16 pixel rows, each MSX sub-tile
// MMAs (M = 128, N = BN) sharing the step's B. Both operands MN-major SW128:
// 64-channel atoms 16 KK rows of 128 bytes apart (LBO), 8-row groups 1024
// bytes apart (SBO); 16 pixel rows are 2048 bytes further. Unrolled at
// compile time, with the atom stride a constant: issued from a loop with
// run-time bounds, the MMAs left the tensor pipe idle between them (the
// supplement's stage 1 took 176 us instead of 142).
template <int KK, int MSX>
__device__ __forceinline__ void block_mmas_t(uint32_t tmem, uint32_t a, uint32_t b, int BN, uint32_t idesc, bool first) {
  constexpr uint32_t AS = 2048u * KK;
#pragma unroll
  for (int kk = 0; kk < KK; ++kk) {
    const uint64_t bd = smem_desc_sw128(b + 2048u * kk, AS, 1024);
#pragma unroll
    for (int h = 0; h < MSX; ++h)
      mma_f16(tmem + (uint32_t)(h * BN), smem_desc_sw128(a + 2u * (uint32_t)h * AS + 2048u * kk, AS, 1024), bd, idesc,
              (!first || kk > 0) ? 1u : 0u);
  }
}

// The MMA issuer's loop over the slice's nblk pixel blocks, for blocks of KK
// 16-row steps and MSX sub-tiles: wait for a stage, issue its MMAs, free it
// when they complete.
template <int KK, int MSX>
__device__ __forceinline__ void mma_loop(int64_t nblk, int stages, int stage_bytes, uint32_t base, uint32_t tmem, int BN,
                                         uint32_t idesc, uint64_t* full, uint64_t* empty,
                                         volatile uint32_t* abort_flag, unsigned* err) {
  constexpr uint32_t MA = 2 * MSX, AS = 2048u * KK;
  int s = 0;
  uint32_t ph = 0;
  for (int64_t j = 0; j < nblk; ++j) {
    if (!mbar_wait(&full[s], ph, abort_flag, err)) break;
    tc_fence_after();
    const uint32_t a = base + (uint32_t)(s * stage_bytes);
    block_mmas_t<KK, MSX>(tmem, a, a + MA * AS, BN, idesc, j == 0);
    mma_commit(&empty[s]);
    if (++s == stages) {
      s = 0;
      ph ^= 1u;
    }
  }
}

template <int MSX>
__device__ __forceinline__ void mma_loop_ms(int kk, int64_t nblk, int stages, int stage_bytes, uint32_t base,
                                            uint32_t tmem, int BN, uint32_t idesc, uint64_t* full, uint64_t* empty,
                                            volatile uint32_t* abort_flag, unsigned* err) {
  switch (kk) {
    case 1: mma_loop<1, MSX>(nblk, stages, stage_bytes, base, tmem, BN, idesc, full, empty, abort_flag, err); break;
    case 2: mma_loop<2, MSX>(nblk, stages, stage_bytes, base, tmem, BN, idesc, full, empty, abort_flag, err); break;
    case 3: mma_loop<3, MSX>(nblk, stages, stage_bytes, base, tmem, BN, idesc, full, empty, abort_flag, err); break;
    case 4: mma_loop<4, MSX>(nblk, stages, stage_bytes, base, tmem, BN, idesc, full, empty, abort_flag, err); break;
    case 5: mma_loop<5, MSX>(nblk, stages, stage_bytes, base, tmem, BN, idesc, full, empty, abort_flag, err); break;
    case 6: mma_loop<6, MSX>(nblk, stages, stage_bytes, base, tmem, BN, idesc, full, empty, abort_flag, err); break;
    case 7: mma_loop<7, MSX>(nblk, stages, stage_bytes, base, tmem, BN, idesc, full, empty, abort_flag, err); break;
    default: mma_loop<8, MSX>(nblk, stages, stage_bytes, base, tmem, BN, idesc, full, empty, abort_flag, err); break;
  }
}

template <typename TI, typename TO>
__global__ void __launch_bounds__(kThreads, 1)
    wgrad_tc_kernel(const __grid_constant__ CUtensorMap tm_dy, const __grid_constant__ CUtensorMap tm_x,
                    const __grid_constant__ CUtensorMap tm_out, bool split, TO* db, float* ws_bias, WtParams wp,
                    unsigned* err) {
  const int AS = wp.BP * 128;          // one 64-channel atom of a pixel block
  const int MA = 2 * wp.MS;            // dY atoms (M)
  const int NA = wp.BN / 64;           // X atoms (N)
  const int stage_bytes = (MA + NA) * AS;
  const int stages = wp.stages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)stages * stage_bytes);
  uint64_t* empty = full + stages;
  uint64_t* tmem_full = empty + stages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tmem_full + 1);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  constexpr uint32_t FMT = std::is_same<TI, __nv_bfloat16>::value ? 1u : 0u;
  const uint32_t idesc = mma_idesc(FMT, 1u, 1u, (uint32_t)wp.BN, 128u);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int64_t tile = blockIdx.x % wp.tiles;
  const int32_t sigma = (int32_t)(blockIdx.x / wp.tiles);
  const int32_t taps = wp.R * wp.S;
  const int32_t tap = (int32_t)(tile % taps);
  const int64_t ct = (tile / taps) % wp.ctiles;
  const int64_t kt = (tile / taps / wp.ctiles) % wp.ktiles;
  const int64_t grp = tile / taps / wp.ctiles / wp.ktiles;
  const int32_t rr = tap / wp.S, ss = tap % wp.S;
  const int32_t k0 = (int32_t)(grp * wp.Kg + kt * 128 * wp.MS);  // first output channel (all groups)
  const int32_t c0 = (int32_t)(ct * wp.BN);                       // first input channel within the group
  const int32_t xc0 = (int32_t)(grp * wp.Cg) + c0;                // ... as a channel of X
  const int64_t b0 = slice_begin(wp.blocks, wp.split, sigma);
  const int64_t nblk = slice_begin(wp.blocks, wp.split, sigma + 1) - b0;
  // The bias gradient of the tile's output channels is shared out over the CTAs of the same
  // channel tile and slice (every input-channel tile and tap reads the same dY): CTA w of them sums
  // the 16-byte chunks [q0, q1) (8 channels each) of the dY atoms, each chunk in exactly one CTA.
  const int nchunk = 8 * 2 * wp.MS;
  const int64_t workers = wp.ctiles * taps, widx = ct * taps + tap;
  const int q0 = (int)(nchunk * widx / workers), q1 = (int)(nchunk * (widx + 1) / workers);
  const bool do_bias = (db != nullptr || ws_bias != nullptr) && q1 > q0;
  const int rows = wp.TR * wp.BW;  // rows TMA writes per atom; [rows, BP) stay zero
  const uint32_t tx = (uint32_t)((MA + NA) * rows * 128);

  // Zero the pad rows of every atom once (TMA never writes them).
  if (rows < wp.BP) {
    const int pad16 = (wp.BP - rows) * 8;  // 16-byte units per atom
    const int units = stages * (MA + NA) * pad16;
    for (int i = threadIdx.x; i < units; i += kThreads) {
      const int atom = i / pad16, u = i % pad16;
      reinterpret_cast<uint4*>(smem + (size_t)atom * AS + (size_t)rows * 128)[u] = make_uint4(0u, 0u, 0u, 0u);
    }
    fence_proxy_async_smem();
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < stages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1 + (do_bias ? 128 : 0));
    }
    mbar_init(tmem_full, 1);
    *abort_flag = 0u;
    mbar_fence_init();
    tma_prefetch(&tm_dy);
    tma_prefetch(&tm_x);
    tma_prefetch(&tm_out);
  }
  if (warp == 2) {
    tmem_alloc(tmem_slot, wp.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---------------------------------------------------- TMA producer
    // Every lane keeps the block position; lane 0 waits for a free stage and
    // arms its full barrier, then lane j issues box j (dY atoms first, then X):
    // one warp-wide instruction instead of MA + NA copies in turn from one
    // thread, each of which costs the issuing thread a few hundred cycles.
    {
      int s = 0;
      uint32_t ph = 0;
      const int64_t per_img = wp.hblocks * wp.wblocks;
      int64_t n = b0 / per_img;
      int64_t hb = (b0 % per_img) / wp.wblocks;
      int64_t wb = b0 % wp.wblocks;
      int64_t it = 0;
      for (; it < nblk; ++it) {
        bool ok = true;
        if (lane == 0) {
          if (it >= stages) ok = mbar_wait(&empty[s], ph ^ 1u, abort_flag, err);
          if (ok) mbar_arrive_expect_tx(&full[s], tx);
        }
        if (!__shfl_sync(0xffffffffu, ok, 0)) break;
        uint8_t* st = smem + (size_t)s * stage_bytes;
        const int32_t ho0 = (int32_t)(hb * wp.TR), wo0 = (int32_t)(wb * wp.BW);
        if (lane < MA)  // dY: the block's pixels x output channels k0 + 64 lane ..
          tma_load_4d(st + lane * AS, &tm_dy, k0 + 64 * lane, wo0, ho0, (int32_t)n, &full[s]);
        else if (lane < MA + NA)  // X through tap (rr, ss): the same pixels' inputs, channels xc0 + 64 (lane - MA) ..
          tma_load_4d(st + lane * AS, &tm_x, xc0 + 64 * (lane - MA), wo0 * wp.sw + ss * wp.dw - wp.pw,
                      ho0 * wp.sh + rr * wp.dh - wp.ph, (int32_t)n, &full[s]);
        __syncwarp();
        if (++wb == wp.wblocks) {
          wb = 0;
          if (++hb == wp.hblocks) {
            hb = 0;
            ++n;
          }
        }
        if (++s == stages) {
          s = 0;
          ph ^= 1u;
        }
      }
      // No copy may still be in flight when the CTA exits.
      if (lane == 0)
        for (int64_t q = it > stages ? it - stages : 0; q < it; ++q)
          mbar_wait(&full[q % stages], (uint32_t)(q / stages) & 1u, nullptr, err);
      __syncwarp();
    }
  } else if (warp == 1) {
    // ---------------------------------------------------- MMA issuer
    if (lane == 0) {
      // kk = BP / 16 (1..8: blocks of at most 128 rows, the atom stride AS = 2048 kk bytes)
      const uint32_t base = smem_u32(smem);
      if (wp.MS == 2)
        mma_loop_ms<2>(wp.BP / 16, nblk, stages, stage_bytes, base, tmem, wp.BN, idesc, full, empty, abort_flag, err);
      else
        mma_loop_ms<1>(wp.BP / 16, nblk, stages, stage_bytes, base, tmem, wp.BN, idesc, full, empty, abort_flag, err);
      if (nblk > 0) mma_commit(tmem_full);
      else mbar_arrive(tmem_full);
    }
  } else if (warp >= 4) {
    const int q = warp - 4;
    const int m = 32 * q + lane;  // row m of each M sub-tile (TMEM lane m)
    // ---------------------------------------------------- bias sums (this CTA's chunks)
    // Thread t sums chunk q0 + t % cc over the rows p = ph, ph + nph, ... of every block
    // (ph = t / cc, nph = 128 / cc phases); the phases are added in order at the end.
    const int t = threadIdx.x - 128;
    const int cc = q1 - q0 > 0 ? q1 - q0 : 1, nph = 128 / cc, ph0 = t / cc, qc = q0 + t % cc;
    float2 bacc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
    if (do_bias) {
      const int catom = qc / 8, cu = qc % 8;  // the chunk's dY atom and 16-byte unit
      int s = 0;
      uint32_t ph = 0;
      for (int64_t j = 0; j < nblk; ++j) {
        if (!mbar_wait(&full[s], ph, abort_flag, err)) break;
        if (ph0 < nph) {
          const uint8_t* at = smem + (size_t)s * stage_bytes + (size_t)catom * AS;
          for (int p = ph0; p < rows; p += nph) {
            const uint4 v = *reinterpret_cast<const uint4*>(at + p * 128 + ((cu ^ (p & 7)) << 4));
            bacc[0] = __fadd2_rn(bacc[0], widen2<TI>(v.x));
            bacc[1] = __fadd2_rn(bacc[1], widen2<TI>(v.y));
            bacc[2] = __fadd2_rn(bacc[2], widen2<TI>(v.z));
            bacc[3] = __fadd2_rn(bacc[3], widen2<TI>(v.w));
          }
        }
        mbar_arrive(&empty[s]);
        if (++s == stages) {
          s = 0;
          ph ^= 1u;
        }
      }
      // The epilogue below reuses the ring as staging: every bias warp must be done reading it
      // (the last MMA can complete before a slower warp has summed the last stages).
      named_bar_sync(1, 128);
    }
    // ---------------------------------------------------- epilogue
    const bool ok = mbar_wait(tmem_full, 0u, nullptr, err) && *abort_flag == 0u;
    signal_dependents();
    tc_fence_after();
    const uint32_t trow = tmem + ((uint32_t)(32 * q) << 16);
    uint8_t* stage = smem;  // the ring is idle: every copy landed, every MMA completed (kEpiBufs x 16 KB)
    const int32_t kend = (int32_t)(grp * wp.Kg + wp.Kg);  // this group's channels end here
#pragma unroll 1
    for (int h = 0; h < wp.MS; ++h) {
      const int32_t kr = k0 + 128 * h;
      if (kr >= kend) break;  // uniform over the 128 threads
      // the box {chunk, 1 tap, 128 output channels, 1} at (c, tap, k, slab), clipped at Cg and K
      auto store = [&](const void* buf, int32_t x) { tma_store_4d(&tm_out, buf, x, tap, kr, split ? sigma : 0); };
      if (split)
        store_rows_tma<float, kEpiBufs>(trow + (uint32_t)(h * wp.BN), stage, wp.BN, c0, wp.Cg, m, nblk > 0,
                                        threadIdx.x == 128, ok, store);
      else
        store_rows_tma<TO, kEpiBufs>(trow + (uint32_t)(h * wp.BN), stage, wp.BN, c0, wp.Cg, m, nblk > 0,
                                     threadIdx.x == 128, ok, store);
    }
    if (do_bias) {
      // The partial sums [phase][chunk][8] after the staging buffers (the ring is idle), then
      // channel j of this CTA's 8 cc channels adds its nph phases in order (deterministic).
      float* red = reinterpret_cast<float*>(smem + kEpiBufs * 128 * 128);
      if (ph0 < nph) {
        float* mine = red + (ph0 * cc + t % cc) * 8;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          mine[2 * i] = bacc[i].x;
          mine[2 * i + 1] = bacc[i].y;
        }
      }
      named_bar_sync(1, 128);
      for (int j = t; j < 8 * cc && ok; j += 128) {
        const int64_t k = (int64_t)k0 + 8 * q0 + j;
        if (k >= kend) continue;
        float sum = 0.f;
        for (int q2 = 0; q2 < nph; ++q2) sum += red[(q2 * cc + j / 8) * 8 + j % 8];
        if (ws_bias) ws_bias[(int64_t)sigma * wp.K + k] = sum;
        else store_out(db + k, sum);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, wp.tmem_cols);
  }
}

// ---------------------------------------------------------------- planning

// M sub-tiles: two (256 output channels sharing each X tile) when the group
// has more than 128 output channels (and, with several groups, a multiple of
// 256 of them, so no tile crosses a group); else one.
int ms_of(const Shape& s) {
  if (s.kg <= 128) return 1;
  return s.groups == 1 || s.kg % 256 == 0 ? 2 : 1;
}

// Input channels of a tile: the group's channels rounded up to 64, at most 256.
int bn_of(const Shape& s) {
  const int64_t c = (s.cg + 63) / 64 * 64;
  return (int)(c < 256 ? c : 256);
}

struct Blocking {
  int64_t tr = 0, bw = 0, bp = 0;
};

// The pixel block: TR x BW output positions with TR*BW <= rmax rows, chosen
// to waste the fewest padded rows over the image (rows are padded to 16 per
// block, and partial blocks at the image's edge are zero-filled), ties to the
// larger block. Its boxes must fit inside the tensors: BW <= Wo, TR <= Ho,
// BW*sw <= W, TR*sh <= H, and at most 256 elements per box dimension.
Blocking choose_blocking(const Shape& s, int64_t rmax) {
  Blocking best;
  int64_t best_cost = -1;
  for (int64_t bw = 1; bw <= s.wo && bw <= rmax; ++bw) {
    if (bw * s.sw > s.w || bw * s.sw > 256) break;
    int64_t tr = rmax / bw;
    if (tr > s.ho) tr = s.ho;
    while (tr > 1 && (tr * s.sh > s.h || tr * s.sh > 256)) --tr;
    if (tr < 1 || tr * s.sh > s.h) continue;
    const int64_t bp = (tr * bw + 15) / 16 * 16;
    const int64_t cost = ((s.ho + tr - 1) / tr) * ((s.wo + bw - 1) / bw) * bp;
    if (best_cost < 0 || cost < best_cost || (cost == best_cost && tr * bw > best.tr * best.bw)) {
      best_cost = cost;
      best.tr = tr;
      best.bw = bw;
      best.bp = bp;
    }
  }
  return best;
}

struct Config {
  int ms = 0, bn = 0, stages = 0;
  Blocking blk;
  size_t smem = 0;
};

Config config_of(const Shape& s) {
  Config cf;
  cf.ms = ms_of(s);
  cf.bn = bn_of(s);
  const int atoms = 2 * cf.ms + cf.bn / 64;
  int64_t rmax = kStageBudget / (atoms * 128) / 16 * 16;
  if (rmax > 128) rmax = 128;
  cf.blk = choose_blocking(s, rmax);
  if (cf.blk.bp == 0) return cf;
  const size_t stage = (size_t)atoms * cf.blk.bp * 128;
  const size_t fixed = 1024 + 256;
  int st = (int)((kSmemMax - fixed) / stage);
  if (st > kMaxStages) st = kMaxStages;
  cf.stages = st;
  cf.smem = fixed + (size_t)st * stage;
  // At least 120 KB, so one CTA runs per SM: its tensor-memory allocation
  // (up to all 512 columns) never waits for another CTA's.
  if (cf.smem < 120 * 1024) cf.smem = 120 * 1024;
  return cf;
}

bool admissible(const Shape& s) {
  if (s.in_dt == CONV_F32) return false;
  if (s.groups != 1 && (s.cg % 64 != 0 || s.kg % 128 != 0)) return false;
  if (s.c < 64 || s.k < 64 || s.cg < 64 || s.c % 8 != 0 || s.k % 8 != 0) return false;
  if (s.sh > 8 || s.sw > 8) return false;  // TMA traversal strides take 1..8
  if (s.n < 1 || s.n > 0x7fffffffLL || s.h > 0x7fffffffLL || s.w > 0x7fffffffLL || s.c > 0x7fffffffLL ||
      s.k > 0x7fffffffLL)
    return false;
  if (s.r * s.s > 0x7fffffffLL) return false;
  const Config cf = config_of(s);
  if (cf.blk.bp == 0 || cf.stages < 2) return false;
  // the box of the epilogue: 128 bytes of channels (32 fp32 or 64 16-bit values) within Cg
  if (s.cg < (s.out_dt == CONV_F32 ? 32 : 64)) return false;
  return true;
}

template <typename TI, typename TO>
cudaError_t launch_typed(const Plan& p, const Args& a, CUtensorMapDataType dt) {
  const Shape& s = p.sh;
  const Config cf = config_of(s);
  WtParams wp;
  wp.K = s.k;
  wp.Ho = s.ho;
  wp.Wo = s.wo;
  wp.Cg = (int32_t)s.cg;
  wp.Kg = (int32_t)s.kg;
  wp.R = (int32_t)s.r;
  wp.S = (int32_t)s.s;
  wp.ph = (int32_t)s.ph;
  wp.pw = (int32_t)s.pw;
  wp.sh = (int32_t)s.sh;
  wp.sw = (int32_t)s.sw;
  wp.dh = (int32_t)s.dh;
  wp.dw = (int32_t)s.dw;
  wp.TR = (int32_t)cf.blk.tr;
  wp.BW = (int32_t)cf.blk.bw;
  wp.BP = (int32_t)cf.blk.bp;
  wp.hblocks = (s.ho + cf.blk.tr - 1) / cf.blk.tr;
  wp.wblocks = (s.wo + cf.blk.bw - 1) / cf.blk.bw;
  wp.blocks = s.n * wp.hblocks * wp.wblocks;
  wp.MS = cf.ms;
  wp.BN = cf.bn;
  wp.ktiles = (s.kg + 128 * cf.ms - 1) / (128 * cf.ms);
  wp.ctiles = (s.cg + cf.bn - 1) / cf.bn;
  wp.tiles = s.groups * wp.ktiles * wp.ctiles * s.r * s.s;
  wp.split = p.split;
  wp.stages = cf.stages;
  uint32_t cols = 32;
  while (cols < (uint32_t)(cf.ms * cf.bn)) cols *= 2;
  wp.tmem_cols = cols;
  CUtensorMap tm_dy, tm_x, tm_out;
  const uint64_t y_dims[4] = {(uint64_t)s.k, (uint64_t)s.wo, (uint64_t)s.ho, (uint64_t)s.n};
  const uint64_t y_strides[3] = {(uint64_t)s.k * 2u, (uint64_t)(s.wo * s.k) * 2u, (uint64_t)(s.ho * s.wo * s.k) * 2u};
  const uint32_t y_box[4] = {64u, (uint32_t)cf.blk.bw, (uint32_t)cf.blk.tr, 1u};
  const uint64_t x_dims[4] = {(uint64_t)s.c, (uint64_t)s.w, (uint64_t)s.h, (uint64_t)s.n};
  const uint64_t x_strides[3] = {(uint64_t)s.c * 2u, (uint64_t)(s.w * s.c) * 2u, (uint64_t)(s.h * s.w * s.c) * 2u};
  const uint32_t x_box[4] = {64u, (uint32_t)(cf.blk.bw * s.sw), (uint32_t)(cf.blk.tr * s.sh), 1u};
  const uint32_t x_estr[4] = {1u, (uint32_t)s.sw, (uint32_t)s.sh, 1u};
  if (!encode_tmap(&tm_dy, dt, 4, a.b, y_dims, y_strides, y_box, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tmap(&tm_x, dt, 4, a.x, x_dims, x_strides, x_box, CU_TENSOR_MAP_SWIZZLE_128B, x_estr))
    return cudaErrorInvalidValue;
  // dW (or the fp32 slabs) as [S][K][R*S][Cg]: boxes of 128 bytes of channels x 1 tap x up to 128
  // output channels, clipped at Cg and at K.
  const bool split = a.ws != nullptr;
  const uint64_t es = split ? 4u : (uint64_t)sizeof(TO);
  const CUtensorMapDataType odt = split || sizeof(TO) == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : dt;
  const uint64_t o_dims[4] = {(uint64_t)s.cg, (uint64_t)(s.r * s.s), (uint64_t)s.k, split ? (uint64_t)p.split : 1u};
  const uint64_t o_strides[3] = {(uint64_t)s.cg * es, (uint64_t)(s.r * s.s * s.cg) * es,
                                 (uint64_t)(s.k * s.r * s.s * s.cg) * es};
  const uint32_t o_box[4] = {(uint32_t)(128 / es), 1u, (uint32_t)(s.k < 128 ? s.k : 128), 1u};
  if (!encode_tmap(&tm_out, odt, 4, split ? (const void*)a.ws : a.out, o_dims, o_strides, o_box,
                   CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  auto kern = wgrad_tc_kernel<TI, TO>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)cf.smem);
  if (err != cudaSuccess) return err;
  const int64_t ctas = wp.tiles * p.split;
  if (ctas > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  kern<<<(unsigned)ctas, kThreads, cf.smem, a.stream>>>(tm_dy, tm_x, tm_out, split,
                                                        p.with_bias ? static_cast<TO*>(a.db) : nullptr,
                                                        p.with_bias ? a.ws_bias : nullptr, wp, device_error_word());
  return cudaGetLastError();
}

}  // namespace

Geometry geometry_wgrad_tc(const Shape& s) {
  Geometry g;
  if (!admissible(s)) return g;
  const Config cf = config_of(s);
  g.ok = true;
  g.ctas_per_sm = 1;
  g.tiles = s.groups * ((s.kg + 128 * cf.ms - 1) / (128 * cf.ms)) * ((s.cg + cf.bn - 1) / cf.bn) * s.r * s.s;
  g.blocks = s.n * ((s.ho + cf.blk.tr - 1) / cf.blk.tr) * ((s.wo + cf.blk.bw - 1) / cf.blk.bw);
  return g;
}

cudaError_t launch_wgrad_tc(const Plan& p, const Args& a) {
  if (p.sh.in_dt == CONV_BF16) {
    if (p.sh.out_dt == CONV_F32) return launch_typed<__nv_bfloat16, float>(p, a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16);
    return launch_typed<__nv_bfloat16, __nv_bfloat16>(p, a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16);
  }
  if (p.sh.out_dt == CONV_F32) return launch_typed<__half, float>(p, a, CU_TENSOR_MAP_DATA_TYPE_FLOAT16);
  return launch_typed<__half, __half>(p, a, CU_TENSOR_MAP_DATA_TYPE_FLOAT16);
}

}  // namespace cig
