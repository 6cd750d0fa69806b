// 16-bit forward convolution on the tcgen05 tensor cores, im2col gathered on
// the fly by TMA, deterministic split-K over the reduction (r, s, c).
//
// GEMM view: M = output pixels, N = output channels k, reduction (r, s, c)
// with c innermost:
//   A[m][(r,s,c)] = X[n, ho + r*dh - ph, wo + s*dw - pw, c],  B[k][(r,s,c)] = W[k,r,s,c].
// Both are K-major in NHWC / channels-last memory, as the bf16/fp16 MMA wants.
// An M tile is TR whole output rows (TR*Wo <= 128 pixels). For a reduction
// block (r, s, 64 channels) its A tile is ONE 4-D TMA box {64 ch, Wo*sw,
// TR*sh, 1} of X starting at (c0, s*dw - pw, ho0*sh + r*dh - ph, n), read
// with traversal strides (1, sw, sh, 1) so it holds exactly the Wo x TR
// input positions the tile's outputs read through tap (r, s): coordinates
// outside the image read zeros, which is exactly the zero padding, and the
// box lands as TR*Wo rows of 128 bytes in the 128B-swizzled K-major layout
// the MMA reads. B is a box {64, BN} of W viewed as [K][R*S*C].
//
// Work units are (tile, slice) pairs. The 256-wide two-stage form runs
// persistent: at most one CTA per SM, each taking units in turn with its ring
// streaming on across them (see Tile).
//
// Split-K ("feat(rocke): split-K forward implicit-GEMM convolution on
// gfx1250", "Two-stage split-K"): unit (tile, sigma) reduces the blocks of
// slice sigma and stores its fp32 partial tile into slab sigma of the
// workspace, every element written once; the fold kernel sums the slabs in
// slice order and rounds into Y. With one slice the epilogue rounds straight
// into Y. No fused epilogue is applied under split-K ("Review follow-ups":
// a bias or activation cannot be applied per slice).
//
// Single-launch form (same page, "Changes": single-launch split-K; its
// testing notes: each slice folds 1/S of the tile's rows): the S slices of a
// tile are one thread-block cluster (S <= 16). Each CTA stages its fp32
// partial tile in its own shared memory; after a cluster barrier, CTA sigma
// sums rows [128 sigma / S, 128 (sigma + 1) / S) of all S partial tiles over
// distributed shared memory, in slice order 0..S-1 (the fold's order, so Y is
// bit-identical to the two-stage form at the same S), and rounds into Y. No
// workspace and no fold launch. A second cluster barrier keeps every CTA (and
// its shared memory) alive until its peers have read it.
//
// Warp roles: 0 TMA producer, 1 MMA issuer, 2 TMEM owner, 4-7 epilogue (and
// 8-11, a second epilogue group, in the persistent form).
#include "tc_store.cuh"
#include "../kernel_entry.h"

namespace cig {
namespace {

constexpr int kThreads = 256;
// The persistent form has two epilogue groups of four warps (warps 4-7 and
// 8-11), which share each unit's column chunks.
constexpr int kThreadsPersist = 384;
constexpr int kBM = 128;
constexpr int kBK = 64;                     // channels per reduction block (128 bytes of 16-bit)
constexpr int kA = kBM * 128;               // A tile bytes (128 rows x 128 B)

// Tile of BN output channels (128, or 256 when K >= 256: an SM then loads
// 48 KB per 2 M multiply-adds instead of 32 KB per 1 M, and its L2 -> shared
// bandwidth, not the tensor pipe, is what bounds a block) and MS M sub-tiles
// of TR output rows each: with MS = 2 two A tiles share the B tile (64 KB per
// 4 M multiply-adds), which is taken when the grid has tiles to spare. Ring:
// 3 stages for BN = 128 (2 CTAs per SM), 4 for BN = 256 (1 CTA per SM), 3 for
// BN = 256 with MS = 2 (64 KB stages). (A deeper ring for
// the cluster form would hold one CTA per SM, and then only 7 clusters of 16
// fit on the GPU at once, fewer than the 8 tiles of the 3x3 small-M layer.)
template <int BN, int MS>
struct Tile {
  static constexpr int kB = BN * 128;              // B tile bytes (BN rows x 128 B)
  static constexpr int kStage = MS * kA + kB;      // MS A tiles (M sub-tiles) share one B tile
  static constexpr int kStages = (BN == 256 && MS == 1) ? 4 : 3;
  static constexpr uint32_t kTmemCols = BN * MS;   // one fp32 accumulator per M sub-tile
  // 256-wide tiles (one CTA per SM) run persistent: a CTA takes unit after
  // unit, its ring streaming on across them, the epilogue staging in its own
  // two 16 KB buffers (+ the bias); with two accumulators in TMEM (when they
  // fit) a unit's epilogue overlaps the next unit's MMAs.
  static constexpr bool kPersist = BN == 256;
  static constexpr int kOwnEpiBufs = 2;
  static constexpr int kOwnEpi = kPersist ? kOwnEpiBufs * kBM * 128 + BN * 4 : 0;
  static constexpr int kAccs = kPersist && 2 * kTmemCols <= 512 ? 2 : 1;
  static constexpr size_t kSmem = 1024 + (size_t)kStages * kStage + kOwnEpi + 256;
  static_assert(kSmem <= 227 * 1024, "shared memory");
  static constexpr int kLD = BN + 4;                // staged partial tile row stride, floats (conflict-free float4s)
  static_assert(BN == 128 || BN == 256, "tile width");
  static_assert(MS == 1 || MS == 2, "M sub-tiles");
  static_assert(kTmemCols <= 512, "TMEM columns");
  static_assert(kBM * kLD * 4 <= kStages * kStage, "staged partial tile must fit in the ring");
  // epilogue staging buffers (16 KB each, up to 8) and the bias, over the idle ring
  static constexpr int kEpiBufs =
      (kStages * kStage - BN * 4) / (kBM * 128) < 8 ? (kStages * kStage - BN * 4) / (kBM * 128) : 8;
  static_assert(kEpiBufs >= 2, "epilogue staging and bias must fit in the ring");
};

struct FwdParams {
  int64_t N, K, Ho, Wo, Cg, S_f;   // S_f: filter width
  int64_t E;                    // output elements N*Ho*Wo*K (one slab)
  int64_t cblocks;              // Cg / 64
  int64_t tiles_m_per_img;      // ceil(Ho / TR)
  int64_t tiles_n;              // ceil(K / 128)
  int64_t tiles;                // N * tiles_m_per_img * tiles_n
  int64_t blocks;               // R * S * cblocks
  int32_t TR;                   // output rows per M tile
  int32_t ph, pw, dh, dw;
  int32_t sh;                   // stride along H (along W it is the X map's traversal stride)
  int32_t a_coff;               // 1: the X channel coordinate starts at the tile's first output channel
                                // (block-diagonal grouped problems), 0: at 0
  int32_t taps;                 // R * S (read by the MN-major B form: tap rs of the problem is tap
                                // taps - 1 - rs of the filter it reads)
  int32_t split;
  // fused epilogue (unsplit only): y = min(max(acc + bias[k], ep_lo), ep_hi)
  const void* ep_bias;
  float ep_lo, ep_hi;
  int32_t ep;
};

// True when the phase with this parity has completed (never suspends).
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

template <typename TO>
__device__ __forceinline__ void store4(TO* dst, float4 v);
template <>
__device__ __forceinline__ void store4<float>(float* dst, float4 v) {
  *reinterpret_cast<float4*>(dst) = v;
}
template <>
__device__ __forceinline__ void store4<__nv_bfloat16>(__nv_bfloat16* dst, float4 v) {
  __nv_bfloat162 h[2] = {__floats2bfloat162_rn(v.x, v.y), __floats2bfloat162_rn(v.z, v.w)};
  *reinterpret_cast<uint2*>(dst) = *reinterpret_cast<uint2*>(h);
}
template <>
__device__ __forceinline__ void store4<__half>(__half* dst, float4 v) {
  __half2 h[2] = {__floats2half2_rn(v.x, v.y), __floats2half2_rn(v.z, v.w)};
  *reinterpret_cast<uint2*>(dst) = *reinterpret_cast<uint2*>(h);
}

// BMN: B is read MN-major from a filter laid out [C'][R][S][K'] (the
// reduction channel outermost, output channels contiguous) with the taps
// reversed: the data gradient's own filter, which as a forward problem is
// W'[c][r'][s'][k] = W[k][R-1-r'][S-1-s'][c]. Each stage then holds BN / 64
// atoms of 64 output channels x 64 reduction rows (128B-swizzled, 8 KB apart).
template <typename TO, uint32_t FMT, bool CL, int BN, int MS, bool BMN = false>
__global__ void __launch_bounds__(BN == 256 ? kThreadsPersist : kThreads, BN == 256 ? 1 : 2)
    fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                  const __grid_constant__ CUtensorMap tm_y, TO* out, float* ws, FwdParams fp, unsigned* err) {
  using T = Tile<BN, MS>;
  constexpr int kStages = T::kStages, kStage = T::kStage, kB = T::kB, kLD = T::kLD;
  constexpr uint32_t kTmemCols = T::kTmemCols;
  constexpr bool kPersist = T::kPersist && !CL;
  constexpr int NACC = T::kAccs;  // TMEM accumulators (2: a unit's epilogue overlaps the next unit's MMAs)
  // One accumulator of two M sub-tiles: the epilogue frees each sub-tile on its
  // own (tmem_empty[h]), so the next unit's sub-tile 0 MMAs start while
  // sub-tile 1 is still being read; its sub-tile 1 MMAs follow, for up to
  // kStages held blocks.
  constexpr bool kSplitRelease = kPersist && NACC == 1 && MS == 2;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)kStages * kStage + T::kOwnEpi);
  uint64_t* empty = full + kStages;
  uint64_t* tmem_full = empty + kStages;
  uint64_t* tmem_empty = tmem_full + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tmem_empty + 2);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  constexpr uint32_t IDESC = mma_idesc(FMT, 0u, BMN ? 1u : 0u, (uint32_t)BN, (uint32_t)kBM);
  constexpr uint32_t kAtom = 64u * 128u;  // one MN-major B atom: 64 reduction rows of 128 bytes

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  // Work units (tile, slice sigma). Two-stage form: unit = sigma * tiles +
  // tile; a persistent CTA takes units blockIdx.x, blockIdx.x + gridDim.x,
  // ... (else the grid has one CTA per unit). Cluster form: one unit a CTA,
  // the S CTAs of a tile consecutive, sigma = rank in the cluster.
  const int64_t units = CL ? (int64_t)gridDim.x : fp.tiles * fp.split;
  const int64_t ustride = (int64_t)gridDim.x;
  struct Unit {
    int64_t img, ho0, k0, b0, nblk;
    int32_t sigma;
  };
  // (units, tiles and their factors fit 32 bits: the host launches at most
  // 2^31 - 1 units; 32-bit divisions keep this off the loads' critical path)
  auto unit_of = [&](int64_t u) {
    Unit w;
    const uint32_t u32 = (uint32_t)u, nt = (uint32_t)fp.tiles, ntn = (uint32_t)fp.tiles_n;
    const uint32_t tile = CL ? u32 / (uint32_t)fp.split : u32 % nt;
    w.sigma = CL ? (int32_t)cluster_ctarank() : (int32_t)(u32 / nt);
    const uint32_t tn = tile % ntn, tm = tile / ntn, tmi = (uint32_t)fp.tiles_m_per_img;
    w.img = tm / tmi;
    w.ho0 = (int64_t)(tm % tmi) * fp.TR * MS;  // sub-tile h starts at row ho0 + h * TR
    w.k0 = (int64_t)tn * BN;
    w.b0 = slice_begin(fp.blocks, fp.split, w.sigma);
    w.nblk = slice_begin(fp.blocks, fp.split, w.sigma + 1) - w.b0;
    return w;
  };
  const int64_t u_first = blockIdx.x;
  const uint32_t tx = (uint32_t)(MS * fp.TR * fp.Wo * 128 + kB);

  // Producer state (every lane of warp 0, kept in step): the ring stage and
  // its round's parity, the unit and block being loaded, and that block's
  // (r, s, c-block), all advanced by increments.
  int ps = 0;
  uint32_t pph = 0;
  const int32_t cblocks = (int32_t)fp.cblocks, cg = (int32_t)fp.Cg, sf = (int32_t)fp.S_f;
  int64_t pu = u_first, pj = 0, it = 0;
  Unit pw = unit_of(pu);
  int32_t cb, rs, r, sx;
  auto unit_start = [&]() {
    pj = 0;
    cb = (int32_t)((uint32_t)pw.b0 % (uint32_t)cblocks);
    rs = (int32_t)((uint32_t)pw.b0 / (uint32_t)cblocks);
    r = rs / sf;
    sx = rs % sf;
  };
  unit_start();
  // true while a block is left to load (moving on past finished units)
  auto pending = [&]() {
    while (pj >= pw.nblk) {
      pu += ustride;
      if (pu >= units) return false;
      pw = unit_of(pu);
      unit_start();
    }
    return true;
  };
  // A block's loads go out as ONE warp-wide 4-D TMA instruction, lane i
  // issuing box i: lanes 0..MS-1 the A sub-tiles, the next lanes the B
  // box(es), rather than one thread issuing them in turn.
  constexpr int kLoads = MS + (BMN ? BN / 64 : 1);
  auto issue = [&]() {
    uint8_t* st = smem + (size_t)ps * kStage;
    if (lane < kLoads) {
      const bool is_a = lane < MS;
      const int j = lane - MS;  // B piece
      const int32_t a_c0 = (fp.a_coff ? (int32_t)pw.k0 : 0) + cb * kBK;
      const int32_t a_c2 = (int32_t)(pw.ho0 + lane * fp.TR) * fp.sh + r * fp.dh - fp.ph;
      const CUtensorMap* map = is_a ? &tm_x : &tm_w;
      uint8_t* dst = is_a ? st + lane * kA : st + MS * kA + (BMN ? j * (int)kAtom : 0);
      int32_t c0, c1, c2;
      if (BMN) {
        c0 = is_a ? a_c0 : (int32_t)pw.k0 + 64 * j;
        c1 = is_a ? sx * fp.dw - fp.pw : fp.taps - 1 - rs;
        c2 = is_a ? a_c2 : cb * kBK;
      } else {
        c0 = is_a ? a_c0 : rs * cg + cb * kBK;
        c1 = is_a ? sx * fp.dw - fp.pw : (int32_t)pw.k0;
        c2 = is_a ? a_c2 : 0;
      }
      // a sub-tile past the image reads zeros (and is not stored)
      tma_load_4d(dst, map, c0, c1, c2, is_a ? (int32_t)pw.img : 0, &full[ps]);
    }
    ++pj;
    ++it;
    if (++cb == cblocks) {
      cb = 0;
      ++rs;
      if (++sx == sf) {
        sx = 0;
        ++r;
      }
    }
    if (++ps == kStages) {
      ps = 0;
      pph ^= 1u;
    }
  };

  // A full barrier's one arrival (with the stage's byte count) is made ahead
  // of its loads: here for the first round, then by the MMA thread as soon
  // as it has seen the previous round's bytes land. The producer only waits
  // for a free stage and issues its copies (an expect-tx just before the
  // copies on the same barrier cost the issuing thread several hundred
  // cycles a block).
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tmem_full[i], 1);
      mbar_init(&tmem_empty[i], kPersist ? 2 : 1);  // one arrival per epilogue group
    }
    *abort_flag = 0u;
    mbar_fence_init();
    for (int i = 0; i < kStages; ++i) mbar_arrive_expect_tx(&full[i], tx);
    tma_prefetch(&tm_x);
    tma_prefetch(&tm_w);
  }
  if (warp == 0) {
    __syncwarp();  // the barriers are initialised
    // The first ring of loads goes out before the CTA-wide sync (which waits
    // for the TMEM allocation), so its latency overlaps the set-up.
    while (it < kStages && pending()) issue();
  }
  if (warp == 2) {
    tmem_alloc(tmem_slot, kTmemCols * NACC);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    while (pending()) {
      bool ok = true;
      if (lane == 0) ok = mbar_wait(&empty[ps], pph ^ 1u, abort_flag, err);
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      issue();
    }
    if (lane == 0)
      for (int64_t q = it > kStages ? it - kStages : 0; q < it; ++q)
        mbar_wait(&full[q % kStages], (uint32_t)(q / kStages) & 1u, nullptr, err);
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t base = smem_u32(smem);
      int s = 0;
      uint32_t ph = 0;
      bool live = true;  // false once a wait gave up: the units left only signal their (empty) accumulators
      int64_t i = 0;
      // The MMAs of one block (ring stage st, the unit's block jb) into sub-tile h.
      auto block_mmas = [&](int st, int64_t jb, int h, uint32_t dacc) {
        const uint32_t a = base + (uint32_t)(st * kStage), b = a + MS * kA;
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk) {
          // K-major SW128: 8-row groups 1024 B apart; a K step of 16 elements is
          // a 32-byte advance inside the swizzled 128-byte row. MN-major SW128
          // (BMN): atoms kAtom apart, 8-row groups 1024 B apart; a K step of 16
          // rows is 2048 B.
          const uint64_t bd =
              BMN ? smem_desc_sw128(b + 2048u * kk, kAtom, 1024) : smem_desc_sw128(b + 32u * kk, 16, 1024);
          mma_f16(dacc + (uint32_t)(h * BN), smem_desc_sw128(a + (uint32_t)(h * kA) + 32u * kk, 16, 1024), bd,
                  IDESC, (jb > 0 || kk > 0) ? 1u : 0u);
        }
      };
      for (int64_t u = u_first; u < units; u += ustride, ++i) {
        const int64_t nblk = unit_of(u).nblk;
        const int buf = (int)(i % NACC);
        const uint32_t use = (uint32_t)(i / NACC);
        // the epilogue has drained this accumulator's previous unit (with one
        // accumulator of two sub-tiles: its first sub-tile; the second is
        // waited for below, while the first one's MMAs run)
        if (live && use > 0 && !mbar_wait(&tmem_empty[buf], (use - 1u) & 1u, abort_flag, err)) live = false;
        tc_fence_after();
        const uint32_t dacc = tmem + (uint32_t)buf * kTmemCols;
        bool any = false;
        bool h1 = !kSplitRelease || use == 0;  // sub-tile 1 of the accumulator is free
        int pend = 0;  // blocks before this one whose sub-tile 1 MMAs wait for it (their stages stay held)
        for (int64_t j = 0; live && j < nblk; ++j) {
          if (!mbar_wait(&full[s], ph, abort_flag, err)) {
            live = false;
            break;
          }
          mbar_arrive_expect_tx(&full[s], tx);  // arms the stage's next round
          tc_fence_after();
          if (!kSplitRelease) {
#pragma unroll
            for (int h = 0; h < MS; ++h) block_mmas(s, j, h, dacc);
            mma_commit(&empty[s]);
          } else {
            block_mmas(s, j, 0, dacc);
            if (!h1) h1 = mbar_test(&tmem_empty[1], (use - 1u) & 1u);
            if (!h1 && pend + 1 == kStages) {  // every stage is held: sub-tile 1 must be free now
              if (!mbar_wait(&tmem_empty[1], (use - 1u) & 1u, abort_flag, err)) {
                live = false;
                break;
              }
              h1 = true;
            }
            if (h1) {
              tc_fence_after();
              for (int t = pend; t > 0; --t) {  // the held blocks first, in order
                const int st = (s - t + kStages) % kStages;
                block_mmas(st, j - t, 1, dacc);
                mma_commit(&empty[st]);
              }
              block_mmas(s, j, 1, dacc);
              mma_commit(&empty[s]);
              pend = 0;
            } else {
              ++pend;
            }
          }
          any = true;
          if (++s == kStages) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (kSplitRelease && live && pend > 0) {  // a unit of fewer blocks than stages
          if (!mbar_wait(&tmem_empty[1], (use - 1u) & 1u, abort_flag, err)) {
            live = false;
          } else {
            tc_fence_after();
            for (int t = pend; t > 0; --t) {
              const int st = (s - t + kStages) % kStages;
              block_mmas(st, nblk - t, 1, dacc);
              mma_commit(&empty[st]);
            }
          }
        }
        if (any) mma_commit(&tmem_full[buf]);
        else mbar_arrive(&tmem_full[buf]);
      }
    }
  } else if (warp >= 4) {
    constexpr int NG = kPersist ? 2 : 1;  // epilogue groups of four warps
    const int g = NG == 2 ? (warp - 4) / 4 : 0;
    const int q = warp % 4;       // TMEM lane quarter of the warp
    const int m = 32 * q + lane;  // tile row = output pixel within the tile
    int64_t i = 0;
    for (int64_t u = u_first; u < units; u += ustride, ++i) {
      const Unit w = unit_of(u);
      const int buf = (int)(i % NACC);
      const uint32_t use = (uint32_t)(i / NACC);
      const bool ok = mbar_wait(&tmem_full[buf], use & 1u, nullptr, err) && *abort_flag == 0u;
      if (!CL && u + ustride >= units) signal_dependents();
      tc_fence_after();
      const uint32_t trow = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)buf * kTmemCols;
      if (CL) {
        // Stage this slice's partial tile: row m at part + m * kLD (the ring is
        // idle: every copy landed and every MMA that read it has completed).
        float* part = reinterpret_cast<float*>(smem) + m * kLD;
#pragma unroll 1
        for (int j = 0; j < BN / 32; ++j) {
          float v[32];
          if (w.nblk > 0) {
            tmem_ld32(trow + 32u * j, v);
          } else {
#pragma unroll
            for (int c = 0; c < 32; ++c) v[c] = 0.f;
          }
#pragma unroll
          for (int c = 0; c < 32; c += 4)
            *reinterpret_cast<float4*>(part + 32 * j + c) = make_float4(v[c], v[c + 1], v[c + 2], v[c + 3]);
        }
      } else {
        // Y (or slab sigma of the workspace, fp32) as [N (x S)][Ho*Wo][K], one
        // M sub-tile (accumulator columns h * BN ..) after the other. Staging:
        // the CTA's last unit (or only one) uses the idle ring, up to 8 16 KB
        // buffers (every copy landed, every MMA completed); earlier units of a
        // persistent CTA use its own two, as the ring keeps loading. The
        // epilogue's bias for the unit's BN channels, fp32 in shared memory
        // past the staging buffers (0 beyond K or without a bias).
        // With two groups, group g takes the chunks g, g + 2, ... through its
        // half of the buffers.
        const bool in_ring = !kPersist || u + ustride >= units;
        const int nbufs = in_ring ? T::kEpiBufs : T::kOwnEpiBufs;
        uint8_t* stage0 = in_ring ? smem : smem + (size_t)kStages * kStage;
        uint8_t* stage = stage0 + (size_t)g * (nbufs / NG) * kBM * 128;
        float* sbias = reinterpret_cast<float*>(stage0 + (size_t)nbufs * kBM * 128);
        if (!ws && fp.ep) {
          const TO* bias = static_cast<const TO*>(fp.ep_bias);
          named_bar_sync(NG == 2 ? 3 : 1, 128 * NG);  // every group is done with the previous unit's bias
          for (int c = threadIdx.x - 128; c < BN; c += 128 * NG)
            sbias[c] = bias && w.k0 + c < fp.K ? to_f32(bias[w.k0 + c]) : 0.f;
          named_bar_sync(NG == 2 ? 3 : 1, 128 * NG);
        }
        // Sub-tiles inside the image (a sub-tile past it is not stored); each
        // group releases the accumulator after its last read of the last one
        // (of each one, with kSplitRelease; a sub-tile past the image at once),
        // and waits for global completion of its stores only at the CTA's
        // last unit.
        const int nsub = (int)((fp.Ho - w.ho0 + fp.TR - 1) / fp.TR) < MS ? (int)((fp.Ho - w.ho0 + fp.TR - 1) / fp.TR)
                                                                           : MS;
        const bool last_unit = !kPersist || u + ustride >= units;
#pragma unroll 1
        for (int h = 0; h < nsub; ++h) {
          const int64_t hrow = w.ho0 + h * fp.TR;
          uint64_t* rel = kSplitRelease ? &tmem_empty[h] : kPersist && h == nsub - 1 ? &tmem_empty[buf] : nullptr;
          const int32_t py = (int32_t)(hrow * fp.Wo);
          // the box {chunk, TR*Wo pixels, 1} at (channel, first pixel, image), clipped at K and Ho*Wo
          const int32_t pz = ws ? (int32_t)(w.sigma * fp.N + w.img) : (int32_t)w.img;
          auto store = [&](const void* sb, int32_t x) { tma_store_3d(&tm_y, sb, x, py, pz); };
          const uint32_t acc = trow + (uint32_t)(h * BN);
          const bool lead = threadIdx.x == 128 + 128 * g;
          const bool epi = !ws && fp.ep != 0;
          if (ws) {
            if (in_ring)
              store_rows_tma<float, T::kEpiBufs / NG>(acc, stage, BN, (int32_t)w.k0, (int32_t)fp.K, m, w.nblk > 0,
                                                      lead, ok, store, nullptr, 0.f, 0.f, false, g, NG, 1 + g, rel,
                                                      last_unit);
            else
              store_rows_tma<float, T::kOwnEpiBufs / NG>(acc, stage, BN, (int32_t)w.k0, (int32_t)fp.K, m,
                                                         w.nblk > 0, lead, ok, store, nullptr, 0.f, 0.f, false, g,
                                                         NG, 1 + g, rel, last_unit);
          } else {
            if (in_ring)
              store_rows_tma<TO, T::kEpiBufs / NG>(acc, stage, BN, (int32_t)w.k0, (int32_t)fp.K, m, w.nblk > 0,
                                                   lead, ok, store, sbias, fp.ep_lo, fp.ep_hi, epi, g, NG, 1 + g, rel,
                                                   last_unit);
            else
              store_rows_tma<TO, T::kOwnEpiBufs / NG>(acc, stage, BN, (int32_t)w.k0, (int32_t)fp.K, m, w.nblk > 0,
                                                      lead, ok, store, sbias, fp.ep_lo, fp.ep_hi, epi, g, NG, 1 + g,
                                                      rel, last_unit);
          }
        }
        if (kSplitRelease && nsub < 2 && threadIdx.x == 128 + 128 * g) mbar_arrive(&tmem_empty[1]);
      }
      if (!kPersist) {  // every TMEM read of the unit is done: the accumulator is free again
        tc_fence_before();
        named_bar_sync(1, 128);
        if (threadIdx.x == 128) mbar_arrive(&tmem_empty[buf]);
      }
    }
  }

  tc_fence_before();
  if (CL) {
    const Unit w0 = unit_of(u_first);  // the cluster form's single unit
    const int32_t sigma = w0.sigma;
    const int64_t ho0 = w0.ho0, img = w0.img, k0 = w0.k0;
    cluster_sync();  // every slice's partial tile is staged
    const int S = fp.split;
    const int r0 = (sigma * kBM) / S, r1 = ((sigma + 1) * kBM) / S;
    const int64_t rows_here = fp.Ho - ho0 < fp.TR ? fp.Ho - ho0 : fp.TR;
    const int valid = (int)(rows_here * fp.Wo);  // rows m < valid are output pixels
    const bool ok = *abort_flag == 0u;
    const uint32_t base = smem_u32(smem);
#pragma unroll 1
    for (int w = threadIdx.x; w < (r1 - r0) * (BN / 4); w += kThreads) {
      const int m = r0 + w / (BN / 4), c4 = w % (BN / 4);
      const int64_t k = k0 + 4 * c4;
      if (!ok || m >= valid || k >= fp.K) continue;  // K % 8 == 0: 4-wide groups are all in or all out
      const uint32_t la = base + (uint32_t)((m * kLD + 4 * c4) * 4);
      float4 part[kMaxClusterSplit];
#pragma unroll
      for (int j = 0; j < kMaxClusterSplit; ++j)
        if (j < S) part[j] = ld_cluster_f4(cluster_map(la, (uint32_t)j));
      float4 acc = part[0];
#pragma unroll
      for (int j = 1; j < kMaxClusterSplit; ++j)
        if (j < S) {
          acc.x += part[j].x;
          acc.y += part[j].y;
          acc.z += part[j].z;
          acc.w += part[j].w;
        }
      const int64_t pix = (img * fp.Ho + ho0 + m / fp.Wo) * fp.Wo + m % fp.Wo;
      store4<TO>(out + pix * fp.K + k, acc);
    }
    cluster_sync();  // peers are done reading this CTA's shared memory
  }
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols * NACC);
  }
}

bool fwd_tc_admissible(const Shape& s) {
  if (s.in_dt == CONV_F32 || s.groups != 1) return false;
  if (s.sh > 8 || s.sw > 8) return false;  // the TMA traversal stride takes 1..8
  if (s.cg % kBK != 0 || s.k % 8 != 0 || s.k < 128) return false;
  // One TMA box spans a whole output row: Wo*sw input columns, no wider than the image.
  if (s.wo > kBM || s.wo * s.sw > 256 || s.wo * s.sw > s.w) return false;
  if (s.n < 1 || s.n > 0x7fffffffLL || s.h > 0x7fffffffLL || s.w > 0x7fffffffLL) return false;
  const int64_t tr = kBM / s.wo;
  const int64_t rows = (tr < s.ho ? tr : s.ho) * s.sh;  // input rows a box spans
  if (rows > s.h || rows > 256) return false;           // no box taller than the image
  if (s.r * s.s * s.cg > 0x7fffffffLL) return false;
  return true;
}

// Tile width: 256 output channels when K >= 256 (the two-stage form), else 128.
int tile_bn(const Shape& s, bool cluster) { return !cluster && s.k >= 256 ? 256 : 128; }

// Output rows of an M sub-tile.
int64_t tile_rows(const Shape& s) { return kBM / s.wo < s.ho ? kBM / s.wo : s.ho; }

// M sub-tiles per CTA: 2 for 256-wide tiles when the grid has at least 512
// such double tiles, else 1: the small-M layers keep their many split-K
// units, and mid-sized grids keep single tiles, whose two TMEM accumulators
// let a unit's epilogue overlap the next unit's MMAs (a 3x3 stride-2 layer
// with 256 double tiles measured 39.3 us, with 512 single ones 38.0 us).
int tile_ms(const Shape& s, bool cluster) {
  if (cluster || tile_bn(s, false) != 256) return 1;
  const int64_t tr = tile_rows(s);
  const int64_t pairs = s.n * ((s.ho + 2 * tr - 1) / (2 * tr)) * ((s.k + 255) / 256);
  return pairs >= 512 ? 2 : 1;
}

FwdParams make_params(const Plan& p, int bn, int ms) {
  const Shape& s = p.sh;
  FwdParams fp;
  fp.N = s.n;
  fp.K = s.k;
  fp.E = s.y_elems();
  fp.Ho = s.ho;
  fp.Wo = s.wo;
  fp.Cg = s.cg;
  fp.S_f = s.s;
  fp.cblocks = s.cg / kBK;
  fp.TR = (int32_t)tile_rows(s);
  fp.tiles_m_per_img = (s.ho + (int64_t)ms * fp.TR - 1) / ((int64_t)ms * fp.TR);
  fp.tiles_n = (s.k + bn - 1) / bn;
  fp.tiles = s.n * fp.tiles_m_per_img * fp.tiles_n;
  fp.blocks = s.r * s.s * fp.cblocks;
  fp.ph = (int32_t)s.ph;
  fp.pw = (int32_t)s.pw;
  fp.dh = (int32_t)s.dh;
  fp.dw = (int32_t)s.dw;
  fp.sh = (int32_t)s.sh;
  fp.a_coff = 0;
  fp.taps = (int32_t)(s.r * s.s);
  fp.split = p.split;
  return fp;
}

template <typename TO, uint32_t FMT, bool CL, int BN, int MS, bool BMN = false>
cudaError_t launch_typed(const Plan& p, const Args& a, CUtensorMapDataType dt, bool block = false) {
  const Shape& s = p.sh;
  FwdParams fp = make_params(p, BN, MS);
  fp.a_coff = block ? 1 : 0;
  fp.ep_bias = a.ep_bias;
  fp.ep_lo = a.ep_lo;
  fp.ep_hi = a.ep_hi;
  fp.ep = a.ep ? 1 : 0;
  if (a.ep && (CL || a.ws)) return cudaErrorInvalidValue;  // the epilogue runs unsplit only
  constexpr size_t smem = Tile<BN, MS>::kSmem;
  CUtensorMap tm_x, tm_w;
  const uint64_t x_dims[4] = {(uint64_t)s.c, (uint64_t)s.w, (uint64_t)s.h, (uint64_t)s.n};
  const uint64_t x_strides[3] = {(uint64_t)s.c * 2u, (uint64_t)(s.w * s.c) * 2u, (uint64_t)(s.h * s.w * s.c) * 2u};
  // Strided problems: the box spans Wo*sw columns and TR*sh rows and the map
  // traverses them with strides (sw, sh), so the TR*Wo rows of 128 bytes land
  // in shared memory exactly as for stride 1.
  const uint32_t x_box[4] = {(uint32_t)kBK, (uint32_t)(s.wo * s.sw), (uint32_t)(fp.TR * s.sh), 1u};
  const uint32_t x_estr[4] = {1u, (uint32_t)s.sw, (uint32_t)s.sh, 1u};
  if (!encode_tmap(&tm_x, dt, 4, a.x, x_dims, x_strides, x_box, CU_TENSOR_MAP_SWIZZLE_128B, x_estr))
    return cudaErrorInvalidValue;
  // The filter maps are 4-D (trailing dimensions of extent 1) so that a
  // block's A and B boxes go out through one 4-D copy instruction.
  if (BMN) {  // the filter [C'][R*S][K']: boxes of 64 output channels x 1 tap x 64 reduction channels
    const uint64_t w_dims[4] = {(uint64_t)s.k, (uint64_t)(s.r * s.s), (uint64_t)s.cg, 1u};
    const uint64_t w_strides[3] = {(uint64_t)s.k * 2u, (uint64_t)(s.r * s.s * s.k) * 2u,
                                   (uint64_t)(s.r * s.s * s.k * s.cg) * 2u};
    const uint32_t w_box[4] = {64u, 1u, (uint32_t)kBK, 1u};
    if (!encode_tmap(&tm_w, dt, 4, a.b, w_dims, w_strides, w_box, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  } else {  // W [K][R*S*Cg]: boxes of 64 reduction elements x BN output channels
    const uint64_t w_dims[4] = {(uint64_t)(s.r * s.s * s.cg), (uint64_t)s.k, 1u, 1u};
    const uint64_t w_strides[3] = {(uint64_t)(s.r * s.s * s.cg) * 2u, (uint64_t)(s.r * s.s * s.cg * s.k) * 2u,
                                   (uint64_t)(s.r * s.s * s.cg * s.k) * 2u};
    const uint32_t w_box[4] = {(uint32_t)kBK, (uint32_t)BN, 1u, 1u};
    if (!encode_tmap(&tm_w, dt, 4, a.b, w_dims, w_strides, w_box, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  // Output map of the two-stage form's epilogue: the slabs (fp32) under
  // split-K, else Y, as [N (x S)][Ho*Wo][K], boxes of 128 bytes x TR*Wo pixels.
  CUtensorMap tm_y;
  if (!CL) {
    const bool slabs = a.ws != nullptr;
    const uint64_t es = slabs ? 4u : (uint64_t)sizeof(TO);
    const CUtensorMapDataType ydt = slabs || sizeof(TO) == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : dt;
    const uint64_t y_dims[3] = {(uint64_t)s.k, (uint64_t)(s.ho * s.wo), (uint64_t)s.n * (slabs ? (uint64_t)p.split : 1u)};
    const uint64_t y_strides[2] = {(uint64_t)s.k * es, (uint64_t)(s.ho * s.wo * s.k) * es};
    const uint32_t y_box[3] = {(uint32_t)(128 / es), (uint32_t)(fp.TR * s.wo), 1u};
    if (s.n * (int64_t)p.split > 0x7fffffffLL ||
        !encode_tmap(&tm_y, ydt, 3, slabs ? (const void*)a.ws : a.out, y_dims, y_strides, y_box,
                     CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  } else {
    tm_y = tm_w;  // unused by the cluster form
  }
  const int64_t ctas = fp.tiles * p.split;
  if (ctas > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  if (!CL) {
    auto kern = fwd_tc_kernel<TO, FMT, false, BN, MS, BMN>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    // The persistent form: at most one CTA per SM, each taking every
    // gridDim-th unit; otherwise one CTA per unit.
    const int sms = current_sm_count() > 0 ? current_sm_count() : 148;
    const int64_t grid = Tile<BN, MS>::kPersist && ctas > sms ? sms : ctas;
    // Slab sigma starts at ws + sigma * E; the kernel indexes pixels within it.
    kern<<<(unsigned)grid, BN == 256 ? kThreadsPersist : kThreads, smem, a.stream>>>(tm_x, tm_w, tm_y,
                                                                                      static_cast<TO*>(a.out), a.ws, fp,
                                                      device_error_word());
    return cudaGetLastError();
  }
  if (p.split < 1 || p.split > kMaxClusterSplit) return cudaErrorInvalidConfiguration;
  auto kern = fwd_tc_kernel<TO, FMT, true, BN, MS>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  if (p.split > 8) {  // above the portable cluster size
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (err != cudaSuccess) return err;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)ctas);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = a.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)p.split;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // A cluster shape the device cannot place fails here, before any launch.
  int clusters = 0;
  err = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg);
  if (err != cudaSuccess) return err;
  if (clusters < 1) return cudaErrorInvalidConfiguration;
  return cudaLaunchKernelEx(&cfg, kern, tm_x, tm_w, tm_y, static_cast<TO*>(a.out), (float*)nullptr, fp,
                            device_error_word());
}

}  // namespace

namespace {
Geometry geometry_of(const Shape& s, bool cluster) {
  Geometry g;
  if (!fwd_tc_admissible(s)) return g;
  const int64_t rows = tile_rows(s) * tile_ms(s, cluster);  // output rows of a CTA's tile
  const int bn = tile_bn(s, cluster);
  g.ok = true;
  g.ctas_per_sm = bn == 256 ? 1 : 2;
  g.tiles = s.n * ((s.ho + rows - 1) / rows) * ((s.k + bn - 1) / bn);
  g.blocks = s.r * s.s * (s.cg / kBK);
  if (cluster) g.max_split = kMaxClusterSplit;
  return g;
}
}  // namespace

Geometry geometry_fwd_tc(const Shape& s) { return geometry_of(s, false); }
Geometry geometry_fwd_tc_cluster(const Shape& s) { return geometry_of(s, true); }

// A channel-block problem (see launch_fwd_tc_block): 128-wide tiles, one M
// sub-tile, 2 CTAs per SM; the cluster form's tiling without its split cap.
Geometry geometry_fwd_tc_block(const Shape& b) {
  Geometry g = geometry_of(b, true);
  g.max_split = 0;
  return g;
}

namespace {
template <bool CL, int BN, int MS, bool BMN = false>
cudaError_t launch_bn(const Plan& p, const Args& a, bool block = false) {
  if (p.sh.in_dt == CONV_BF16) {
    if (p.sh.out_dt == CONV_F32)
      return launch_typed<float, 1u, CL, BN, MS, BMN>(p, a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, block);
    return launch_typed<__nv_bfloat16, 1u, CL, BN, MS, BMN>(p, a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, block);
  }
  if (p.sh.out_dt == CONV_F32)
    return launch_typed<float, 0u, CL, BN, MS, BMN>(p, a, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, block);
  return launch_typed<__half, 0u, CL, BN, MS, BMN>(p, a, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, block);
}
}  // namespace

cudaError_t launch_fwd_tc(const Plan& p, const Args& a) {
  if (tile_bn(p.sh, false) == 128) return launch_bn<false, 128, 1>(p, a);
  return tile_ms(p.sh, false) == 2 ? launch_bn<false, 256, 2>(p, a) : launch_bn<false, 256, 1>(p, a);
}
cudaError_t launch_fwd_tc_cluster(const Plan& p, const Args& a) { return launch_bn<true, 128, 1>(p, a); }
cudaError_t launch_fwd_tc_block(const Plan& p, const Args& a) { return launch_bn<false, 128, 1>(p, a, true); }
// The forward form of a data gradient with B read MN-major from the data
// gradient's own filter (see fwd_tc_kernel's BMN).
cudaError_t launch_fwd_tc_filter_mn(const Plan& p, const Args& a) {
  if (tile_bn(p.sh, false) == 128) return launch_bn<false, 128, 1, true>(p, a);
  return tile_ms(p.sh, false) == 2 ? launch_bn<false, 256, 2, true>(p, a) : launch_bn<false, 256, 1, true>(p, a);
}

}  // namespace cig
