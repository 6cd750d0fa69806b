// 16-bit data gradient on the tensor cores, for stride 1 and one group.
//
// With stride 1 the data gradient is itself a forward convolution:
//   dX[n,h,w,c] = sum over r', s', k of dY[n, h + r'*dh - ph', w + s'*dw - pw', k] * W'[c,r',s',k]
// with W'[c,r',s',k] = W[k, R-1-r', S-1-s', c] (the filter turned by 180
// degrees, input and output channels swapped) and ph' = dh*(R-1) - ph,
// pw' = dw*(S-1) - pw: substituting r = R-1-r' in ho = h + ph - r*dh gives
// ho = h + r'*dh - ph'. The input is dY (Ho x Wo, K channels) and the output
// extent Ho + 2 ph' - dh (R-1) = H. So stage 1 is two launches: the filter
// transform into the first bytes of the workspace, then the forward
// tensor-core kernel (im2col by TMA, tcgen05, split-K slabs) on that
// problem; the fold is the forward's.
#include "common.cuh"

namespace cig {
namespace {

constexpr int kT = 64;        // transpose tile: 64 k x 64 c (one 128-byte row of c per k)
constexpr int kTP = kT + 2;   // padded row: 33 words, so rows and columns spread over the banks

// W [K][R][S][C] -> W' [C][R][S][K] with the taps reversed. A block (256
// threads) moves one 64 x 64 (k, c) tile of one tap through shared memory:
// 16-byte loads along c, 16-byte stores along k. Tiles cut by K or C fall
// back to element copies at the edge.
template <typename T>
__global__ void __launch_bounds__(256) transform_filter_kernel(const T* __restrict__ w, T* __restrict__ wt,
                                                              int64_t K, int64_t R, int64_t S, int64_t C) {
  __shared__ __align__(16) T tile[kT][kTP];
  static_assert(sizeof(T) == 2, "16-bit filters");
  const int64_t c0 = (int64_t)blockIdx.x * kT, k0 = (int64_t)blockIdx.y * kT;
  const int64_t tap = blockIdx.z;  // destination tap r' * S + s'
  const int64_t rd = tap / S, sd = tap % S;
  const int64_t src_tap = (R - 1 - rd) * S + (S - 1 - sd);
  const int t = threadIdx.x;
  const bool vec = (C % 8 == 0) && (K % 8 == 0);
  // load: 64 rows k x 8 units of 8 c
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int u = t + 256 * i, row = u >> 3, cu = (u & 7) * 8;
    const int64_t k = k0 + row, c = c0 + cu;
    const T* src = w + (k * R * S + src_tap) * C + c;
    if (vec && k < K && c + 8 <= C) {
      const uint4 v = *reinterpret_cast<const uint4*>(src);
      uint32_t* d = reinterpret_cast<uint32_t*>(&tile[row][cu]);  // 4-byte aligned (cu even, 132-byte rows)
      d[0] = v.x;
      d[1] = v.y;
      d[2] = v.z;
      d[3] = v.w;
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (k < K && c + j < C) tile[row][cu + j] = src[j];
    }
  }
  __syncthreads();
  // store: 64 rows c x 8 units of 8 k
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int u = t + 256 * i, row = u >> 3, ku = (u & 7) * 8;
    const int64_t c = c0 + row, k = k0 + ku;
    T* dst = wt + (c * R * S + tap) * K + k;
    if (c >= C) continue;
    if (vec && k + 8 <= K) {
      __align__(16) T v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = tile[ku + j][row];
      *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(v);
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (k + j < K) dst[j] = tile[ku + j][row];
    }
  }
}

}  // namespace

// The forward problem a stride-1, ungrouped data gradient is (see above).
Shape dgrad_as_forward(const Shape& s) {
  Shape t = s;
  t.h = s.ho;
  t.w = s.wo;
  t.c = s.k;
  t.k = s.c;
  t.sh = t.sw = 1;
  t.ph = s.dh * (s.r - 1) - s.ph;
  t.pw = s.dw * (s.s - 1) - s.pw;
  t.groups = 1;
  t.cg = t.c;
  t.kg = t.k;
  t.ho = s.h;
  t.wo = s.w;
  return t;
}

Geometry geometry_dgrad_tc(const Shape& s) {
  if (s.in_dt == CONV_F32 || s.groups != 1 || s.sh != 1 || s.sw != 1) return Geometry{};
  if (s.ph > s.dh * (s.r - 1) || s.pw > s.dw * (s.s - 1)) return Geometry{};  // ph' and pw' >= 0
  if (s.k > 65535LL * kT || s.r * s.s > 65535) return Geometry{};  // transform grid (y, z)
  return geometry_fwd_tc(dgrad_as_forward(s));
}

cudaError_t launch_dgrad_tc(const Plan& p, const Args& a) {
  const Shape& s = p.sh;
  if (!a.aux) return cudaErrorInvalidValue;
  const dim3 grid((unsigned)((s.c + kT - 1) / kT), (unsigned)((s.k + kT - 1) / kT), (unsigned)(s.r * s.s));
  const dim3 block(256);
  if (s.in_dt == CONV_BF16)
    transform_filter_kernel<__nv_bfloat16><<<grid, block, 0, a.stream>>>(
        static_cast<const __nv_bfloat16*>(a.b), static_cast<__nv_bfloat16*>(a.aux), s.k, s.r, s.s, s.c);
  else
    transform_filter_kernel<__half><<<grid, block, 0, a.stream>>>(static_cast<const __half*>(a.b),
                                                                  static_cast<__half*>(a.aux), s.k, s.r, s.s, s.c);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  Plan fp = p;
  fp.sh = dgrad_as_forward(s);
  fp.dir = CONV_DIR_FWD;
  fp.kernel = CONV_KERNEL_FWD_TC;
  fp.geo = geometry_fwd_tc(fp.sh);
  Args fa = a;
  fa.b = a.aux;  // W'
  fa.aux = nullptr;
  return launch_fwd_tc(fp, fa);
}

}  // namespace cig
