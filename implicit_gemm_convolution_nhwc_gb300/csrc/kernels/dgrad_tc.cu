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

constexpr int kT = 32;  // transpose tile (k x c)

// W [K][R][S][C] -> W' [C][R][S][K] with the taps reversed. Block (32 x 8
// threads) moves one 32 x 32 (k, c) tile of one tap through shared memory, so
// reads run along c and writes along k.
template <typename T>
__global__ void __launch_bounds__(kT * 8) transform_filter_kernel(const T* __restrict__ w, T* __restrict__ wt,
                                                                  int64_t K, int64_t R, int64_t S, int64_t C) {
  __shared__ T tile[kT][kT + 1];
  const int64_t c0 = (int64_t)blockIdx.x * kT, k0 = (int64_t)blockIdx.y * kT;
  const int64_t tap = blockIdx.z;  // destination tap r' * S + s'
  const int64_t rd = tap / S, sd = tap % S;
  const int64_t src_tap = (R - 1 - rd) * S + (S - 1 - sd);
  const int tx = threadIdx.x, ty = threadIdx.y;
#pragma unroll
  for (int i = ty; i < kT; i += 8) {
    const int64_t k = k0 + i, c = c0 + tx;
    if (k < K && c < C) tile[i][tx] = w[(k * R * S + src_tap) * C + c];
  }
  __syncthreads();
#pragma unroll
  for (int i = ty; i < kT; i += 8) {
    const int64_t c = c0 + i, k = k0 + tx;
    if (k < K && c < C) wt[(c * R * S + tap) * K + k] = tile[tx][i];
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
  if (s.c > 65535LL * kT || s.k > 65535LL * kT || s.r * s.s > 65535) return Geometry{};  // transform grid
  return geometry_fwd_tc(dgrad_as_forward(s));
}

cudaError_t launch_dgrad_tc(const Plan& p, const Args& a) {
  const Shape& s = p.sh;
  if (!a.aux) return cudaErrorInvalidValue;
  const dim3 grid((unsigned)((s.c + kT - 1) / kT), (unsigned)((s.k + kT - 1) / kT), (unsigned)(s.r * s.s));
  const dim3 block(kT, 8);
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
