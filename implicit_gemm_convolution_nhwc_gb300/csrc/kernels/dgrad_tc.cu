// 16-bit data gradient on the tensor cores, for stride 1 and one group.
//
// With stride 1 the data gradient is itself a forward convolution:
//   dX[n,h,w,c] = sum over r', s', k of dY[n, h + r'*dh - ph', w + s'*dw - pw', k] * W'[c,r',s',k]
// with W'[c,r',s',k] = W[k, R-1-r', S-1-s', c] (the filter turned by 180
// degrees, input and output channels swapped) and ph' = dh*(R-1) - ph,
// pw' = dw*(S-1) - pw: substituting r = R-1-r' in ho = h + ph - r*dh gives
// ho = h + r'*dh - ph'. The input is dY (Ho x Wo, K channels) and the output
// extent Ho + 2 ph' - dh (R-1) = H. Stage 1 is the forward tensor-core kernel
// (im2col by TMA, tcgen05, split-K slabs) on that problem, reading W' straight
// from W: for a tap, W is a [k][c] matrix with c contiguous, which is W'
// read MN-major (output channels c contiguous), at tap R*S - 1 - (r'*S + s').
// The fold is the forward's.
#include "common.cuh"

namespace cig {

// The forward kernel with B read MN-major from the data gradient's filter.
cudaError_t launch_fwd_tc_filter_mn(const Plan& p, const Args& a);

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
  return geometry_fwd_tc(dgrad_as_forward(s));
}

cudaError_t launch_dgrad_tc(const Plan& p, const Args& a) {
  Plan fp = p;
  fp.sh = dgrad_as_forward(p.sh);
  fp.dir = CONV_DIR_FWD;
  fp.kernel = CONV_KERNEL_FWD_TC;
  fp.geo = geometry_fwd_tc(fp.sh);
  return launch_fwd_tc_filter_mn(fp, a);
}

}  // namespace cig
