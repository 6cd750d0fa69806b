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
//
// Grouped and depthwise data gradients at stride 1 take the same identity
// with the groups kept (below, and the grouped one in grouped_tc.cu).
#include "common.cuh"
#include "../kernel_entry.h"

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

// The same identity with the groups kept: output channel c of the forward
// problem (group g) reads dY channels g*Kg .. g*Kg + Kg - 1 through
// W'[c, r', s', kk] = W[g*Kg + kk, R-1-r', S-1-s', c - g*Cg].
Shape dgrad_as_forward_grouped(const Shape& s) {
  Shape t = dgrad_as_forward(s);
  t.groups = s.groups;
  t.cg = s.kg;
  t.kg = s.cg;
  return t;
}

// Depthwise data gradient ("feat(rocke): split-K forward implicit-GEMM
// convolution on gfx1250", the depthwise data gradient pasted into it: at
// stride 1 it is the depthwise forward with the filter turned by 180 degrees
// and padding F - 1 - pad): for groups = C = K the turned filter W'[c, r', s']
// = W[c, R-1-r', S-1-s'] is W itself with its taps read backwards, so the
// depthwise forward kernels run on dY with reversed taps and the padding
// dil * (f - 1) - pad. Unsplit (the reduction is R*S taps).
Geometry geometry_dgrad_depthwise(const Shape& s) {
  const bool depthwise = s.groups == s.c && s.groups == s.k;
  if (!depthwise || s.sh != 1 || s.sw != 1) return Geometry{};
  if (s.ph > s.dh * (s.r - 1) || s.pw > s.dw * (s.s - 1)) return Geometry{};
  return geometry_fwd_depthwise(dgrad_as_forward_grouped(s));
}

cudaError_t launch_dgrad_depthwise(const Plan& p, const Args& a) {
  Plan fp = p;
  fp.sh = dgrad_as_forward_grouped(p.sh);
  fp.dir = CONV_DIR_FWD;
  fp.kernel = CONV_KERNEL_FWD_DEPTHWISE;
  fp.geo = geometry_fwd_depthwise(fp.sh);
  Args fa = a;
  fa.rev_taps = true;
  return launch_fwd_depthwise(fp, fa);
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
