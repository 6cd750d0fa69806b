// C-ABI layer: argument validation, the split-K planner and dispatch.
//
// Everything here is host code. Validation happens before the first launch,
// so an error status means nothing was enqueued (the loud-failure rule of
// "ROCm/rocm-libraries PR #11188", "Motivation": a silently wrong dW is the
// failure being designed out). All sizes are 64-bit and checked for overflow.
#include <cmath>
#include <cstdint>
#include <cstring>

#include <cuda_runtime.h>

#include "conv_internal.h"
#include "kernel_entry.h"

namespace cig {
namespace {

int g_kernel_override = CONV_KERNEL_AUTO;

bool mul_ok(int64_t a, int64_t b, int64_t* out) { return !__builtin_mul_overflow(a, b, out); }
bool add_ok(int64_t a, int64_t b, int64_t* out) { return !__builtin_add_overflow(a, b, out); }

int esize(int dt) { return dt == CONV_F32 ? 4 : 2; }

uint64_t round256(uint64_t v) { return (v + 255u) & ~uint64_t(255u); }

// Output extent floor((in + 2 pad - dil (f - 1) - 1) / stride) + 1, computed
// with overflow checks; returns -1 on overflow, 0 when nothing fits.
int64_t out_extent(int64_t in, int64_t pad, int64_t dil, int64_t f, int64_t stride) {
  int64_t twice_pad, reach, span;
  if (!mul_ok(2, pad, &twice_pad) || !mul_ok(dil, f - 1, &reach)) return -1;
  if (!add_ok(in, twice_pad, &span)) return -1;
  span = span - reach - 1;
  if (span < 0) return 0;
  return span / stride + 1;
}

conv_status validate(const conv_problem* p, Shape* out) {
  if (!p) return CONV_ERR_INVALID_ARG;
  if (p->n < 0 || p->h < 1 || p->w < 1 || p->c < 1 || p->k < 1 || p->r < 1 || p->s < 1)
    return CONV_ERR_INVALID_ARG;
  if (p->stride_h < 1 || p->stride_w < 1 || p->dil_h < 1 || p->dil_w < 1) return CONV_ERR_INVALID_ARG;
  if (p->pad_h < 0 || p->pad_w < 0 || p->groups < 1) return CONV_ERR_INVALID_ARG;
  if (p->c % p->groups != 0 || p->k % p->groups != 0) return CONV_ERR_INVALID_ARG;
  if (p->in_dtype < CONV_F32 || p->in_dtype > CONV_F16) return CONV_ERR_INVALID_ARG;
  if (p->out_dtype != CONV_F32 && p->out_dtype != p->in_dtype) return CONV_ERR_INVALID_ARG;
  Shape s;
  s.n = p->n; s.h = p->h; s.w = p->w; s.c = p->c; s.k = p->k; s.r = p->r; s.s = p->s;
  s.sh = p->stride_h; s.sw = p->stride_w; s.ph = p->pad_h; s.pw = p->pad_w;
  s.dh = p->dil_h; s.dw = p->dil_w; s.groups = p->groups;
  s.cg = p->c / p->groups; s.kg = p->k / p->groups;
  s.in_dt = p->in_dtype; s.out_dt = p->out_dtype;
  s.ho = out_extent(s.h, s.ph, s.dh, s.r, s.sh);
  s.wo = out_extent(s.w, s.pw, s.dw, s.s, s.sw);
  if (s.ho < 0 || s.wo < 0) return CONV_ERR_OVERFLOW;
  if (s.ho == 0 || s.wo == 0) return CONV_ERR_INVALID_ARG;
  // Every element and byte count used anywhere must fit in int64 (with room
  // for the 4-byte fp32 slabs).
  int64_t t;
  const int64_t xs[4] = {s.n, s.h, s.w, s.c};
  const int64_t ws_[4] = {s.k, s.r, s.s, s.cg};
  const int64_t ys[4] = {s.n, s.ho, s.wo, s.k};
  const int64_t* lists[3] = {xs, ws_, ys};
  for (auto* l : lists) {
    t = 4;
    for (int i = 0; i < 4; ++i)
      if (!mul_ok(t, l[i], &t)) return CONV_ERR_OVERFLOW;
  }
  *out = s;
  return CONV_OK;
}

Geometry geometry_of(conv_kernel k, const Shape& s, conv_dir dir) {
  switch (k) {
    case CONV_KERNEL_GENERIC: return geometry_generic(s, dir);
    case CONV_KERNEL_WGRAD_1X1_FFMA: return dir == CONV_DIR_WGRAD ? geometry_wgrad1x1_ffma(s) : Geometry{};
    case CONV_KERNEL_WGRAD_1X1_TF32X3: return dir == CONV_DIR_WGRAD ? geometry_wgrad1x1_tf32x3(s) : Geometry{};
    case CONV_KERNEL_FWD_TC: return dir == CONV_DIR_FWD ? geometry_fwd_tc(s) : Geometry{};
    case CONV_KERNEL_FWD_TC_CLUSTER: return dir == CONV_DIR_FWD ? geometry_fwd_tc_cluster(s) : Geometry{};
    case CONV_KERNEL_DGRAD_TC: return dir == CONV_DIR_DGRAD ? geometry_dgrad_tc(s) : Geometry{};
    case CONV_KERNEL_FWD_DEPTHWISE: return dir == CONV_DIR_FWD ? geometry_fwd_depthwise(s) : Geometry{};
    case CONV_KERNEL_FWD_GROUPED_TC: return dir == CONV_DIR_FWD ? geometry_fwd_grouped_tc(s) : Geometry{};
    case CONV_KERNEL_WGRAD_GROUPED_TC: return dir == CONV_DIR_WGRAD ? geometry_wgrad_grouped_tc(s) : Geometry{};
    case CONV_KERNEL_WGRAD_TC: return dir == CONV_DIR_WGRAD ? geometry_wgrad_tc(s) : Geometry{};
    case CONV_KERNEL_WGRAD_GROUPED_MMA: return dir == CONV_DIR_WGRAD ? geometry_wgrad_grouped_mma(s) : Geometry{};
    case CONV_KERNEL_FFMA: return geometry_ffma(s, dir);
    case CONV_KERNEL_WGRAD_DEPTHWISE_MMA: return dir == CONV_DIR_WGRAD ? geometry_wgrad_depthwise_mma(s) : Geometry{};
    case CONV_KERNEL_FWD_GROUPED_MMA: return dir == CONV_DIR_FWD ? geometry_fwd_grouped_mma(s) : Geometry{};
    case CONV_KERNEL_DGRAD_GROUPED_MMA: return dir == CONV_DIR_DGRAD ? geometry_dgrad_grouped_mma(s) : Geometry{};
    case CONV_KERNEL_DGRAD_DEPTHWISE: return dir == CONV_DIR_DGRAD ? geometry_dgrad_depthwise(s) : Geometry{};
    case CONV_KERNEL_DGRAD_GROUPED_TC: return dir == CONV_DIR_DGRAD ? geometry_dgrad_grouped_tc(s) : Geometry{};
    case CONV_KERNEL_WGRAD_DEPTHWISE: return dir == CONV_DIR_WGRAD ? geometry_wgrad_depthwise(s) : Geometry{};
    case CONV_KERNEL_WGRAD_GROUPED: return dir == CONV_DIR_WGRAD ? geometry_wgrad_grouped(s) : Geometry{};
    default: return Geometry{};
  }
}

// Width fold ("feat(rocke): split-K forward implicit-GEMM convolution on
// gfx1250", the fold_width commit): when f divides the filter width, the W
// stride, the input width and the W padding (unit W dilation, one group), the
// problem equals one with W/f positions of f*C channels, filter width S/f and
// W stride sw/f, on the same memory: X [N][H][W][C] is [N][H][W/f][f*C], W
// [K][R][S][C] is [K][R][S/f][f*C] (tap s = f*s' + j, channel j*C + c), and
// Y is unchanged. f is the largest such factor (1: no fold).
int64_t gcd64(int64_t a, int64_t b) {
  while (b != 0) {
    const int64_t t = a % b;
    a = b;
    b = t;
  }
  return a;
}

int64_t fold_width_of(const Shape& s) {
  if (s.groups != 1 || s.dw != 1) return 1;
  return gcd64(gcd64(gcd64(s.s, s.sw), s.w), s.pw);
}

Shape fold_width(const Shape& s, int64_t f) {
  Shape t = s;
  t.w = s.w / f;
  t.s = s.s / f;
  t.sw = s.sw / f;
  t.pw = s.pw / f;
  t.c = s.c * f;
  t.cg = t.c;
  return t;
}

// The kernel a call runs: the override if set, else the first fast kernel
// that takes the problem, else the generic one.
conv_status choose_kernel(const Shape& s, conv_dir dir, conv_kernel* kernel, Geometry* geo) {
  if (g_kernel_override != CONV_KERNEL_AUTO) {
    Geometry g = geometry_of((conv_kernel)g_kernel_override, s, dir);
    if (!g.ok) return CONV_ERR_UNSUPPORTED;
    *kernel = (conv_kernel)g_kernel_override;
    *geo = g;
    return CONV_OK;
  }
  static const conv_kernel wgrad_order[] = {CONV_KERNEL_WGRAD_1X1_TF32X3,  CONV_KERNEL_WGRAD_1X1_FFMA,
                                            CONV_KERNEL_WGRAD_DEPTHWISE,    CONV_KERNEL_WGRAD_GROUPED_MMA,
                                            CONV_KERNEL_WGRAD_GROUPED_TC,   CONV_KERNEL_WGRAD_TC,
                                            CONV_KERNEL_FFMA,               CONV_KERNEL_WGRAD_GROUPED,
                                            CONV_KERNEL_GENERIC};
  // The cluster form of the forward is reached only through the override:
  // on the 3x3 small-M layer it measured slower than the two-stage form. So is
  // the depthwise weight gradient's MMA form: bound by shared-memory traffic
  // (0.65 bytes a useful multiply-add), it measured slower than the CUDA-core
  // ring kernel on the 7x7 layer.
  static const conv_kernel fwd_order[] = {CONV_KERNEL_FWD_TC,         CONV_KERNEL_FWD_DEPTHWISE,
                                          CONV_KERNEL_FWD_GROUPED_MMA, CONV_KERNEL_FWD_GROUPED_TC,
                                          CONV_KERNEL_FFMA,            CONV_KERNEL_GENERIC};
  static const conv_kernel dgrad_order[] = {CONV_KERNEL_DGRAD_TC,         CONV_KERNEL_DGRAD_DEPTHWISE,
                                            CONV_KERNEL_DGRAD_GROUPED_MMA, CONV_KERNEL_DGRAD_GROUPED_TC,
                                            CONV_KERNEL_FFMA,              CONV_KERNEL_GENERIC};
  const conv_kernel* order = dir == CONV_DIR_WGRAD ? wgrad_order : dir == CONV_DIR_FWD ? fwd_order : dgrad_order;
  const int count = dir == CONV_DIR_WGRAD ? 9 : 6;
  for (int i = 0; i < count; ++i) {
    Geometry g = geometry_of(order[i], s, dir);
    if (g.ok) {
      *kernel = order[i];
      *geo = g;
      return CONV_OK;
    }
  }
  return CONV_ERR_UNSUPPORTED;
}

// Split-K degree: see resolve_split_k_for in conv_igemm.h. The forward
// policy restates "feat(rocke): split-K forward implicit-GEMM convolution on
// gfx1250" ("Auto-deduced degree"): split only a grid under half the target,
// over a reduction at least 512 deep; a power of two toward the target, at
// most 32 (at most the kernel's own limit, 16 for the cluster form), with at
// least 2 reduction blocks per slice; pointwise stays whole.
conv_status resolve_degree(const Shape& s, conv_dir dir, const Geometry& g, int32_t request,
                           int32_t sm_count, int32_t* degree) {
  if (request < -1) return CONV_ERR_INVALID_ARG;
  if (request == 0) {
    *degree = 1;
    return CONV_OK;
  }
  if (request > 0) {
    const int64_t cap = g.blocks > 0 ? g.blocks : 1;
    if ((int64_t)request > cap) return CONV_ERR_INVALID_ARG;
    *degree = request;
    return CONV_OK;
  }
  if (sm_count < 1) return CONV_ERR_INVALID_ARG;
  const int64_t target = (int64_t)sm_count * g.ctas_per_sm;
  int64_t d = 1;
  if (dir == CONV_DIR_FWD || dir == CONV_DIR_DGRAD) {
    // The data gradient takes the forward's policy over its own reduction
    // depth R*S*Kg (the pages name a dgrad policy but do not describe it).
    const bool pointwise = s.r == 1 && s.s == 1;
    const int64_t depth = dir == CONV_DIR_DGRAD ? s.r * s.s * s.kg : s.D();
    const int64_t cap = g.max_split > 0 && g.max_split < 32 ? g.max_split : 32;
    if (!pointwise && 2 * g.tiles < target && depth >= 512) {
      while (2 * d <= cap && g.tiles * (2 * d) <= target) d *= 2;
      while (d > 1 && g.blocks < 2 * d) d /= 2;
    }
  } else if (g.tiles < target) {
    d = target / g.tiles;
    if (d > g.blocks / 2) d = g.blocks / 2;
    if (d > 4096) d = 4096;
    if (d < 1) d = 1;
  }
  *degree = (int32_t)d;
  return CONV_OK;
}

// epilogue: a non-identity fused forward epilogue, which runs unsplit
// ("feat(rocke): split-K forward implicit-GEMM convolution on gfx1250",
// "Review follow-ups": split-K rejects it; "Auto-deduced degree": such specs
// resolve to 1).
// The kernel for a problem, folding its width when only the folded problem
// has a kernel faster than the generic one (then *s becomes the folded shape
// and *fold its factor).
// A forced kernel (the testing override) applies to the problem as given:
// no fold is tried, so a kernel that cannot take it fails the call.
conv_status choose_kernel_folded(Shape* s, conv_dir dir, conv_kernel* kernel, Geometry* geo, int64_t* fold) {
  *fold = 1;
  conv_status st = choose_kernel(*s, dir, kernel, geo);
  if (g_kernel_override != CONV_KERNEL_AUTO) return st;
  if (st == CONV_OK && *kernel != CONV_KERNEL_GENERIC) return st;
  const int64_t f = fold_width_of(*s);
  if (f < 2) return st;
  const Shape t = fold_width(*s, f);
  conv_kernel kt;
  Geometry gt;
  if (choose_kernel(t, dir, &kt, &gt) != CONV_OK || kt == CONV_KERNEL_GENERIC) return st;
  *s = t;
  *kernel = kt;
  *geo = gt;
  *fold = f;
  return CONV_OK;
}

conv_status make_plan(const conv_problem* prob, conv_dir dir, int32_t request, bool with_bias,
                      int32_t sm_count, Plan* plan, bool epilogue = false, int64_t* fold_out = nullptr) {
  if (dir != CONV_DIR_FWD && dir != CONV_DIR_WGRAD && dir != CONV_DIR_DGRAD) return CONV_ERR_INVALID_ARG;
  Plan p;
  conv_status st = validate(prob, &p.sh);
  if (st != CONV_OK) return st;
  if (request < -1) return CONV_ERR_INVALID_ARG;
  p.dir = dir;
  p.with_bias = with_bias && dir == CONV_DIR_WGRAD;
  p.epilogue = epilogue;
  if (epilogue) {
    if (dir != CONV_DIR_FWD || request > 1) return CONV_ERR_INVALID_ARG;
    request = 1;
  }
  int64_t fold = 1;
  st = choose_kernel_folded(&p.sh, dir, &p.kernel, &p.geo, &fold);
  if (st != CONV_OK) return st;
  if (fold_out) *fold_out = fold;
  if (epilogue && p.kernel == CONV_KERNEL_FWD_TC_CLUSTER) return CONV_ERR_UNSUPPORTED;
  // The cluster form takes at most 16 slices (one cluster per tile).
  if (p.kernel == CONV_KERNEL_FWD_TC_CLUSTER && request > p.geo.max_split && request <= p.geo.blocks)
    return CONV_ERR_UNSUPPORTED;
  st = resolve_degree(p.sh, dir, p.geo, request, sm_count, &p.split);
  if (st != CONV_OK) return st;
  p.fold = p.split > 1 && p.kernel != CONV_KERNEL_FWD_TC_CLUSTER;
  p.out_elems = dir == CONV_DIR_FWD ? p.sh.y_elems() : dir == CONV_DIR_WGRAD ? p.sh.w_elems() : p.sh.x_elems();
  p.slab_bytes = p.bias_slab_bytes = 0;
  // The grouped forward's tensor-core path writes its block-diagonal filter
  // ([K][R][S][128] in_dtype elements) at the start of the workspace; the
  // grouped data gradient its turned one ([C][R][S][128]).
  p.aux_bytes = 0;
  if (p.kernel == CONV_KERNEL_FWD_GROUPED_TC)
    p.aux_bytes = round256((uint64_t)(p.sh.k * p.sh.r * p.sh.s) * 128u * (uint64_t)esize(p.sh.in_dt));
  if (p.kernel == CONV_KERNEL_DGRAD_GROUPED_TC)
    p.aux_bytes = round256((uint64_t)(p.sh.c * p.sh.r * p.sh.s) * 128u * (uint64_t)esize(p.sh.in_dt));
  if (p.fold) {
    int64_t b;
    if (!mul_ok(p.out_elems, 4, &b) || !mul_ok(b, p.split, &b)) return CONV_ERR_OVERFLOW;
    p.slab_bytes = round256((uint64_t)b);
    if (p.with_bias) p.bias_slab_bytes = round256((uint64_t)p.sh.k * 4u * (uint64_t)p.split);
  }
  *plan = p;
  return CONV_OK;
}

bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

// Which stages a call enqueues.
enum Stages { kStage1 = 1, kStage2 = 2, kBoth = 3 };

// A fused epilogue that changes nothing (no bias, bounds -inf / +inf).
bool identity_epilogue(const conv_epilogue* ep) {
  return !ep || (!ep->bias && std::isinf(ep->lo) && ep->lo < 0 && std::isinf(ep->hi) && ep->hi > 0);
}

conv_status run(const conv_problem* prob, conv_dir dir, const void* x, const void* b, void* out,
                void* db, void* ws, uint64_t ws_bytes, int32_t split_k, void* stream, bool with_bias,
                int stages, const conv_epilogue* ep = nullptr) {
  Shape sh;
  conv_status st = validate(prob, &sh);
  if (st != CONV_OK) return st;
  if (dir != CONV_DIR_FWD && dir != CONV_DIR_WGRAD && dir != CONV_DIR_DGRAD) return CONV_ERR_INVALID_ARG;
  if (split_k < -1) return CONV_ERR_INVALID_ARG;
  if (with_bias && dir != CONV_DIR_WGRAD) return CONV_ERR_INVALID_ARG;
  // Elements of the two inputs and the output, per direction.
  const int64_t x_elems = dir == CONV_DIR_DGRAD ? sh.y_elems() : sh.x_elems();
  const int64_t b_elems = dir == CONV_DIR_WGRAD ? sh.y_elems() : sh.w_elems();
  const int64_t out_elems =
      dir == CONV_DIR_FWD ? sh.y_elems() : dir == CONV_DIR_WGRAD ? sh.w_elems() : sh.x_elems();
  const bool needs_inputs = (stages & kStage1) != 0;
  if ((needs_inputs && x_elems > 0 && !x) || (needs_inputs && b_elems > 0 && !b) ||
      (out_elems > 0 && !out) || (with_bias && !db))
    return CONV_ERR_INVALID_ARG;
  const bool epilogue = !identity_epilogue(ep);
  if (epilogue) {
    if (std::isnan(ep->lo) || std::isnan(ep->hi) || ep->lo > ep->hi) return CONV_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(ep->bias) % (uintptr_t)esize(sh.out_dt) != 0) return CONV_ERR_ALIGNMENT;
    if (dir != CONV_DIR_FWD || split_k > 1) return CONV_ERR_INVALID_ARG;  // never split (make_plan too)
  }
  if (!aligned16(x) || !aligned16(b) || !aligned16(out) || !aligned16(db) || !aligned16(ws))
    return CONV_ERR_ALIGNMENT;
  const int sms = current_sm_count();
  if (sms < 1) return CONV_ERR_CUDA;
  Plan plan;
  st = make_plan(prob, dir, split_k, with_bias, sms, &plan, epilogue);
  if (st != CONV_OK) return st;
  if (plan.ws_bytes() > 0 && (!ws || ws_bytes < plan.ws_bytes())) return CONV_ERR_WORKSPACE_TOO_SMALL;
  if (out_elems == 0) return CONV_OK;  // an empty forward batch: nothing to write
  Args a;
  a.x = x;
  a.b = b;
  a.out = out;
  a.db = plan.with_bias ? db : nullptr;
  a.aux = plan.aux_bytes > 0 ? ws : nullptr;
  a.ws = plan.fold ? reinterpret_cast<float*>(static_cast<char*>(ws) + plan.aux_bytes) : nullptr;
  a.ws_bias = plan.fold && plan.with_bias
                  ? reinterpret_cast<float*>(static_cast<char*>(ws) + plan.aux_bytes + plan.slab_bytes)
                  : nullptr;
  a.stream = static_cast<cudaStream_t>(stream);
  if (epilogue) {
    a.ep = true;
    a.ep_bias = ep->bias;
    a.ep_lo = ep->lo;
    a.ep_hi = ep->hi;
  }
  cudaError_t err = cudaSuccess;
  if (stages & kStage1) {
    switch (plan.kernel) {
      case CONV_KERNEL_GENERIC: err = launch_generic(plan, a); break;
      case CONV_KERNEL_WGRAD_1X1_FFMA: err = launch_wgrad1x1_ffma(plan, a); break;
      case CONV_KERNEL_WGRAD_1X1_TF32X3: err = launch_wgrad1x1_tf32x3(plan, a); break;
      case CONV_KERNEL_FWD_TC: err = launch_fwd_tc(plan, a); break;
      case CONV_KERNEL_FWD_TC_CLUSTER: err = launch_fwd_tc_cluster(plan, a); break;
      case CONV_KERNEL_DGRAD_TC: err = launch_dgrad_tc(plan, a); break;
      case CONV_KERNEL_FWD_DEPTHWISE: err = launch_fwd_depthwise(plan, a); break;
      case CONV_KERNEL_FWD_GROUPED_TC: err = launch_fwd_grouped_tc(plan, a); break;
      case CONV_KERNEL_WGRAD_GROUPED_TC: err = launch_wgrad_grouped_tc(plan, a); break;
      case CONV_KERNEL_WGRAD_TC: err = launch_wgrad_tc(plan, a); break;
      case CONV_KERNEL_WGRAD_GROUPED_MMA: err = launch_wgrad_grouped_mma(plan, a); break;
      case CONV_KERNEL_FFMA: err = launch_ffma(plan, a); break;
      case CONV_KERNEL_WGRAD_DEPTHWISE_MMA: err = launch_wgrad_depthwise_mma(plan, a); break;
      case CONV_KERNEL_FWD_GROUPED_MMA: err = launch_fwd_grouped_mma(plan, a); break;
      case CONV_KERNEL_DGRAD_GROUPED_MMA: err = launch_dgrad_grouped_mma(plan, a); break;
      case CONV_KERNEL_DGRAD_DEPTHWISE: err = launch_dgrad_depthwise(plan, a); break;
      case CONV_KERNEL_DGRAD_GROUPED_TC: err = launch_dgrad_grouped_tc(plan, a); break;
      case CONV_KERNEL_WGRAD_DEPTHWISE: err = launch_wgrad_depthwise(plan, a); break;
      case CONV_KERNEL_WGRAD_GROUPED: err = launch_wgrad_grouped(plan, a); break;
      default: return CONV_ERR_UNSUPPORTED;
    }
    if (err != cudaSuccess) return CONV_ERR_CUDA;
  }
  if ((stages & kStage2) && plan.fold) {
    err = launch_fold(plan, a);
    if (err != cudaSuccess) return CONV_ERR_CUDA;
  }
  return CONV_OK;
}

}  // namespace

int current_sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) {
    cudaGetLastError();
    return -1;
  }
  if (dev < 64 && cached[dev] > 0) return cached[dev];
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return -1;
  }
  if (dev < 64) cached[dev] = sms;
  return sms;
}

}  // namespace cig

using namespace cig;

extern "C" {

const char* conv_status_string(conv_status status) {
  switch (status) {
    case CONV_OK: return "CONV_OK";
    case CONV_ERR_INVALID_ARG: return "CONV_ERR_INVALID_ARG";
    case CONV_ERR_UNSUPPORTED: return "CONV_ERR_UNSUPPORTED";
    case CONV_ERR_WORKSPACE_TOO_SMALL: return "CONV_ERR_WORKSPACE_TOO_SMALL";
    case CONV_ERR_OVERFLOW: return "CONV_ERR_OVERFLOW";
    case CONV_ERR_ALIGNMENT: return "CONV_ERR_ALIGNMENT";
    case CONV_ERR_CUDA: return "CONV_ERR_CUDA";
  }
  return "CONV_ERR_UNKNOWN";
}

conv_status conv_output_dims(const conv_problem* p, int64_t* ho, int64_t* wo) {
  Shape s;
  conv_status st = validate(p, &s);
  if (st != CONV_OK) return st;
  if (!ho || !wo) return CONV_ERR_INVALID_ARG;
  *ho = s.ho;
  *wo = s.wo;
  return CONV_OK;
}

conv_status resolve_split_k_for(const conv_problem* p, conv_dir dir, int32_t request,
                                int32_t sm_count, int32_t* degree) {
  if (!degree) return CONV_ERR_INVALID_ARG;
  Plan plan;
  conv_status st = make_plan(p, dir, request, false, sm_count, &plan);
  if (st == CONV_OK) *degree = plan.split;
  return st;
}

conv_status resolve_split_k(const conv_problem* p, conv_dir dir, int32_t request, int32_t* degree) {
  const int sms = current_sm_count();
  if (sms < 1) return CONV_ERR_CUDA;
  return resolve_split_k_for(p, dir, request, sms, degree);
}

conv_status conv_workspace_bytes_for(const conv_problem* p, conv_dir dir, int32_t split_k,
                                     int32_t with_bias, int32_t sm_count, uint64_t* bytes) {
  if (!bytes) return CONV_ERR_INVALID_ARG;
  Plan plan;
  conv_status st = make_plan(p, dir, split_k, with_bias != 0, sm_count, &plan);
  if (st == CONV_OK) *bytes = plan.ws_bytes();
  return st;
}

conv_status conv_workspace_bytes(const conv_problem* p, conv_dir dir, int32_t split_k,
                                 int32_t with_bias, uint64_t* bytes) {
  const int sms = current_sm_count();
  if (sms < 1) return CONV_ERR_CUDA;
  return conv_workspace_bytes_for(p, dir, split_k, with_bias, sms, bytes);
}

conv_status conv_describe_plan(const conv_problem* p, conv_dir dir, int32_t split_k,
                               int32_t with_bias, int32_t sm_count, conv_plan_info* info) {
  if (!info) return CONV_ERR_INVALID_ARG;
  Plan plan;
  int64_t fold = 1;
  conv_status st = make_plan(p, dir, split_k, with_bias != 0, sm_count, &plan, false, &fold);
  if (st != CONV_OK) return st;
  info->kernel = plan.kernel;
  info->fold_width = (int32_t)fold;
  info->split_k = plan.split;
  info->needs_fold = plan.fold ? 1 : 0;
  info->ctas_per_sm = plan.geo.ctas_per_sm;
  info->tiles = plan.geo.tiles;
  info->reduction_blocks = plan.geo.blocks;
  info->ctas = plan.geo.tiles * plan.split;
  info->workspace_bytes = plan.ws_bytes();
  info->max_split = plan.geo.max_split > 0 && plan.geo.max_split < plan.geo.blocks
                        ? plan.geo.max_split
                        : (int32_t)(plan.geo.blocks < 0x7fffffff ? plan.geo.blocks : 0x7fffffff);
  return CONV_OK;
}

conv_status conv_fwd(const conv_problem* p, const void* x, const void* w, void* y, void* ws,
                     uint64_t ws_bytes, int32_t split_k, void* stream) {
  return run(p, CONV_DIR_FWD, x, w, y, nullptr, ws, ws_bytes, split_k, stream, false, kBoth);
}

conv_status conv_fwd_epilogue(const conv_problem* p, const void* x, const void* w, const conv_epilogue* ep,
                              void* y, void* ws, uint64_t ws_bytes, int32_t split_k, void* stream) {
  return run(p, CONV_DIR_FWD, x, w, y, nullptr, ws, ws_bytes, split_k, stream, false, kBoth, ep);
}

conv_status conv_dgrad(const conv_problem* p, const void* dy, const void* w, void* dx, void* ws,
                       uint64_t ws_bytes, int32_t split_k, void* stream) {
  return run(p, CONV_DIR_DGRAD, dy, w, dx, nullptr, ws, ws_bytes, split_k, stream, false, kBoth);
}

conv_status conv_wgrad(const conv_problem* p, const void* x, const void* dy, void* dw, void* ws,
                       uint64_t ws_bytes, int32_t split_k, void* stream) {
  return run(p, CONV_DIR_WGRAD, x, dy, dw, nullptr, ws, ws_bytes, split_k, stream, false, kBoth);
}

conv_status conv_wgrad_bias(const conv_problem* p, const void* x, const void* dy, void* dw,
                            void* db, void* ws, uint64_t ws_bytes, int32_t split_k, void* stream) {
  return run(p, CONV_DIR_WGRAD, x, dy, dw, db, ws, ws_bytes, split_k, stream, true, kBoth);
}

conv_status conv_stage1(const conv_problem* p, conv_dir dir, const void* x, const void* b, void* out,
                        void* db, void* ws, uint64_t ws_bytes, int32_t split_k, void* stream) {
  return run(p, dir, x, b, out, db, ws, ws_bytes, split_k, stream, db != nullptr, kStage1);
}

conv_status conv_stage2(const conv_problem* p, conv_dir dir, void* out, void* db, void* ws,
                        uint64_t ws_bytes, int32_t split_k, void* stream) {
  return run(p, dir, nullptr, nullptr, out, db, ws, ws_bytes, split_k, stream, db != nullptr, kStage2);
}

int64_t conv_batch_split_count(int64_t n, int64_t max_n) {
  if (n < 0 || max_n < 1) return -1;
  if (n == 0) return 1;
  return (n - 1) / max_n + 1;  // == (n + max_n - 1) / max_n without the overflow
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Weight + bias gradient without any device allocation by the caller.
//
// Some callers cannot allocate device memory at the point where they run the
// convolution: code whose device memory budget is owned by a framework's
// pool, and plugin or enqueue-time paths of inference runtimes that forbid
// cudaMalloc after set-up. They may also have no workspace of their own to
// pass. For them the split-K slabs live in this fixed, library-owned device
// array instead of a caller workspace.
namespace {

constexpr uint64_t kStaticScratchBytes = 8ull << 20;  // 8 MiB on every device that loads the library
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

// The array's device address in the current context, looked up on every call
// (no cache: after a device reset the module reloads and the array may move).
// The first lookup on a device loads the library's module there, which commits
// the array's 8 MiB.
void* static_scratch_address() {
  void* ptr = nullptr;
  if (cudaGetSymbolAddress(&ptr, g_static_scratch) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return ptr;
}

}  // namespace

extern "C" {

conv_status conv_wgrad_bias_static_ws(const conv_problem* p, const void* x, const void* dy, void* dw, void* db,
                                      int32_t split_k, void* stream) {
  const int sms = current_sm_count();
  if (sms < 1) return CONV_ERR_CUDA;
  uint64_t need = 0;
  conv_status st = conv_workspace_bytes_for(p, CONV_DIR_WGRAD, split_k, 1, sms, &need);
  if (st != CONV_OK) return st;
  if (need > kStaticScratchBytes) return CONV_ERR_WORKSPACE_TOO_SMALL;
  // Looked up even when this call needs no slabs, so an empty-batch call
  // (n = 0) serves as the set-up call that loads the module.
  void* scratch = static_scratch_address();
  if (!scratch) return CONV_ERR_CUDA;
  return run(p, CONV_DIR_WGRAD, x, dy, dw, db, scratch, need > 0 ? kStaticScratchBytes : 0, split_k, stream, true,
             kBoth);
}


conv_status conv_set_kernel_override(int32_t kernel) {
  if (kernel < CONV_KERNEL_AUTO || kernel > CONV_KERNEL_DGRAD_GROUPED_MMA) return CONV_ERR_INVALID_ARG;
  g_kernel_override = kernel;
  return CONV_OK;
}

}  // extern "C"
