/*
 * conv_igemm.h — C ABI of the GB300 (sm_103a) NHWC implicit-GEMM convolution
 * library: forward Y = conv(X, W), weight gradient dW and bias gradient db,
 * each with deterministic two-stage split-K.
 *
 * Sources of the operations (web pages, cited by title and section):
 *  [P1] "ROCm/rocm-libraries PR #11188" (MIOpen NHWC wgrad batch split):
 *       "Motivation", "Technical Details", "Test Plan".
 *  [P2] "feat(rocke): split-K forward implicit-GEMM convolution on gfx1250"
 *       (PR #14393): "Two-stage split-K", "Auto-deduced degree",
 *       "ABI, AOT and runtime", "Review follow-ups".
 *  [P3] "perf(rocke): depthwise 7x7 and grouped cpg4/8 wgrad on batched
 *       mfma 4x4x4" (PR #14157): "Technical Details".
 *
 * Conventions shared by every entry point
 *  - Layouts are dense and contiguous: X [n][h][w][c], W and dW
 *    [k][r][s][c/groups] (channels-last weight), Y and dY [n][ho][wo][k],
 *    db [k]. Output channel k reads input channels g*Cg .. g*Cg+Cg-1 with
 *    g = k / (k/groups) (contiguous groups; depthwise is groups = c = k).
 *  - The operation is a cross-correlation:
 *      Y[n,ho,wo,k]  = sum_{r,s,c<Cg} X[n, ho*sh + r*dh - ph, wo*sw + s*dw - pw, g*Cg + c] * W[k,r,s,c]
 *      dW[k,r,s,c]   = sum_{n,ho,wo}  dY[n,ho,wo,k] * X[n, ho*sh + r*dh - ph, wo*sw + s*dw - pw, g*Cg + c]
 *      db[k]         = sum_{n,ho,wo}  dY[n,ho,wo,k]
 *    with X = 0 outside [0,h) x [0,w), and
 *      ho extent = floor((h + 2 ph - dh (r - 1) - 1) / sh) + 1 (likewise wo).
 *  - Every index and byte offset is 64-bit. A tensor larger than 4 GB is
 *    handled in one call; there is no batch split and nothing wraps [P1].
 *    A size whose byte count does not fit in int64 is rejected.
 *  - Ownership: the caller owns every buffer (device memory for tensors and
 *    workspace). The library allocates nothing, never synchronises, and
 *    enqueues its kernels on `stream` (a cudaStream_t; NULL = the legacy
 *    default stream). Pointers must be 16-byte aligned device pointers.
 *  - Errors are loud [P1 "Motivation"]: every argument is checked before the
 *    first launch, so a status other than CONV_OK and CONV_ERR_CUDA means
 *    nothing was enqueued. CONV_ERR_CUDA reports a failed CUDA call; when a
 *    call enqueues two kernels (stage 1, then the fold or the bias sum) and
 *    the second launch fails, the first is already enqueued on the stream, so
 *    after CONV_ERR_CUDA the outputs (and the workspace) are undefined.
 *  - Split-K [P2 "Two-stage split-K"]: the reduction (N*Ho*Wo for the weight
 *    gradient, R*S*Cg for the forward) is cut into S slices. Stage 1 writes
 *    one fp32 partial slab per slice into the caller's workspace, each
 *    element exactly once, so the workspace needs no clearing and its
 *    contents on entry do not matter. Stage 2 (the fold) sums the slabs in
 *    the fixed order 0..S-1 and rounds once (round-to-nearest-even) into the
 *    output type. No atomics are used: a call repeated with the same inputs
 *    and the same degree gives bit-identical outputs. With S = 1 stage 1
 *    writes the output directly and no workspace is needed.
 *  - The degree request: -1 = auto (the policy of resolve_split_k), 0 = no
 *    split (S = 1), n >= 1 = exactly n slices, which must not exceed the
 *    number of reduction blocks of the chosen kernel (else
 *    CONV_ERR_INVALID_ARG). Values below -1 are rejected [P2 "Review
 *    follow-ups": split_k <= 0 is rejected there; this ABI keeps 0 = none].
 */
#ifndef CONV_IGEMM_H
#define CONV_IGEMM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum conv_status {
  CONV_OK = 0,
  CONV_ERR_INVALID_ARG = 1,          /* a NULL pointer, a bad size, dtype or degree */
  CONV_ERR_UNSUPPORTED = 2,          /* a valid problem no kernel here takes */
  CONV_ERR_WORKSPACE_TOO_SMALL = 3,  /* ws_bytes < conv_workspace_bytes(...) */
  CONV_ERR_OVERFLOW = 4,             /* a byte size does not fit in int64 */
  CONV_ERR_ALIGNMENT = 5,            /* a pointer is not 16-byte aligned */
  CONV_ERR_CUDA = 6                  /* a CUDA call failed (no device, launch error) */
} conv_status;

typedef enum conv_dtype { CONV_F32 = 0, CONV_BF16 = 1, CONV_F16 = 2 } conv_dtype;

/* Direction: forward (Y from X, W), weight gradient (dW, db from X, dY) or
 * data gradient (dX from dY, W: the gradient of the forward with respect to
 * X, the "dgrad" the split-K resolver of [P2 "Auto-deduced degree"] also
 * covers). */
typedef enum conv_dir { CONV_DIR_FWD = 0, CONV_DIR_WGRAD = 1, CONV_DIR_DGRAD = 2 } conv_dir;

/* One convolution. in_dtype is the type of X and W (forward), X and dY
 * (weight gradient) or dY and W (data gradient). out_dtype is the type of Y,
 * of dW and db, or of dX; it must be
 * CONV_F32 or in_dtype (the pages require a non-NULL output type [P2 "Review
 * follow-ups"]). Sizes: n >= 0 (n = 0 gives dW = db = 0); h, w, c, k, r, s,
 * strides, dilations, groups >= 1; pads >= 0; groups divides c and k; the
 * output extent must be >= 1. */
typedef struct conv_problem {
  int64_t n, h, w, c, k, r, s;
  int64_t stride_h, stride_w, pad_h, pad_w, dil_h, dil_w, groups;
  int32_t in_dtype, out_dtype;
} conv_problem;

/* The kernels stage 1 can run. Chosen from the problem and the degree
 * request alone (never from timing), so a degree and a workspace size
 * resolved ahead of a call hold for that call. Automatic choice never takes
 * CONV_KERNEL_FWD_TC_CLUSTER (on the 3x3 small-M layer it measured slower than
 * the two-stage form) nor CONV_KERNEL_WGRAD_DEPTHWISE_MMA (on the 7x7 layer it
 * measured slower than CONV_KERNEL_WGRAD_DEPTHWISE); the override selects
 * them. */
typedef enum conv_kernel {
  CONV_KERNEL_AUTO = 0,
  CONV_KERNEL_GENERIC = 1,           /* direct, CUDA cores: any shape and type */
  CONV_KERNEL_WGRAD_1X1_FFMA = 2,    /* fp32 1x1 weight gradient, FFMA tiles */
  CONV_KERNEL_WGRAD_1X1_TF32X3 = 3,  /* fp32 1x1 weight gradient, tcgen05 3xTF32 */
  CONV_KERNEL_FWD_TC = 4,            /* 16-bit forward, tcgen05 + TMA im2col */
  CONV_KERNEL_WGRAD_DEPTHWISE = 5,   /* depthwise weight gradient, CUDA cores */
  CONV_KERNEL_WGRAD_GROUPED = 6,     /* 4/8 channels per group, CUDA cores */
  CONV_KERNEL_FWD_TC_CLUSTER = 7,    /* 16-bit forward, the S <= 16 slices of a tile as one
                                        thread-block cluster folding through distributed
                                        shared memory [P2 "Changes": single-launch split-K]:
                                        no workspace, no stage 2 */
  CONV_KERNEL_DGRAD_TC = 8,          /* 16-bit, stride-1, ungrouped data gradient: the forward
                                        tensor-core kernel over dY with the filter rotated 180
                                        degrees and k and c swapped, read in place (MN-major) */
  CONV_KERNEL_FWD_DEPTHWISE = 9,     /* depthwise forward (C = K = groups, C even, filter
                                        width 3/5/7, W stride 1/2), CUDA cores, unsplit */
  CONV_KERNEL_FWD_GROUPED_TC = 10,   /* 16-bit grouped forward (Cg = Kg dividing 128, C % 128 = 0):
                                        each 128-channel block as a dense tensor-core forward with
                                        a block-diagonal filter written into the workspace */
  CONV_KERNEL_WGRAD_GROUPED_TC = 11, /* 16-bit grouped weight gradient (Cg = Kg in 2..32, C % 128 = 0,
                                        filter width <= 4): per 128-channel block and tap, the dense
                                        product on the tensor cores with MN-major operands, of which
                                        the diagonal group blocks are kept */
  CONV_KERNEL_WGRAD_TC = 12,         /* 16-bit dense weight gradient (one group, or Cg % 64 = 0 and
                                        Kg % 128 = 0; C, K >= 64 and multiples of 8): per filter tap
                                        the product dY^T X over the output pixels on the tensor
                                        cores, both operands MN-major straight from TMA boxes */
  CONV_KERNEL_DGRAD_DEPTHWISE = 13,  /* stride-1 depthwise data gradient: the depthwise forward
                                        kernels over dY with the filter's taps read backwards
                                        (turned 180 degrees), padding dil*(f-1)-pad; unsplit */
  CONV_KERNEL_DGRAD_GROUPED_TC = 14, /* stride-1 16-bit grouped data gradient (Cg = Kg dividing 128,
                                        C % 128 = 0): the block-diagonal grouped forward over dY
                                        with the turned filter written into the workspace */
  CONV_KERNEL_WGRAD_GROUPED_MMA = 15, /* 16-bit grouped weight gradient (Cg = Kg in 2..32, C % 64 = 0,
                                        unit stride and dilation, 1x1, 3 x (1..4) or 5 x (1..6)
                                        filters): warp-level m16n8k16 MMAs over input columns with
                                        the filter column applied as a shift of dY, so every product
                                        is a gradient element (8 or more channels per group) */
  CONV_KERNEL_FFMA = 16,             /* fp32, one group, C and K multiples of 4: implicit-GEMM FFMA
                                        tiles (128 x 128, 8 x 8 a thread) for the forward, the
                                        stride-1 data gradient (the turned problem, filter read in
                                        place) and the weight gradient (+ bias gradient) */
  CONV_KERNEL_WGRAD_DEPTHWISE_MMA = 17, /* 16-bit depthwise weight gradient (filters up to 7 x 7, unit
                                        stride and dilation, rows of at most 64 input and output
                                        columns, C % 8 = 0): per channel and output row, warp-level
                                        m16n8k16 MMAs of the filter rows' input rows against dY
                                        shifted by each filter column (a Toeplitz operand), rows
                                        transposed in shared memory; the bias summed from the
                                        transposed dY rows */
  CONV_KERNEL_FWD_GROUPED_MMA = 18,  /* 16-bit grouped forward (Cg = Kg = 4 or 8, C % 64 = 0, unit stride
                                        and dilation, 1x1 / 3x3 / 5x5 filters, Wo <= 64): per output
                                        row and 16 columns, warp-level m16n8k16 MMAs over pairs of taps
                                        with the tap as a pixel shift of X and the group's filter in
                                        registers; unsplit, fused epilogue supported */
  CONV_KERNEL_DGRAD_GROUPED_MMA = 19 /* the stride-1 grouped data gradient on the same kernel: the
                                        forward over dY with the turned filter read in place */
} conv_kernel;

/* What a call with these arguments would run. */
typedef struct conv_plan_info {
  int32_t kernel;            /* conv_kernel of stage 1 */
  int32_t split_k;           /* resolved degree S >= 1 */
  int32_t needs_fold;        /* 1 when stage 2 runs (S > 1, slices not folded in-launch) */
  int32_t ctas_per_sm;       /* resident stage-1 CTAs per SM the policy assumes */
  int64_t tiles;             /* output tiles of stage 1 */
  int64_t reduction_blocks;  /* reduction blocks; a pinned degree may not exceed it */
  int64_t ctas;              /* stage-1 work units = tiles * S (one CTA each; the 256-wide
                                tensor-core forward runs them on at most one persistent CTA
                                per SM) */
  uint64_t workspace_bytes;  /* bytes the call needs (0 without stage 2, except the grouped
                                forward's block-diagonal filter) */
  int32_t max_split;         /* largest degree a pinned request may ask of this kernel */
  int32_t fold_width;        /* f > 1: the call runs the width-folded problem (f adjacent W
                                positions as f*C channels, filter width S/f, W stride sw/f, on
                                the same memory), chosen when only it has a kernel faster than
                                the generic one; 1: no fold */
} conv_plan_info;

/* Human-readable name of a status. Never NULL. */
const char* conv_status_string(conv_status status);

/* Output extent (ho, wo) of a problem after validation. */
conv_status conv_output_dims(const conv_problem* p, int64_t* ho, int64_t* wo);

/* Resolve a degree request for this problem on a GPU with sm_count SMs
 * (pure host function). request -1 runs the auto policy
 * [P2 "Auto-deduced degree"], restated for this hardware:
 *  - target = sm_count x (resident stage-1 CTAs per SM of the chosen kernel);
 *  - forward: split only when the unsplit grid is under half the target and
 *    the reduction R*S*Cg is at least 512 deep, and never for a pointwise
 *    (1x1) forward; the degree is the largest power of two <= 32 (<= 16,
 *    the largest cluster, for the cluster form) with tiles x degree <=
 *    target, halved until every slice has >= 2 reduction blocks;
 *  - weight gradient (no policy on the pages): degree = floor(target / tiles)
 *    when tiles < target, at most half the reduction blocks (>= 2 blocks per
 *    slice) and at most 4096, else 1.
 * request 0 gives 1; request n >= 1 gives n if n <= reduction blocks (and
 * n <= 16 for the cluster form, else CONV_ERR_UNSUPPORTED). */
conv_status resolve_split_k_for(const conv_problem* p, conv_dir dir, int32_t request,
                                int32_t sm_count, int32_t* degree);

/* resolve_split_k_for on the current CUDA device (CONV_ERR_CUDA without one). */
conv_status resolve_split_k(const conv_problem* p, conv_dir dir, int32_t request, int32_t* degree);

/* Workspace bytes a call with this degree request needs: 0 when the degree
 * resolves to 1, else S x E x 4 rounded up to 256 bytes (E = output elements),
 * plus S x k x 4 (rounded up to 256) when with_bias and dir is the weight
 * gradient; the grouped forward's and grouped data gradient's tensor-core
 * paths add their block-diagonal filter (k x r x s x 128 elements of
 * in_dtype, rounded up to 256; c x r x s x 128 for the data gradient) in
 * front, at every degree. */
conv_status conv_workspace_bytes_for(const conv_problem* p, conv_dir dir, int32_t split_k,
                                     int32_t with_bias, int32_t sm_count, uint64_t* bytes);
conv_status conv_workspace_bytes(const conv_problem* p, conv_dir dir, int32_t split_k,
                                 int32_t with_bias, uint64_t* bytes);

/* The full plan for a call (kernel, degree, grid, workspace) on sm_count SMs. */
conv_status conv_describe_plan(const conv_problem* p, conv_dir dir, int32_t split_k,
                               int32_t with_bias, int32_t sm_count, conv_plan_info* info);

/* Forward [P2 "Two-stage split-K"]: y = conv(x, w). x, w in in_dtype, y in
 * out_dtype. ws may be NULL when the resolved degree is 1. */
conv_status conv_fwd(const conv_problem* p, const void* x, const void* w, void* y, void* ws,
                     uint64_t ws_bytes, int32_t split_k, void* stream);

/* Weight gradient [P1 "Motivation"; P3 "Technical Details"]: dw from x and
 * dy, in out_dtype. */
conv_status conv_wgrad(const conv_problem* p, const void* x, const void* dy, void* dw, void* ws,
                       uint64_t ws_bytes, int32_t split_k, void* stream);

/* A fused forward epilogue: y = min(max(conv(x, w) + bias[k], lo), hi),
 * with the bias added to the fp32 accumulator and one rounding into
 * out_dtype [P2 "Review follow-ups": bias / ReLU / clamp are the
 * non-identity epilogues]. The clamp gives the values it would give before
 * the rounding (the tensor-core forward clamps 16-bit outputs after it,
 * against the rounded bounds: rounding to nearest is monotone); a NaN sum
 * becomes lo (the identity epilogue leaves it NaN). bias is [k] in out_dtype, or NULL for none; ReLU is
 * {lo = 0, hi = +inf}; {-inf, +inf} with no bias is the identity. lo <= hi,
 * neither NaN. */
typedef struct conv_epilogue {
  const void* bias;
  float lo, hi;
} conv_epilogue;

/* Forward with a fused epilogue. A non-identity epilogue cannot be applied
 * per slice, so it runs unsplit [P2 "Review follow-ups": split-K rejects
 * it; "Auto-deduced degree": such specs resolve to 1]: split_k -1, 0 or 1
 * gives one slice, any other degree is CONV_ERR_INVALID_ARG; the workspace
 * is what conv_workspace_bytes reports at degree 1 (0 except for the grouped
 * forward's block-diagonal filter). An identity epilogue (or ep == NULL) is exactly
 * conv_fwd. */
conv_status conv_fwd_epilogue(const conv_problem* p, const void* x, const void* w, const conv_epilogue* ep,
                              void* y, void* ws, uint64_t ws_bytes, int32_t split_k, void* stream);

/* Data gradient: dx[n,h,w,c] = sum over k, r, s of dy[n,ho,wo,k] * w[k,r,s,c]
 * for the (ho, wo) with ho*sh + r*dh - ph = h and wo*sw + s*dw - pw = w (the
 * forward's taps read backwards), k running over the output channels of c's
 * group. dy and w in in_dtype, dx [n,h,w,c] in out_dtype. The reduction
 * (r, s, k) splits like the forward's; the workspace is the slabs (none at
 * degree 1), after the turned block-diagonal filter of the grouped
 * tensor-core path (see conv_workspace_bytes). */
conv_status conv_dgrad(const conv_problem* p, const void* dy, const void* w, void* dx, void* ws,
                       uint64_t ws_bytes, int32_t split_k, void* stream);

/* Weight and bias gradient together [P1 "Motivation": weight.grad and
 * bias.grad]: dw as conv_wgrad, db[k] = sum of dy over n, ho, wo, both in
 * out_dtype, from one pass over dy. */
conv_status conv_wgrad_bias(const conv_problem* p, const void* x, const void* dy, void* dw,
                            void* db, void* ws, uint64_t ws_bytes, int32_t split_k, void* stream);

/* The two stages of a call, enqueued separately [P2 "Two-stage split-K";
 * "Benchmark": both stages are bound and launched one after the other].
 * conv_stage1 followed by conv_stage2 on the same stream, with the same
 * arguments, is exactly conv_fwd (dir = FWD, b = w, db = NULL), conv_wgrad
 * (dir = WGRAD, b = dy, db = NULL), conv_wgrad_bias (db != NULL) or
 * conv_dgrad (dir = DGRAD, x = dy, b = w, out = dx, db = NULL).
 * conv_stage1 writes the slabs (or, at degree 1, the outputs);
 * conv_stage2 folds the slabs into out (and db) and enqueues nothing when the
 * degree resolves to 1. Each validates all of its arguments. */
conv_status conv_stage1(const conv_problem* p, conv_dir dir, const void* x, const void* b, void* out,
                        void* db, void* ws, uint64_t ws_bytes, int32_t split_k, void* stream);
conv_status conv_stage2(const conv_problem* p, conv_dir dir, void* out, void* db, void* ws,
                        uint64_t ws_bytes, int32_t split_k, void* stream);

/* Batch split count [P1 "Technical Details"]: the smallest m with
 * m * max_n >= n, i.e. the integer ceiling (n + max_n - 1) / max_n, or 1 for
 * n = 0. Returns -1 when n < 0 or max_n < 1. The library itself never splits
 * a batch (all indexing is 64-bit); this is the exact form of the count for
 * callers that must. */
int64_t conv_batch_split_count(int64_t n, int64_t max_n);

/* Weight + bias gradient for callers that cannot allocate device memory.
 * The pages have no counterpart to this entry point; it exists for users of
 * this library. Some callers cannot call cudaMalloc where they run the
 * convolution: their device memory is owned by a framework's pool, or they
 * run at plugin/enqueue time in a runtime that forbids allocation after
 * set-up, and they may hold no spare workspace either. This call computes
 * exactly what conv_wgrad_bias computes, with the split-K slabs placed in
 * one fixed device array owned by the library (8 MiB on every GPU that loads
 * the library, held until the process exits) instead of a caller workspace.
 *  - The caller still passes x, dy, dw and db (device pointers, 16-byte
 *    aligned); nothing is allocated or freed by this call.
 *  - A degree whose slabs need more than 8 MiB (conv_workspace_bytes with
 *    with_bias = 1 above 8388608) is rejected with
 *    CONV_ERR_WORKSPACE_TOO_SMALL before anything is enqueued.
 *  - Every call looks up the array's device address in the current context
 *    (cudaGetSymbolAddress). The first call on a device loads the library's
 *    module there, which commits the array's 8 MiB of device memory: that
 *    first call is a one-time allocation by the CUDA runtime and can fail
 *    with CONV_ERR_CUDA when the device memory is exhausted, so make it
 *    during set-up and before any stream capture. A call with an empty batch
 *    (p->n = 0, NULL tensors allowed where they hold no elements) does only
 *    that set-up and writes dw = db = 0.
 *  - Every call shares the one array. Its contents between calls do not
 *    matter (every slab element is written before it is read), but two calls
 *    whose kernels overlap on the GPU (different streams, no ordering) race
 *    on it; order such calls on one stream or with events. */
conv_status conv_wgrad_bias_static_ws(const conv_problem* p, const void* x, const void* dy, void* dw,
                                      void* db, int32_t split_k, void* stream);

/* Device-side error word of the current device (synchronous read). The
 * tensor-core kernels bound every pipeline wait; a wait that gives up sets
 * bit 0 (1 = a pipeline wait timed out; that call's outputs are invalid) and
 * the kernel ends early instead of hanging. clear != 0 resets the word. */
conv_status conv_device_errors(uint32_t* flags, int32_t clear);

/* Testing aid for the bounded waits: one CTA waits on a pipeline barrier that
 * nothing ever completes, giving up after limit_ns (1 .. 1e9 ns) of global
 * time. The kernel returns (no fault, no hang), bit 0 of the device error
 * word is set (see conv_device_errors) and *gave_up = 1 when the wait gave up
 * and raised its abort word. Synchronises the stream. */
conv_status conv_selftest_wait_timeout(uint64_t limit_ns, uint32_t* gave_up, void* stream);

/* Testing aid: force stage 1 to one kernel (CONV_KERNEL_AUTO restores the
 * normal choice). The forced kernel runs the problem as given (no width fold
 * is tried); a forced kernel that cannot take it makes the call fail with
 * CONV_ERR_UNSUPPORTED. Process-wide, not thread-safe. */
conv_status conv_set_kernel_override(int32_t kernel);

#ifdef __cplusplus
}
#endif

#endif /* CONV_IGEMM_H */
