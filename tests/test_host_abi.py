"""Host-side logic of the C ABI, run without a GPU: exports, validation, the
split-K planner, workspace arithmetic and the batch-split count."""
import ctypes

import pytest

import implicit_gemm_convolution_nhwc_gb300 as cig
from implicit_gemm_convolution_nhwc_gb300 import BF16, DIR_FWD, DIR_WGRAD, F16, F32, Problem

SMS = 152

CONFIG1 = Problem(n=4, h=16, w=16, c=8, k=16)
CONFIG2 = Problem(n=64, h=512, w=512, c=96, k=64)
CONFIG3 = Problem(n=1, h=14, w=14, c=2048, k=512, r=3, s=3, pad_h=1, pad_w=1, in_dtype=BF16, out_dtype=BF16)
CONFIG4 = Problem(n=32, h=56, w=56, c=384, k=384, r=7, s=7, pad_h=3, pad_w=3, groups=384,
                  in_dtype=BF16, out_dtype=BF16)
CONFIG5A = Problem(n=64, h=28, w=28, c=512, k=512, r=3, s=3, pad_h=1, pad_w=1, groups=64,
                   in_dtype=F16, out_dtype=F16)
CONFIG5B = Problem(n=64, h=28, w=28, c=512, k=512, r=3, s=3, pad_h=1, pad_w=1, groups=128,
                   in_dtype=F16, out_dtype=F16)
CONFIGS = [(CONFIG1, DIR_WGRAD), (CONFIG2, DIR_WGRAD), (CONFIG3, DIR_FWD), (CONFIG4, DIR_WGRAD),
           (CONFIG5A, DIR_WGRAD), (CONFIG5B, DIR_WGRAD)]


@pytest.fixture(autouse=True)
def _no_override():
    cig.set_kernel_override("auto")
    yield
    cig.set_kernel_override("auto")


def test_library_exports_every_declared_symbol():
    import re
    import os
    lib = cig.load()
    header = open(os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "conv_igemm.h")).read()
    declared = set(re.findall(r"^\S.*?\b(\w+)\s*\(", header, re.M)) - {"if", "while"}
    declared = {d for d in declared if d.startswith(("conv_", "resolve_"))}
    assert declared == set(cig.EXPORTS)
    for name in declared:
        assert hasattr(lib, name)
    assert lib.conv_status_string(0) == b"CONV_OK"
    assert lib.conv_status_string(99) == b"CONV_ERR_UNKNOWN"


def test_output_dims():
    assert cig.output_dims(CONFIG3) == (14, 14)
    assert cig.output_dims(CONFIG4) == (56, 56)
    assert cig.output_dims(Problem(n=1, h=9, w=10, c=1, k=1, r=3, s=2, stride_h=2, stride_w=3,
                                   pad_h=1, pad_w=0, dil_h=2, dil_w=1)) == (4, 3)


@pytest.mark.parametrize("bad", [
    dict(n=-1), dict(h=0), dict(c=0), dict(k=0), dict(r=0), dict(stride_h=0), dict(dil_w=0),
    dict(pad_h=-1), dict(groups=0), dict(groups=3), dict(in_dtype=3), dict(in_dtype=F16, out_dtype=BF16),
    dict(h=2, w=2, r=5, s=5),
])
def test_validation_rejects(bad):
    base = dict(n=2, h=8, w=8, c=8, k=4, r=3, s=3, pad_h=1, pad_w=1, groups=2)
    base.update(bad)
    with pytest.raises(cig.ConvError) as e:
        cig.resolve_split_k(Problem(**base), DIR_WGRAD, -1, sm_count=SMS)
    assert e.value.status == 1


def test_overflow_is_loud():
    huge = Problem(n=1 << 30, h=1 << 20, w=1 << 20, c=64, k=64)
    with pytest.raises(cig.ConvError) as e:
        cig.resolve_split_k(huge, DIR_WGRAD, -1, sm_count=SMS)
    assert e.value.status == 4
    with pytest.raises(cig.ConvError) as e:
        cig.resolve_split_k(Problem(n=1, h=1 << 62, w=1, c=1, k=1, pad_h=1 << 62), DIR_FWD, 0, sm_count=SMS)
    assert e.value.status == 4


def test_degree_request_semantics():
    p = CONFIG1
    plan = cig.describe_plan(p, DIR_WGRAD, 1, sm_count=SMS)
    assert cig.resolve_split_k(p, DIR_WGRAD, 0, sm_count=SMS) == 1
    assert cig.resolve_split_k(p, DIR_WGRAD, 3, sm_count=SMS) == 3
    blocks = plan["reduction_blocks"]
    assert cig.resolve_split_k(p, DIR_WGRAD, blocks, sm_count=SMS) == blocks
    for bad in (blocks + 1, -2, -100):
        with pytest.raises(cig.ConvError) as e:
            cig.resolve_split_k(p, DIR_WGRAD, bad, sm_count=SMS)
        assert e.value.status == 1
    with pytest.raises(cig.ConvError):
        cig.resolve_split_k(p, 7, -1, sm_count=SMS)


def test_auto_is_deterministic_and_within_bounds():
    for p, d in CONFIGS:
        for sms in (1, 2, 16, 148, 152, 160):
            a = cig.describe_plan(p, d, -1, sm_count=sms)
            b = cig.describe_plan(p, d, -1, sm_count=sms)
            assert a == b
            S = a["split_k"]
            assert 1 <= S <= max(1, a["reduction_blocks"])
            assert a["ctas"] == a["tiles"] * S
            assert a["needs_fold"] == (S > 1 and a["kernel_name"] != "fwd_tc_cluster")


def test_forward_policy_properties():
    """Forward auto degree ("Auto-deduced degree" of the split-K forward page):
    power of two <= 32 (<= 16 for the cluster form), 1 for a grid >= half the
    target, a reduction < 512 or a pointwise problem, >= 2 reduction blocks
    per slice."""
    shapes = [CONFIG3,
              Problem(n=1, h=7, w=7, c=512, k=512, r=7, s=7, pad_h=3, pad_w=3, in_dtype=BF16, out_dtype=BF16),
              Problem(n=1, h=14, w=14, c=2048, k=512, in_dtype=BF16, out_dtype=BF16),   # pointwise
              Problem(n=1, h=14, w=14, c=16, k=64, r=3, s=3, pad_h=1, pad_w=1, in_dtype=BF16, out_dtype=BF16),
              Problem(n=64, h=56, w=56, c=256, k=256, r=3, s=3, pad_h=1, pad_w=1, in_dtype=BF16, out_dtype=BF16)]
    for p in shapes:
        for sms in (8, 76, 152):
            info = cig.describe_plan(p, DIR_FWD, -1, sm_count=sms)
            S, tiles, blocks = info["split_k"], info["tiles"], info["reduction_blocks"]
            target = sms * info["ctas_per_sm"]
            depth = p.r * p.s * (p.c // p.groups)
            cap = 16 if info["kernel_name"] == "fwd_tc_cluster" else 32
            assert S & (S - 1) == 0 and S <= cap
            if p.r == 1 and p.s == 1 or 2 * tiles >= target or depth < 512:
                assert S == 1
            else:
                assert tiles * S <= target and blocks >= 2 * S
                assert S == cap or tiles * 2 * S > target or blocks < 4 * S


def test_wgrad_policy_fills_the_gpu_in_whole_waves():
    info = cig.describe_plan(CONFIG2, DIR_WGRAD, -1, with_bias=True, sm_count=SMS)
    target = SMS * info["ctas_per_sm"]
    assert info["ctas"] <= target and info["ctas"] > target - info["tiles"]
    assert info["reduction_blocks"] >= 2 * info["split_k"]


def test_workspace_bytes_arithmetic():
    for p, d in CONFIGS:
        for req in (-1, 0, 1, 2, 5):
            for bias in (False, True):
                info = cig.describe_plan(p, d, req, with_bias=bias, sm_count=SMS)
                S = info["split_k"]
                ho, wo = p.out_hw
                E = p.n * ho * wo * p.k if d == DIR_FWD else p.k * p.r * p.s * (p.c // p.groups)
                r256 = lambda v: (v + 255) // 256 * 256  # noqa: E731
                fold = S > 1 and info["kernel_name"] != "fwd_tc_cluster"
                want = 0 if not fold else r256(S * E * 4) + (r256(S * p.k * 4) if bias and d == DIR_WGRAD else 0)
                assert info["workspace_bytes"] == want
                assert cig.workspace_bytes(p, d, req, bias, sm_count=SMS) == want


def test_forward_cluster_form_selection():
    """Single-launch split-K ("feat(rocke): split-K forward implicit-GEMM
    convolution on gfx1250", "Changes"): only through the override; degrees
    1..16, no workspace and no fold; past 16 it is refused. Automatic choice
    keeps the two-stage form."""
    auto = cig.describe_plan(CONFIG3, DIR_FWD, -1, sm_count=SMS)
    assert auto["kernel_name"] == "fwd_tc" and auto["split_k"] == 32 and auto["needs_fold"] == 1
    assert auto["max_split"] == auto["reduction_blocks"] == 288
    cig.set_kernel_override("fwd_tc_cluster")
    info = cig.describe_plan(CONFIG3, DIR_FWD, -1, sm_count=SMS)
    assert (info["kernel_name"], info["split_k"], info["workspace_bytes"], info["needs_fold"]) == (
        "fwd_tc_cluster", 16, 0, 0)
    assert info["max_split"] == 16
    for req in (0, 1, 2, 3, 9, 16):
        info = cig.describe_plan(CONFIG3, DIR_FWD, req, sm_count=SMS)
        assert (info["kernel_name"], info["split_k"], info["workspace_bytes"]) == ("fwd_tc_cluster", max(req, 1), 0)
        assert cig.workspace_bytes(p=CONFIG3, direction=DIR_FWD, split_k=req, sm_count=SMS) == 0
    for req, status in ((17, 2), (288, 2), (289, 1)):
        with pytest.raises(cig.ConvError) as e:
            cig.describe_plan(CONFIG3, DIR_FWD, req, sm_count=SMS)
        assert e.value.status == status
    with pytest.raises(cig.ConvError) as e:
        cig.describe_plan(CONFIG4, DIR_WGRAD, -1, sm_count=SMS)
    assert e.value.status == 2


def test_dgrad_plans():
    """Data gradient: the tensor-core path (16-bit, stride 1, one group) reads
    the filter in place, so its workspace is the slabs alone; grouped and
    depthwise stride-1 problems take the turned-filter forwards; strided ones
    take the generic kernel."""
    r256 = lambda v: (v + 255) // 256 * 256  # noqa: E731
    p = CONFIG3
    E = p.n * p.h * p.w * p.c
    for req in (-1, 1, 2, 8):
        info = cig.describe_plan(p, cig.DIR_DGRAD, req, sm_count=SMS)
        S = info["split_k"]
        assert info["kernel_name"] == "dgrad_tc" and info["needs_fold"] == (S > 1)
        assert info["workspace_bytes"] == (r256(S * E * 4) if S > 1 else 0)
        assert cig.workspace_bytes(p, cig.DIR_DGRAD, req, sm_count=SMS) == info["workspace_bytes"]
    auto = cig.describe_plan(p, cig.DIR_DGRAD, -1, sm_count=SMS)
    assert auto["split_k"] & (auto["split_k"] - 1) == 0 and auto["ctas"] <= SMS * auto["ctas_per_sm"]
    strided = Problem(n=2, h=9, w=11, c=128, k=128, r=3, s=3, stride_h=2, stride_w=2, pad_h=1, pad_w=1,
                      in_dtype=BF16, out_dtype=BF16)
    info = cig.describe_plan(strided, cig.DIR_DGRAD, 1, sm_count=SMS)
    assert info["kernel_name"] == "generic" and info["workspace_bytes"] == 0
    # grouped and depthwise data gradients at stride 1 take the turned-filter forwards: 4 or 8 channels
    # per group the MMA kernel (filter read in place, unsplit), else (Cg = Kg dividing 128) the
    # block-diagonal one (the turned block-diagonal filter in the workspace)
    info = cig.describe_plan(CONFIG5A, cig.DIR_DGRAD, -1, sm_count=SMS)
    assert (info["kernel_name"], info["split_k"], info["workspace_bytes"]) == ("dgrad_grouped_mma", 1, 0)
    cpg2 = Problem(n=2, h=8, w=8, c=128, k=128, r=5, s=5, pad_h=2, pad_w=2, groups=64, in_dtype=F16, out_dtype=F16)
    info = cig.describe_plan(cpg2, cig.DIR_DGRAD, -1, sm_count=SMS)
    assert info["kernel_name"] == "dgrad_grouped_tc"
    assert info["workspace_bytes"] == r256(cpg2.c * 25 * 128 * 2)  # the turned block-diagonal filter
    info = cig.describe_plan(CONFIG4, cig.DIR_DGRAD, -1, sm_count=SMS)
    assert (info["kernel_name"], info["split_k"], info["workspace_bytes"]) == ("dgrad_depthwise", 1, 0)
    strided_dw = Problem(n=2, h=9, w=9, c=64, k=64, r=3, s=3, stride_h=2, stride_w=2, pad_h=1, pad_w=1,
                         groups=64, in_dtype=BF16, out_dtype=BF16)
    assert cig.describe_plan(strided_dw, cig.DIR_DGRAD, -1, sm_count=SMS)["kernel_name"] == "generic"
    # the planner ignores with_bias outside the weight gradient
    assert cig.describe_plan(p, cig.DIR_DGRAD, -1, with_bias=True, sm_count=SMS) == auto
    with pytest.raises(cig.ConvError) as e:
        cig.describe_plan(p, 3, -1, sm_count=SMS)
    assert e.value.status == 1


def test_empty_batch_plans_one_slice():
    p = Problem(n=0, h=8, w=8, c=8, k=8)
    assert cig.resolve_split_k(p, DIR_WGRAD, -1, sm_count=SMS) == 1
    assert cig.resolve_split_k(p, DIR_WGRAD, 1, sm_count=SMS) == 1
    with pytest.raises(cig.ConvError):
        cig.resolve_split_k(p, DIR_WGRAD, 2, sm_count=SMS)


def test_batch_split_count_exhaustive():
    """Exact integer ceiling (PR #11188, "Technical Details"): minimal m with m * max_n >= n."""
    for n in range(0, 2001):
        for max_n in range(1, 2001, 7):
            m = cig.batch_split_count(n, max_n)
            assert m * max_n >= n and (m == 1 or (m - 1) * max_n < n)
    assert cig.batch_split_count(-1, 3) == -1 and cig.batch_split_count(3, 0) == -1
    big = (1 << 62) + 1
    assert cig.batch_split_count(big, 1 << 61) == 3


def test_kernel_override():
    assert cig.describe_plan(CONFIG1, DIR_WGRAD, -1, sm_count=SMS)["kernel_name"] != "generic"
    cig.set_kernel_override("generic")
    assert cig.describe_plan(CONFIG1, DIR_WGRAD, -1, sm_count=SMS)["kernel_name"] == "generic"
    cig.set_kernel_override("wgrad_1x1_ffma")
    with pytest.raises(cig.ConvError) as e:
        cig.describe_plan(CONFIG3, DIR_FWD, -1, sm_count=SMS)
    assert e.value.status == 2
    with pytest.raises(cig.ConvError):
        cig.set_kernel_override(42)


def test_calls_validate_before_touching_the_device():
    lib = cig.load()
    p = cig._cp(CONFIG1)
    null = ctypes.c_void_p(0)
    # NULL problem, NULL tensors, misaligned pointer: rejected without a device
    assert lib.conv_wgrad(None, null, null, null, null, 0, -1, null) == 1
    assert lib.conv_wgrad(p, null, null, null, null, 0, -1, null) == 1
    assert lib.conv_wgrad_bias(p, 16, 16, 16, None, None, 0, -1, None) == 1
    assert lib.conv_fwd(p, 18, 32, 32, None, 0, -1, None) == 5
    assert lib.conv_wgrad(p, 16, 16, 16, None, 0, -3, None) == 1


def test_fused_epilogue_validation_without_a_device():
    """conv_fwd_epilogue: bounds and bias alignment are checked before anything else runs;
    a non-identity epilogue is never split ("feat(rocke): split-K forward implicit-GEMM
    convolution on gfx1250", "Review follow-ups")."""
    lib = cig.load()
    p = cig._cp(CONFIG3)
    inf = float("inf")
    ep = cig._CEpilogue(None, 1.0, 0.0)          # lo > hi
    assert lib.conv_fwd_epilogue(p, 16, 16, ctypes.byref(ep), 16, None, 0, -1, None) == 1
    ep = cig._CEpilogue(None, float("nan"), inf)  # NaN bound
    assert lib.conv_fwd_epilogue(p, 16, 16, ctypes.byref(ep), 16, None, 0, -1, None) == 1
    ep = cig._CEpilogue(17, 0.0, inf)            # bf16 bias at an odd address
    assert lib.conv_fwd_epilogue(p, 16, 16, ctypes.byref(ep), 16, None, 0, -1, None) == 5
    ep = cig._CEpilogue(None, 0.0, inf)          # ReLU with a pinned split: rejected
    assert lib.conv_fwd_epilogue(p, 16, 16, ctypes.byref(ep), 16, None, 0, 4, None) == 1
    ep = cig._CEpilogue(None, 0.0, inf)          # ReLU with NULL tensors
    assert lib.conv_fwd_epilogue(p, None, None, ctypes.byref(ep), None, None, 0, -1, None) == 1


def test_selftest_arguments_checked_without_a_device():
    lib = cig.load()
    out = ctypes.c_uint32()
    assert lib.conv_selftest_wait_timeout(0, ctypes.byref(out), None) == 1           # no limit
    assert lib.conv_selftest_wait_timeout(2_000_000_000, ctypes.byref(out), None) == 1  # over 1 s
    assert lib.conv_selftest_wait_timeout(1000, None, None) == 1


def dw(**kw):
    """A 16-bit depthwise problem (C = K = groups)."""
    base = dict(n=2, h=12, w=14, c=64, r=7, s=7, pad_h=3, pad_w=3, in_dtype=BF16, out_dtype=BF16)
    base.update(kw)
    return Problem(k=base["c"], groups=base["c"], **base)


def test_depthwise_ring_selection():
    """Which depthwise shapes the row-ring kernels take (16-bit, square 3/5/7 filters, unit stride and
    dilation, pad_w <= F-1, C % 8 == 0 and C >= 64, rows of at most 256 columns that fit the ring),
    told apart by what the plan reports: the weight gradient's shared-memory form needs C % 64 == 0
    and 16-bit inputs; the forward's shared-weight form runs 4 CTAs per SM, the ring form 1."""
    wg = lambda p: cig.describe_plan(p, DIR_WGRAD, -1, sm_count=SMS)  # noqa: E731
    fw = lambda p: cig.describe_plan(p, DIR_FWD, -1, sm_count=SMS)  # noqa: E731
    # C = 72: only the ring takes the weight gradient (two 64-channel tiles, the last 8 wide)
    info = wg(dw(c=72))
    assert info["kernel_name"] == "wgrad_depthwise" and info["tiles"] == 2 and info["ctas_per_sm"] == 1
    assert fw(dw(c=72))["kernel_name"] == "fwd_depthwise" and fw(dw(c=72))["ctas_per_sm"] == 1
    # C % 8 != 0 or C < 64: neither TMA ring; the weight gradient falls to the generic kernel, the
    # forward to its shared-weight form
    for c in (34, 32):
        assert wg(dw(c=c))["kernel_name"] == "generic"
        assert fw(dw(c=c))["kernel_name"] == "fwd_depthwise" and fw(dw(c=c))["ctas_per_sm"] == 4
    # fp32 inputs: no ring (and no shared-memory weight-gradient form)
    assert wg(dw(in_dtype=F32, out_dtype=F32))["kernel_name"] == "generic"
    assert fw(dw(in_dtype=F32, out_dtype=F32))["ctas_per_sm"] == 4
    # pad_w = F: past the ring's padding; C % 64 == 0 keeps the shared-memory weight-gradient form
    p = dw(r=3, s=3, pad_h=1, pad_w=3)
    assert wg(p)["kernel_name"] == "wgrad_depthwise" and fw(p)["ctas_per_sm"] == 4
    # non-square and strided filters: the forward's shared-weight form
    assert fw(dw(r=3, s=7, pad_h=1))["ctas_per_sm"] == 4
    assert fw(dw(r=3, s=3, pad_h=1, pad_w=1, stride_w=2))["ctas_per_sm"] == 4
    # a row too wide for the forward's ring (28 rows of 64 channels x W columns) but not for the
    # weight gradient's (whose ring is shallower)
    wide = dw(h=20, w=80)
    assert fw(wide)["ctas_per_sm"] == 4 and wg(wide)["ctas_per_sm"] == 1
    # the ring grids: the forward spreads (n, ho) rows over about one CTA per SM
    info = fw(CONFIG4)
    assert info["ctas_per_sm"] == 1 and info["ctas"] == 150 and info["split_k"] == 1
    assert cig.workspace_bytes(CONFIG4, DIR_FWD, -1, sm_count=SMS) == 0


SUPPLEMENT = Problem(n=64, h=56, w=56, c=256, k=256, r=3, s=3, pad_h=1, pad_w=1, in_dtype=BF16, out_dtype=BF16)


def test_depthwise_mma_wgrad_admission():
    """Which depthwise weight gradients the MMA kernel (reached through the override only: it measured
    slower than the ring kernel) takes: 16-bit, filters up to 7 x 7 (any R, S), unit stride and
    dilation, pad <= F - 1, rows of at most 64 input and output columns, C % 8 == 0; 64 channels a CTA,
    split-K over the (n, ho) rows. Automatic choice keeps the ring kernel."""
    wg = lambda p: cig.describe_plan(p, DIR_WGRAD, -1, sm_count=SMS)  # noqa: E731
    assert wg(CONFIG4)["kernel_name"] == "wgrad_depthwise"
    cig.set_kernel_override("wgrad_depthwise_mma")
    try:
        info = wg(CONFIG4)
        assert info["kernel_name"] == "wgrad_depthwise_mma" and info["tiles"] == 6 and info["ctas_per_sm"] == 1
        assert info["reduction_blocks"] == 32 * 56 and info["ctas"] == 6 * info["split_k"] <= SMS
        for p in (dw(r=3, s=5, pad_h=1, pad_w=2), dw(r=1, s=1, pad_h=0, pad_w=0), dw(w=64), dw(w=58, pad_w=6),
                  dw(c=8), dw(in_dtype=F16, out_dtype=F32)):
            assert wg(p)["kernel_name"] == "wgrad_depthwise_mma", p
        # rows past 64 columns (input or output), a 9-wide filter, padding F, stride or dilation 2, fp32
        # inputs, C % 8 != 0: not this kernel
        for p in (dw(w=65), dw(w=59, pad_w=6), dw(r=9, s=9, pad_h=4, pad_w=4), dw(r=3, s=3, pad_h=1, pad_w=3),
                  dw(stride_w=2), dw(dil_h=2), dw(in_dtype=F32, out_dtype=F32), dw(c=12)):
            with pytest.raises(RuntimeError):
                wg(p)
    finally:
        cig.set_kernel_override("auto")


def test_grouped_mma_forward_selection():
    """Which grouped forwards (and stride-1 data gradients) the MMA kernel takes: 16-bit, Cg = Kg = 4 or
    8, C % 64 == 0, unit stride and dilation, 1x1 / 3x3 / 5x5 filters with pad <= F - 1, at most 64
    output columns; unsplit, about two CTAs per SM over the 64-channel blocks, no workspace."""
    fw = lambda p: cig.describe_plan(p, DIR_FWD, -1, sm_count=SMS)  # noqa: E731
    dg = lambda p: cig.describe_plan(p, cig.DIR_DGRAD, -1, sm_count=SMS)  # noqa: E731

    def grp(**kw):
        base = dict(n=2, h=12, w=14, c=128, k=128, r=3, s=3, pad_h=1, pad_w=1, groups=16, in_dtype=F16,
                    out_dtype=F16)
        base.update(kw)
        return Problem(**base)
    for p in (CONFIG5A, CONFIG5B, grp(), grp(groups=32), grp(r=1, s=1, pad_h=0, pad_w=0), grp(r=5, s=5, pad_h=2),
              grp(w=64), grp(in_dtype=BF16, out_dtype=F32)):
        info = fw(p)
        assert (info["kernel_name"], info["split_k"], info["workspace_bytes"]) == ("fwd_grouped_mma", 1, 0), p
        assert info["ctas"] <= 2 * SMS + p.c // 64 and info["ctas_per_sm"] == 2
        assert dg(p)["kernel_name"] == "dgrad_grouped_mma", p
    info = fw(CONFIG5A)
    assert info["ctas"] == 304  # 8 channel blocks x 38 runs of (n, ho) rows (a multiple of the step)
    # 2 or 16 channels per group, C % 64 != 0, stride 2, a 7x7 filter, 65 output columns, fp32: not this
    # kernel (the data gradient at stride 2 is not a forward)
    for p in (grp(groups=64), grp(groups=8), grp(c=96, k=96, groups=12), grp(stride_h=2, stride_w=2),
              grp(r=7, s=7, pad_h=3, pad_w=3), grp(w=65), grp(in_dtype=F32, out_dtype=F32)):
        assert fw(p)["kernel_name"] != "fwd_grouped_mma", p
    assert dg(grp(r=3, s=3, pad_h=1, pad_w=1, dil_h=2, dil_w=2))["kernel_name"] != "dgrad_grouped_mma"


def test_dense_wgrad_tensor_core_selection():
    """Which weight gradients the dense tensor-core kernel takes (16-bit, one group or Cg % 64 == 0 with
    Kg % 128 == 0, C and K >= 64 and multiples of 8), and its tiling: 256 output channels x up to 256
    input channels x one tap per CTA, split-K over pixel blocks to fill the SMs once."""
    r256 = lambda v: (v + 255) // 256 * 256  # noqa: E731
    wg = lambda p, req=-1, bias=True: cig.describe_plan(p, DIR_WGRAD, req, with_bias=bias, sm_count=SMS)  # noqa
    info = wg(SUPPLEMENT)
    # 9 taps x one 256 x 256 tile; 56x56 images in 8x8 pixel blocks (no padded row): 64 * 49 blocks
    assert (info["kernel_name"], info["tiles"], info["reduction_blocks"]) == ("wgrad_tc", 9, 64 * 49)
    assert info["split_k"] == SMS // 9 and info["ctas"] == 9 * (SMS // 9) and info["ctas_per_sm"] == 1
    E = 256 * 9 * 256
    assert info["workspace_bytes"] == r256(info["split_k"] * E * 4) + r256(info["split_k"] * 256 * 4)
    assert wg(SUPPLEMENT, bias=False)["workspace_bytes"] == r256(info["split_k"] * E * 4)
    assert wg(SUPPLEMENT, 1)["workspace_bytes"] == 0 and wg(SUPPLEMENT, 1)["needs_fold"] == 0
    # the small-M layer's weight gradient: 2 x 8 x 9 = 144 tiles fill the GPU unsplit
    info = wg(CONFIG3)
    assert (info["kernel_name"], info["tiles"], info["split_k"]) == ("wgrad_tc", 144, 1)
    # 1x1 16-bit, groups with Kg % 128 == 0, fp16
    assert wg(Problem(n=4, h=16, w=16, c=128, k=256, in_dtype=F16, out_dtype=F32))["kernel_name"] == "wgrad_tc"
    g2 = Problem(n=2, h=12, w=12, c=128, k=256, r=3, s=3, pad_h=1, pad_w=1, groups=2, in_dtype=BF16,
                 out_dtype=BF16)
    info = wg(g2)
    assert info["kernel_name"] == "wgrad_tc" and info["tiles"] == 2 * 9
    # not taken: fp32 (the FFMA tiles take it), fewer than 64 channels, channels not a multiple of 8,
    # groups with Kg = 64
    assert wg(Problem(n=4, h=16, w=16, c=128, k=256, r=3, s=3, pad_h=1, pad_w=1))["kernel_name"] == "ffma"
    for c, k in ((32, 128), (128, 32), (100, 128)):
        p = Problem(n=2, h=8, w=8, c=c, k=k, r=3, s=3, pad_h=1, pad_w=1, in_dtype=BF16, out_dtype=BF16)
        assert wg(p)["kernel_name"] == "generic", (c, k)
    g8 = Problem(n=2, h=8, w=8, c=512, k=512, r=3, s=3, pad_h=1, pad_w=1, groups=8, in_dtype=BF16, out_dtype=BF16)
    assert wg(g8)["kernel_name"] == "generic"
    # the grouped configurations take the warp-level MMA kernel: 8 channel blocks of 64, split over the SMs
    for cfg in (CONFIG5A, CONFIG5B):
        info = wg(cfg)
        assert (info["kernel_name"], info["tiles"], info["reduction_blocks"]) == ("wgrad_grouped_mma", 8, 64 * 28)
        assert info["split_k"] == SMS // 8 and info["ctas_per_sm"] == 1
    # strided grouped problems keep the block-diagonal tensor-core kernel
    strided = Problem(n=1, h=12, w=12, c=128, k=128, groups=8, r=3, s=3, stride_h=2, stride_w=2, pad_h=1, pad_w=1,
                      in_dtype=F16, out_dtype=F16)
    assert wg(strided)["kernel_name"] == "wgrad_grouped_tc"


def test_fp32_ffma_tiles_selection():
    """fp32 problems with one group and channel counts that are multiples of 4 take the FFMA implicit-GEMM
    tiles in every direction (the data gradient at stride 1); others keep the generic kernel."""
    p = Problem(n=4, h=16, w=16, c=128, k=256, r=3, s=3, pad_h=1, pad_w=1)
    for d, tiles in ((DIR_FWD, 8 * 2), (cig.DIR_DGRAD, 8 * 1), (DIR_WGRAD, 2 * 1 * 9)):
        info = cig.describe_plan(p, d, -1, sm_count=SMS)
        assert info["kernel_name"] == "ffma" and info["tiles"] == tiles and info["ctas_per_sm"] == 2, (d, info)
        assert info["ctas"] <= 2 * SMS, (d, info)
    strided = Problem(n=2, h=9, w=9, c=16, k=16, r=3, s=3, stride_h=2, stride_w=2, pad_h=1, pad_w=1)
    assert cig.describe_plan(strided, cig.DIR_DGRAD, -1, sm_count=SMS)["kernel_name"] == "generic"
    assert cig.describe_plan(strided, DIR_FWD, -1, sm_count=SMS)["kernel_name"] == "ffma"
    for bad in (Problem(n=2, h=8, w=8, c=6, k=8, r=3, s=3), Problem(n=2, h=8, w=8, c=8, k=8, r=3, s=3, groups=2),
                Problem(n=2, h=8, w=8, c=8, k=6, r=3, s=3)):
        assert cig.describe_plan(bad, DIR_FWD, -1, sm_count=SMS)["kernel_name"] == "generic"
    # 16-bit inputs never take the fp32 tiles
    b = Problem(n=2, h=8, w=8, c=8, k=8, r=3, s=3, in_dtype=BF16, out_dtype=BF16)
    assert cig.describe_plan(b, DIR_FWD, -1, sm_count=SMS)["kernel_name"] != "ffma"
    # the tiles' spatial index arithmetic is 32-bit: a row whose padded width reaches 2^31, or a weight
    # gradient with 2^31 - 16 output pixels or more, keeps the generic kernel (no memory is touched here)
    wide = Problem(n=1, h=1, w=2**31 - 2, c=4, k=4, r=1, s=3, pad_w=1)
    for d in (DIR_FWD, DIR_WGRAD):
        assert cig.describe_plan(wide, d, -1, sm_count=SMS)["kernel_name"] == "generic", d
    narrower = Problem(n=1, h=1, w=2**31 - 4, c=4, k=4, r=1, s=3, pad_w=1)  # W + 2 pw = 2^31 - 2
    assert cig.describe_plan(narrower, DIR_FWD, -1, sm_count=SMS)["kernel_name"] == "ffma"
    many = Problem(n=2**16, h=2**7, w=2**8 - 1, c=4, k=4)  # 2^31 - 2^23 output pixels: still 32-bit
    assert cig.describe_plan(many, DIR_WGRAD, -1, sm_count=SMS)["kernel_name"] in ("ffma", "wgrad_1x1_tf32x3",
                                                                                   "wgrad_1x1_ffma")
