"""GPU parity through the C ABI against the CPU oracle, element by element,
on seeded inputs spanning several tiles with ragged tails; determinism;
workspace needing no clearing; canaries around every output."""
import numpy as np
import pytest
import torch

import oracle
import synth
import implicit_gemm_convolution_nhwc_gb300 as cig
from gpu_util import TORCH_DT, Guarded, inputs, oproblem, relerr, run_dgrad, run_fwd, run_wgrad, tol

pytestmark = pytest.mark.gpu

BF16, F16, F32 = cig.BF16, cig.F16, cig.F32


@pytest.fixture(autouse=True)
def _reset_override():
    cig.set_kernel_override("auto")
    yield
    cig.set_kernel_override("auto")


def _max_degree(p, d):
    """The largest degree the current kernel takes: the reduction blocks, or
    the cluster limit of the single-launch forward."""
    return cig.describe_plan(p, d, 1, sm_count=torch.cuda.get_device_properties(0).multi_processor_count)[
        "max_split"]


def check_wgrad(p, seed, kernels, splits, dist="normal", a=0.0, b=1.0, bias=True):
    orc = oracle.get()
    x, dy = inputs(p, seed, dist, a, b)
    ref_w = orc.wgrad(oproblem(p), x, dy)
    ref_b = orc.bgrad(oproblem(p), dy) if bias else None
    for kern in kernels:
        cig.set_kernel_override(kern)
        top = _max_degree(p, cig.DIR_WGRAD)
        for sk in splits:
            sk = top if sk == "max" else sk
            if sk > top:  # more slices than reduction blocks: rejected, checked elsewhere
                continue
            dw, db = run_wgrad(p, x, dy, sk, bias)
            e = relerr(dw, ref_w)
            assert e <= tol(p), f"{kern} split {sk}: dW err {e:.3e}"
            if bias:
                eb = relerr(db, ref_b)
                assert eb <= tol(p), f"{kern} split {sk}: db err {eb:.3e}"
    cig.set_kernel_override("auto")


def check_fwd(p, seed, kernels, splits, dist="normal", a=0.0, b=1.0):
    orc = oracle.get()
    x, w = inputs(p, seed, dist, a, b, cig.DIR_FWD)
    ref = orc.fwd(oproblem(p), x, w)
    for kern in kernels:
        cig.set_kernel_override(kern)
        top = _max_degree(p, cig.DIR_FWD)
        for sk in splits:
            sk = top if sk == "max" else sk
            if sk > top:
                continue
            y = run_fwd(p, x, w, sk)
            e = relerr(y, ref)
            assert e <= tol(p), f"{kern} split {sk}: Y err {e:.3e}"
    cig.set_kernel_override("auto")


# ---------------------------------------------------------------- 1x1 fp32


def test_config1_exact():
    """1x1 wgrad+db fp32, N=4, 16x16, C=8 -> K=16, uniform [-1, 1], seed 0."""
    p = cig.Problem(n=4, h=16, w=16, c=8, k=16)
    check_wgrad(p, 0, ["auto", "generic", "wgrad_1x1_ffma"], [-1, 0, 1, 2, 5, "max"], "uniform", -1.0, 1.0)
    assert cig.device_errors() == 0


@pytest.mark.parametrize("shape", [
    dict(n=3, h=37, w=29, c=100, k=68),     # ragged rows, one c tile with a tail, two k tiles
    dict(n=2, h=19, w=23, c=196, k=16),     # two c tiles (128 + 68)
    dict(n=1, h=5, w=7, c=4, k=4),          # fewer rows than one block
    dict(n=5, h=16, w=16, c=96, k=64),      # the large config's channels on a small image
    dict(n=2, h=33, w=31, c=40, k=36),      # tensor-core tile with channel tails in both operands
    dict(n=3, h=8, w=8, c=128, k=128),      # two k tiles, one full 128-wide c tile
])
def test_1x1_fp32_ragged(shape):
    p = cig.Problem(**shape)
    kernels = ["auto", "wgrad_1x1_ffma", "generic"]
    if p.c >= 32 and p.k >= 32 and p.h * p.w >= 32:
        kernels.append("wgrad_1x1_tf32x3")
    check_wgrad(p, 1, kernels, [-1, 1, 3, 17])
    assert cig.device_errors() == 0


def test_1x1_without_bias_and_empty_batch():
    p = cig.Problem(n=2, h=9, w=9, c=32, k=32)
    check_wgrad(p, 3, ["auto"], [-1, 1], bias=False)
    empty = cig.Problem(n=0, h=9, w=9, c=32, k=32)
    x, dy = inputs(empty, 3)
    dw, db = run_wgrad(empty, x, dy, -1, True)
    assert not dw.any() and not db.any()


# ------------------------------------------------------------ generic path

GENERIC_SHAPES = [
    dict(n=2, h=7, w=9, c=6, k=4, r=3, s=2, stride_h=1, stride_w=2, pad_h=1, pad_w=0),
    dict(n=1, h=8, w=8, c=8, k=6, r=3, s=3, stride_h=2, stride_w=2, pad_h=1, pad_w=1, dil_h=2, groups=2),
    dict(n=3, h=5, w=6, c=4, k=4, r=5, s=3, pad_h=2, pad_w=3, dil_w=2, groups=4),
    dict(n=2, h=9, w=7, c=12, k=8, r=1, s=4, stride_h=3, pad_w=2, groups=4),
]
DTYPES = [(F32, F32), (BF16, BF16), (BF16, F32), (F16, F16), (F16, F32)]


@pytest.mark.parametrize("shape", GENERIC_SHAPES)
@pytest.mark.parametrize("dt", DTYPES, ids=lambda d: f"{d[0]}{d[1]}")
def test_generic_wgrad(shape, dt):
    p = cig.Problem(**shape, in_dtype=dt[0], out_dtype=dt[1])
    check_wgrad(p, 4, ["generic"], [-1, 0, 3])


@pytest.mark.parametrize("shape", GENERIC_SHAPES)
@pytest.mark.parametrize("dt", DTYPES, ids=lambda d: f"{d[0]}{d[1]}")
def test_generic_fwd(shape, dt):
    p = cig.Problem(**shape, in_dtype=dt[0], out_dtype=dt[1])
    check_fwd(p, 5, ["generic"], [-1, 0, 2])


# ------------------------------------------------------------ determinism


def test_repeated_runs_are_bit_identical():
    for p, direction in [(cig.Problem(n=3, h=37, w=29, c=100, k=68), cig.DIR_WGRAD),
                         (cig.Problem(n=2, h=9, w=7, c=12, k=8, r=3, s=3, pad_h=1, pad_w=1, groups=4,
                                      in_dtype=BF16, out_dtype=BF16), cig.DIR_WGRAD),
                         (cig.Problem(n=1, h=8, w=8, c=64, k=32, r=3, s=3, pad_h=1, pad_w=1,
                                      in_dtype=BF16, out_dtype=BF16), cig.DIR_FWD)]:
        x, other = inputs(p, 9, direction=direction)
        for sk in (-1, min(3, _max_degree(p, direction))):
            if direction == cig.DIR_WGRAD:
                outs = [run_wgrad(p, x, other, sk, True) for _ in range(3)]
                for o in outs[1:]:
                    assert torch.equal(o[0], outs[0][0]) and torch.equal(o[1], outs[0][1])
            else:
                outs = [run_fwd(p, x, other, sk) for _ in range(3)]
                for o in outs[1:]:
                    assert torch.equal(o, outs[0])


# ---------------------------------------------------------------- errors


def test_device_call_errors():
    p = cig.Problem(n=2, h=16, w=16, c=8, k=16)
    x, dy = inputs(p, 0)
    xd, dyd = x.cuda(), dy.cuda()
    dw = torch.empty((16, 1, 1, 8), device="cuda")
    db = torch.empty(16, device="cuda")
    need = cig.workspace_bytes(p, cig.DIR_WGRAD, 4, True)
    small = torch.empty(need - 1, dtype=torch.uint8, device="cuda")
    with pytest.raises(cig.ConvError) as e:
        cig.conv_wgrad_bias(p, xd, dyd, dw, db, small, 4)
    assert e.value.status == 3
    with pytest.raises(cig.ConvError) as e:
        cig.conv_wgrad_bias(p, xd, dyd, dw, db, None, 4)
    assert e.value.status == 3
    big = torch.empty(need + 4, dtype=torch.uint8, device="cuda")
    with pytest.raises(cig.ConvError) as e:
        cig.conv_wgrad_bias(p, xd, dyd, dw, db, big[4:], 4)
    assert e.value.status == 5
    flat = torch.empty(2 * 16 * 16 * 8 + 1, device="cuda")
    with pytest.raises(cig.ConvError) as e:
        cig.conv_wgrad_bias(p, flat[1:], dyd, dw, db, big[:need], 4)
    assert e.value.status == 5


# ------------------------------------------------------- tensor-core forward


def test_config3_forward_split_sweep():
    """3x3 fwd bf16, N=1, 14x14, C=2048 -> K=512, pad 1, N(0, 0.02) seed 2; split auto and 1..32."""
    p = cig.Problem(n=1, h=14, w=14, c=2048, k=512, r=3, s=3, pad_h=1, pad_w=1, in_dtype=BF16, out_dtype=BF16)
    assert cig.describe_plan(p, cig.DIR_FWD, -1)["kernel_name"] == "fwd_tc"
    check_fwd(p, 2, ["auto"], [-1, 1, 2, 4, 8, 16, 32], "normal", 0.0, 0.02)
    check_fwd(p, 2, ["fwd_tc_cluster"], [-1, 2, 16], "normal", 0.0, 0.02)
    assert cig.device_errors() == 0


@pytest.mark.parametrize("shape", [
    dict(n=1, h=14, w=14, c=2048, k=512, r=3, s=3, pad_h=1, pad_w=1),          # the 3x3 small-M layer
    dict(n=2, h=10, w=12, c=128, k=136, r=3, s=3, pad_h=1, pad_w=1),           # K tail, 2 M tiles per image
    dict(n=1, h=9, w=11, c=64, k=128, r=5, s=5, pad_h=4, pad_w=4, dil_h=2, dil_w=2),
    dict(n=1, h=20, w=40, c=256, k=192, r=3, s=1, pad_h=1, pad_w=0),           # last N tile half empty
])
def test_forward_cluster_equals_two_stage(shape):
    """The single-launch form folds the same per-slice partial tiles in the
    same slice order as the fold kernel ("feat(rocke): split-K forward
    implicit-GEMM convolution on gfx1250", "Changes"), so Y is bit-identical
    to the two-stage form at every degree, and reruns are bit-identical."""
    p = cig.Problem(**shape, in_dtype=BF16, out_dtype=BF16)
    x, w = inputs(p, 2, "normal", 0.0, 0.02, cig.DIR_FWD)
    top = cig.describe_plan(p, cig.DIR_FWD, 1)["reduction_blocks"]
    for sk in (2, 3, 5, 8, 13, 16):
        if sk > top:
            continue
        cig.set_kernel_override("fwd_tc_cluster")
        assert cig.describe_plan(p, cig.DIR_FWD, sk)["workspace_bytes"] == 0
        y1 = run_fwd(p, x, w, sk)
        y2 = run_fwd(p, x, w, sk)
        cig.set_kernel_override("fwd_tc")
        y0 = run_fwd(p, x, w, sk)
        cig.set_kernel_override("auto")
        assert torch.equal(y1.view(torch.int16), y0.view(torch.int16)), f"split {sk}: cluster != two-stage"
        assert torch.equal(y1.view(torch.int16), y2.view(torch.int16)), f"split {sk}: rerun differs"
    assert cig.device_errors() == 0


@pytest.mark.parametrize("shape", [
    dict(n=2, h=10, w=12, c=128, k=136, r=3, s=3, pad_h=1, pad_w=1),           # K tail, 2 M tiles per image
    dict(n=1, h=9, w=11, c=64, k=128, r=5, s=5, pad_h=4, pad_w=4, dil_h=2, dil_w=2),  # dilation, wide pad
    dict(n=3, h=9, w=9, c=64, k=128),                                           # pointwise
    dict(n=1, h=20, w=40, c=192, k=256, r=3, s=1, pad_h=1, pad_w=0),           # non-square filter
    dict(n=1, h=20, w=40, c=256, k=192, r=3, s=1, pad_h=1, pad_w=0),           # last N tile half empty
])
@pytest.mark.parametrize("dt", [(BF16, BF16), (F16, F32), (F16, F16)], ids=lambda d: f"{d[0]}{d[1]}")
def test_forward_tc_ragged(shape, dt):
    p = cig.Problem(**shape, in_dtype=dt[0], out_dtype=dt[1])
    check_fwd(p, 6, ["fwd_tc", "fwd_tc_cluster", "generic"], [-1, 1, 3])
    check_fwd(p, 6, ["fwd_tc", "fwd_tc_cluster"], ["max"])
    assert cig.device_errors() == 0


@pytest.mark.parametrize("shape", [
    dict(n=2, h=16, w=16, c=128, k=128, r=3, s=3, stride_h=2, stride_w=2, pad_h=1, pad_w=1),   # 3x3 downsample
    dict(n=2, h=14, w=14, c=64, k=256, r=1, s=1, stride_h=2, stride_w=2),                       # 1x1 projection
    dict(n=1, h=21, w=24, c=128, k=136, r=3, s=3, stride_h=3, stride_w=2, pad_h=1, pad_w=1),   # unequal strides, K tail
    dict(n=1, h=16, w=16, c=64, k=128, r=3, s=3, stride_h=2, stride_w=2, pad_h=2, pad_w=2, dil_h=2, dil_w=2),
])
@pytest.mark.parametrize("dt", [(BF16, BF16), (F16, F32)], ids=lambda d: f"{d[0]}{d[1]}")
def test_forward_tc_strided(shape, dt):
    """Strided forwards on the tensor cores: the X box is read with TMA traversal strides."""
    p = cig.Problem(**shape, in_dtype=dt[0], out_dtype=dt[1])
    assert cig.describe_plan(p, cig.DIR_FWD, -1)["kernel_name"] == "fwd_tc"
    check_fwd(p, 7, ["fwd_tc", "generic"], [-1, 1, 3])
    check_fwd(p, 7, ["fwd_tc_cluster"], [2])
    assert cig.device_errors() == 0


@pytest.mark.parametrize("shape", [
    dict(n=2, h=13, w=17, c=128, k=128, groups=128, r=7, s=7, pad_h=3, pad_w=3),   # 7x7, ragged W chunks
    dict(n=3, h=9, w=10, c=96, k=96, groups=96, r=3, s=3, pad_h=1, pad_w=1),       # a half channel block
    dict(n=2, h=14, w=15, c=64, k=64, groups=64, r=3, s=3, stride_h=2, stride_w=2, pad_h=1, pad_w=1),
    dict(n=1, h=12, w=20, c=64, k=64, groups=64, r=5, s=5, pad_h=4, pad_w=2, dil_h=2),  # H dilation
    dict(n=2, h=10, w=12, c=32, k=32, groups=32, r=7, s=7),                         # no padding
    dict(n=1, h=9, w=23, c=64, k=64, groups=64, r=3, s=7, stride_h=3, stride_w=2, pad_h=0, pad_w=3),
    dict(n=3, h=5, w=9, c=72, k=72, groups=72, r=5, s=5, pad_h=4, pad_w=4),        # pad F-1, 8-channel tile, steps across images
    dict(n=4, h=3, w=30, c=64, k=64, groups=64, r=3, s=3, pad_h=0, pad_w=2),       # one output row an image
    dict(n=1, h=40, w=60, c=64, k=64, groups=64, r=7, s=7, pad_h=3, pad_w=3),      # a wide row ring
])
@pytest.mark.parametrize("dt", [(BF16, BF16), (F16, F32), (F32, F32)], ids=lambda d: f"{d[0]}{d[1]}")
def test_forward_depthwise(shape, dt):
    p = cig.Problem(**shape, in_dtype=dt[0], out_dtype=dt[1])
    assert cig.describe_plan(p, cig.DIR_FWD, -1)["kernel_name"] == "fwd_depthwise"
    check_fwd(p, 13, ["auto", "generic"], [-1, 1])
    assert cig.device_errors() == 0


@pytest.mark.parametrize("shape", [
    dict(n=2, h=10, w=12, c=128, k=128, groups=16, r=3, s=3, pad_h=1, pad_w=1),     # cpg 8
    dict(n=3, h=9, w=9, c=256, k=256, groups=64, r=3, s=3, pad_h=1, pad_w=1),       # cpg 4, two blocks
    dict(n=1, h=14, w=13, c=128, k=128, groups=64, r=5, s=5, pad_h=2, pad_w=2),     # cpg 2
    dict(n=2, h=16, w=16, c=384, k=384, groups=24, r=3, s=3, stride_h=2, stride_w=2, pad_h=1, pad_w=1),  # cpg 16
    dict(n=2, h=7, w=9, c=128, k=128, groups=32, r=1, s=1),                          # pointwise cpg 4
])
@pytest.mark.parametrize("dt", [(BF16, BF16), (F16, F32), (F16, F16)], ids=lambda d: f"{d[0]}{d[1]}")
def test_forward_grouped_tc(shape, dt):
    """Grouped forwards as block-diagonal dense 128-channel blocks on the tensor cores (automatic choice
    for 4 or 8 channels per group at stride 1: the warp-MMA kernel)."""
    p = cig.Problem(**shape, in_dtype=dt[0], out_dtype=dt[1])
    assert cig.describe_plan(p, cig.DIR_FWD, -1)["kernel_name"] in ("fwd_grouped_tc", "fwd_grouped_mma")
    check_fwd(p, 14, ["fwd_grouped_tc", "generic"], [-1, 1, 3])
    check_fwd(p, 14, ["fwd_grouped_tc"], ["max"])
    assert cig.device_errors() == 0


# ------------------------------------------------------- fused forward epilogue

INF = float("inf")


def run_fwd_ep(p, x, w, bias, lo, hi, split_k=-1):
    ho, wo = p.out_hw
    y = Guarded(p.n * ho * wo * p.k, TORCH_DT[p.out_dtype])
    ws = cig.workspace(p, cig.DIR_FWD, 1, False)  # unsplit: a kernel's transformed filter at most
    cig.conv_fwd_epilogue(p, x.cuda(), w.cuda(), y.view, None if bias is None else bias.cuda(), lo, hi,
                          ws, split_k)
    torch.cuda.synchronize()
    assert y.intact(), "a write left its buffer"
    return y.view.cpu().reshape(p.n, ho, wo, p.k)


@pytest.mark.parametrize("shape", [
    dict(n=2, h=10, w=12, c=128, k=136, r=3, s=3, pad_h=1, pad_w=1),          # tensor cores, K tail
    dict(n=1, h=14, w=14, c=256, k=256, r=3, s=3, pad_h=1, pad_w=1),          # 128 x 256 tiles; conv_fwd would split
    dict(n=2, h=9, w=11, c=12, k=8, r=3, s=3, stride_h=2, stride_w=2, pad_h=1, pad_w=1),  # generic
    dict(n=2, h=13, w=17, c=96, k=96, groups=96, r=7, s=7, pad_h=3, pad_w=3),             # depthwise kernel
    dict(n=2, h=10, w=12, c=128, k=128, groups=16, r=3, s=3, pad_h=1, pad_w=1),           # grouped, warp MMAs
    dict(n=2, h=8, w=8, c=128, k=128, groups=64, r=5, s=5, pad_h=2, pad_w=2),             # grouped, tensor cores
])
@pytest.mark.parametrize("dt", [(BF16, BF16), (F16, F16), (F16, F32), (F32, F32)], ids=lambda d: f"{d[0]}{d[1]}")
def test_forward_fused_epilogue(shape, dt):
    """Bias / ReLU / clamp fused into the unsplit forward ("feat(rocke): split-K forward
    implicit-GEMM convolution on gfx1250", "Review follow-ups"), against the oracle."""
    p = cig.Problem(**shape, in_dtype=dt[0], out_dtype=dt[1])
    x, w = inputs(p, 21, "normal", 0.0, 0.05, cig.DIR_FWD)
    bias = synth.tensor((p.k,), TORCH_DT[p.out_dtype], "normal", 0.0, 0.1, 21, synth.BIAS_ID)
    orc = oracle.get()
    # the last bounds lie past fp16's range: 16-bit outputs are clamped after the rounding, against
    # the rounded (here infinite) bounds
    for use_bias, lo, hi in [(True, 0.0, INF), (True, -INF, INF), (False, 0.0, INF), (True, -0.05, 0.03),
                             (True, -7e4, 7e4)]:
        b = bias if use_bias else None
        ref = orc.fwd_epilogue(oproblem(p), x, w, b, lo, hi)
        # bias and clamp are exact; the error is the sum's, so it is measured against the
        # magnitude of the sum before the clamp
        scale = np.abs(orc.fwd_epilogue(oproblem(p), x, w, b)).max()
        for sk in (-1, 1):
            got = run_fwd_ep(p, x, w, b, lo, hi, sk).double().numpy()
            e = np.abs(got - ref).max() / scale
            assert e <= tol(p), f"bias {use_bias} [{lo}, {hi}] split {sk}: err {e:.3e}"
    # the identity epilogue is conv_fwd itself, bit for bit (same degree, same kernels)
    ho, wo = p.out_hw
    ident = Guarded(p.n * ho * wo * p.k, TORCH_DT[p.out_dtype])
    ws = cig.workspace(p, cig.DIR_FWD, -1, False)
    cig.conv_fwd_epilogue(p, x.cuda(), w.cuda(), ident.view, None, -INF, INF, ws, -1)
    torch.cuda.synchronize()
    plain = run_fwd(p, x, w, -1)
    assert torch.equal(ident.view.cpu().view(torch.uint8), plain.reshape(-1).view(torch.uint8))
    with pytest.raises(cig.ConvError) as err:
        run_fwd_ep(p, x, w, bias, 0.0, INF, 2)
    assert err.value.status == 1
    assert cig.device_errors() == 0



@pytest.mark.parametrize("shape", [
    dict(n=2, h=10, w=12, c=128, k=136, r=3, s=3, pad_h=1, pad_w=1),          # tensor cores
    dict(n=2, h=9, w=11, c=12, k=8, r=3, s=3, stride_h=2, stride_w=2, pad_h=1, pad_w=1),  # generic
    dict(n=2, h=13, w=17, c=96, k=96, groups=96, r=7, s=7, pad_h=3, pad_w=3),             # depthwise kernel
    dict(n=2, h=10, w=12, c=128, k=128, groups=16, r=3, s=3, pad_h=1, pad_w=1),           # grouped, warp MMAs
])
@pytest.mark.parametrize("dt", [(BF16, BF16), (F16, F16), (BF16, F32)], ids=lambda d: f"{d[0]}{d[1]}")
def test_forward_fused_epilogue_nan_becomes_lo(shape, dt):
    """A NaN in X makes NaN sums; a non-identity epilogue turns each into lo, as fminf(fmaxf(nan, lo), hi)
    does, in every kernel (the tensor-core forward clamps 16-bit outputs after the rounding)."""
    p = cig.Problem(**shape, in_dtype=dt[0], out_dtype=dt[1])
    x, w = inputs(p, 23, "normal", 0.0, 0.05, cig.DIR_FWD)
    x[1, 4, 5, 3] = float("nan")
    bias = synth.tensor((p.k,), TORCH_DT[p.out_dtype], "normal", 0.0, 0.1, 23, synth.BIAS_ID)
    ref = oracle.get().fwd_epilogue(oproblem(p), x, w, bias, -0.05, 0.03)
    nan = np.isnan(ref)
    assert nan.any() and not nan.all()
    got = run_fwd_ep(p, x, w, bias, -0.05, 0.03).double().numpy()
    lo = torch.tensor(-0.05, dtype=TORCH_DT[p.out_dtype]).double().item()
    assert (got[nan] == lo).all()
    scale = np.abs(np.nan_to_num(oracle.get().fwd_epilogue(oproblem(p), x, w, bias))).max()
    assert np.abs(got[~nan] - ref[~nan]).max() / scale <= tol(p)
    assert cig.device_errors() == 0

# ------------------------------------------------------- persistent forward


@pytest.mark.parametrize("dt", [(BF16, BF16), (F16, F32)], ids=lambda d: f"{d[0]}{d[1]}")
def test_persistent_forward_units(dt):
    """The 256-wide tensor-core forward runs persistent: with more work units than SMs a CTA takes several
    (tile, slice) units in turn, its two TMEM accumulators alternating and its two epilogue groups sharing
    each unit's column chunks. K = 320 leaves the last channel tile a single 64-channel chunk (the second
    epilogue group stores nothing there). Every element against the oracle at pinned degrees 3 and 4 (168
    and 224 units), unsplit, with the data gradient of the layer with C and K swapped (the same forward form);
    then 168 unsplit units with the fused
    bias + ReLU, which a CTA reloads per unit."""
    p = cig.Problem(n=4, h=28, w=28, c=64, k=320, r=3, s=3, pad_h=1, pad_w=1, in_dtype=dt[0], out_dtype=dt[1])
    info = cig.describe_plan(p, cig.DIR_FWD, 4)
    assert info["kernel_name"] == "fwd_tc" and info["ctas"] == 56 * 4, info  # 28 row tiles x 2 channel tiles x 4
    check_fwd(p, 31, ["auto"], [-1, 1, 3, 4], "normal", 0.0, 0.05)
    pd = cig.Problem(n=4, h=28, w=28, c=320, k=64, r=3, s=3, pad_h=1, pad_w=1, in_dtype=dt[0], out_dtype=dt[1])
    assert cig.describe_plan(pd, cig.DIR_DGRAD, 4)["kernel_name"] == "dgrad_tc"
    check_dgrad(pd, 32, ["auto"], [-1, 1, 3, 4], "normal", 0.0, 0.05)
    p12 = cig.Problem(n=12, h=28, w=28, c=64, k=320, r=3, s=3, pad_h=1, pad_w=1, in_dtype=dt[0], out_dtype=dt[1])
    assert cig.describe_plan(p12, cig.DIR_FWD, 1)["ctas"] == 168
    x, w = inputs(p12, 33, "normal", 0.0, 0.05, cig.DIR_FWD)
    bias = synth.tensor((p12.k,), TORCH_DT[p12.out_dtype], "normal", 0.0, 0.1, 33, synth.BIAS_ID)
    orc = oracle.get()
    ref = orc.fwd_epilogue(oproblem(p12), x, w, bias, 0.0, INF)
    scale = np.abs(orc.fwd_epilogue(oproblem(p12), x, w, bias)).max()
    got = run_fwd_ep(p12, x, w, bias, 0.0, INF, 1).double().numpy()
    assert np.abs(got - ref).max() / scale <= tol(p12)
    assert cig.device_errors() == 0


# ------------------------------------------------------------- data gradient


def check_dgrad(p, seed, kernels, splits, dist="normal", a=0.0, b=1.0):
    orc = oracle.get()
    dy, w = inputs(p, seed, dist, a, b, cig.DIR_DGRAD)
    ref = orc.dgrad(oproblem(p), dy, w)
    for kern in kernels:
        cig.set_kernel_override(kern)
        top = _max_degree(p, cig.DIR_DGRAD)
        for sk in splits:
            sk = top if sk == "max" else sk
            if sk > top:
                continue
            dx = run_dgrad(p, dy, w, sk)
            e = relerr(dx, ref)
            assert e <= tol(p), f"{kern} split {sk}: dX err {e:.3e}"
    cig.set_kernel_override("auto")


@pytest.mark.parametrize("shape", [
    dict(n=2, h=9, w=11, c=12, k=8, r=3, s=3, stride_h=2, stride_w=2, pad_h=1, pad_w=1),   # stride 2
    dict(n=1, h=13, w=10, c=6, k=9, r=3, s=2, stride_h=3, stride_w=1, pad_h=2, pad_w=0, dil_h=2, dil_w=1),
    dict(n=2, h=8, w=8, c=16, k=24, r=3, s=3, pad_h=1, pad_w=1, groups=4),                # groups
    dict(n=3, h=7, w=9, c=32, k=32, r=5, s=5, pad_h=2, pad_w=2, groups=32),               # depthwise
    dict(n=2, h=6, w=5, c=40, k=20, r=1, s=1),                                              # pointwise
])
@pytest.mark.parametrize("dt", [(F32, F32), (BF16, BF16), (F16, F32)], ids=lambda d: f"{d[0]}{d[1]}")
def test_dgrad_generic(shape, dt):
    p = cig.Problem(**shape, in_dtype=dt[0], out_dtype=dt[1])
    check_dgrad(p, 11, ["auto", "generic"], [-1, 1, 3, "max"])
    assert cig.device_errors() == 0


@pytest.mark.parametrize("shape", [
    dict(n=2, h=10, w=12, c=136, k=128, r=3, s=3, pad_h=1, pad_w=1),          # C tail (the output channels)
    dict(n=1, h=9, w=11, c=128, k=192, r=5, s=5, pad_h=4, pad_w=4, dil_h=2, dil_w=2),
    dict(n=3, h=9, w=9, c=256, k=64),                                          # pointwise
    dict(n=1, h=20, w=40, c=192, k=256, r=3, s=1, pad_h=1, pad_w=0),          # non-square filter
])
@pytest.mark.parametrize("dt", [(BF16, BF16), (F16, F32), (F16, F16)], ids=lambda d: f"{d[0]}{d[1]}")
def test_dgrad_tc_ragged(shape, dt):
    p = cig.Problem(**shape, in_dtype=dt[0], out_dtype=dt[1])
    assert cig.describe_plan(p, cig.DIR_DGRAD, -1)["kernel_name"] == "dgrad_tc"
    check_dgrad(p, 12, ["dgrad_tc", "generic"], [-1, 1, 3])
    check_dgrad(p, 12, ["dgrad_tc"], ["max"])
    assert cig.device_errors() == 0


def test_dgrad_config3_layer():
    """The 3x3 small-M layer (N=1, 14x14, C=2048, K=512, pad 1, bf16) run
    backwards: dX [1,14,14,2048] from dY [1,14,14,512]; auto and pinned
    degrees; reruns bit-identical."""
    p = cig.Problem(n=1, h=14, w=14, c=2048, k=512, r=3, s=3, pad_h=1, pad_w=1, in_dtype=BF16, out_dtype=BF16)
    assert cig.describe_plan(p, cig.DIR_DGRAD, -1)["kernel_name"] == "dgrad_tc"
    check_dgrad(p, 2, ["auto"], [-1, 1, 8, 32], "normal", 0.0, 0.02)
    dy, w = inputs(p, 2, "normal", 0.0, 0.02, cig.DIR_DGRAD)
    a, b = run_dgrad(p, dy, w, -1), run_dgrad(p, dy, w, -1)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert cig.device_errors() == 0


@pytest.mark.parametrize("shape, ring", [
    (dict(n=3, h=13, w=17, c=72, r=7, s=7, pad_h=3, pad_w=3), True),     # channel tail, the ring form
    (dict(n=2, h=11, w=9, c=64, r=5, s=5, pad_h=1, pad_w=2), True),      # turned padding 3 / 2
    (dict(n=2, h=6, w=30, c=128, r=3, s=3), True),                       # no padding: turned padding 2
    (dict(n=2, h=12, w=10, c=34, r=3, s=5, pad_h=1, pad_w=2), False),    # non-square, C < 64: shared form
    (dict(n=1, h=15, w=11, c=40, r=3, s=3, pad_h=2, pad_w=1, dil_h=2), False),  # H dilation
])
@pytest.mark.parametrize("dt", [(BF16, BF16), (F16, F32), (F32, F32)], ids=lambda d: f"{d[0]}{d[1]}")
def test_dgrad_depthwise(shape, ring, dt):
    """Depthwise data gradient at stride 1 as the depthwise forward over dY with the filter's taps read
    backwards (the turned-filter identity of the depthwise data gradient pasted into "feat(rocke):
    split-K forward implicit-GEMM convolution on gfx1250")."""
    c = shape["c"]
    p = cig.Problem(**shape, k=c, groups=c, in_dtype=dt[0], out_dtype=dt[1])
    info = cig.describe_plan(p, cig.DIR_DGRAD, -1)
    assert info["kernel_name"] == "dgrad_depthwise" and info["split_k"] == 1
    assert (info["ctas_per_sm"] == 1) == (ring and dt[0] != F32)
    check_dgrad(p, 13, ["auto", "generic"], [-1, 1])
    assert cig.device_errors() == 0


@pytest.mark.parametrize("shape", [
    dict(n=2, h=10, w=12, c=256, k=256, r=3, s=3, pad_h=1, pad_w=1, groups=32),    # 8 per group
    dict(n=1, h=9, w=11, c=128, k=128, r=3, s=3, pad_h=1, pad_w=1, groups=32),     # 4 per group
    dict(n=2, h=8, w=8, c=128, k=128, r=5, s=5, pad_h=2, pad_w=2, groups=64),      # 2 per group
    dict(n=1, h=12, w=12, c=256, k=256, r=3, s=3, pad_h=2, pad_w=2, dil_h=2, dil_w=2, groups=8),  # 32
    dict(n=2, h=7, w=13, c=128, k=128, r=1, s=1, groups=8),                         # pointwise, 16
])
@pytest.mark.parametrize("dt", [(F16, F16), (BF16, F32)], ids=lambda d: f"{d[0]}{d[1]}")
def test_dgrad_grouped_tc(shape, dt):
    """Grouped data gradient at stride 1 as the block-diagonal grouped forward over dY with the turned
    filter in the group blocks."""
    p = cig.Problem(**shape, in_dtype=dt[0], out_dtype=dt[1])
    info = cig.describe_plan(p, cig.DIR_DGRAD, -1)
    assert info["kernel_name"] in ("dgrad_grouped_tc", "dgrad_grouped_mma")
    check_dgrad(p, 14, ["auto", "dgrad_grouped_tc"], [-1, 1, 2, "max"])
    check_dgrad(p, 14, ["generic"], [1])
    assert cig.device_errors() == 0


@pytest.mark.parametrize("shape", [
    dict(n=2, h=10, w=13, c=128, k=128, groups=16, r=3, s=3, pad_h=1, pad_w=1),   # cpg 8, two channel blocks
    dict(n=3, h=9, w=9, c=64, k=64, groups=16, r=3, s=3, pad_h=1, pad_w=1),       # cpg 4
    dict(n=1, h=12, w=40, c=64, k=64, groups=8, r=3, s=3),                         # no padding, 3 column tiles
    dict(n=2, h=7, w=9, c=128, k=128, groups=32, r=5, s=5, pad_h=2, pad_w=2),     # cpg 4, 5x5
    dict(n=2, h=6, w=17, c=64, k=64, groups=8, r=1, s=1),                          # pointwise
    dict(n=1, h=5, w=64, c=64, k=64, groups=8, r=3, s=3, pad_h=2, pad_w=1),       # widest rows, Ho > H
    dict(n=5, h=3, w=6, c=64, k=64, groups=16, r=5, s=5, pad_h=4, pad_w=4),       # pad F - 1: rows past the image
])
@pytest.mark.parametrize("dt", [(F16, F16), (BF16, F32), (BF16, BF16)], ids=lambda d: f"{d[0]}{d[1]}")
def test_grouped_mma_forward_and_dgrad(shape, dt):
    """The grouped warp-MMA kernel (taps as pixel shifts, the group's filter in registers, unsplit):
    the forward and, on the turned problem with the filter read in place, the stride-1 data gradient,
    against the oracle; reruns bit-identical."""
    p = cig.Problem(**shape, in_dtype=dt[0], out_dtype=dt[1])
    assert cig.describe_plan(p, cig.DIR_FWD, -1)["kernel_name"] == "fwd_grouped_mma"
    assert cig.describe_plan(p, cig.DIR_DGRAD, -1)["kernel_name"] == "dgrad_grouped_mma"
    check_fwd(p, 16, ["auto"], [-1, 1])
    check_dgrad(p, 16, ["auto"], [-1, 1])
    x, w = inputs(p, 16, direction=cig.DIR_FWD)
    assert torch.equal(run_fwd(p, x, w, -1), run_fwd(p, x, w, -1))
    assert cig.device_errors() == 0


# ------------------------------------------------------- depthwise / grouped


def test_config4_depthwise_full():
    """Depthwise 7x7 wgrad bf16, N=32, 56x56, C=K=384 (groups=384), pad 3, N(0,1) seed 3."""
    p = cig.Problem(n=32, h=56, w=56, c=384, k=384, r=7, s=7, pad_h=3, pad_w=3, groups=384,
                    in_dtype=BF16, out_dtype=BF16)
    assert cig.describe_plan(p, cig.DIR_WGRAD, -1)["kernel_name"] == "wgrad_depthwise"
    check_wgrad(p, 3, ["auto", "wgrad_depthwise_mma"], [-1, 1, 7], bias=False)
    check_wgrad(p, 3, ["auto"], [-1], bias=True)
    x, dy = inputs(p, 3)
    a, b = run_wgrad(p, x, dy, -1, True), run_wgrad(p, x, dy, -1, True)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    assert cig.device_errors() == 0


@pytest.mark.parametrize("shape", [
    dict(n=2, h=14, w=14, c=64, r=7, s=7, pad_h=3, pad_w=3),
    dict(n=3, h=13, w=17, c=128, r=5, s=5, pad_h=2, pad_w=2),     # two 16-column chunks
    dict(n=2, h=9, w=33, c=72, r=3, s=3),                          # three chunks, no padding, 8-channel tail
    dict(n=2, h=11, w=58, c=96, r=7, s=7, pad_h=6, pad_w=6),      # Wo = 64 > W: bias columns past the input
    dict(n=1, h=7, w=64, c=64, r=7, s=7, pad_h=3, pad_w=3),       # the widest rows
    dict(n=3, h=5, w=9, c=8, r=3, s=5, pad_h=1, pad_w=2),         # one warp's channels, non-square filter
    dict(n=4, h=3, w=16, c=64, r=1, s=1),                          # pointwise, one chunk
    dict(n=2, h=6, w=20, c=40, r=7, s=3, pad_h=5, pad_w=1),       # fewer input rows than filter rows
    dict(n=5, h=2, w=5, c=16, r=2, s=4, pad_h=1, pad_w=3),        # even filter sizes, rows spanning images
])
@pytest.mark.parametrize("dt", [(BF16, BF16), (BF16, F32), (F16, F16)], ids=lambda d: f"{d[0]}{d[1]}")
def test_depthwise_mma(shape, dt):
    """The depthwise MMA weight gradient (Toeplitz dY operand, rows transposed in shared memory) against
    the oracle at several degrees, with the bias gradient; reruns bit-identical."""
    shp = dict(shape, k=shape["c"], groups=shape["c"])
    p = cig.Problem(**shp, in_dtype=dt[0], out_dtype=dt[1])
    check_wgrad(p, 9, ["wgrad_depthwise_mma"], [-1, 1, 4, "max"], bias=True)
    x, dy = inputs(p, 9)
    cig.set_kernel_override("wgrad_depthwise_mma")
    try:
        assert cig.describe_plan(p, cig.DIR_WGRAD, -1)["kernel_name"] == "wgrad_depthwise_mma"
        a, b = run_wgrad(p, x, dy, 3, True), run_wgrad(p, x, dy, 3, True)
    finally:
        cig.set_kernel_override("auto")
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    assert cig.device_errors() == 0


@pytest.mark.parametrize("shape", [
    dict(n=3, h=13, w=17, c=128, k=128, groups=128, r=5, s=5, pad_h=2, pad_w=2),
    dict(n=2, h=9, w=30, c=64, k=64, groups=64, r=3, s=3, pad_h=1, pad_w=1),
    dict(n=1, h=12, w=20, c=64, k=64, groups=64, r=3, s=11, pad_h=1, pad_w=5),
    dict(n=2, h=10, w=12, c=64, k=64, groups=64, r=7, s=7),                  # no padding: Wo = W - 6
    dict(n=3, h=5, w=9, c=192, k=192, groups=192, r=7, s=7, pad_h=3, pad_w=3),  # fewer rows than taps
    dict(n=2, h=11, w=13, c=96, k=96, groups=96, r=7, s=7, pad_h=6, pad_w=6),   # pad F-1, C % 64 != 0
    dict(n=1, h=4, w=5, c=72, k=72, groups=72, r=3, s=3, pad_h=2, pad_w=0),     # 8 channels in the last tile
    dict(n=2, h=6, w=70, c=136, k=136, groups=136, r=5, s=5, pad_h=1, pad_w=4),
    dict(n=2, h=9, w=10, c=64, k=64, groups=64, r=3, s=3, pad_h=1, pad_w=3),    # pad_w = F: shared-memory form
    dict(n=1, h=3, w=90, c=64, k=64, groups=64, r=7, s=7, pad_h=3, pad_w=3),    # rings one row ahead
])
@pytest.mark.parametrize("dt", [(BF16, BF16), (BF16, F32), (F16, F16)], ids=lambda d: f"{d[0]}{d[1]}")
def test_depthwise_ragged(shape, dt):
    p = cig.Problem(**shape, in_dtype=dt[0], out_dtype=dt[1])
    check_wgrad(p, 8, ["wgrad_depthwise", "generic"], [-1, 1, 4], bias=True)
    assert cig.device_errors() == 0


@pytest.mark.parametrize("groups", [64, 128], ids=["cpg8", "cpg4"])
def test_config5_grouped_full(groups):
    """Grouped 3x3 wgrad fp16, N=64, 28x28, C=K=512, groups 64 / 128, pad 1, N(0,1) seed 4."""
    p = cig.Problem(n=64, h=28, w=28, c=512, k=512, r=3, s=3, pad_h=1, pad_w=1, groups=groups,
                    in_dtype=F16, out_dtype=F16)
    assert cig.describe_plan(p, cig.DIR_WGRAD, -1)["kernel_name"] == "wgrad_grouped_mma"
    check_wgrad(p, 4, ["auto", "wgrad_grouped_tc"], [-1, 1, 9], bias=False)
    check_wgrad(p, 4, ["auto"], [-1], bias=True)
    x, dy = inputs(p, 4)
    a, b = run_wgrad(p, x, dy, -1, True), run_wgrad(p, x, dy, -1, True)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    assert cig.device_errors() == 0


@pytest.mark.parametrize("shape", [
    dict(n=3, h=11, w=13, c=128, k=128, groups=16, r=3, s=3, pad_h=1, pad_w=1),   # cpg 8
    dict(n=2, h=9, w=30, c=64, k=64, groups=16, r=3, s=3, pad_h=1, pad_w=1),      # cpg 4
    dict(n=2, h=7, w=9, c=64, k=64, groups=16, r=5, s=5, pad_h=2, pad_w=2),       # cpg 4, 5x5
    dict(n=4, h=6, w=6, c=192, k=192, groups=24, r=1, s=1),                         # cpg 8, pointwise
    dict(n=1, h=4, w=5, c=64, k=64, groups=8, r=3, s=3),                            # no padding
])
@pytest.mark.parametrize("dt", [(F16, F16), (BF16, F32)], ids=lambda d: f"{d[0]}{d[1]}")
def test_grouped_ragged(shape, dt):
    p = cig.Problem(**shape, in_dtype=dt[0], out_dtype=dt[1])
    check_wgrad(p, 9, ["wgrad_grouped", "generic"], [-1, 1, 3], bias=True)
    assert cig.device_errors() == 0


@pytest.mark.parametrize("shape", [
    dict(n=3, h=11, w=13, c=128, k=128, groups=16, r=3, s=3, pad_h=1, pad_w=1),    # cpg 8
    dict(n=2, h=9, w=30, c=256, k=256, groups=64, r=3, s=3, pad_h=1, pad_w=1),     # cpg 4, two blocks
    dict(n=2, h=7, w=9, c=128, k=128, groups=32, r=3, s=1),                         # cpg 4, 3x1, no padding
    dict(n=1, h=12, w=12, c=128, k=128, groups=8, r=3, s=3, stride_h=2, stride_w=2, pad_h=1, pad_w=1),  # cpg 16
    dict(n=2, h=6, w=5, c=128, k=128, groups=4, r=3, s=3, pad_h=1, pad_w=1),       # cpg 32
    dict(n=2, h=8, w=8, c=128, k=128, groups=64, r=3, s=3, pad_h=1, pad_w=1),      # cpg 2
])
@pytest.mark.parametrize("dt", [(F16, F16), (BF16, F32)], ids=lambda d: f"{d[0]}{d[1]}")
def test_wgrad_grouped_tc(shape, dt):
    """Grouped weight gradients as block-diagonal dense blocks on the tensor cores (MN-major
    operands), with the bias gradient summed from the dY tiles (the automatic choice for the strided
    problem, through the override for the others)."""
    p = cig.Problem(**shape, in_dtype=dt[0], out_dtype=dt[1])
    assert cig.describe_plan(p, cig.DIR_WGRAD, -1)["kernel_name"] in ("wgrad_grouped_tc", "wgrad_grouped_mma")
    check_wgrad(p, 15, ["wgrad_grouped_tc", "generic"], [-1, 1, 3], bias=True)
    check_wgrad(p, 15, ["wgrad_grouped_tc"], ["max"], bias=True)
    assert cig.device_errors() == 0


@pytest.mark.parametrize("shape", [
    dict(n=3, h=11, w=13, c=128, k=128, groups=16, r=3, s=3, pad_h=1, pad_w=1),    # cpg 8, 3 columns past W
    dict(n=2, h=9, w=30, c=256, k=256, groups=64, r=3, s=3, pad_h=1, pad_w=1),     # cpg 4, two 16-column steps
    dict(n=2, h=7, w=9, c=128, k=128, groups=32, r=3, s=1),                         # cpg 4, 3x1, no padding
    dict(n=2, h=6, w=5, c=128, k=128, groups=4, r=3, s=3, pad_h=1, pad_w=1),       # cpg 32: 4 pairs a warp
    dict(n=2, h=8, w=8, c=128, k=128, groups=64, r=3, s=3, pad_h=1, pad_w=1),      # cpg 2
    dict(n=2, h=10, w=17, c=128, k=128, groups=8, r=3, s=2, pad_h=1, pad_w=1),     # cpg 16, 3x2
    dict(n=2, h=7, w=9, c=64, k=64, groups=16, r=5, s=5, pad_h=2, pad_w=2),        # cpg 4, 5x5
    dict(n=4, h=6, w=6, c=192, k=192, groups=24, r=1, s=1),                         # cpg 8, pointwise
    dict(n=1, h=4, w=5, c=64, k=64, groups=8, r=3, s=3),                            # no padding, Wo = 3
    dict(n=2, h=9, w=40, c=64, k=64, groups=8, r=3, s=4, pad_h=1, pad_w=2),        # even filter width
    dict(n=1, h=5, w=100, c=64, k=64, groups=8, r=3, s=3, pad_h=1, pad_w=1),       # 7 column steps
])
@pytest.mark.parametrize("dt", [(F16, F16), (BF16, F32)], ids=lambda d: f"{d[0]}{d[1]}")
def test_wgrad_grouped_mma(shape, dt):
    """Grouped weight gradients on warp-level MMAs with the filter column applied as a shift of dY
    ("perf(rocke): depthwise 7x7 and grouped cpg4/8 wgrad on batched mfma 4x4x4", "Technical
    Details"), with and without the bias gradient; reruns bit-identical."""
    p = cig.Problem(**shape, in_dtype=dt[0], out_dtype=dt[1])
    info = cig.describe_plan(p, cig.DIR_WGRAD, -1, True)
    assert info["kernel_name"] == "wgrad_grouped_mma"
    check_wgrad(p, 16, ["auto"], [-1, 1, 3, "max"], bias=True)
    check_wgrad(p, 16, ["auto"], [-1, 2], bias=False)
    x, dy = inputs(p, 16)
    sk = min(3, info["max_split"])
    a, b = run_wgrad(p, x, dy, sk, True), run_wgrad(p, x, dy, sk, True)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    assert cig.device_errors() == 0


def test_bounded_wait_gives_up_and_the_context_survives():
    """A pipeline wait that can never complete gives up after its limit (here 1 ms), records
    the timeout in the device error word and lets the kernel return; the context stays usable
    (no device fault is involved: the wait simply ends)."""
    cig.device_errors(clear=True)
    assert cig.selftest_wait_timeout(1_000_000)
    assert cig.device_errors(clear=True) & 1
    assert cig.device_errors(clear=True) == 0
    # a convolution right after it is correct
    p = cig.Problem(n=4, h=16, w=16, c=8, k=16)
    check_wgrad(p, 0, ["auto"], [-1], "uniform", -1.0, 1.0)
    assert cig.device_errors() == 0


@pytest.mark.parametrize("shape", [
    dict(h=9, w=11, c=128, k=128, groups=16, r=3, s=3, pad_h=1, pad_w=1, in_dtype=F16, out_dtype=F16),   # grouped
    dict(h=9, w=11, c=64, k=64, groups=64, r=7, s=7, pad_h=3, pad_w=3, in_dtype=BF16, out_dtype=BF16),   # depthwise
    dict(h=14, w=14, c=128, k=256, r=3, s=3, pad_h=1, pad_w=1, in_dtype=BF16, out_dtype=F32),            # dense 16-bit
])
def test_empty_batch_every_direction(shape):
    """N = 0: the weight and bias gradients are exactly zero, the forward, the fused forward
    and the data gradient write nothing and fail nothing."""
    p = cig.Problem(n=0, **shape)
    x, dy = inputs(p, 3)
    dw, db = run_wgrad(p, x, dy, -1, True)
    assert torch.count_nonzero(dw.float()) == 0 and torch.count_nonzero(db.float()) == 0
    xw = inputs(p, 3, direction=cig.DIR_FWD)
    assert run_fwd(p, xw[0], xw[1], -1).numel() == 0
    assert run_dgrad(p, dy, xw[1], -1).numel() == 0
    ho, wo = p.out_hw
    y = torch.empty(0, dtype=TORCH_DT[p.out_dtype], device="cuda")
    cig.conv_fwd_epilogue(p, xw[0].cuda(), xw[1].cuda(), y, None, 0.0, INF, None, -1)
    torch.cuda.synchronize()
    assert cig.device_errors() == 0


# ------------------------------------------------------------- width fold


@pytest.mark.parametrize("shape,direction,dt,kernel", [
    (dict(n=2, h=16, w=16, c=32, k=128, r=2, s=2, stride_h=2, stride_w=2), cig.DIR_FWD, (BF16, BF16), "fwd_tc"),
    (dict(n=3, h=20, w=24, c=16, k=256, r=4, s=4, stride_h=4, stride_w=4), cig.DIR_FWD, (F16, F32), "fwd_tc"),
    (dict(n=2, h=9, w=16, c=32, k=136, r=3, s=2, stride_w=2, pad_h=1), cig.DIR_FWD, (BF16, BF16), "fwd_tc"),
    (dict(n=2, h=8, w=64, c=18, k=64, r=1, s=2, stride_w=2), cig.DIR_WGRAD, (F32, F32), "wgrad_1x1_tf32x3"),
    (dict(n=2, h=8, w=16, c=64, k=128, r=1, s=2, stride_w=2), cig.DIR_DGRAD, (BF16, BF16), "dgrad_tc"),
], ids=["2x2s2", "4x4s4", "3x2ws2", "wgrad1x2", "dgrad1x2"])
def test_width_fold(shape, direction, dt, kernel):
    """Calls the planner width-folds ("feat(rocke): split-K forward implicit-GEMM convolution on gfx1250",
    the fold_width commit) run the folded problem on the same tensors; checked against the oracle on the
    original problem."""
    p = cig.Problem(**shape, in_dtype=dt[0], out_dtype=dt[1])
    info = cig.describe_plan(p, direction, -1)
    assert info["kernel_name"] == kernel and info["fold_width"] > 1
    if direction == cig.DIR_FWD:
        check_fwd(p, 21, ["auto", "generic"], [-1, 1, 2])
    elif direction == cig.DIR_WGRAD:
        check_wgrad(p, 21, ["auto"], [-1, 1, 2], bias=True)
    else:
        check_dgrad(p, 21, ["auto", "generic"], [-1, 1, 2])
    assert cig.device_errors() == 0


# ------------------------------------------------------------- fp32 FFMA tiles

FFMA_SHAPES = [
    dict(n=2, h=9, w=11, c=20, k=36, r=3, s=3, pad_h=1, pad_w=1),                   # channel tails in a step and a tile
    dict(n=3, h=13, w=10, c=16, k=132, r=3, s=2, stride_h=2, stride_w=1, pad_h=1, dil_h=2),  # strided, dilated
    dict(n=1, h=17, w=19, c=64, k=64, r=5, s=5, pad_h=2, pad_w=2),
    dict(n=2, h=12, w=12, c=136, k=8, r=1, s=1),                                   # pointwise, ragged M
    dict(n=1, h=20, w=21, c=8, k=260, r=3, s=3, stride_h=2, stride_w=2, pad_h=1, pad_w=1),  # 3 N tiles
    dict(n=5, h=7, w=1, c=12, k=20, r=3, s=1, pad_h=1),                            # Wo = 1: steps span images
]


@pytest.mark.parametrize("shape", FFMA_SHAPES)
def test_ffma_fp32_all_directions(shape):
    """fp32 implicit-GEMM FFMA tiles: forward, data gradient (stride 1; else generic) and weight gradient with
    its bias gradient, against the oracle at the fp32 tolerance, automatic, pinned and maximal degrees."""
    p = cig.Problem(**shape)
    assert cig.describe_plan(p, cig.DIR_FWD, -1)["kernel_name"] == "ffma"
    assert cig.describe_plan(p, cig.DIR_WGRAD, -1)["kernel_name"] in ("ffma", "wgrad_1x1_tf32x3", "wgrad_1x1_ffma")
    check_fwd(p, 17, ["ffma"], [-1, 1, 3, "max"])
    check_wgrad(p, 17, ["ffma"], [-1, 1, 3, "max"], bias=True)
    check_wgrad(p, 17, ["ffma"], [2], bias=False)
    if p.stride_h == 1 and p.stride_w == 1:
        assert cig.describe_plan(p, cig.DIR_DGRAD, -1)["kernel_name"] == "ffma"
        check_dgrad(p, 17, ["ffma"], [-1, 1, 3, "max"])
    x, w = inputs(p, 17, direction=cig.DIR_FWD)
    assert torch.equal(run_fwd(p, x, w, 3), run_fwd(p, x, w, 3))
    assert cig.device_errors() == 0


def test_ffma_fp32_exact_on_small_integers():
    """Small-integer inputs keep every fp32 product and partial sum exact, so every degree gives exactly the
    oracle's value in all three directions."""
    p = cig.Problem(n=2, h=10, w=9, c=24, k=40, r=3, s=3, pad_h=1, pad_w=1)
    orc = oracle.get()
    x, w = inputs(p, 18, "integer", -3, 3, cig.DIR_FWD)
    dy, _ = inputs(p, 18, "integer", -3, 3, cig.DIR_DGRAD)
    cig.set_kernel_override("ffma")
    try:
        for sk in (-1, 1, 2, 5):
            assert np.array_equal(run_fwd(p, x, w, sk).double().numpy(), orc.fwd(oproblem(p), x, w)), sk
            assert np.array_equal(run_dgrad(p, dy, w, sk).double().numpy(), orc.dgrad(oproblem(p), dy, w)), sk
            dw, db = run_wgrad(p, x, dy, sk, True)
            assert np.array_equal(dw.double().numpy(), orc.wgrad(oproblem(p), x, dy)), sk
            assert np.array_equal(db.double().numpy(), orc.bgrad(oproblem(p), dy)), sk
    finally:
        cig.set_kernel_override("auto")


# ------------------------------------------------------------- staged calls

STAGED = [  # (problem, direction): kernels with and without a fold, every direction
    (dict(n=1, h=14, w=14, c=256, k=512, r=3, s=3, pad_h=1, pad_w=1, in_dtype=BF16, out_dtype=BF16), cig.DIR_FWD),
    (dict(n=4, h=28, w=28, c=64, k=320, r=3, s=3, pad_h=1, pad_w=1, in_dtype=BF16, out_dtype=BF16), cig.DIR_FWD),
    (dict(n=1, h=14, w=14, c=512, k=256, r=3, s=3, pad_h=1, pad_w=1, in_dtype=F16, out_dtype=F32), cig.DIR_DGRAD),
    (dict(n=2, h=16, w=16, c=64, k=128, r=3, s=3, pad_h=1, pad_w=1, in_dtype=BF16, out_dtype=BF16), cig.DIR_WGRAD),
    (dict(n=2, h=12, w=12, c=16, k=32, r=3, s=3, pad_h=1, pad_w=1), cig.DIR_WGRAD),                     # fp32 FFMA
    (dict(n=2, h=20, w=20, c=64, k=64, groups=64, r=7, s=7, pad_h=3, pad_w=3, in_dtype=BF16, out_dtype=BF16),
     cig.DIR_WGRAD),                                                                                   # depthwise
]


@pytest.mark.parametrize("case", STAGED, ids=lambda c: f"{c[1]}-{c[0]['c']}x{c[0]['k']}")
def test_staged_calls_equal_one_call(case):
    """conv_stage1 then conv_stage2 with the same arguments is the one call, bit for bit (same kernels, same
    degree), at the automatic degree, degree 1 (stage 2 enqueues nothing) and a pinned degree with a fold."""
    shape, d = case
    p = cig.Problem(**shape)
    a, b = inputs(p, 41, "normal", 0.0, 0.05, d)
    a, b = a.cuda(), b.cuda()
    ho, wo = p.out_hw
    odt = TORCH_DT[p.out_dtype]
    n_out = {cig.DIR_FWD: p.n * ho * wo * p.k, cig.DIR_DGRAD: p.n * p.h * p.w * p.c,
             cig.DIR_WGRAD: p.k * p.r * p.s * (p.c // p.groups)}[d]
    bias = d == cig.DIR_WGRAD
    for sk in (-1, 1, 2):
        ws = cig.workspace(p, d, sk, bias)
        one, db1 = torch.empty(n_out, dtype=odt, device="cuda"), torch.empty(p.k, dtype=odt, device="cuda")
        two, db2 = torch.full((n_out,), float("nan"), dtype=odt, device="cuda"), torch.full((p.k,), float("nan"), dtype=odt, device="cuda")
        if d == cig.DIR_FWD:
            cig.conv_fwd(p, a, b, one, ws, sk)
        elif d == cig.DIR_DGRAD:
            cig.conv_dgrad(p, a, b, one, ws, sk)
        else:
            cig.conv_wgrad_bias(p, a, b, one, db1, ws, sk)
        cig.conv_stage1(p, d, a, b, two, db2 if bias else None, ws, sk)
        cig.conv_stage2(p, d, two, db2 if bias else None, ws, sk)
        torch.cuda.synchronize()
        assert torch.equal(one.view(torch.uint8), two.view(torch.uint8)), (d, sk)
        if bias:
            assert torch.equal(db1.view(torch.uint8), db2.view(torch.uint8)), (d, sk)
    assert cig.device_errors() == 0


# ------------------------------------------------------------- CUDA graphs


@pytest.mark.parametrize("case", STAGED, ids=lambda c: f"{c[1]}-{c[0]['c']}x{c[0]['k']}")
def test_calls_capture_into_a_cuda_graph(case):
    """A call (stage 1 and the fold, PDL-linked) captured into a CUDA graph replays to the eager result, bit
    for bit, at a pinned degree with a fold; the graph replays again after the inputs change in place."""
    shape, d = case
    p = cig.Problem(**shape)
    a, b = inputs(p, 43, "normal", 0.0, 0.05, d)
    a, b = a.cuda(), b.cuda()
    ho, wo = p.out_hw
    odt = TORCH_DT[p.out_dtype]
    n_out = {cig.DIR_FWD: p.n * ho * wo * p.k, cig.DIR_DGRAD: p.n * p.h * p.w * p.c,
             cig.DIR_WGRAD: p.k * p.r * p.s * (p.c // p.groups)}[d]
    bias = d == cig.DIR_WGRAD
    sk = 2
    ws = cig.workspace(p, d, sk, bias)
    out = torch.empty(n_out, dtype=odt, device="cuda")
    db = torch.empty(p.k, dtype=odt, device="cuda") if bias else None

    def call():
        if d == cig.DIR_FWD:
            cig.conv_fwd(p, a, b, out, ws, sk)
        elif d == cig.DIR_DGRAD:
            cig.conv_dgrad(p, a, b, out, ws, sk)
        else:
            cig.conv_wgrad_bias(p, a, b, out, db, ws, sk)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        call()  # warm-up outside the capture (module, attributes, tensor maps)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    eager = out.clone()
    eager_db = db.clone() if bias else None
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    for trial in range(2):
        out.fill_(float("nan"))
        if bias:
            db.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.uint8), eager.view(torch.uint8)), trial
        if bias:
            assert torch.equal(db.view(torch.uint8), eager_db.view(torch.uint8)), trial
    # new inputs in place: the replay computes on them
    a.mul_(-1)
    g.replay()
    torch.cuda.synchronize()
    flipped = out.clone()
    a.mul_(-1)
    call()
    torch.cuda.synchronize()
    assert torch.equal(flipped.float(), -out.float()), "replay on negated inputs"
    assert cig.device_errors() == 0
