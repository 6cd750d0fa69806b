"""The width fold ("feat(rocke): split-K forward implicit-GEMM convolution on
gfx1250", the fold_width commit): when f divides the filter width, the W
stride, the input width and the W padding (unit W dilation, one group), the
convolution equals one on W/f positions of f*C channels with filter width S/f
and W stride sw/f, on the same memory. Checked here with torch's float64
conv2d and its autograd (independent of the library and of the oracle), and
against the planner's choices; the GPU parity of folded calls is in
test_gpu_parity.py."""
import pytest
import torch

import implicit_gemm_convolution_nhwc_gb300 as cig
from implicit_gemm_convolution_nhwc_gb300 import BF16, DIR_DGRAD, DIR_FWD, DIR_WGRAD, Problem

SMS = 152


def conv(x, w, sh, sw, ph, pw):
    """NHWC x, KRSC w -> NHWC y with torch float64 conv2d."""
    y = torch.nn.functional.conv2d(x.permute(0, 3, 1, 2), w.permute(0, 3, 1, 2), stride=(sh, sw), padding=(ph, pw))
    return y.permute(0, 2, 3, 1)


def folded(t, f):
    """[.., W, C] viewed as [.., W/f, f*C] (the same memory)."""
    return t.reshape(*t.shape[:-2], t.shape[-2] // f, f * t.shape[-1])


CASES = [  # (n, h, w, c, k, r, s, sh, sw, ph, pw, f)
    (2, 8, 12, 3, 5, 2, 2, 2, 2, 0, 0, 2),      # 2x2 stride-2 downsample
    (1, 8, 16, 3, 4, 4, 4, 4, 4, 0, 0, 4),      # a 4x4 patch embedding
    (2, 5, 12, 2, 3, 3, 4, 1, 2, 1, 2, 2),      # padding and a W stride both divisible by 2
    (1, 6, 18, 2, 3, 2, 6, 2, 3, 0, 3, 3),      # f = 3
]


@pytest.mark.parametrize("case", CASES)
def test_fold_identity(case):
    n, h, w, c, k, r, s, sh, sw, ph, pw, f = case
    g = torch.Generator().manual_seed(7)
    x = torch.randn(n, h, w, c, dtype=torch.float64, generator=g)
    wt = torch.randn(k, r, s, c, dtype=torch.float64, generator=g)
    y = conv(x, wt, sh, sw, ph, pw)
    yf = conv(folded(x, f), folded(wt, f), sh, sw // f, ph, pw // f)
    assert yf.shape == y.shape
    assert torch.allclose(yf, y, rtol=0, atol=1e-12)
    # the gradients: dW and dX of the folded problem are the folded views of the originals'
    dy = torch.randn(*y.shape, dtype=torch.float64, generator=g)
    xa, wa = x.clone().requires_grad_(), wt.clone().requires_grad_()
    conv(xa, wa, sh, sw, ph, pw).backward(dy)
    xb, wb = folded(x, f).clone().requires_grad_(), folded(wt, f).clone().requires_grad_()
    conv(xb, wb, sh, sw // f, ph, pw // f).backward(dy)
    assert torch.allclose(wb.grad, folded(wa.grad, f), rtol=0, atol=1e-12)
    assert torch.allclose(xb.grad, folded(xa.grad, f), rtol=0, atol=1e-12)


def fw(p, d=DIR_FWD):
    return cig.describe_plan(p, d, -1, sm_count=SMS)


def test_planner_folds_when_only_the_folded_problem_has_a_fast_kernel():
    # 2x2 stride 2, C = 32: the forward tensor-core kernel wants 64-channel blocks; folded C = 64
    p = Problem(n=2, h=16, w=16, c=32, k=128, r=2, s=2, stride_h=2, stride_w=2, in_dtype=BF16, out_dtype=BF16)
    info = fw(p)
    assert info["kernel_name"] == "fwd_tc" and info["fold_width"] == 2
    # 4x4 stride 4, C = 16: folded by 4
    p = Problem(n=2, h=32, w=32, c=16, k=128, r=4, s=4, stride_h=4, stride_w=4, in_dtype=BF16, out_dtype=BF16)
    assert fw(p)["kernel_name"] == "fwd_tc" and fw(p)["fold_width"] == 4
    # a 1x2 W-stride-2 weight gradient in fp32 with 18 channels (no FFMA tiles: not a multiple of 4)
    # becomes a 1x1 one of 36 channels
    p = Problem(n=2, h=8, w=64, c=18, k=64, r=1, s=2, stride_w=2)
    assert fw(p, DIR_WGRAD)["kernel_name"] == "wgrad_1x1_tf32x3" and fw(p, DIR_WGRAD)["fold_width"] == 2
    # with 64 channels the FFMA tiles take it as given: no fold
    p = Problem(n=2, h=8, w=16, c=64, k=64, r=1, s=2, stride_w=2)
    assert fw(p, DIR_WGRAD)["kernel_name"] == "ffma" and fw(p, DIR_WGRAD)["fold_width"] == 1
    # and its data gradient (16-bit) becomes stride 1
    p = Problem(n=2, h=8, w=16, c=64, k=128, r=1, s=2, stride_w=2, in_dtype=BF16, out_dtype=BF16)
    assert fw(p, DIR_DGRAD)["kernel_name"] == "dgrad_tc" and fw(p, DIR_DGRAD)["fold_width"] == 2
    # the workspace of a folded plan is that of the folded problem (the same output count)
    assert cig.workspace_bytes(p, DIR_DGRAD, -1, sm_count=SMS) == fw(p, DIR_DGRAD)["workspace_bytes"]


def test_planner_keeps_what_needs_no_fold():
    # already on a fast kernel: no fold (the 2x2 stride-2 forward with C = 64 takes strided boxes)
    p = Problem(n=2, h=16, w=16, c=64, k=128, r=2, s=2, stride_h=2, stride_w=2, in_dtype=BF16, out_dtype=BF16)
    assert fw(p)["kernel_name"] == "fwd_tc" and fw(p)["fold_width"] == 1
    # folding would not reach a fast kernel: a 16x16 patch of 3 channels (48 after the fold)
    p = Problem(n=1, h=32, w=32, c=3, k=64, r=16, s=16, stride_h=16, stride_w=16, in_dtype=BF16, out_dtype=BF16)
    assert fw(p)["kernel_name"] == "generic" and fw(p)["fold_width"] == 1
    # not foldable: groups, W dilation, a padding or width not divisible by the filter/stride factor
    base = dict(n=2, h=16, w=16, c=32, k=128, r=2, s=2, stride_h=2, stride_w=2, in_dtype=BF16, out_dtype=BF16)
    for kw in (dict(groups=2), dict(dil_w=2, pad_w=1), dict(pad_w=1), dict(w=15)):
        p = Problem(**{**base, **kw})
        assert fw(p)["fold_width"] == 1, kw
