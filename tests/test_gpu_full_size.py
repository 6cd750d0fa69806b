"""Full-size parity of the >4 GB 1x1 fp32 weight + bias gradient, in the launch
configuration the bench times (auto split-K).

The oracle computes every output (all 64 x 96 of dW and all of db), streaming
the inputs sample by sample from the seeded generator, and the GPU result is
compared element by element. The last batch sample is also run alone at its
>6 GB offset: the failure on the pages was a silently zero or wrong weight
gradient once a dispatch addressed more than ~4 GB ("ROCm/rocm-libraries PR
#11188", "Motivation")."""
import numpy as np
import pytest
import torch

import oracle
import synth
import implicit_gemm_convolution_nhwc_gb300 as cig
from gpu_util import oproblem, relerr

pytestmark = pytest.mark.gpu

C, K, HW = 96, 64, 512


def device_inputs(n, seed=1):
    """X [n,512,512,96] and dY [n,512,512,64] fp32 ~ N(0,1), streamed to the device."""
    x = torch.empty((n, HW, HW, C), dtype=torch.float32, device="cuda")
    dy = torch.empty((n, HW, HW, K), dtype=torch.float32, device="cuda")
    for t, tid in ((x, synth.X_ID), (dy, synth.DY_ID)):
        per = t[0].numel()
        stage = torch.empty(per, dtype=torch.float32, pin_memory=True)
        for i in range(n):
            synth.fill(stage, "normal", 0.0, 1.0, seed, tid, offset=i * per)
            t[i].view(-1).copy_(stage)
    return x, dy


def oracle_rows(n_begin, n_end, seed=1, dw=None, db=None):
    """Oracle dW (every row) and db over samples [n_begin, n_end), added into dw / db."""
    orc = oracle.get()
    p1 = oracle.Problem(n=1, h=HW, w=HW, c=C, k=K)
    dw = np.zeros((K, 1, 1, C)) if dw is None else dw
    db = np.zeros(K) if db is None else db
    x = np.empty((1, HW, HW, C), np.float32)
    dy = np.empty((1, HW, HW, K), np.float32)
    for i in range(n_begin, n_end):
        synth.fill(x, "normal", 0.0, 1.0, seed, synth.X_ID, offset=i * x.size)
        synth.fill(dy, "normal", 0.0, 1.0, seed, synth.DY_ID, offset=i * dy.size)
        orc.wgrad_acc(p1, x, dy, dw)
        orc.bgrad_acc(p1, dy, db)
    return dw, db


def gpu_wgrad(x, dy, n):
    p = cig.Problem(n=n, h=HW, w=HW, c=C, k=K)
    dw = torch.empty((K, 1, 1, C), device="cuda")
    db = torch.empty(K, device="cuda")
    ws = cig.workspace(p, cig.DIR_WGRAD, -1, True)
    cig.conv_wgrad_bias(p, x, dy, dw, db, ws, -1)
    torch.cuda.synchronize()
    return dw.cpu(), db.cpu()


def test_config2_n64_sampled_rows_and_last_sample():
    x, dy = device_inputs(64)
    assert x.numel() * 4 > 2 ** 32 and dy.numel() * 4 >= 2 ** 32
    dw, db = gpu_wgrad(x, dy, 64)
    ref_w, ref_b = oracle_rows(0, 64)
    assert relerr(dw, ref_w) <= 1e-5
    assert relerr(db, ref_b) <= 1e-5
    # every row non-zero, including rows 32..63 (the second 32-channel dY box)
    assert float(dw.abs().amax(dim=(1, 2, 3)).min()) > 100.0
    # run-to-run bit identity at the same (auto) degree
    dw2, db2 = gpu_wgrad(x, dy, 64)
    assert torch.equal(dw, dw2) and torch.equal(db, db2)
    # the last sample alone, read at its offset past 6 GB: non-zero and correct
    last_w, last_b = gpu_wgrad(x[63:], dy[63:], 1)
    ref_lw, ref_lb = oracle_rows(63, 64)
    assert float(last_w.abs().amax(dim=(1, 2, 3)).min()) > 100.0
    assert relerr(last_w, ref_lw) <= 1e-5
    assert relerr(last_b, ref_lb) <= 1e-5


def test_config2_batch_sweep():
    """N = 43, 59, ..., 187 (the pages' sweep range, step 16): every N against the oracle."""
    ns = list(range(43, 193, 16))
    free, _ = torch.cuda.mem_get_info()
    need = ns[-1] * HW * HW * (C + K) * 4
    if need > free * 0.9:
        pytest.skip(f"needs {need / 1e9:.1f} GB of device memory")
    x, dy = device_inputs(ns[-1])
    dw_ref, db_ref = np.zeros((K, 1, 1, C)), np.zeros(K)
    done = 0
    for n in ns:
        oracle_rows(done, n, dw=dw_ref, db=db_ref)  # the prefix sums, extended
        done = n
        dw, db = gpu_wgrad(x[:n], dy[:n], n)
        assert relerr(dw, dw_ref) <= 1e-5, n
        assert relerr(db, db_ref) <= 1e-5, n


def test_fwd3x3_compute_bound_supplement_sampled_images():
    """3x3 fwd bf16, N=64, 56x56, C=K=256, pad 1, in the bench's launch
    configuration (auto). An image's output depends on that image alone, so the
    oracle runs images 0, 31 and 63 as N=1 problems on the same W."""
    n, hw, c, k = 64, 56, 256, 256
    p = cig.Problem(n=n, h=hw, w=hw, c=c, k=k, r=3, s=3, pad_h=1, pad_w=1, in_dtype=cig.BF16, out_dtype=cig.BF16)
    x = synth.tensor((n, hw, hw, c), torch.bfloat16, "normal", 0.0, 0.02, 5, synth.X_ID)
    w = synth.tensor((k, 3, 3, c), torch.bfloat16, "normal", 0.0, 0.02, 5, synth.W_ID)
    y = torch.empty((n, hw, hw, k), dtype=torch.bfloat16, device="cuda")
    ws = cig.workspace(p, cig.DIR_FWD, -1, False)
    assert cig.describe_plan(p, cig.DIR_FWD, -1)["kernel_name"] == "fwd_tc"
    cig.conv_fwd(p, x.cuda(), w.cuda(), y, ws, -1)
    torch.cuda.synchronize()
    yc = y.cpu()
    orc = oracle.get()
    p1 = cig.Problem(n=1, h=hw, w=hw, c=c, k=k, r=3, s=3, pad_h=1, pad_w=1, in_dtype=cig.BF16, out_dtype=cig.BF16)
    for i in (0, 31, 63):
        ref = orc.fwd(oproblem(p1), x[i:i + 1], w)
        e = relerr(yc[i:i + 1], ref)
        assert e <= 1e-2, f"image {i}: err {e:.3e}"
    assert cig.device_errors() == 0


def test_dgrad3x3_compute_bound_supplement_sampled_images():
    """The supplement backwards (dX of the 3x3 bf16 N=64, 56x56, C=K=256
    layer, auto): images 0 and 63 against the oracle as N=1 problems."""
    n, hw, c, k = 64, 56, 256, 256
    p = cig.Problem(n=n, h=hw, w=hw, c=c, k=k, r=3, s=3, pad_h=1, pad_w=1, in_dtype=cig.BF16, out_dtype=cig.BF16)
    dy = synth.tensor((n, hw, hw, k), torch.bfloat16, "normal", 0.0, 0.02, 5, synth.DY_ID)
    w = synth.tensor((k, 3, 3, c), torch.bfloat16, "normal", 0.0, 0.02, 5, synth.W_ID)
    dx = torch.empty((n, hw, hw, c), dtype=torch.bfloat16, device="cuda")
    assert cig.describe_plan(p, cig.DIR_DGRAD, -1)["kernel_name"] == "dgrad_tc"
    ws = cig.workspace(p, cig.DIR_DGRAD, -1, False)
    cig.conv_dgrad(p, dy.cuda(), w.cuda(), dx, ws, -1)
    torch.cuda.synchronize()
    dxc = dx.cpu()
    orc = oracle.get()
    p1 = cig.Problem(n=1, h=hw, w=hw, c=c, k=k, r=3, s=3, pad_h=1, pad_w=1, in_dtype=cig.BF16, out_dtype=cig.BF16)
    for i in (0, 63):
        ref = orc.dgrad(oproblem(p1), dy[i:i + 1], w)
        e = relerr(dxc[i:i + 1], ref)
        assert e <= 1e-2, f"image {i}: err {e:.3e}"
    assert cig.device_errors() == 0


@pytest.mark.parametrize("direction", ["fwd", "dgrad"])
def test_two_m_subtiles_with_a_partial_second(direction):
    """512 images of 14x14 (K = C = 256, 3x3, pad 1, bf16): enough tiles for CTAs with two M
    sub-tiles of 9 output rows sharing the weight tile, the second one cut at row 14.
    Images 0, 1 and 511 against the oracle as N=1 problems."""
    n, hw, c, k = 512, 14, 256, 256
    p = cig.Problem(n=n, h=hw, w=hw, c=c, k=k, r=3, s=3, pad_h=1, pad_w=1, in_dtype=cig.BF16, out_dtype=cig.BF16)
    p1 = cig.Problem(n=1, h=hw, w=hw, c=c, k=k, r=3, s=3, pad_h=1, pad_w=1, in_dtype=cig.BF16, out_dtype=cig.BF16)
    w = synth.tensor((k, 3, 3, c), torch.bfloat16, "normal", 0.0, 0.05, 8, synth.W_ID)
    orc = oracle.get()
    if direction == "fwd":
        info = cig.describe_plan(p, cig.DIR_FWD, -1)
        assert info["kernel_name"] == "fwd_tc" and info["tiles"] == n  # one double tile per image
        a = synth.tensor((n, hw, hw, c), torch.bfloat16, "normal", 0.0, 0.05, 8, synth.X_ID)
        out = torch.empty((n, hw, hw, k), dtype=torch.bfloat16, device="cuda")
        cig.conv_fwd(p, a.cuda(), w.cuda(), out, cig.workspace(p, cig.DIR_FWD, -1, False), -1)
    else:
        info = cig.describe_plan(p, cig.DIR_DGRAD, -1)
        assert info["kernel_name"] == "dgrad_tc" and info["tiles"] == n
        a = synth.tensor((n, hw, hw, k), torch.bfloat16, "normal", 0.0, 0.05, 8, synth.DY_ID)
        out = torch.empty((n, hw, hw, c), dtype=torch.bfloat16, device="cuda")
        cig.conv_dgrad(p, a.cuda(), w.cuda(), out, cig.workspace(p, cig.DIR_DGRAD, -1, False), -1)
    torch.cuda.synchronize()
    got = out.cpu()
    for i in (0, 1, 511):
        ref = orc.fwd(oproblem(p1), a[i:i + 1], w) if direction == "fwd" else orc.dgrad(oproblem(p1), a[i:i + 1], w)
        e = relerr(got[i:i + 1], ref)
        assert e <= 1e-2, f"{direction} image {i}: err {e:.3e}"
    assert cig.device_errors() == 0


@pytest.mark.parametrize("direction", ["fwd", "fwd_bias_relu", "dgrad"])
def test_two_m_subtiles_the_last_pair_single(direction):
    """128 images of 28x28 (K = C = 256, 3x3, pad 1, bf16): 512 double tiles of two M sub-tiles of 4
    output rows, over 152 persistent CTAs (the accumulator of a unit freed one sub-tile at a time); each
    image's last double tile holds rows 24..27 only, so its second sub-tile lies past the image.
    Images 0, 1 and 127 against the oracle as N=1 problems."""
    n, hw, c, k = 128, 28, 256, 256
    p = cig.Problem(n=n, h=hw, w=hw, c=c, k=k, r=3, s=3, pad_h=1, pad_w=1, in_dtype=cig.BF16, out_dtype=cig.BF16)
    p1 = cig.Problem(n=1, h=hw, w=hw, c=c, k=k, r=3, s=3, pad_h=1, pad_w=1, in_dtype=cig.BF16, out_dtype=cig.BF16)
    w = synth.tensor((k, 3, 3, c), torch.bfloat16, "normal", 0.0, 0.05, 9, synth.W_ID)
    bias = synth.tensor((k,), torch.bfloat16, "normal", 0.0, 0.1, 9, synth.BIAS_ID)
    orc = oracle.get()
    if direction != "dgrad":
        info = cig.describe_plan(p, cig.DIR_FWD, -1)
        assert info["kernel_name"] == "fwd_tc" and info["tiles"] == 4 * n and info["split_k"] == 1, info
        a = synth.tensor((n, hw, hw, c), torch.bfloat16, "normal", 0.0, 0.05, 9, synth.X_ID)
        out = torch.empty((n, hw, hw, k), dtype=torch.bfloat16, device="cuda")
        if direction == "fwd":
            cig.conv_fwd(p, a.cuda(), w.cuda(), out, cig.workspace(p, cig.DIR_FWD, -1, False), -1)
        else:
            cig.conv_fwd_epilogue(p, a.cuda(), w.cuda(), out, bias.cuda(), 0.0, float("inf"), None, -1)
    else:
        info = cig.describe_plan(p, cig.DIR_DGRAD, -1)
        assert info["kernel_name"] == "dgrad_tc" and info["tiles"] == 4 * n and info["split_k"] == 1, info
        a = synth.tensor((n, hw, hw, k), torch.bfloat16, "normal", 0.0, 0.05, 9, synth.DY_ID)
        out = torch.empty((n, hw, hw, c), dtype=torch.bfloat16, device="cuda")
        cig.conv_dgrad(p, a.cuda(), w.cuda(), out, cig.workspace(p, cig.DIR_DGRAD, -1, False), -1)
    torch.cuda.synchronize()
    got = out.cpu()
    for i in (0, 1, 127):
        if direction == "fwd":
            ref = orc.fwd(oproblem(p1), a[i:i + 1], w)
        elif direction == "fwd_bias_relu":
            ref = orc.fwd_epilogue(oproblem(p1), a[i:i + 1], w, bias, 0.0, float("inf"))
        else:
            ref = orc.dgrad(oproblem(p1), a[i:i + 1], w)
        e = relerr(got[i:i + 1], ref)
        assert e <= 1e-2, f"{direction} image {i}: err {e:.3e}"
    assert cig.device_errors() == 0

def test_depthwise_7x7_forward_full_sampled_images():
    """Depthwise 7x7 forward bf16, N=32, 56x56, C=K=384, pad 3 (the depthwise configuration's
    forward twin), auto: images 0, 17 and 31 against the oracle as N=1 problems."""
    n, hw, c = 32, 56, 384
    p = cig.Problem(n=n, h=hw, w=hw, c=c, k=c, r=7, s=7, pad_h=3, pad_w=3, groups=c,
                    in_dtype=cig.BF16, out_dtype=cig.BF16)
    assert cig.describe_plan(p, cig.DIR_FWD, -1)["kernel_name"] == "fwd_depthwise"
    x = synth.tensor((n, hw, hw, c), torch.bfloat16, "normal", 0.0, 1.0, 3, synth.X_ID)
    w = synth.tensor((c, 7, 7, 1), torch.bfloat16, "normal", 0.0, 1.0, 3, synth.W_ID)
    y = torch.empty((n, hw, hw, c), dtype=torch.bfloat16, device="cuda")
    cig.conv_fwd(p, x.cuda(), w.cuda(), y, None, -1)
    torch.cuda.synchronize()
    yc = y.cpu()
    orc = oracle.get()
    p1 = cig.Problem(n=1, h=hw, w=hw, c=c, k=c, r=7, s=7, pad_h=3, pad_w=3, groups=c,
                     in_dtype=cig.BF16, out_dtype=cig.BF16)
    for i in (0, 17, 31):
        e = relerr(yc[i:i + 1], orc.fwd(oproblem(p1), x[i:i + 1], w))
        assert e <= 1e-2, f"image {i}: err {e:.3e}"
    assert cig.device_errors() == 0


@pytest.mark.parametrize("groups", [64, 128], ids=["cpg8", "cpg4"])
def test_grouped_3x3_forward_full_sampled_images(groups):
    """Grouped 3x3 forward fp16, N=64, 28x28, C=K=512 (the grouped configuration's forward
    twin), auto (the grouped warp-MMA kernel): images 0 and 63 against the oracle."""
    n, hw, c = 64, 28, 512
    p = cig.Problem(n=n, h=hw, w=hw, c=c, k=c, r=3, s=3, pad_h=1, pad_w=1, groups=groups,
                    in_dtype=cig.F16, out_dtype=cig.F16)
    assert cig.describe_plan(p, cig.DIR_FWD, -1)["kernel_name"] == "fwd_grouped_mma"
    x = synth.tensor((n, hw, hw, c), torch.float16, "normal", 0.0, 1.0, 4, synth.X_ID)
    w = synth.tensor((c, 3, 3, c // groups), torch.float16, "normal", 0.0, 1.0, 4, synth.W_ID)
    y = torch.empty((n, hw, hw, c), dtype=torch.float16, device="cuda")
    cig.conv_fwd(p, x.cuda(), w.cuda(), y, cig.workspace(p, cig.DIR_FWD, -1, False), -1)
    torch.cuda.synchronize()
    yc = y.cpu()
    orc = oracle.get()
    p1 = cig.Problem(n=1, h=hw, w=hw, c=c, k=c, r=3, s=3, pad_h=1, pad_w=1, groups=groups,
                     in_dtype=cig.F16, out_dtype=cig.F16)
    for i in (0, 63):
        e = relerr(yc[i:i + 1], orc.fwd(oproblem(p1), x[i:i + 1], w))
        assert e <= 1e-2, f"image {i}: err {e:.3e}"
    assert cig.device_errors() == 0


def test_depthwise_7x7_dgrad_full():
    """Depthwise 7x7 data gradient bf16, N=32, 56x56, C=K=384, pad 3 (the depthwise configuration's layer
    backwards; dY ~ N(0, 1) seed 3, W as in the forward), auto: every element against the oracle."""
    n, hw, c = 32, 56, 384
    p = cig.Problem(n=n, h=hw, w=hw, c=c, k=c, r=7, s=7, pad_h=3, pad_w=3, groups=c,
                    in_dtype=cig.BF16, out_dtype=cig.BF16)
    assert cig.describe_plan(p, cig.DIR_DGRAD, -1)["kernel_name"] == "dgrad_depthwise"
    dy = synth.tensor((n, hw, hw, c), torch.bfloat16, "normal", 0.0, 1.0, 3, synth.DY_ID)
    w = synth.tensor((c, 7, 7, 1), torch.bfloat16, "normal", 0.0, 1.0, 3, synth.W_ID)
    dx = torch.empty((n, hw, hw, c), dtype=torch.bfloat16, device="cuda")
    cig.conv_dgrad(p, dy.cuda(), w.cuda(), dx, None, -1)
    torch.cuda.synchronize()
    e = relerr(dx.cpu(), oracle.get().dgrad(oproblem(p), dy, w))
    assert e <= 1e-2, f"err {e:.3e}"
    assert cig.device_errors() == 0


@pytest.mark.parametrize("groups", [64, 128], ids=["cpg8", "cpg4"])
def test_grouped_3x3_dgrad_full(groups):
    """Grouped 3x3 data gradient fp16, N=64, 28x28, C=K=512 (the grouped configuration's layer backwards;
    dY ~ N(0, 1) seed 4), auto: every element against the oracle."""
    n, hw, c = 64, 28, 512
    p = cig.Problem(n=n, h=hw, w=hw, c=c, k=c, r=3, s=3, pad_h=1, pad_w=1, groups=groups,
                    in_dtype=cig.F16, out_dtype=cig.F16)
    assert cig.describe_plan(p, cig.DIR_DGRAD, -1)["kernel_name"] == "dgrad_grouped_mma"
    dy = synth.tensor((n, hw, hw, c), torch.float16, "normal", 0.0, 1.0, 4, synth.DY_ID)
    w = synth.tensor((c, 3, 3, c // groups), torch.float16, "normal", 0.0, 1.0, 4, synth.W_ID)
    dx = torch.empty((n, hw, hw, c), dtype=torch.float16, device="cuda")
    cig.conv_dgrad(p, dy.cuda(), w.cuda(), dx, cig.workspace(p, cig.DIR_DGRAD, -1, False), -1)
    torch.cuda.synchronize()
    e = relerr(dx.cpu(), oracle.get().dgrad(oproblem(p), dy, w))
    assert e <= 1e-2, f"err {e:.3e}"
    assert cig.device_errors() == 0
