"""GPU parity of the dense 16-bit weight gradient on the tensor cores
(CONV_KERNEL_WGRAD_TC) against the CPU oracle, element by element, through the
C ABI: ragged pixel blocks, channel tails in both operands, output-channel
tails in the second M sub-tile, strides, dilations, non-square filters, a
1x1, a wide image and a grouped problem; every output type; automatic,
pinned and maximal split-K degrees with the workspace pre-filled with NaN
bytes; canaries around every output; bit-identical reruns. Plus the
compute-bound 3x3 bf16 N=64 56x56 C=K=256 layer at full size."""
import numpy as np
import pytest
import torch

import oracle
import synth
import implicit_gemm_convolution_nhwc_gb300 as cig
from gpu_util import inputs, oproblem, relerr, run_wgrad, tol

pytestmark = pytest.mark.gpu

BF16, F16, F32 = cig.BF16, cig.F16, cig.F32

SHAPES = [
    dict(n=2, h=9, w=11, c=72, k=136, r=3, s=3, pad_h=1, pad_w=1),          # c tail, 8-row second sub-tile
    dict(n=3, h=13, w=10, c=64, k=64, r=3, s=2, stride_h=2, pad_h=1, dil_h=2),  # strided, dilated, 3x2
    dict(n=1, h=17, w=19, c=256, k=264, r=5, s=5, pad_h=2, pad_w=2),        # two k tiles, the second 8 rows
    dict(n=4, h=16, w=16, c=128, k=256),                                     # 1x1
    dict(n=2, h=20, w=21, c=96, k=200, r=3, s=3, stride_h=2, stride_w=2, pad_h=1, pad_w=1),
    dict(n=2, h=12, w=12, c=128, k=256, r=3, s=3, pad_h=1, pad_w=1, groups=2),  # Cg = 64, Kg = 128
    dict(n=1, h=6, w=150, c=64, k=128, r=1, s=3, pad_w=1),                  # several pixel blocks per row
    dict(n=2, h=10, w=14, c=64, k=128, r=3, s=3, pad_h=2, pad_w=2, dil_h=2, dil_w=2),
]
DTYPES = [(BF16, BF16), (BF16, F32), (F16, F16), (F16, F32)]


@pytest.fixture(autouse=True)
def _reset_override():
    cig.set_kernel_override("auto")
    yield
    cig.set_kernel_override("auto")


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("dt", DTYPES, ids=lambda d: f"{d[0]}{d[1]}")
def test_wgrad_tc_parity(shape, dt):
    p = cig.Problem(**shape, in_dtype=dt[0], out_dtype=dt[1])
    info = cig.describe_plan(p, cig.DIR_WGRAD, -1, True)
    assert info["kernel_name"] == "wgrad_tc"
    orc = oracle.get()
    x, dy = inputs(p, 31)
    ref_w = orc.wgrad(oproblem(p), x, dy)
    ref_b = orc.bgrad(oproblem(p), dy)
    top = info["max_split"]
    for sk in sorted({-1, 1, 2, min(5, top), top}):
        dw, db = run_wgrad(p, x, dy, sk, True)
        e = relerr(dw, ref_w)
        assert e <= tol(p), f"split {sk}: dW err {e:.3e}"
        eb = relerr(db, ref_b)
        assert eb <= tol(p), f"split {sk}: db err {eb:.3e}"
    assert cig.device_errors() == 0


def test_wgrad_tc_without_bias_and_reruns_bit_identical():
    p = cig.Problem(n=3, h=14, w=14, c=192, k=320, r=3, s=3, pad_h=1, pad_w=1, in_dtype=BF16, out_dtype=BF16)
    assert cig.describe_plan(p, cig.DIR_WGRAD, -1)["kernel_name"] == "wgrad_tc"
    x, dy = inputs(p, 32)
    ref = oracle.get().wgrad(oproblem(p), x, dy)
    for sk in (-1, 3):
        outs = [run_wgrad(p, x, dy, sk, False)[0] for _ in range(3)]
        assert relerr(outs[0], ref) <= tol(p)
        for o in outs[1:]:
            assert torch.equal(o, outs[0])
    # with the bias at the same degree: the same dW bits
    dw_b, _ = run_wgrad(p, x, dy, 3, True)
    assert torch.equal(dw_b, run_wgrad(p, x, dy, 3, False)[0])
    assert cig.device_errors() == 0


def test_wgrad_tc_uniform_small_integers_exact():
    """Small-integer inputs make every product and partial sum exact in fp32, so
    any degree must give exactly the oracle's value (catches a dropped or doubled
    pixel block, which tolerance could hide on random data)."""
    p = cig.Problem(n=2, h=11, w=9, c=64, k=136, r=3, s=3, pad_h=1, pad_w=1, in_dtype=BF16, out_dtype=F32)
    x = synth.tensor((p.n, p.h, p.w, p.c), torch.bfloat16, "integer", -3, 3, 33, synth.X_ID)
    ho, wo = p.out_hw
    dy = synth.tensor((p.n, ho, wo, p.k), torch.bfloat16, "integer", -3, 3, 33, synth.DY_ID)
    ref_w = oracle.get().wgrad(oproblem(p), x, dy)
    ref_b = oracle.get().bgrad(oproblem(p), dy)
    for sk in (-1, 1, 2, 4):
        dw, db = run_wgrad(p, x, dy, sk, True)
        assert np.array_equal(dw.double().numpy(), ref_w), sk
        assert np.array_equal(db.double().numpy(), ref_b), sk


def test_wgrad_tc_compute_bound_supplement_full():
    """3x3 wgrad + db bf16, N=64, 56x56, C=K=256, pad 1, N(0, 0.02) seed 5, in the bench's launch
    configuration (auto split-K). The oracle computes rows 120..135 (across the two M sub-tiles) and
    248..255 of dW over the whole batch, and all of db."""
    n, hw, c, k = 64, 56, 256, 256
    p = cig.Problem(n=n, h=hw, w=hw, c=c, k=k, r=3, s=3, pad_h=1, pad_w=1, in_dtype=BF16, out_dtype=BF16)
    info = cig.describe_plan(p, cig.DIR_WGRAD, -1, True, torch.cuda.get_device_properties(0).multi_processor_count)
    assert info["kernel_name"] == "wgrad_tc" and info["split_k"] > 1
    x = synth.tensor((n, hw, hw, c), torch.bfloat16, "normal", 0.0, 0.02, 5, synth.X_ID)
    dy = synth.tensor((n, hw, hw, k), torch.bfloat16, "normal", 0.0, 0.02, 5, synth.DY_ID)
    dw, db = run_wgrad(p, x, dy, -1, True)
    dw2, db2 = run_wgrad(p, x, dy, -1, True)
    assert torch.equal(dw, dw2) and torch.equal(db, db2)
    orc = oracle.get()
    ref = np.zeros((k, 3, 3, c))
    for rows in ((120, 136), (248, 256)):
        orc.wgrad_acc(oproblem(p), x, dy, ref, rows)
    ref_b = orc.bgrad(oproblem(p), dy)
    for k0, k1 in ((120, 136), (248, 256)):
        e = relerr(dw[k0:k1], ref[k0:k1])
        assert e <= 1e-2, f"rows {k0}..{k1}: err {e:.3e}"
    assert relerr(db, ref_b) <= 1e-2
    assert cig.device_errors() == 0
