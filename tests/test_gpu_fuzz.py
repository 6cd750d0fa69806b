"""Seeded random shapes through every path the planner picks, against the oracle: forward and data
gradient (tensor-core tiles, persistent or not, block-diagonal, generic), weight gradient (dense 16-bit
tensor cores, fp32 FFMA tiles, grouped warp MMAs, depthwise rings, generic), at the automatic degree and
pinned ones; then grouped, depthwise, dilated and fp32 forwards and data gradients. The shapes are drawn
from fixed seeds, so every run tests the same ones."""
import random

import pytest

import implicit_gemm_convolution_nhwc_gb300 as cig
import oracle
from gpu_util import inputs, oproblem, relerr, run_dgrad, run_fwd, run_wgrad, tol

pytestmark = pytest.mark.gpu
FLOP_CAP = 3e9  # keeps each oracle call near a second


def _fwd_shapes(count, seed):
    rnd = random.Random(seed)
    out = []
    while len(out) < count:
        r = rnd.choice([1, 3, 5])
        s = rnd.choice([1, 3, 5]) if r > 1 else 1
        st = rnd.choice([1, 1, 2])
        ph = rnd.randint(0, r // 2 + 1) if r > 1 else 0
        pw = rnd.randint(0, s // 2 + 1) if s > 1 else 0
        shape = dict(n=rnd.choice([1, 2, 4, 8]), h=rnd.choice([7, 12, 14, 19, 28]), w=rnd.choice([7, 10, 14, 21, 28]),
                     c=rnd.choice([64, 128, 256]), k=rnd.choice([128, 136, 256, 320, 512]), r=r, s=s, stride_h=st,
                     stride_w=st, pad_h=ph, pad_w=pw)
        dt = rnd.choice([(cig.BF16, cig.BF16), (cig.F16, cig.F16), (cig.F16, cig.F32)])
        p = cig.Problem(**shape, in_dtype=dt[0], out_dtype=dt[1])
        if min(p.out_hw) > 0 and p.flops() <= FLOP_CAP:
            out.append(p)
    return out


def _wgrad_shapes(count, seed):
    rnd = random.Random(seed)
    out = []
    kinds = ["dense16", "fp32", "grouped", "depthwise"]
    while len(out) < count:
        kind = kinds[len(out) % 4]
        st = rnd.choice([1, 1, 2])
        if kind == "dense16":
            c, k, g = rnd.choice([64, 128, 192]), rnd.choice([128, 256, 384]), 1
            dt = rnd.choice([(cig.BF16, cig.BF16), (cig.F16, cig.F32)])
            r = rnd.choice([1, 3, 5])
        elif kind == "fp32":
            c, k, g, dt, r = rnd.choice([8, 20, 64]), rnd.choice([12, 32, 132]), 1, (cig.F32, cig.F32), rnd.choice([1, 3])
        elif kind == "grouped":
            cg, g = rnd.choice([4, 8]), rnd.choice([16, 32])
            c = k = cg * g
            dt, r = rnd.choice([(cig.F16, cig.F16), (cig.BF16, cig.F32)]), rnd.choice([3, 5])
        else:
            c = k = g = rnd.choice([64, 128])
            dt, r = rnd.choice([(cig.BF16, cig.BF16), (cig.F16, cig.F32)]), rnd.choice([3, 5, 7])
        ph, pw = rnd.randint(0, r // 2), rnd.randint(0, r // 2)
        p = cig.Problem(n=rnd.choice([1, 2, 3, 5]), h=rnd.choice([6, 9, 14, 17, 28]), w=rnd.choice([5, 8, 14, 19, 28]),
                        c=c, k=k, r=r, s=r, stride_h=st, stride_w=st, pad_h=ph, pad_w=pw, groups=g,
                        in_dtype=dt[0], out_dtype=dt[1])
        if min(p.out_hw) > 0 and p.flops() <= FLOP_CAP:
            out.append(p)
    return out


def _other_fwd_shapes(count, seed):
    """Grouped (4 or 8 channels a group: warp MMAs; 16 to 64: block-diagonal tiles), depthwise, dilated
    16-bit and fp32 problems."""
    rnd = random.Random(seed)
    out = []
    kinds = ["grouped_mma", "grouped_tc", "depthwise", "dilated16", "fp32"]
    while len(out) < count:
        kind = kinds[len(out) % len(kinds)]
        st, dil = 1, 1
        dt = rnd.choice([(cig.BF16, cig.BF16), (cig.F16, cig.F16), (cig.BF16, cig.F32)])
        if kind == "grouped_mma":
            cg, g, r = rnd.choice([4, 8]), rnd.choice([16, 32, 64]), rnd.choice([1, 3, 5])
            c = k = cg * g
        elif kind == "grouped_tc":
            cg, g, r = rnd.choice([16, 32, 64]), rnd.choice([2, 4, 8]), rnd.choice([3, 5])
            c = k = cg * g
        elif kind == "depthwise":
            c = k = g = rnd.choice([32, 64, 96, 128])
            r, st = rnd.choice([3, 5, 7]), rnd.choice([1, 1, 2])
        elif kind == "dilated16":
            c, k, g, r, dil = rnd.choice([64, 128]), rnd.choice([128, 256]), 1, 3, rnd.choice([2, 3])
        else:
            c, k, g, r = rnd.choice([8, 24, 64]), rnd.choice([16, 40, 128]), 1, rnd.choice([1, 3])
            st, dil, dt = rnd.choice([1, 2]), rnd.choice([1, 2]), (cig.F32, cig.F32)
        ph = rnd.randint(0, dil * (r - 1))
        pw = rnd.randint(0, dil * (r - 1))
        p = cig.Problem(n=rnd.choice([1, 2, 4]), h=rnd.choice([8, 13, 16, 21]), w=rnd.choice([8, 11, 16, 24]), c=c, k=k,
                        r=r, s=r, stride_h=st, stride_w=st, pad_h=ph, pad_w=pw, dil_h=dil, dil_w=dil, groups=g,
                        in_dtype=dt[0], out_dtype=dt[1])
        if min(p.out_hw) > 0 and p.flops() <= FLOP_CAP:
            out.append(p)
    return out


def _top(p, direction, bias=False):
    """The largest degree a pinned request may take on this problem's kernel."""
    return cig.describe_plan(p, direction, -1, bias)["max_split"]


@pytest.mark.parametrize("i", range(24))
def test_fuzz_forward_and_dgrad(i):
    p = _fwd_shapes(24, 7)[i]
    orc = oracle.get()
    top = _top(p, cig.DIR_FWD)
    x, w = inputs(p, 50 + i, "normal", 0.0, 0.05, cig.DIR_FWD)
    ref = orc.fwd(oproblem(p), x, w)
    for sk in (-1, 1, 3):
        if sk <= top:
            e = relerr(run_fwd(p, x, w, sk), ref)
            assert e <= tol(p), (p, sk, e)
    if p.stride_h == 1:
        top = _top(p, cig.DIR_DGRAD)
        dy, w2 = inputs(p, 150 + i, "normal", 0.0, 0.05, cig.DIR_DGRAD)
        dref = orc.dgrad(oproblem(p), dy, w2)
        for sk in (-1, 2):
            if sk <= top:
                e = relerr(run_dgrad(p, dy, w2, sk), dref)
                assert e <= tol(p), (p, sk, e)
    assert cig.device_errors() == 0


@pytest.mark.parametrize("i", range(32))
def test_fuzz_wgrad(i):
    p = _wgrad_shapes(32, 11)[i]
    orc = oracle.get()
    top = _top(p, cig.DIR_WGRAD, True)
    x, dy = inputs(p, 250 + i, "normal", 0.0, 0.05, cig.DIR_WGRAD)
    ref, bref = orc.wgrad(oproblem(p), x, dy), orc.bgrad(oproblem(p), dy)
    for sk in (-1, 1, 3):
        if sk <= top:
            dw, db = run_wgrad(p, x, dy, sk, True)
            assert relerr(dw, ref) <= tol(p) and relerr(db, bref) <= tol(p), (p, sk)
    assert cig.device_errors() == 0


@pytest.mark.parametrize("i", range(30))
def test_fuzz_other_forward_and_dgrad(i):
    p = _other_fwd_shapes(30, 13)[i]
    orc = oracle.get()
    x, w = inputs(p, 350 + i, "normal", 0.0, 0.05, cig.DIR_FWD)
    ref = orc.fwd(oproblem(p), x, w)
    top = _top(p, cig.DIR_FWD)
    for sk in (-1, 1, 2):
        if sk <= top:
            assert relerr(run_fwd(p, x, w, sk), ref) <= tol(p), (p, sk)
    dy, w2 = inputs(p, 450 + i, "normal", 0.0, 0.05, cig.DIR_DGRAD)
    dref = orc.dgrad(oproblem(p), dy, w2)
    top = _top(p, cig.DIR_DGRAD)
    for sk in (-1, 2):
        if sk <= top:
            assert relerr(run_dgrad(p, dy, w2, sk), dref) <= tol(p), (p, sk)
    assert cig.device_errors() == 0
