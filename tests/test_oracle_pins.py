"""Pins for the CPU oracle against things other than itself.

Each check below is independent of the oracle's own loops: closed forms
(a 1x1 weight gradient is a GEMM; the bias gradient is a sum; an all-ones
problem counts valid taps), a library routine (torch's float64 conv2d and its
weight gradient; scipy's 2-D correlation for depthwise), brute force through
an explicitly built im2col matrix, and the adjoint identity that ties the
forward and the weight gradient. The last test plants mistakes in copies of
the oracle's source and checks that some pin catches every one.
"""
import itertools
import os

import numpy as np
import pytest
import torch

import oracle
import synth
from oracle import Oracle, Problem

RNG = np.random.default_rng(1234)


def rand(shape, seed, tid, dist="uniform", a=-1.0, b=1.0):
    arr = np.empty(shape, dtype=np.float32)
    synth.fill(arr, dist, a, b, seed, tid)
    return arr


def torch_fwd(p: Problem, x, w):
    """Y via torch.nn.functional.conv2d in float64 (NCHW inside, NHWC out)."""
    xt = torch.from_numpy(np.asarray(x, np.float64)).permute(0, 3, 1, 2)
    wt = torch.from_numpy(np.asarray(w, np.float64)).permute(0, 3, 1, 2)
    y = torch.nn.functional.conv2d(xt, wt, stride=(p.stride_h, p.stride_w),
                                   padding=(p.pad_h, p.pad_w), dilation=(p.dil_h, p.dil_w),
                                   groups=p.groups)
    return y.permute(0, 2, 3, 1).numpy()


def torch_wgrad(p: Problem, x, dy):
    """dW via autograd of torch's float64 conv2d."""
    xt = torch.from_numpy(np.asarray(x, np.float64)).permute(0, 3, 1, 2)
    wt = torch.zeros((p.k, p.c // p.groups, p.r, p.s), dtype=torch.float64, requires_grad=True)
    y = torch.nn.functional.conv2d(xt, wt, stride=(p.stride_h, p.stride_w),
                                   padding=(p.pad_h, p.pad_w), dilation=(p.dil_h, p.dil_w),
                                   groups=p.groups)
    y.backward(torch.from_numpy(np.asarray(dy, np.float64)).permute(0, 3, 1, 2))
    return wt.grad.permute(0, 2, 3, 1).numpy()


def relerr(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    scale = max(np.abs(b).max(), 1e-300)
    return float(np.abs(a - b).max() / scale)


# A spread of shapes: strides, dilations, asymmetric padding, groups,
# non-square filters, ragged sizes, padding larger than the filter reach.
SHAPES = [
    Problem(n=2, h=7, w=9, c=6, k=4, r=3, s=2, stride_h=1, stride_w=2, pad_h=1, pad_w=0, dil_h=1, dil_w=1, groups=1),
    Problem(n=1, h=8, w=8, c=8, k=6, r=3, s=3, stride_h=2, stride_w=2, pad_h=1, pad_w=1, dil_h=2, dil_w=1, groups=2),
    Problem(n=3, h=5, w=6, c=4, k=4, r=5, s=3, stride_h=1, stride_w=1, pad_h=2, pad_w=3, dil_h=1, dil_w=2, groups=4),
    Problem(n=2, h=9, w=7, c=12, k=8, r=1, s=4, stride_h=3, stride_w=1, pad_h=0, pad_w=2, dil_h=1, dil_w=1, groups=4),
    Problem(n=1, h=6, w=6, c=3, k=5, r=2, s=2, stride_h=1, stride_w=1, pad_h=0, pad_w=0, dil_h=3, dil_w=3, groups=1),
]


def _inputs(p: Problem, orc: Oracle, seed=7):
    ho, wo = orc.out_hw(p)
    x = rand((p.n, p.h, p.w, p.c), seed, synth.X_ID)
    w = rand((p.k, p.r, p.s, p.c // p.groups), seed, synth.W_ID)
    dy = rand((p.n, ho, wo, p.k), seed, synth.DY_ID)
    return x, w, dy


# --------------------------------------------------------------- pins


def pin_1x1_gemm(orc: Oracle):
    """A 1x1 weight gradient is dY^T X on the [N*H*W, C] view (the F.linear form)."""
    p = Problem(n=4, h=16, w=16, c=8, k=16)
    x = rand((4, 16, 16, 8), 0, synth.X_ID)
    dy = rand((4, 16, 16, 16), 0, synth.DY_ID)
    ref = dy.reshape(-1, 16).astype(np.float64).T @ x.reshape(-1, 8).astype(np.float64)
    return relerr(orc.wgrad(p, x, dy).reshape(16, 8), ref) <= 1e-12


def pin_bias_sum(orc: Oracle):
    p = SHAPES[1]
    _, _, dy = _inputs(p, orc)
    return relerr(orc.bgrad(p, dy), dy.astype(np.float64).sum(axis=(0, 1, 2))) <= 1e-12


def pin_torch_fwd(orc: Oracle):
    for p in SHAPES:
        x, w, _ = _inputs(p, orc)
        y = orc.fwd(p, x, w)
        ref = torch_fwd(p, x, w)
        if y.shape != ref.shape or relerr(y, ref) > 1e-12:
            return False
    return True


def pin_torch_wgrad(orc: Oracle):
    for p in SHAPES:
        x, _, dy = _inputs(p, orc)
        if relerr(orc.wgrad(p, x, dy), torch_wgrad(p, x, dy)) > 1e-12:
            return False
    return True


def pin_all_ones(orc: Oracle):
    """X = dY = 1: dW[k,r,s,c] = N * (#valid ho for tap r) * (#valid wo for tap s)."""
    for p in SHAPES:
        ho, wo = orc.out_hw(p)
        x = np.ones((p.n, p.h, p.w, p.c), np.float32)
        dy = np.ones((p.n, ho, wo, p.k), np.float32)
        dw = orc.wgrad(p, x, dy)

        def count(extent, out, stride, pad, dil, tap):
            # ho valid iff 0 <= ho*stride + tap*dil - pad <= extent-1
            lo = max(0, -(-(pad - tap * dil) // stride))
            hi = min(out - 1, (extent - 1 + pad - tap * dil) // stride)
            return max(0, hi - lo + 1)

        for r in range(p.r):
            for s in range(p.s):
                want = p.n * count(p.h, ho, p.stride_h, p.pad_h, p.dil_h, r) * \
                    count(p.w, wo, p.stride_w, p.pad_w, p.dil_w, s)
                if not np.all(dw[:, r, s, :] == want):
                    return False
    return True


def pin_adjoint(orc: Oracle):
    """<conv(X, W), dY> = <W, wgrad(X, dY)> (exact in real arithmetic)."""
    for p in SHAPES:
        x, w, dy = _inputs(p, orc)
        lhs = float((orc.fwd(p, x, w) * dy.astype(np.float64)).sum())
        rhs = float((orc.wgrad(p, x, dy) * w.astype(np.float64)).sum())
        if abs(lhs - rhs) > 1e-12 * max(1.0, abs(lhs)):
            return False
    return True


def torch_dgrad(p: Problem, w, dy):
    """dX via autograd of torch's float64 conv2d with respect to its input."""
    xt = torch.zeros((p.n, p.c, p.h, p.w), dtype=torch.float64, requires_grad=True)
    wt = torch.from_numpy(np.asarray(w, np.float64)).permute(0, 3, 1, 2)
    y = torch.nn.functional.conv2d(xt, wt, stride=(p.stride_h, p.stride_w),
                                   padding=(p.pad_h, p.pad_w), dilation=(p.dil_h, p.dil_w),
                                   groups=p.groups)
    y.backward(torch.from_numpy(np.asarray(dy, np.float64)).permute(0, 3, 1, 2))
    return xt.grad.permute(0, 2, 3, 1).numpy()


def pin_torch_dgrad(orc: Oracle):
    for p in SHAPES:
        _, w, dy = _inputs(p, orc)
        if relerr(orc.dgrad(p, dy, w), torch_dgrad(p, w, dy)) > 1e-12:
            return False
    return True


def pin_adjoint_dgrad(orc: Oracle):
    """<conv(X, W), dY> = <X, dgrad(dY, W)> (exact in real arithmetic)."""
    for p in SHAPES:
        x, w, dy = _inputs(p, orc)
        lhs = float((orc.fwd(p, x, w) * dy.astype(np.float64)).sum())
        rhs = float((orc.dgrad(p, dy, w) * x.astype(np.float64)).sum())
        if abs(lhs - rhs) > 1e-12 * max(1.0, abs(lhs)):
            return False
    return True


def pin_1x1_dgrad_gemm(orc: Oracle):
    """A 1x1, stride-1 data gradient is dY W on the [N*H*W, K] view."""
    p = Problem(n=3, h=5, w=7, c=12, k=10)
    dy = rand((3, 5, 7, 10), 3, synth.DY_ID)
    w = rand((10, 1, 1, 12), 3, synth.W_ID)
    ref = dy.reshape(-1, 10).astype(np.float64) @ w.reshape(10, 12).astype(np.float64)
    return relerr(orc.dgrad(p, dy, w).reshape(-1, 12), ref) <= 1e-12


def pin_torch_fwd_bias_relu(orc: Oracle):
    """The fused epilogue against torch's float64 conv2d with its own bias, then relu / clamp."""
    for p in SHAPES:
        x, w, _ = _inputs(p, orc)
        b = rand((p.k,), 9, synth.W_ID + 7)
        xt = torch.from_numpy(np.asarray(x, np.float64)).permute(0, 3, 1, 2)
        wt = torch.from_numpy(np.asarray(w, np.float64)).permute(0, 3, 1, 2)
        y = torch.nn.functional.conv2d(xt, wt, torch.from_numpy(b.astype(np.float64)),
                                       stride=(p.stride_h, p.stride_w), padding=(p.pad_h, p.pad_w),
                                       dilation=(p.dil_h, p.dil_w), groups=p.groups).permute(0, 2, 3, 1)
        if relerr(orc.fwd_epilogue(p, x, w, b, 0.0), torch.relu(y).numpy()) > 1e-12:
            return False
        if relerr(orc.fwd_epilogue(p, x, w, b, -0.25, 0.5), torch.clamp(y, -0.25, 0.5).numpy()) > 1e-12:
            return False
    return True


PINS = [pin_1x1_gemm, pin_bias_sum, pin_torch_fwd, pin_torch_wgrad, pin_all_ones, pin_adjoint,
        pin_torch_dgrad, pin_adjoint_dgrad, pin_1x1_dgrad_gemm, pin_torch_fwd_bias_relu]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_pin(orc, pin):
    assert pin(orc)


def test_output_extent_matches_torch(orc):
    for p in SHAPES:
        x, w, _ = _inputs(p, orc)
        assert orc.out_hw(p) == torch_fwd(p, x, w).shape[1:3]
    # a filter that does not fit gives an empty output
    assert orc.out_hw(Problem(n=1, h=2, w=2, c=1, k=1, r=5, s=5)) == (0, 0)


def test_bruteforce_im2col(orc):
    """Tiny problems through an explicitly materialised im2col matrix."""
    for p in [Problem(n=2, h=4, w=5, c=4, k=3, r=3, s=2, stride_h=1, stride_w=2, pad_h=1, pad_w=1,
                      dil_h=1, dil_w=1, groups=1),
              Problem(n=3, h=5, w=5, c=4, k=4, r=2, s=3, stride_h=2, stride_w=1, pad_h=0, pad_w=2,
                      dil_h=2, dil_w=1, groups=2)]:
        x, w, dy = _inputs(p, orc, seed=11)
        ho, wo = orc.out_hw(p)
        cg, kg = p.c // p.groups, p.k // p.groups
        y = np.zeros((p.n, ho, wo, p.k))
        dw = np.zeros((p.k, p.r, p.s, cg))
        for g in range(p.groups):
            rows = []
            for n, i, j in itertools.product(range(p.n), range(ho), range(wo)):
                col = []
                for r, s, c in itertools.product(range(p.r), range(p.s), range(cg)):
                    hh, ww = i * p.stride_h - p.pad_h + r * p.dil_h, j * p.stride_w - p.pad_w + s * p.dil_w
                    inside = 0 <= hh < p.h and 0 <= ww < p.w
                    col.append(float(x[n, hh, ww, g * cg + c]) if inside else 0.0)
                rows.append(col)
            a = np.array(rows)                                       # [P, R*S*Cg]
            wm = w[g * kg:(g + 1) * kg].reshape(kg, -1).astype(np.float64)  # [Kg, R*S*Cg]
            y[..., g * kg:(g + 1) * kg] = (a @ wm.T).reshape(p.n, ho, wo, kg)
            dym = dy[..., g * kg:(g + 1) * kg].reshape(-1, kg).astype(np.float64)
            dw[g * kg:(g + 1) * kg] = (dym.T @ a).reshape(kg, p.r, p.s, cg)
        assert relerr(orc.fwd(p, x, w), y) <= 1e-12
        assert relerr(orc.wgrad(p, x, dy), dw) <= 1e-12


def test_depthwise_is_per_channel_correlation(orc):
    """Depthwise wgrad: dW[c] = sum_n correlate2d(Xpad[n, :, :, c], dY[n, :, :, c], 'valid')."""
    from scipy.signal import correlate2d
    p = Problem(n=2, h=9, w=8, c=5, k=5, r=7, s=7, pad_h=3, pad_w=3, groups=5)
    x, _, dy = _inputs(p, orc, seed=3)
    dw = orc.wgrad(p, x, dy)
    xp = np.pad(x.astype(np.float64), ((0, 0), (3, 3), (3, 3), (0, 0)))
    for c in range(p.c):
        ref = sum(correlate2d(xp[n, :, :, c], dy[n, :, :, c].astype(np.float64), mode="valid")
                  for n in range(p.n))
        assert relerr(dw[c, :, :, 0], ref) <= 1e-12


def test_batch_chunks_sum_to_whole(orc):
    """The weight gradient does not depend on how the batch is split (PR #11188 "Motivation")."""
    p = Problem(n=7, h=6, w=5, c=4, k=6, r=3, s=3, pad_h=1, pad_w=1, groups=2)
    x, _, dy = _inputs(p, orc, seed=5)
    whole = orc.wgrad(p, x, dy)
    for m in (2, 3, 7):
        acc = np.zeros_like(whole)
        bounds = [p.n * i // m for i in range(m + 1)]
        for a, b in zip(bounds[:-1], bounds[1:]):
            q = Problem(**{**p.__dict__, "n": b - a})
            orc.wgrad_acc(q, x[a:b], dy[a:b], acc)
        # same terms, same order: bit-identical
        assert np.array_equal(acc, whole)


def test_wgrad_channel_subset_is_a_slice(orc):
    p = SHAPES[2]
    x, _, dy = _inputs(p, orc)
    whole = orc.wgrad(p, x, dy)
    part = orc.wgrad(p, x, dy, k_range=(1, 3))
    assert np.array_equal(part[1:3], whole[1:3]) and not part[0].any() and not part[3:].any()


def test_batch_split_count_is_ceil_div(orc):
    """The brute-force count equals the page's fixed integer ceiling (n + max_n - 1) / max_n
    (PR #11188, "Technical Details"), and the page's broken form n / max_n differs exactly
    where max_n does not divide n."""
    for n in range(0, 400):
        for max_n in range(1, 60):
            m = orc.batch_split_count(n, max_n)
            assert m == max(1, (n + max_n - 1) // max_n)
            assert m * max_n >= n and (m == 1 or (m - 1) * max_n < n)
    assert orc.batch_split_count(5, 0) == -1


def test_golden_batch_split_ticket(orc):
    """The ticket shape of PR #11188 ("Motivation", "Test Plan"), stored by tests/golden/make_golden.py."""
    import json
    path = os.path.join(os.path.dirname(__file__), "golden", "batch_split_ticket.json")
    g = json.load(open(path))
    assert g["bytes_per_sample"] == 96 * 512 * 512 * 4
    assert g["max_n"] == (2 ** 32) // g["bytes_per_sample"] == 42
    for n, m in g["split_count"].items():
        assert orc.batch_split_count(int(n), g["max_n"]) == m
    assert g["split_count"]["64"] == 2  # the ticket's batch needs two dispatches


def test_1x1_wgrad_large_batch_streams(orc):
    """Config-shaped 1x1 (C=96, K=64) on a reduced image: GEMM closed form, streamed per sample."""
    p = Problem(n=3, h=32, w=32, c=96, k=64)
    dw = np.zeros((64, 1, 1, 96))
    ref = np.zeros((64, 96))
    for n in range(p.n):
        x = np.empty((1, 32, 32, 96), np.float32)
        dy = np.empty((1, 32, 32, 64), np.float32)
        synth.fill(x, "normal", 0, 1, 1, synth.X_ID, offset=n * x.size)
        synth.fill(dy, "normal", 0, 1, 1, synth.DY_ID, offset=n * dy.size)
        orc.wgrad_acc(Problem(**{**p.__dict__, "n": 1}), x, dy, dw)
        ref += dy.reshape(-1, 64).astype(np.float64).T @ x.reshape(-1, 96).astype(np.float64)
    assert relerr(dw.reshape(64, 96), ref) <= 1e-12


# ----------------------------------------------------- planted mistakes

MUTANTS = {
    # a transposed operand: dW written with its filter taps in (s, r) order
    "wgrad_taps_transposed": ("double* d = j->out + ((k * p->r + r) * p->s + s) * Cg;",
                              "double* d = j->out + ((k * p->s + s) * p->r + r) * Cg;"),
    # a dropped factor: dilation ignored along w
    "wgrad_no_dilation": ("const int64_t w = wo * p->stride_w + s * p->dil_w - p->pad_w;\n              if (w < 0 || w >= p->w) continue;\n              const float* xp = j->x + ((n * p->h + h) * p->w + w) * p->c + g * Cg;\n              double* d",
                          "const int64_t w = wo * p->stride_w + s - p->pad_w;\n              if (w < 0 || w >= p->w) continue;\n              const float* xp = j->x + ((n * p->h + h) * p->w + w) * p->c + g * Cg;\n              double* d"),
    # a wrong sign: padding added instead of subtracted
    "wgrad_pad_sign": ("const int64_t h = ho * p->stride_h + r * p->dil_h - p->pad_h;\n            if (h < 0 || h >= p->h) continue;\n            for (int64_t s = 0; s < p->s; ++s) {\n              const int64_t w",
                       "const int64_t h = ho * p->stride_h + r * p->dil_h + p->pad_h;\n            if (h < 0 || h >= p->h) continue;\n            for (int64_t s = 0; s < p->s; ++s) {\n              const int64_t w"),
    # a wrong index: groups interleaved instead of contiguous
    "wgrad_group_modulo": ("const double gk = (double)dyp[k];\n          const int64_t g = k / Kg;",
                           "const double gk = (double)dyp[k];\n          const int64_t g = k % p->groups;"),
    "fwd_weight_transposed": ("const float* wp = j->wt + ((k * p->r + r) * p->s + s) * Cg;",
                              "const float* wp = j->wt + ((k * p->s + s) * p->r + r) * Cg;"),
    # dropped terms
    "bias_dropped_term": ("for (int64_t q = 0; q < P; ++q)", "for (int64_t q = 1; q < P; ++q)"),
    "wgrad_dropped_last_sample": ("  for (int64_t n = 0; n < p->n; ++n) {\n    for (int64_t ho = 0; ho < Ho; ++ho) {\n      for (int64_t wo = 0; wo < Wo; ++wo) {\n        const float* dyp",
                                  "  for (int64_t n = 0; n + 1 < p->n; ++n) {\n    for (int64_t ho = 0; ho < Ho; ++ho) {\n      for (int64_t wo = 0; wo < Wo; ++wo) {\n        const float* dyp"),
    "fwd_stride_ignored": ("const int64_t h = ho * p->stride_h + r * p->dil_h - p->pad_h;\n          if (h < 0 || h >= p->h) continue;\n          for (int64_t s = 0; s < p->s; ++s) {\n            const int64_t w = wo * p->stride_w",
                           "const int64_t h = ho + r * p->dil_h - p->pad_h;\n          if (h < 0 || h >= p->h) continue;\n          for (int64_t s = 0; s < p->s; ++s) {\n            const int64_t w = wo * p->stride_w"),
    "extent_off_by_one": ("return span / stride + 1;", "return span / stride;"),
    # data gradient: a wrong sign, a dropped stride test, a transposed tap, the
    # wrong group block
    "dgrad_pad_sign": ("const int64_t hn = h + p->pad_h - r * p->dil_h;",
                       "const int64_t hn = h - p->pad_h + r * p->dil_h;"),
    "dgrad_stride_not_checked": ("if (wn < 0 || wn % p->stride_w != 0) continue;", "if (wn < 0) continue;"),
    "dgrad_taps_transposed": ("const float* wp = j->wt + ((g * Kg * p->r + r) * p->s + s) * Cg + c;",
                              "const float* wp = j->wt + ((g * Kg * p->s + s) * p->r + r) * Cg + c;"),
    "dgrad_group_block": ("const int64_t g = ci / Cg, c = ci % Cg;", "const int64_t g = ci % p->groups, c = ci / p->groups;"),
    "dgrad_dropped_last_k": ("for (int64_t kk = 0; kk < Kg; ++kk)", "for (int64_t kk = 0; kk + 1 < Kg; ++kk)"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(tmp_path, name):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "conv_oracle.c")).read()
    old, repl = MUTANTS[name]
    assert src.count(old) == 1, name
    mutated = src.replace(old, repl)
    path = tmp_path / "mutant.c"
    path.write_text(mutated)
    lib = oracle.build(force=True, source=str(path), out_path=str(tmp_path / "libmutant.so"))
    mut = Oracle(lib)

    def fails(pin):
        try:
            return not pin(mut)
        except (AssertionError, ValueError, RuntimeError):  # a shape mismatch is a caught mistake too
            return True

    failed = [pin.__name__ for pin in PINS if fails(pin)]
    assert failed, f"no pin caught the planted mistake {name}"
