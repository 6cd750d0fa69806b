"""The allocation-free weight + bias gradient entry point.

conv_wgrad_bias_static_ws serves callers that cannot call cudaMalloc where
they run the convolution (a framework pool owns the device memory, or a
plugin/enqueue path forbids allocation after set-up) and hold no workspace:
its split-K slabs live in one fixed 8 MiB device array inside the library.
These tests call it through the C ABI and compare it with conv_wgrad_bias on
the same inputs, twice in a row (the array keeps the previous call's
contents, which must not matter). Both calls run the same kernels at the same
split-K degree, so the outputs must be bit-identical. This file is collected
last on purpose.
"""
import ctypes

import pytest
import torch

import implicit_gemm_convolution_nhwc_gb300 as cig
from gpu_util import inputs, relerr, tol

pytestmark = pytest.mark.gpu


def _regular(p, x, dy, split_k):
    dw = torch.empty((p.k, p.r, p.s, p.c // p.groups), dtype=x.dtype, device="cuda")
    db = torch.empty(p.k, dtype=x.dtype, device="cuda")
    ws = cig.workspace(p, cig.DIR_WGRAD, split_k, True)
    cig.conv_wgrad_bias(p, x, dy, dw, db, ws, split_k)
    return dw, db


def _static_into(p, x, dy, dw, db, split_k):
    lib = cig.load()
    st = lib.conv_wgrad_bias_static_ws(cig._cp(p), x.data_ptr(), dy.data_ptr(), dw.data_ptr(), db.data_ptr(),
                                       split_k, torch.cuda.current_stream().cuda_stream)
    assert st == 0, cig.STATUS[st]


def _setup_call():
    """The documented set-up call: an empty batch loads the module and commits the array."""
    p0 = cig.Problem(n=0, h=8, w=8, c=8, k=8)
    dw = torch.empty((8, 1, 1, 8), device="cuda")
    db = torch.empty(8, device="cuda")
    lib = cig.load()
    st = lib.conv_wgrad_bias_static_ws(cig._cp(p0), None, None, dw.data_ptr(), db.data_ptr(), -1,
                                       torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert st == 0, cig.STATUS[st]
    assert not dw.any() and not db.any()


@pytest.mark.parametrize("shape, split_k", [
    (dict(n=8, h=64, w=64, c=96, k=64), -1),                 # tensor-core 1x1 path, auto degree
    (dict(n=2, h=14, w=14, c=64, k=64, r=3, s=3, pad_h=1, pad_w=1, groups=8), 5),  # grouped path, pinned
])
def test_static_workspace_matches_the_workspace_call(shape, split_k):
    p = cig.Problem(**shape)
    x, dy = inputs(p, 11)
    x, dy = x.cuda(), dy.cuda()
    assert 0 < cig.workspace_bytes(p, cig.DIR_WGRAD, split_k, True) <= cig.STATIC_WS_BYTES
    _setup_call()
    ref_w, ref_b = _regular(p, x, dy, split_k)
    torch.cuda.synchronize()
    for i in range(2):  # two calls in a row share (and overwrite) the array
        dw = torch.full((p.k, p.r, p.s, p.c // p.groups), float("nan"), dtype=x.dtype, device="cuda")
        db = torch.full((p.k,), float("nan"), dtype=x.dtype, device="cuda")
        torch.cuda.synchronize()
        before = (torch.cuda.memory_allocated(), torch.cuda.mem_get_info()[0])
        _static_into(p, x, dy, dw, db, split_k)
        torch.cuda.synchronize()
        after = (torch.cuda.memory_allocated(), torch.cuda.mem_get_info()[0])
        assert after == before, f"call {i}: device memory changed {before} -> {after}"
        # same kernels, same degree: bit-identical to the workspace call
        assert torch.equal(dw, ref_w), f"call {i}: dW differs"
        assert torch.equal(db, ref_b), f"call {i}: db differs"
        assert relerr(dw.cpu(), ref_w.cpu().double().numpy()) <= tol(p)
    assert cig.device_errors() == 0


def test_static_workspace_rejects_a_degree_it_cannot_hold():
    p = cig.Problem(n=8, h=64, w=64, c=96, k=64)
    too_many = 400  # 400 slabs of 64 x 96 fp32 plus bias slabs exceed 8 MiB
    assert cig.workspace_bytes(p, cig.DIR_WGRAD, too_many, True) > cig.STATIC_WS_BYTES
    x, dy = inputs(p, 11)
    dw = torch.empty((64, 1, 1, 96), device="cuda")
    db = torch.empty(64, device="cuda")
    lib = cig.load()
    st = lib.conv_wgrad_bias_static_ws(cig._cp(p), x.cuda().data_ptr(), dy.cuda().data_ptr(), dw.data_ptr(),
                                       db.data_ptr(), too_many, None)
    assert st == 3  # CONV_ERR_WORKSPACE_TOO_SMALL, nothing enqueued
