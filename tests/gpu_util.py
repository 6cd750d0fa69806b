"""Helpers for the GPU parity tests: seeded inputs, guarded device buffers,
calls through the C ABI, and the oracle comparison with the stated tolerances.

Tolerances (normwise, max |gpu - oracle| <= tol * max |oracle|):
  fp32 inputs: 1e-5; bf16/fp16 inputs with fp32 accumulation: 1e-2.
The oracle is fed exactly the values the GPU sees (16-bit inputs widen to
fp32 exactly), so only accumulation order and the output rounding differ.
"""
import numpy as np
import torch

import oracle
import synth
import implicit_gemm_convolution_nhwc_gb300 as cig

TORCH_DT = {cig.F32: torch.float32, cig.BF16: torch.bfloat16, cig.F16: torch.float16}
GUARD = 64  # elements of canary on each side of an output
GUARD_BYTES = 256


def tol(p: cig.Problem) -> float:
    return 1e-5 if p.in_dtype == cig.F32 else 1e-2


def oproblem(p: cig.Problem) -> oracle.Problem:
    return oracle.Problem(n=p.n, h=p.h, w=p.w, c=p.c, k=p.k, r=p.r, s=p.s, stride_h=p.stride_h,
                          stride_w=p.stride_w, pad_h=p.pad_h, pad_w=p.pad_w, dil_h=p.dil_h, dil_w=p.dil_w,
                          groups=p.groups)


def inputs(p: cig.Problem, seed: int, dist: str = "normal", a: float = 0.0, b: float = 1.0, direction=cig.DIR_WGRAD):
    """Seeded CPU tensors: (x, w) forward, (x, dy) weight gradient, (dy, w) data gradient."""
    dt = TORCH_DT[p.in_dtype]
    ho, wo = p.out_hw
    x = synth.tensor((p.n, p.h, p.w, p.c), dt, dist, a, b, seed, synth.X_ID)
    if direction == cig.DIR_FWD:
        other = synth.tensor((p.k, p.r, p.s, p.c // p.groups), dt, dist, a, b, seed, synth.W_ID)
    elif direction == cig.DIR_DGRAD:  # (dy, w)
        dy = synth.tensor((p.n, ho, wo, p.k), dt, dist, a, b, seed, synth.DY_ID)
        return dy, synth.tensor((p.k, p.r, p.s, p.c // p.groups), dt, dist, a, b, seed, synth.W_ID)
    else:
        other = synth.tensor((p.n, ho, wo, p.k), dt, dist, a, b, seed, synth.DY_ID)
    return x, other


class Guarded:
    """A device tensor of `numel` elements with canary elements on both sides."""

    def __init__(self, numel: int, dtype, fill=12345.0, device="cuda"):
        self.numel = numel
        self.fill = fill
        self.buf = torch.full((numel + 2 * GUARD,), fill, dtype=dtype, device=device)
        self.view = self.buf[GUARD:GUARD + numel]
        self.ref = self.buf[:1].clone()  # the fill as stored in this dtype

    def intact(self) -> bool:
        b = self.buf
        return bool((b[:GUARD] == self.ref).all() and (b[GUARD + self.numel:] == self.ref).all())


class GuardedWs:
    """A device workspace pre-filled with NaN bit patterns, with byte canaries around it."""

    def __init__(self, nbytes: int, device="cuda"):
        self.nbytes = nbytes
        self.buf = torch.full((nbytes + 2 * GUARD_BYTES,), 0xFF, dtype=torch.uint8, device=device)
        self.buf[:GUARD_BYTES] = 0xAB
        self.buf[GUARD_BYTES + nbytes:] = 0xAB
        self.view = self.buf[GUARD_BYTES:GUARD_BYTES + nbytes] if nbytes else None

    def intact(self) -> bool:
        b = self.buf
        return bool((b[:GUARD_BYTES] == 0xAB).all() and (b[GUARD_BYTES + self.nbytes:] == 0xAB).all())


def run_wgrad(p: cig.Problem, x, dy, split_k=-1, bias=True, check_guards=True):
    """dW (and db) from the GPU as CPU tensors, with guard and workspace checks."""
    dev = torch.device("cuda")
    odt = TORCH_DT[p.out_dtype]
    dw = Guarded(p.k * p.r * p.s * (p.c // p.groups), odt)
    db = Guarded(p.k, odt) if bias else None
    ws = GuardedWs(cig.workspace_bytes(p, cig.DIR_WGRAD, split_k, bias))
    xd, dyd = x.to(dev), dy.to(dev)
    if bias:
        cig.conv_wgrad_bias(p, xd, dyd, dw.view, db.view, ws.view, split_k)
    else:
        cig.conv_wgrad(p, xd, dyd, dw.view, ws.view, split_k)
    torch.cuda.synchronize()
    if check_guards:
        assert dw.intact() and ws.intact() and (db is None or db.intact()), "a write left its buffer"
    out_w = dw.view.cpu().reshape(p.k, p.r, p.s, p.c // p.groups)
    return out_w, (db.view.cpu() if bias else None)


def run_fwd(p: cig.Problem, x, w, split_k=-1, check_guards=True):
    dev = torch.device("cuda")
    ho, wo = p.out_hw
    y = Guarded(p.n * ho * wo * p.k, TORCH_DT[p.out_dtype])
    ws = GuardedWs(cig.workspace_bytes(p, cig.DIR_FWD, split_k, False))
    cig.conv_fwd(p, x.to(dev), w.to(dev), y.view, ws.view, split_k)
    torch.cuda.synchronize()
    if check_guards:
        assert y.intact() and ws.intact(), "a write left its buffer"
    return y.view.cpu().reshape(p.n, ho, wo, p.k)


def run_dgrad(p: cig.Problem, dy, w, split_k=-1, check_guards=True):
    """dX from the GPU as a CPU tensor [n, h, w, c], with guard and workspace checks."""
    dev = torch.device("cuda")
    dx = Guarded(p.n * p.h * p.w * p.c, TORCH_DT[p.out_dtype])
    ws = GuardedWs(cig.workspace_bytes(p, cig.DIR_DGRAD, split_k, False))
    cig.conv_dgrad(p, dy.to(dev), w.to(dev), dx.view, ws.view, split_k)
    torch.cuda.synchronize()
    if check_guards:
        assert dx.intact() and ws.intact(), "a write left its buffer"
    return dx.view.cpu().reshape(p.n, p.h, p.w, p.c)


def relerr(gpu, ref) -> float:
    g = gpu.double().numpy() if isinstance(gpu, torch.Tensor) else np.asarray(gpu, np.float64)
    r = np.asarray(ref, np.float64)
    assert g.shape == r.shape, (g.shape, r.shape)
    assert np.isfinite(g).all(), "non-finite output"
    scale = np.abs(r).max()
    if scale == 0:
        return float(np.abs(g).max())
    return float(np.abs(g - r).max() / scale)
