"""CPU fp64 oracle for NHWC convolution (forward, weight, bias and data gradients).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
bench's CPU-baseline leg are the only code allowed to import this package.
The product path never calls it. The arithmetic is in ``conv_oracle.c``;
this module only compiles it and marshals numpy arrays in and out.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, fields

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "conv_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libconv_oracle.so")
CFLAGS = ["-O2", "-fPIC", "-shared", "-pthread", "-ffp-contract=off"]


@dataclass(frozen=True)
class Problem:
    """One convolution: X [n,h,w,c], W [k,r,s,c/groups], Y/dY [n,ho,wo,k]."""
    n: int
    h: int
    w: int
    c: int
    k: int
    r: int = 1
    s: int = 1
    stride_h: int = 1
    stride_w: int = 1
    pad_h: int = 0
    pad_w: int = 0
    dil_h: int = 1
    dil_w: int = 1
    groups: int = 1


class _CProblem(ctypes.Structure):
    _fields_ = [(f.name, ctypes.c_int64) for f in fields(Problem)]


def build(force: bool = False, source: str = _SRC, out_path: str = _LIB_PATH) -> str:
    """Compile the oracle with the system C compiler."""
    if not force and os.path.exists(out_path) and os.path.getmtime(out_path) >= os.path.getmtime(source):
        return out_path
    os.makedirs(os.path.dirname(out_path), exist_ok=True)
    tmp = out_path + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *CFLAGS, "-o", tmp, source], check=True)
    os.replace(tmp, out_path)
    return out_path


def _threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _f32(a) -> np.ndarray:
    """A C-contiguous float32 numpy view/copy of a numpy array or CPU torch tensor.

    16-bit inputs widen to float32 exactly."""
    try:
        import torch
        if isinstance(a, torch.Tensor):
            a = a.detach().to("cpu").float().contiguous().numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(a, dtype=np.float32)


_P = ctypes.c_void_p


class Oracle:
    """The oracle library at ``path`` (the committed source by default)."""

    def __init__(self, path: str | None = None):
        lib = ctypes.CDLL(path or build())
        lib.oracle_out_extent.argtypes = [ctypes.c_int64] * 5
        lib.oracle_out_extent.restype = ctypes.c_int64
        lib.oracle_conv_fwd.argtypes = [ctypes.POINTER(_CProblem), _P, _P, _P, ctypes.c_int]
        lib.oracle_conv_fwd.restype = None
        lib.oracle_conv_wgrad_acc.argtypes = [ctypes.POINTER(_CProblem), _P, _P, ctypes.c_int64,
                                              ctypes.c_int64, _P, ctypes.c_int]
        lib.oracle_conv_wgrad_acc.restype = None
        lib.oracle_conv_dgrad.argtypes = [ctypes.POINTER(_CProblem), _P, _P, _P, ctypes.c_int]
        lib.oracle_conv_dgrad.restype = None
        lib.oracle_conv_bgrad_acc.argtypes = [ctypes.POINTER(_CProblem), _P, _P]
        lib.oracle_conv_bgrad_acc.restype = None
        lib.oracle_batch_split_count.argtypes = [ctypes.c_int64, ctypes.c_int64]
        lib.oracle_batch_split_count.restype = ctypes.c_int64
        self._lib = lib

    # -- shapes ------------------------------------------------------------
    def out_hw(self, p: Problem) -> tuple[int, int]:
        ho = self._lib.oracle_out_extent(p.h, p.pad_h, p.dil_h, p.r, p.stride_h)
        wo = self._lib.oracle_out_extent(p.w, p.pad_w, p.dil_w, p.s, p.stride_w)
        return int(ho), int(wo)

    @staticmethod
    def _cp(p: Problem):
        return ctypes.byref(_CProblem(*[getattr(p, f.name) for f in fields(Problem)]))

    # -- operations ----------------------------------------------------------
    def fwd(self, p: Problem, x, w, nthreads: int | None = None) -> np.ndarray:
        """Y [n, ho, wo, k] in float64."""
        ho, wo = self.out_hw(p)
        x, w = _f32(x), _f32(w)
        assert x.size == p.n * p.h * p.w * p.c and w.size == p.k * p.r * p.s * (p.c // p.groups)
        y = np.zeros((p.n, ho, wo, p.k), dtype=np.float64)
        self._lib.oracle_conv_fwd(self._cp(p), x.ctypes.data, w.ctypes.data, y.ctypes.data,
                                  nthreads or _threads())
        return y

    def fwd_epilogue(self, p: Problem, x, w, bias=None, lo: float = -np.inf, hi: float = np.inf,
                     nthreads: int | None = None) -> np.ndarray:
        """min(max(Y + bias[k], lo), hi) in float64: the fused bias / ReLU / clamp epilogue
        ("feat(rocke): split-K forward implicit-GEMM convolution on gfx1250", "Review follow-ups"),
        applied to the forward's exact sum."""
        y = self.fwd(p, x, w, nthreads)
        if bias is not None:
            y = y + _f32(bias).astype(np.float64).reshape(1, 1, 1, p.k)
        return np.minimum(np.maximum(y, lo), hi)

    def dgrad(self, p: Problem, dy, w, nthreads: int | None = None) -> np.ndarray:
        """dX [n, h, w, c] in float64: the gradient of the forward with respect to X."""
        ho, wo = self.out_hw(p)
        dy, w = _f32(dy), _f32(w)
        assert dy.size == p.n * ho * wo * p.k and w.size == p.k * p.r * p.s * (p.c // p.groups)
        dx = np.zeros((p.n, p.h, p.w, p.c), dtype=np.float64)
        self._lib.oracle_conv_dgrad(self._cp(p), dy.ctypes.data, w.ctypes.data, dx.ctypes.data,
                                    nthreads or _threads())
        return dx

    def wgrad_acc(self, p: Problem, x, dy, dw: np.ndarray, k_range=None, nthreads: int | None = None):
        """dw += the weight gradient of the samples in x / dy (p.n of them)."""
        ho, wo = self.out_hw(p)
        x, dy = _f32(x), _f32(dy)
        assert x.size == p.n * p.h * p.w * p.c and dy.size == p.n * ho * wo * p.k
        assert dw.dtype == np.float64 and dw.flags["C_CONTIGUOUS"]
        assert dw.size == p.k * p.r * p.s * (p.c // p.groups)
        k0, k1 = k_range if k_range is not None else (0, p.k)
        self._lib.oracle_conv_wgrad_acc(self._cp(p), x.ctypes.data, dy.ctypes.data, k0, k1,
                                        dw.ctypes.data, nthreads or _threads())
        return dw

    def wgrad(self, p: Problem, x, dy, k_range=None, nthreads: int | None = None) -> np.ndarray:
        """dW [k, r, s, c/groups] in float64."""
        dw = np.zeros((p.k, p.r, p.s, p.c // p.groups), dtype=np.float64)
        return self.wgrad_acc(p, x, dy, dw, k_range, nthreads)

    def bgrad_acc(self, p: Problem, dy, db: np.ndarray):
        ho, wo = self.out_hw(p)
        dy = _f32(dy)
        assert dy.size == p.n * ho * wo * p.k and db.dtype == np.float64 and db.size == p.k
        self._lib.oracle_conv_bgrad_acc(self._cp(p), dy.ctypes.data, db.ctypes.data)
        return db

    def bgrad(self, p: Problem, dy) -> np.ndarray:
        """db [k] in float64."""
        return self.bgrad_acc(p, dy, np.zeros(p.k, dtype=np.float64))

    def batch_split_count(self, n: int, max_n: int) -> int:
        return int(self._lib.oracle_batch_split_count(n, max_n))


_default: Oracle | None = None


def get() -> Oracle:
    """The oracle built from the committed source."""
    global _default
    if _default is None:
        _default = Oracle()
    return _default
