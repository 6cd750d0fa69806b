"""Python binding of the NHWC implicit-GEMM convolution library (libconv_igemm.so).

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI declared in include/conv_igemm.h. There is no CPU
or PyTorch fallback: if the library is missing or a call fails, an exception
is raised. PyTorch provides device memory (tensors) and the current stream.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass, fields

from . import _build

F32, BF16, F16 = 0, 1, 2
DIR_FWD, DIR_WGRAD, DIR_DGRAD = 0, 1, 2
KERNELS = {"auto": 0, "generic": 1, "wgrad_1x1_ffma": 2, "wgrad_1x1_tf32x3": 3, "fwd_tc": 4,
           "wgrad_depthwise": 5, "wgrad_grouped": 6, "fwd_tc_cluster": 7, "dgrad_tc": 8,
           "fwd_depthwise": 9, "fwd_grouped_tc": 10, "wgrad_grouped_tc": 11, "wgrad_tc": 12,
           "dgrad_depthwise": 13, "dgrad_grouped_tc": 14, "wgrad_grouped_mma": 15,
           "ffma": 16, "wgrad_depthwise_mma": 17,
           "fwd_grouped_mma": 18, "dgrad_grouped_mma": 19}
KERNEL_NAMES = {v: k for k, v in KERNELS.items()}
STATUS = ["CONV_OK", "CONV_ERR_INVALID_ARG", "CONV_ERR_UNSUPPORTED", "CONV_ERR_WORKSPACE_TOO_SMALL",
          "CONV_ERR_OVERFLOW", "CONV_ERR_ALIGNMENT", "CONV_ERR_CUDA"]

# Every symbol include/conv_igemm.h declares.
EXPORTS = ["conv_status_string", "conv_output_dims", "resolve_split_k_for", "resolve_split_k",
           "conv_workspace_bytes_for", "conv_workspace_bytes", "conv_describe_plan", "conv_fwd",
           "conv_fwd_epilogue", "conv_dgrad", "conv_wgrad", "conv_wgrad_bias", "conv_stage1", "conv_stage2", "conv_batch_split_count",
           "conv_wgrad_bias_static_ws", "conv_device_errors", "conv_selftest_wait_timeout",
           "conv_set_kernel_override"]


class ConvError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        name = STATUS[status] if 0 <= status < len(STATUS) else f"status {status}"
        super().__init__(f"{what}: {name}")


@dataclass(frozen=True)
class Problem:
    """Mirror of conv_problem. dtypes: F32 / BF16 / F16 codes."""
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
    in_dtype: int = F32
    out_dtype: int = F32

    @property
    def out_hw(self) -> tuple[int, int]:
        ho = (self.h + 2 * self.pad_h - self.dil_h * (self.r - 1) - 1) // self.stride_h + 1
        wo = (self.w + 2 * self.pad_w - self.dil_w * (self.s - 1) - 1) // self.stride_w + 1
        return ho, wo

    def flops(self) -> int:
        ho, wo = self.out_hw
        return 2 * self.n * ho * wo * self.k * (self.c // self.groups) * self.r * self.s


class _CEpilogue(ctypes.Structure):
    _fields_ = [("bias", ctypes.c_void_p), ("lo", ctypes.c_float), ("hi", ctypes.c_float)]


class _CProblem(ctypes.Structure):
    _fields_ = [(f.name, ctypes.c_int64) for f in fields(Problem) if not f.name.endswith("dtype")] + \
               [("in_dtype", ctypes.c_int32), ("out_dtype", ctypes.c_int32)]


class PlanInfo(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_int32), ("split_k", ctypes.c_int32), ("needs_fold", ctypes.c_int32),
                ("ctas_per_sm", ctypes.c_int32), ("tiles", ctypes.c_int64),
                ("reduction_blocks", ctypes.c_int64), ("ctas", ctypes.c_int64),
                ("workspace_bytes", ctypes.c_uint64), ("max_split", ctypes.c_int32),
                ("fold_width", ctypes.c_int32)]

    def as_dict(self) -> dict:
        d = {f[0]: getattr(self, f[0]) for f in self._fields_}
        d["kernel_name"] = KERNEL_NAMES.get(self.kernel, str(self.kernel))
        return d


_lib = None


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """Load libconv_igemm.so (building it first if allowed). Raises if it cannot."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB
    if not _build.up_to_date():
        if not build_if_missing:
            raise RuntimeError(f"{path} is missing or stale; run __graft_entry__.build()")
        _build.build()
    lib = ctypes.CDLL(path)
    P, V, I32, I64, U64 = ctypes.POINTER(_CProblem), ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64
    sig = {
        "conv_status_string": ([ctypes.c_int], ctypes.c_char_p),
        "conv_output_dims": ([P, ctypes.POINTER(I64), ctypes.POINTER(I64)], ctypes.c_int),
        "resolve_split_k_for": ([P, ctypes.c_int, I32, I32, ctypes.POINTER(I32)], ctypes.c_int),
        "resolve_split_k": ([P, ctypes.c_int, I32, ctypes.POINTER(I32)], ctypes.c_int),
        "conv_workspace_bytes_for": ([P, ctypes.c_int, I32, I32, I32, ctypes.POINTER(U64)], ctypes.c_int),
        "conv_workspace_bytes": ([P, ctypes.c_int, I32, I32, ctypes.POINTER(U64)], ctypes.c_int),
        "conv_describe_plan": ([P, ctypes.c_int, I32, I32, I32, ctypes.POINTER(PlanInfo)], ctypes.c_int),
        "conv_fwd": ([P, V, V, V, V, U64, I32, V], ctypes.c_int),
        "conv_dgrad": ([P, V, V, V, V, U64, I32, V], ctypes.c_int),
        "conv_fwd_epilogue": ([P, V, V, ctypes.POINTER(_CEpilogue), V, V, U64, I32, V], ctypes.c_int),
        "conv_wgrad": ([P, V, V, V, V, U64, I32, V], ctypes.c_int),
        "conv_wgrad_bias": ([P, V, V, V, V, V, U64, I32, V], ctypes.c_int),
        "conv_stage1": ([P, ctypes.c_int, V, V, V, V, V, U64, I32, V], ctypes.c_int),
        "conv_stage2": ([P, ctypes.c_int, V, V, V, U64, I32, V], ctypes.c_int),
        "conv_batch_split_count": ([I64, I64], I64),
        "conv_set_kernel_override": ([I32], ctypes.c_int),
        "conv_device_errors": ([ctypes.POINTER(ctypes.c_uint32), I32], ctypes.c_int),
        "conv_wgrad_bias_static_ws": ([P, V, V, V, V, I32, V], ctypes.c_int),
        "conv_selftest_wait_timeout": ([U64, ctypes.POINTER(ctypes.c_uint32), V], ctypes.c_int),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


def _cp(p: Problem):
    return ctypes.byref(_CProblem(*[getattr(p, f[0]) for f in _CProblem._fields_]))


def _check(st: int, what: str):
    if st != 0:
        raise ConvError(st, what)


# ------------------------------------------------------------ host logic


def output_dims(p: Problem) -> tuple[int, int]:
    ho, wo = ctypes.c_int64(), ctypes.c_int64()
    _check(load().conv_output_dims(_cp(p), ctypes.byref(ho), ctypes.byref(wo)), "conv_output_dims")
    return ho.value, wo.value


def resolve_split_k(p: Problem, direction: int, request: int = -1, sm_count: int | None = None) -> int:
    d = ctypes.c_int32()
    lib = load()
    if sm_count is None:
        _check(lib.resolve_split_k(_cp(p), direction, request, ctypes.byref(d)), "resolve_split_k")
    else:
        _check(lib.resolve_split_k_for(_cp(p), direction, request, sm_count, ctypes.byref(d)),
               "resolve_split_k_for")
    return d.value


def workspace_bytes(p: Problem, direction: int, split_k: int = -1, with_bias: bool = False,
                    sm_count: int | None = None) -> int:
    b = ctypes.c_uint64()
    lib = load()
    if sm_count is None:
        _check(lib.conv_workspace_bytes(_cp(p), direction, split_k, int(with_bias), ctypes.byref(b)),
               "conv_workspace_bytes")
    else:
        _check(lib.conv_workspace_bytes_for(_cp(p), direction, split_k, int(with_bias), sm_count,
                                            ctypes.byref(b)), "conv_workspace_bytes_for")
    return b.value


def describe_plan(p: Problem, direction: int, split_k: int = -1, with_bias: bool = False,
                  sm_count: int = 152) -> dict:
    info = PlanInfo()
    _check(load().conv_describe_plan(_cp(p), direction, split_k, int(with_bias), sm_count, ctypes.byref(info)),
           "conv_describe_plan")
    return info.as_dict()


def batch_split_count(n: int, max_n: int) -> int:
    return int(load().conv_batch_split_count(n, max_n))


def set_kernel_override(name: str | int):
    code = KERNELS[name] if isinstance(name, str) else int(name)
    _check(load().conv_set_kernel_override(code), "conv_set_kernel_override")


# ------------------------------------------------------------ device calls


def _ptr(t) -> int:
    return 0 if t is None else t.data_ptr()


def _stream(stream) -> int:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _dtype_code(t) -> int:
    import torch
    return {torch.float32: F32, torch.bfloat16: BF16, torch.float16: F16}[t.dtype]


def _need(t, name, numel, dtype_code):
    if t is None:
        raise ValueError(f"{name} is required")
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if t.numel() != numel:
        raise ValueError(f"{name} has {t.numel()} elements, expected {numel}")
    if _dtype_code(t) != dtype_code:
        raise ValueError(f"{name} has dtype {t.dtype}, expected code {dtype_code}")


def workspace(p: Problem, direction: int, split_k: int = -1, with_bias: bool = False, device=None):
    """A device workspace (torch uint8 tensor) large enough for the call, or None."""
    import torch
    n = workspace_bytes(p, direction, split_k, with_bias)
    return None if n == 0 else torch.empty(n, dtype=torch.uint8, device=device or "cuda")


def conv_fwd(p: Problem, x, w, y, ws=None, split_k: int = -1, stream=None):
    ho, wo = p.out_hw
    _need(x, "x", p.n * p.h * p.w * p.c, p.in_dtype)
    _need(w, "w", p.k * p.r * p.s * (p.c // p.groups), p.in_dtype)
    _need(y, "y", p.n * ho * wo * p.k, p.out_dtype)
    st = load().conv_fwd(_cp(p), _ptr(x), _ptr(w), _ptr(y), _ptr(ws), 0 if ws is None else ws.numel(),
                         split_k, _stream(stream))
    _check(st, "conv_fwd")
    return y


def conv_fwd_epilogue(p: Problem, x, w, y, bias=None, lo: float = float("-inf"), hi: float = float("inf"),
                      ws=None, split_k: int = -1, stream=None):
    """Forward with a fused y = min(max(conv + bias[k], lo), hi) (ReLU: lo = 0). bias: [k] in out_dtype or None."""
    ho, wo = p.out_hw
    _need(x, "x", p.n * p.h * p.w * p.c, p.in_dtype)
    _need(w, "w", p.k * p.r * p.s * (p.c // p.groups), p.in_dtype)
    _need(y, "y", p.n * ho * wo * p.k, p.out_dtype)
    if bias is not None:
        _need(bias, "bias", p.k, p.out_dtype)
    ep = _CEpilogue(_ptr(bias), lo, hi)
    st = load().conv_fwd_epilogue(_cp(p), _ptr(x), _ptr(w), ctypes.byref(ep), _ptr(y), _ptr(ws),
                                  0 if ws is None else ws.numel(), split_k, _stream(stream))
    _check(st, "conv_fwd_epilogue")
    return y


def conv_dgrad(p: Problem, dy, w, dx, ws=None, split_k: int = -1, stream=None):
    ho, wo = p.out_hw
    _need(dy, "dy", p.n * ho * wo * p.k, p.in_dtype)
    _need(w, "w", p.k * p.r * p.s * (p.c // p.groups), p.in_dtype)
    _need(dx, "dx", p.n * p.h * p.w * p.c, p.out_dtype)
    st = load().conv_dgrad(_cp(p), _ptr(dy), _ptr(w), _ptr(dx), _ptr(ws), 0 if ws is None else ws.numel(),
                           split_k, _stream(stream))
    _check(st, "conv_dgrad")
    return dx


def conv_wgrad(p: Problem, x, dy, dw, ws=None, split_k: int = -1, stream=None):
    ho, wo = p.out_hw
    _need(x, "x", p.n * p.h * p.w * p.c, p.in_dtype)
    _need(dy, "dy", p.n * ho * wo * p.k, p.in_dtype)
    _need(dw, "dw", p.k * p.r * p.s * (p.c // p.groups), p.out_dtype)
    st = load().conv_wgrad(_cp(p), _ptr(x), _ptr(dy), _ptr(dw), _ptr(ws), 0 if ws is None else ws.numel(),
                           split_k, _stream(stream))
    _check(st, "conv_wgrad")
    return dw


def conv_wgrad_bias(p: Problem, x, dy, dw, db, ws=None, split_k: int = -1, stream=None):
    ho, wo = p.out_hw
    _need(x, "x", p.n * p.h * p.w * p.c, p.in_dtype)
    _need(dy, "dy", p.n * ho * wo * p.k, p.in_dtype)
    _need(dw, "dw", p.k * p.r * p.s * (p.c // p.groups), p.out_dtype)
    _need(db, "db", p.k, p.out_dtype)
    st = load().conv_wgrad_bias(_cp(p), _ptr(x), _ptr(dy), _ptr(dw), _ptr(db), _ptr(ws),
                                0 if ws is None else ws.numel(), split_k, _stream(stream))
    _check(st, "conv_wgrad_bias")
    return dw, db


def conv_stage1(p: Problem, direction: int, x, b, out, db=None, ws=None, split_k: int = -1, stream=None):
    """Stage 1 only (slabs, or the outputs at degree 1). x is dy for the data
    gradient; b is w (forward, data gradient) or dy (weight gradient)."""
    st = load().conv_stage1(_cp(p), direction, _ptr(x), _ptr(b), _ptr(out), _ptr(db), _ptr(ws),
                            0 if ws is None else ws.numel(), split_k, _stream(stream))
    _check(st, "conv_stage1")


def conv_stage2(p: Problem, direction: int, out, db=None, ws=None, split_k: int = -1, stream=None):
    """Stage 2 only: fold the slabs (no-op at degree 1)."""
    st = load().conv_stage2(_cp(p), direction, _ptr(out), _ptr(db), _ptr(ws), 0 if ws is None else ws.numel(),
                            split_k, _stream(stream))
    _check(st, "conv_stage2")


def selftest_wait_timeout(limit_ns: int = 1_000_000, stream=None) -> bool:
    """Runs a kernel whose pipeline wait can never complete, bounded by limit_ns: True when
    the wait gave up as designed (the device error word then has bit 0 set)."""
    out = ctypes.c_uint32()
    _check(load().conv_selftest_wait_timeout(limit_ns, ctypes.byref(out), _stream(stream)),
           "conv_selftest_wait_timeout")
    return bool(out.value)


def device_errors(clear: bool = True) -> int:
    """The device error word (bit 0: a pipeline wait timed out); synchronous."""
    v = ctypes.c_uint32()
    _check(load().conv_device_errors(ctypes.byref(v), int(clear)), "conv_device_errors")
    return v.value


STATIC_WS_BYTES = 8 << 20


def conv_wgrad_bias_static_ws(p: Problem, x, dy, dw, db, split_k: int = -1, stream=None):
    """conv_wgrad_bias with the split-K slabs in the library's fixed 8 MiB device
    array: for callers that cannot allocate device memory (or hold no workspace)
    where they run. Calls that overlap on the GPU share that array and race."""
    ho, wo = p.out_hw
    _need(x, "x", p.n * p.h * p.w * p.c, p.in_dtype)
    _need(dy, "dy", p.n * ho * wo * p.k, p.in_dtype)
    _need(dw, "dw", p.k * p.r * p.s * (p.c // p.groups), p.out_dtype)
    _need(db, "db", p.k, p.out_dtype)
    st = load().conv_wgrad_bias_static_ws(_cp(p), _ptr(x), _ptr(dy), _ptr(dw), _ptr(db), split_k, _stream(stream))
    _check(st, "conv_wgrad_bias_static_ws")
    return dw, db
