"""Seeded counter-based synthetic inputs (no convolution arithmetic here).

The generator's definition is in ``synth.c``. Element ``i`` of tensor
``(seed, tensor_id)`` depends only on those three numbers, so a tensor can be
produced in pieces (``offset``) and a large input never needs one host copy.

Tensor ids used across the repository: X = 0, W = 1, dY = 2.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libsynth.so")
_lib = None

X_ID, W_ID, DY_ID, BIAS_ID = 0, 1, 2, 3
DISTS = {"uniform": 0, "normal": 1, "integer": 2}


def build(force: bool = False) -> str:
    """Compile the generator with the system C compiler (no GPU needed)."""
    src = os.path.join(_HERE, "synth.c")
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(src):
        return _LIB_PATH
    os.makedirs(_BUILD, exist_ok=True)
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.run(["gcc", "-O2", "-fPIC", "-shared", "-pthread", "-ffp-contract=off",
                    "-o", tmp, src, "-lm"], check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        lib.synth_fill.argtypes = [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_int, ctypes.c_int,
                                   ctypes.c_double, ctypes.c_double, ctypes.c_uint64,
                                   ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int]
        lib.synth_fill.restype = ctypes.c_int
        lib.synth_f32_to_bf16.argtypes = [ctypes.c_float]
        lib.synth_f32_to_bf16.restype = ctypes.c_uint16
        lib.synth_f32_to_f16.argtypes = [ctypes.c_float]
        lib.synth_f32_to_f16.restype = ctypes.c_uint16
        _lib = lib
    return _lib


def _threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _code_of(dst) -> tuple[int, int, int]:
    """(dtype code, data pointer, element count) of a contiguous numpy array or CPU torch tensor."""
    try:
        import torch
    except ImportError:  # pragma: no cover
        torch = None
    if torch is not None and isinstance(dst, torch.Tensor):
        if dst.device.type != "cpu" or not dst.is_contiguous():
            raise ValueError("synth.fill needs a contiguous CPU tensor")
        code = {torch.float32: 0, torch.bfloat16: 1, torch.float16: 2}.get(dst.dtype)
        if code is None:
            raise ValueError(f"unsupported dtype {dst.dtype}")
        return code, dst.data_ptr(), dst.numel()
    arr = dst
    if not arr.flags["C_CONTIGUOUS"]:
        raise ValueError("synth.fill needs a C-contiguous array")
    if arr.dtype == np.float32:
        code = 0
    elif arr.dtype == np.float16:
        code = 2
    elif arr.dtype == np.uint16:  # raw bf16 bit patterns
        code = 1
    else:
        raise ValueError(f"unsupported dtype {arr.dtype}")
    return code, arr.ctypes.data, arr.size


def fill(dst, dist: str, a: float, b: float, seed: int, tensor_id: int, offset: int = 0,
         nthreads: int | None = None):
    """Write elements ``offset .. offset+numel`` of tensor (seed, tensor_id) into ``dst``.

    dist "uniform": [a, b); "normal": mean a, std b; "integer": integers in [a, b].
    """
    code, ptr, count = _code_of(dst)
    rc = _load().synth_fill(ptr, count, code, DISTS[dist], float(a), float(b), int(seed),
                            int(tensor_id), int(offset), int(nthreads or _threads()))
    if rc != 0:
        raise RuntimeError("synth_fill rejected its arguments")
    return dst


def tensor(shape, dtype, dist: str, a: float, b: float, seed: int, tensor_id: int, pin: bool = False):
    """A new CPU torch tensor of ``shape``/``dtype`` filled from (seed, tensor_id)."""
    import torch
    t = torch.empty(tuple(shape), dtype=dtype, pin_memory=pin)
    return fill(t, dist, a, b, seed, tensor_id)


def f32_to_bf16_bits(f: float) -> int:
    return int(_load().synth_f32_to_bf16(f))


def f32_to_f16_bits(f: float) -> int:
    return int(_load().synth_f32_to_f16(f))
