"""Host sanitizer builds (CPU only): the oracle and the library's host code (validation and the split-K
planner) compiled with AddressSanitizer and UndefinedBehaviorSanitizer and run on small problems. The
CUDA kernels are compiled into the planner harness but never launched; the device code is checked by the
GPU parity tests and the bounded pipeline waits (a device-side sanitizer is closed on this machine)."""
import glob
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HERE = os.path.join(ROOT, "tests", "sanitize")
SAN = ["-fsanitize=address", "-fsanitize=undefined", "-fno-sanitize-recover=all", "-fno-omit-frame-pointer", "-g",
       "-O1"]
ENV = dict(os.environ, ASAN_OPTIONS="detect_leaks=0:abort_on_error=0", UBSAN_OPTIONS="print_stacktrace=1")


def _run(exe):
    res = subprocess.run([exe], capture_output=True, text=True, env=ENV, timeout=600)
    out = res.stdout + res.stderr
    assert res.returncode == 0, out[-4000:]
    assert "runtime error" not in out and "AddressSanitizer" not in out, out[-4000:]
    return out


def test_oracle_under_asan_ubsan(tmp_path):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not found")
    exe = str(tmp_path / "oracle_san")
    subprocess.run([gcc, *SAN, "-pthread", "-o", exe, os.path.join(ROOT, "oracle", "conv_oracle.c"),
                    os.path.join(HERE, "oracle_main.c"), "-lm"], check=True)
    assert "oracle harness ok" in _run(exe)


def test_planner_under_asan_ubsan(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not found")
    csrc = os.path.join(ROOT, "implicit_gemm_convolution_nhwc_gb300", "csrc")
    srcs = sorted(glob.glob(os.path.join(csrc, "*.cu")) + glob.glob(os.path.join(csrc, "kernels", "*.cu")))
    host = [f"-Xcompiler={f}" for f in SAN]  # one flag each: nvcc splits -Xcompiler values at commas
    flags = ["-gencode", "arch=compute_103a,code=sm_103a", "-std=c++17", *host,
             "-I", os.path.join(ROOT, "include"), "-I", csrc]

    def compile_one(src):
        obj = str(tmp_path / (os.path.relpath(src, csrc).replace(os.sep, "_") + ".o"))
        subprocess.run([nvcc, *flags, "-c", src, "-o", obj], check=True, capture_output=True)
        return obj

    with ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_one, srcs))
    main_obj = str(tmp_path / "planner_main.o")
    subprocess.run([nvcc, *flags, "-x", "cu", "-c", os.path.join(HERE, "planner_main.cpp"), "-o", main_obj],
                   check=True, capture_output=True)
    exe = str(tmp_path / "planner_san")
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", *host, "-o", exe, main_obj, *objs],
                   check=True, capture_output=True)
    out = _run(exe)
    assert "planner harness ok" in out
