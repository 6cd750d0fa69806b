"""Benchmark of the NHWC implicit-GEMM convolution library on one GB300.

Default workload (the headline): the 1x1 fp32 weight + bias gradient,
N=64, H=W=512, C=96 -> K=64 (X 6.4 GB, dY 4.3 GB, over the 4 GB mark),
X, dY ~ N(0, 1) from seed 1, split-K degree resolved automatically.
One step = stage 1 + fold of one conv_wgrad_bias call over that batch.

Prints one JSON line. `value` is effective TFLOP/s (2 N Ho Wo K Cg R S per
step) with inputs resident in HBM; `e2e` is the same metric through the C ABI
with the inputs copied from pinned host memory and dW/db read back inside the
timed region; `roofline` rates the dominant kernel (stage 1) against the
measured HBM copy bandwidth (or the FP32/tensor peak for other workloads);
`cpu_baseline` times the CPU oracle on a bounded sample of the workload.

  python bench.py [--steps K] [--warmup W] [--workload NAME] [--split-k S]
  python bench.py --impl reference ...   (the CPU oracle as the reference arm)
Under torchrun (N > 1) every rank runs an independent replica (replicas only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "conv wgrad/fwd effective TFLOP/s + % of roofline (tensor or HBM), 1 GB300"

# name -> (problem kwargs, direction, dist, dist args, seed, description)
WORKLOADS = {
    "wgrad1x1_f32_n64": (dict(n=64, h=512, w=512, c=96, k=64), "wgrad", "normal", (0.0, 1.0), 1,
                         "1x1 wgrad+db fp32 NHWC N=64 H=W=512 C=96 K=64 (X 6.4 GB, dY 4.3 GB)"),
    "wgrad1x1_f32_n4": (dict(n=4, h=16, w=16, c=8, k=16), "wgrad", "uniform", (-1.0, 1.0), 0,
                        "1x1 wgrad+db fp32 NHWC N=4 H=W=16 C=8 K=16"),
    "fwd3x3_bf16_n1": (dict(n=1, h=14, w=14, c=2048, k=512, r=3, s=3, pad_h=1, pad_w=1, in_dtype=1, out_dtype=1),
                       "fwd", "normal", (0.0, 0.02), 2,
                       "3x3 fwd bf16 NHWC N=1 H=W=14 C=2048 K=512 pad 1, split-K"),
    "fwd3x3_bf16_n64_c256": (dict(n=64, h=56, w=56, c=256, k=256, r=3, s=3, pad_h=1, pad_w=1, in_dtype=1,
                                  out_dtype=1), "fwd", "normal", (0.0, 0.02), 5,
                             "3x3 fwd bf16 NHWC N=64 H=W=56 C=K=256 pad 1 (compute-bound supplement)"),
    "fwd3x3s2_bf16_n64": (dict(n=64, h=56, w=56, c=128, k=256, r=3, s=3, stride_h=2, stride_w=2, pad_h=1, pad_w=1,
                               in_dtype=1, out_dtype=1), "fwd", "normal", (0.0, 0.02), 6,
                          "3x3 stride-2 fwd bf16 NHWC N=64 H=W=56 C=128 K=256 pad 1 (a downsampling layer)"),
    "fwd2x2s2_bf16_n64_c32": (dict(n=64, h=112, w=112, c=32, k=128, r=2, s=2, stride_h=2, stride_w=2,
                                   in_dtype=1, out_dtype=1), "fwd", "normal", (0.0, 0.02), 7,
                              "2x2 stride-2 fwd bf16 NHWC N=64 H=W=112 C=32 K=128 (a downsampling layer; width-folded)"),
    "dgrad3x3_bf16_n1": (dict(n=1, h=14, w=14, c=2048, k=512, r=3, s=3, pad_h=1, pad_w=1, in_dtype=1, out_dtype=1),
                         "dgrad", "normal", (0.0, 0.02), 2,
                         "3x3 dgrad bf16 NHWC N=1 H=W=14 C=2048 K=512 pad 1 (the small-M layer backwards), split-K"),
    "dgrad3x3_bf16_n64_c256": (dict(n=64, h=56, w=56, c=256, k=256, r=3, s=3, pad_h=1, pad_w=1, in_dtype=1,
                                    out_dtype=1), "dgrad", "normal", (0.0, 0.02), 5,
                               "3x3 dgrad bf16 NHWC N=64 H=W=56 C=K=256 pad 1 (compute-bound supplement backwards)"),
    "dw7x7_wgrad_bf16": (dict(n=32, h=56, w=56, c=384, k=384, r=7, s=7, pad_h=3, pad_w=3, groups=384,
                              in_dtype=1, out_dtype=1), "wgrad", "normal", (0.0, 1.0), 3,
                         "depthwise 7x7 wgrad bf16 NHWC N=32 H=W=56 C=K=384 pad 3"),
    "dw7x7_fwd_bf16": (dict(n=32, h=56, w=56, c=384, k=384, r=7, s=7, pad_h=3, pad_w=3, groups=384,
                            in_dtype=1, out_dtype=1), "fwd", "normal", (0.0, 1.0), 3,
                       "depthwise 7x7 fwd bf16 NHWC N=32 H=W=56 C=K=384 pad 3"),
    "dw7x7_dgrad_bf16": (dict(n=32, h=56, w=56, c=384, k=384, r=7, s=7, pad_h=3, pad_w=3, groups=384,
                              in_dtype=1, out_dtype=1), "dgrad", "normal", (0.0, 1.0), 3,
                         "depthwise 7x7 dgrad bf16 NHWC N=32 H=W=56 C=K=384 pad 3"),
    "wgrad3x3_bf16_n64_c256": (dict(n=64, h=56, w=56, c=256, k=256, r=3, s=3, pad_h=1, pad_w=1, in_dtype=1,
                                    out_dtype=1), "wgrad", "normal", (0.0, 0.02), 5,
                               "3x3 wgrad+db bf16 NHWC N=64 H=W=56 C=K=256 pad 1 (compute-bound supplement, "
                               "weight gradient)"),
    "grp3x3_dgrad_f16_g64": (dict(n=64, h=28, w=28, c=512, k=512, r=3, s=3, pad_h=1, pad_w=1, groups=64,
                                  in_dtype=2, out_dtype=2), "dgrad", "normal", (0.0, 1.0), 4,
                             "grouped 3x3 dgrad fp16 NHWC N=64 H=W=28 C=K=512 groups=64 (8 ch/group)"),
    "fwd3x3_f32_n16_c256": (dict(n=16, h=56, w=56, c=256, k=256, r=3, s=3, pad_h=1, pad_w=1), "fwd", "normal",
                            (0.0, 1.0), 9, "3x3 fwd fp32 NHWC N=16 H=W=56 C=K=256 pad 1 (FFMA tiles)"),
    "wgrad3x3_f32_n16_c256": (dict(n=16, h=56, w=56, c=256, k=256, r=3, s=3, pad_h=1, pad_w=1), "wgrad", "normal",
                              (0.0, 1.0), 9, "3x3 wgrad+db fp32 NHWC N=16 H=W=56 C=K=256 pad 1 (FFMA tiles)"),
    "grp3x3_fwd_f16_g64": (dict(n=64, h=28, w=28, c=512, k=512, r=3, s=3, pad_h=1, pad_w=1, groups=64,
                                in_dtype=2, out_dtype=2), "fwd", "normal", (0.0, 1.0), 4,
                           "grouped 3x3 fwd fp16 NHWC N=64 H=W=28 C=K=512 groups=64 (8 ch/group)"),
    "grp3x3_fwd_f16_g128": (dict(n=64, h=28, w=28, c=512, k=512, r=3, s=3, pad_h=1, pad_w=1, groups=128,
                                 in_dtype=2, out_dtype=2), "fwd", "normal", (0.0, 1.0), 4,
                            "grouped 3x3 fwd fp16 NHWC N=64 H=W=28 C=K=512 groups=128 (4 ch/group)"),
    "grp3x3_wgrad_f16_g64": (dict(n=64, h=28, w=28, c=512, k=512, r=3, s=3, pad_h=1, pad_w=1, groups=64,
                                  in_dtype=2, out_dtype=2), "wgrad", "normal", (0.0, 1.0), 4,
                             "grouped 3x3 wgrad fp16 NHWC N=64 H=W=28 C=K=512 groups=64 (8 ch/group)"),
    "grp3x3_wgrad_f16_g128": (dict(n=64, h=28, w=28, c=512, k=512, r=3, s=3, pad_h=1, pad_w=1, groups=128,
                                   in_dtype=2, out_dtype=2), "wgrad", "normal", (0.0, 1.0), 4,
                              "grouped 3x3 wgrad fp16 NHWC N=64 H=W=28 C=K=512 groups=128 (4 ch/group)"),
}
DEFAULT = "wgrad1x1_f32_n64"
L2_BYTES = 129 * 10 ** 6
DT_NAME = {0: "f32", 1: "bf16", 2: "f16"}
ESIZE = {0: 4, 1: 2, 2: 2}


def rank_info():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), \
        int(os.environ.get("LOCAL_RANK", "0"))


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return dict(hbm=d["hbm_gbs"], bf16=d["bf16_tflops"], bf16_sust=d.get("bf16_tflops_sustained"),
                    sm_max_mhz=d.get("sm_max_mhz", 2070.0), source="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sust=1700.0, sm_max_mhz=2070.0, source="fallback")


def problem_bytes(p, direction):
    """Algorithmic bytes: read the two inputs once, write the outputs once."""
    ho, wo = p.out_hw
    es, eo = ESIZE[p.in_dtype], ESIZE[p.out_dtype]
    x = p.n * p.h * p.w * p.c * es
    w = p.k * p.r * p.s * (p.c // p.groups)
    y = p.n * ho * wo * p.k
    if direction == "wgrad":
        return x + y * es + (w + p.k) * eo
    if direction == "dgrad":  # dY and W in, dX out
        return y * es + w * es + p.n * p.h * p.w * p.c * eo
    return x + w * es + y * eo


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi samples (SM clock, reasons) while the timed region runs."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.samples = []
        self.proc = None
        self.dev = device_index
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.dev}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def mark(self, begin: bool):
        if begin:
            self.t0 = time.time()
        else:
            self.t1 = time.time()

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for t, line in self.samples:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            rows.append((t, f))
        inside = [f for t, f in rows if self.t0 is not None and self.t0 - 0.1 <= t <= (self.t1 or t) + 0.1]
        use = inside or [f for t, f in rows]
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}

        def num(v):
            try:
                return float(v)
            except ValueError:
                return None
        sm = [num(f[1]) for f in use if num(f[1]) is not None]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for f in use:
            for name, v in zip(names, f[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(num(f[2]) or 0 for f in use),
                "reasons": sorted(reasons), "samples": len(use), "in_timed_region": bool(inside),
                "power_w_max": max(num(f[3]) or 0 for f in use)}


# ------------------------------------------------------------------ inputs

def make_inputs_on_device(p, direction, dist, args, seed, device, pinned_copy=False):
    """Seeded inputs streamed sample by sample from host to device (no full host copy).
    Returns (x_dev, b_dev, pinned host copies or None)."""
    import torch
    import synth
    import implicit_gemm_convolution_nhwc_gb300 as cig
    dt = {0: torch.float32, 1: torch.bfloat16, 2: torch.float16}[p.in_dtype]
    ho, wo = p.out_hw
    x = torch.empty((p.n, p.h, p.w, p.c), dtype=dt, device=device)
    x_id = synth.X_ID
    if direction == "fwd":
        b = torch.empty((p.k, p.r, p.s, p.c // p.groups), dtype=dt, device=device)
        b_id = synth.W_ID
    elif direction == "dgrad":  # the first input is dY, the second W
        x = torch.empty((p.n, ho, wo, p.k), dtype=dt, device=device)
        x_id = synth.DY_ID
        b = torch.empty((p.k, p.r, p.s, p.c // p.groups), dtype=dt, device=device)
        b_id = synth.W_ID
    else:
        b = torch.empty((p.n, ho, wo, p.k), dtype=dt, device=device)
        b_id = synth.DY_ID
    hosts = None
    if pinned_copy:
        hosts = (torch.empty(x.shape, dtype=dt, pin_memory=True), torch.empty(b.shape, dtype=dt, pin_memory=True))
        synth.fill(hosts[0], dist, args[0], args[1], seed, x_id)
        synth.fill(hosts[1], dist, args[0], args[1], seed, b_id)
        x.copy_(hosts[0])
        b.copy_(hosts[1])
        return x, b, hosts
    for t, tid in ((x, x_id), (b, b_id)):
        flat = t.view(-1)
        chunk = max(1, min(flat.numel(), 64 << 20))
        stage = torch.empty(chunk, dtype=dt, pin_memory=True)
        for off in range(0, flat.numel(), chunk):
            m = min(chunk, flat.numel() - off)
            synth.fill(stage[:m], dist, args[0], args[1], seed, tid, offset=off)
            flat[off:off + m].copy_(stage[:m], non_blocking=False)
    del cig
    return x, b, hosts


# --------------------------------------------------------------- replicas

def max_over_ranks(value: float, device) -> float:
    """The largest of every rank's value (all ranks get it), then a barrier.
    Used for the step time of replicas: the job is as slow as its slowest rank."""
    import torch
    import torch.distributed as dist_
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist_.all_reduce(t, op=dist_.ReduceOp.MAX)
    dist_.barrier()
    return float(t.item())


# --------------------------------------------------------------- traffic

def recorded_traffic(kernel_name: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if the kernel's source
    has not changed since the capture (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    try:
        table = json.load(open(path))
    except ValueError:
        return None
    entry = table.get(f"{kernel_name}:{workload}")
    if not entry:
        return None
    if sources_digest(entry["sources"]) != entry.get("sources_sha256_16"):
        return None
    return entry["dram_bytes_per_launch"]


def sources_digest(rel_paths) -> str | None:
    """sha256 (first 16 hex digits) over the listed csrc files, in order."""
    h = hashlib.sha256()
    for rel in rel_paths:
        path = os.path.join(ROOT, "implicit_gemm_convolution_nhwc_gb300", "csrc", rel)
        if not os.path.exists(path):
            return None
        h.update(open(path, "rb").read())
    return h.hexdigest()[:16]


# ------------------------------------------------------------------ oracle

def oracle_sample(p, direction, dist, args, seed, n_samples: int):
    """Inputs for the first n_samples batch samples (CPU float32 numpy)."""
    import numpy as np
    import synth
    ho, wo = p.out_hw
    x = np.empty((n_samples, p.h, p.w, p.c), np.float32)
    synth.fill(x, dist, args[0], args[1], seed, synth.X_ID)
    if direction == "dgrad":  # (dY, W)
        x = np.empty((n_samples, ho, wo, p.k), np.float32)
        synth.fill(x, dist, args[0], args[1], seed, synth.DY_ID)
        b = np.empty((p.k, p.r, p.s, p.c // p.groups), np.float32)
        synth.fill(b, dist, args[0], args[1], seed, synth.W_ID)
    elif direction == "fwd":
        b = np.empty((p.k, p.r, p.s, p.c // p.groups), np.float32)
        synth.fill(b, dist, args[0], args[1], seed, synth.W_ID)
    else:
        b = np.empty((n_samples, ho, wo, p.k), np.float32)
        synth.fill(b, dist, args[0], args[1], seed, synth.DY_ID)
    if p.in_dtype != 0:  # the GPU sees 16-bit values: round the same way
        import torch
        tdt = {1: torch.bfloat16, 2: torch.float16}[p.in_dtype]
        x = torch.from_numpy(x).to(tdt).float().numpy()
        b = torch.from_numpy(b).to(tdt).float().numpy()
    return x, b


def time_oracle(p, direction, dist, args, seed, target_s: float):
    """Run the oracle on growing batch samples until one run takes >= 0.6 target_s
    (or covers the whole batch), then report that run.
    Returns (flops/s, seconds, samples, threads)."""
    import oracle
    orc = oracle.get()
    threads = max(1, len(os.sched_getaffinity(0)))
    n = 1
    while True:
        x, b = oracle_sample(p, direction, dist, args, seed, n)
        op = oracle.Problem(n=n, h=p.h, w=p.w, c=p.c, k=p.k, r=p.r, s=p.s, stride_h=p.stride_h,
                            stride_w=p.stride_w, pad_h=p.pad_h, pad_w=p.pad_w, dil_h=p.dil_h,
                            dil_w=p.dil_w, groups=p.groups)
        t0 = time.perf_counter()
        if direction == "fwd":
            orc.fwd(op, x, b, threads)
        elif direction == "dgrad":
            orc.dgrad(op, x, b, threads)
        else:
            orc.wgrad(op, x, b, None, threads)
            orc.bgrad(op, b)
        dt = time.perf_counter() - t0
        flops = 2 * n * p.out_hw[0] * p.out_hw[1] * p.k * (p.c // p.groups) * p.r * p.s
        if dt >= 0.6 * target_s or n >= p.n:
            used = min(threads, p.k) if direction == "wgrad" else \
                min(threads, n * (p.h if direction == "dgrad" else p.out_hw[0]))
            return flops / dt, dt, n, used
        n = min(p.n, max(n + 1, int(n * target_s / max(dt, 1e-3))))


# --------------------------------------------------------------- our arm

# The configurations (and the compute-bound supplement) timed after the
# headline and reported under "per_config", each at its own automatic plan.
PER_CONFIG = ["wgrad1x1_f32_n4", "fwd3x3_bf16_n1", "dgrad3x3_bf16_n1", "dw7x7_wgrad_bf16", "dw7x7_dgrad_bf16",
              "grp3x3_wgrad_f16_g64", "grp3x3_wgrad_f16_g128", "grp3x3_dgrad_f16_g64", "fwd3x3_bf16_n64_c256",
              "dgrad3x3_bf16_n64_c256", "wgrad3x3_bf16_n64_c256", "fwd3x3_f32_n16_c256", "wgrad3x3_f32_n16_c256"]
# The split-K degrees swept on the small-M layer (auto first).
SWEEP = {"fwd3x3_bf16_n1": [-1, 1, 2, 4, 8, 16, 32]}
# The fold on slabs far larger than L2: the dense forward at a pinned degree,
# whose stage 2 reads S fp32 slabs of the whole output from HBM.
FOLD_HBM = [("fwd3x3_bf16_n64_c256", 4)]


def fold_bytes(split, out, db):
    """Bytes the fold moves: S fp32 slabs read, the output (and db) written once."""
    e = out.numel() + (db.numel() if db is not None else 0)
    return split * e * 4 + e * out.element_size()


def roofline_for(kname, p, direction, flops, in_bytes, stage1_ms, pk, sms):
    """The dominant kernel (stage 1) against the roofline that bounds it."""
    alu_peak = sms * 128 * 2 * pk["sm_max_mhz"] * 1e6 / 1e12  # FP32 FMA lanes x 2 flop x max clock
    if kname in ("wgrad_1x1_tf32x3", "wgrad_1x1_ffma") or direction == "wgrad" and kname == "generic" and p.r == 1:
        bound = "hbm"
    elif kname in ("fwd_tc", "fwd_tc_cluster", "dgrad_tc", "wgrad_tc"):
        # past the ridge point (flop per byte of the measured peaks) the tensor
        # pipe bounds it, else HBM
        bound = "tensor" if flops / in_bytes > pk["bf16"] * 1e12 / (pk["hbm"] * 1e9) else "hbm"
    elif kname in ("fwd_grouped_tc", "wgrad_grouped_tc", "dgrad_grouped_tc"):
        bound = "tensor_blockdiag"
    elif kname in ("wgrad_depthwise", "wgrad_grouped", "fwd_depthwise", "dgrad_depthwise", "ffma") or \
            kname == "generic":
        bound = "alu"
    else:
        bound = "hbm"
    tens_src = pk["source"] + " (dense bf16 GEMM, burst; fp16 runs at the same nominal rate)"
    if bound == "tensor_blockdiag":
        # Each 128-channel block runs as a dense MMA with a block-diagonal filter:
        # the tensor pipe executes 128 / Cg times the useful multiply-adds.
        waste = 128 // (p.c // p.groups)
        achieved = flops * waste / (stage1_ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": round(achieved, 2), "peak": pk["bf16"], "unit": "TFLOP/s",
                "frac": round(achieved / pk["bf16"], 4), "peak_source": tens_src,
                "executed_per_useful": waste,
                "useful_tflops": round(flops / (stage1_ms * 1e-3) / 1e12, 3),
                "useful_frac_of_fp32_pipe": round(flops / (stage1_ms * 1e-3) / 1e12 / alu_peak, 4)}
    elif bound == "tensor":
        achieved = flops / (stage1_ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": round(achieved, 2), "peak": pk["bf16"], "unit": "TFLOP/s",
                "frac": round(achieved / pk["bf16"], 4), "peak_source": tens_src}
    elif bound == "hbm":
        achieved = in_bytes / (stage1_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": pk["hbm"], "unit": "GB/s",
                "frac": round(achieved / pk["hbm"], 4), "peak_source": pk["source"] + " (HBM copy)"}
    else:
        achieved = flops / (stage1_ms * 1e-3) / 1e12
        roof = {"bound": "alu", "achieved": round(achieved, 3), "peak": round(alu_peak, 2), "unit": "TFLOP/s",
                "frac": round(achieved / alu_peak, 4),
                "peak_source": f"derived: {sms} SMs x 128 FP32 lanes x 2 flop x max SM clock"}
    # HBM fraction beside any other bound (the bandwidth-bound kernels' targets are stated against HBM)
    roof["hbm_frac"] = round(in_bytes / (stage1_ms * 1e-3) / 1e9 / pk["hbm"], 4)
    return roof


class Workload:
    """One workload on the device: inputs, outputs, workspace and plan, and the
    step (one call through the public API) and staged step (stage 1, then
    stage 2, with an event between them)."""

    def __init__(self, name, dev, sms, split_k=-1, fused=False, batch=0):
        import torch
        import implicit_gemm_convolution_nhwc_gb300 as cig
        kw, direction, dist, args, seed, desc = WORKLOADS[name]
        if batch:
            kw = dict(kw, n=batch)
            desc = f"{desc} [batch overridden to N={batch}]"
        self.name, self.desc, self.direction = name, desc, direction
        self.dist, self.args, self.seed = dist, args, seed
        self.cig, self.torch = cig, torch
        self.dev, self.sms = dev, sms
        self.split_k, self.fused = split_k, fused
        p = self.p = cig.Problem(**kw)
        self.d = {"fwd": cig.DIR_FWD, "wgrad": cig.DIR_WGRAD, "dgrad": cig.DIR_DGRAD}[direction]
        self.bias = direction == "wgrad"
        self.x, self.b, _ = make_inputs_on_device(p, direction, dist, args, seed, dev)
        ho, wo = p.out_hw
        self.odt = odt = {0: torch.float32, 1: torch.bfloat16, 2: torch.float16}[p.out_dtype]
        if direction == "fwd":
            self.out, self.db = torch.empty((p.n, ho, wo, p.k), dtype=odt, device=dev), None
        elif direction == "dgrad":
            self.out, self.db = torch.empty((p.n, p.h, p.w, p.c), dtype=odt, device=dev), None
        else:
            self.out = torch.empty((p.k, p.r, p.s, p.c // p.groups), dtype=odt, device=dev)
            self.db = torch.empty(p.k, dtype=odt, device=dev)
        if fused and direction != "fwd":
            raise SystemExit("--bias-relu applies to forward workloads only")
        self.ep_bias = None
        if fused:  # the fused bias + ReLU epilogue runs unsplit
            import synth
            self.ep_bias = synth.tensor((p.k,), odt, "normal", 0.0, 0.1, seed, synth.BIAS_ID).to(dev)
            if split_k > 1:
                raise SystemExit("--bias-relu runs unsplit: use --split-k -1, 0 or 1")
        self.plan = cig.describe_plan(p, self.d, 1 if fused else split_k, self.bias, sm_count=sms)
        self.ws = cig.workspace(p, self.d, 1 if fused else split_k, self.bias, dev)
        self.in_bytes = problem_bytes(p, direction)
        self.flush = None
        if self.in_bytes < 4 * L2_BYTES:  # small inputs: flush L2 between steps
            self.flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
        self.stream = torch.cuda.current_stream(dev)

    def call(self, x, b):
        cig, p, s = self.cig, self.p, self.stream
        if self.fused:
            cig.conv_fwd_epilogue(p, x, b, self.out, self.ep_bias, 0.0, float("inf"), self.ws, self.split_k, s)
        elif self.direction == "fwd":
            cig.conv_fwd(p, x, b, self.out, self.ws, self.split_k, s)
        elif self.direction == "dgrad":
            cig.conv_dgrad(p, x, b, self.out, self.ws, self.split_k, s)
        else:
            cig.conv_wgrad_bias(p, x, b, self.out, self.db, self.ws, self.split_k, s)

    def step(self, ev=None):
        """One step through the user-facing call (stage 1 + fold)."""
        if self.flush is not None:
            self.flush.fill_(1.0)
        if ev is not None:
            ev[0].record(self.stream)
        self.call(self.x, self.b)
        if ev is not None:
            ev[1].record(self.stream)

    def staged(self, ev):
        """The same step with an event between the stages (per-kernel times)."""
        cig, p, s = self.cig, self.p, self.stream
        if self.flush is not None:
            self.flush.fill_(1.0)
        ev[0].record(s)
        if self.fused:  # one unsplit launch: all of it is stage 1
            self.call(self.x, self.b)
            ev[1].record(s)
        else:
            cig.conv_stage1(p, self.d, self.x, self.b, self.out, self.db, self.ws, self.split_k, s)
            ev[1].record(s)
            cig.conv_stage2(p, self.d, self.out, self.db, self.ws, self.split_k, s)
        ev[2].record(s)

    def launches_per_step(self):
        kname = self.plan["kernel_name"]
        return (1 + (1 if self.plan["needs_fold"] else 0) + (1 if kname == "generic" and self.bias else 0) +
                (1 if kname in ("fwd_grouped_tc", "dgrad_grouped_tc") else 0))  # the filter expansion

    def time(self, steps, warmup, world=1, sampler=None):
        """(ms per step, stage-1 ms list, fold ms list). With an L2 flush between
        steps only each step's call is timed; otherwise the whole back-to-back
        region is."""
        torch, dev, stream = self.torch, self.dev, self.stream
        for _ in range(warmup):
            self.step()
        torch.cuda.synchronize(dev)
        if world > 1:
            import torch.distributed as dist_
            dist_.barrier()
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        if sampler is not None:
            sampler.mark(True)
        start.record(stream)
        for i in range(steps):
            self.step(evs[i] if self.flush is not None else None)
        end.record(stream)
        torch.cuda.synchronize(dev)
        if sampler is not None:
            sampler.mark(False)
        total_ms = sum(e[0].elapsed_time(e[1]) for e in evs) if self.flush is not None else start.elapsed_time(end)
        if world > 1:
            total_ms = max_over_ranks(total_ms, dev)
        sev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
        for i in range(steps):
            self.staged(sev[i])
        torch.cuda.synchronize(dev)
        s1 = [e[0].elapsed_time(e[1]) for e in sev]
        s2 = [e[1].elapsed_time(e[2]) for e in sev]
        return total_ms / steps, s1, s2

    def free(self):
        self.x = self.b = self.out = self.db = self.ws = self.flush = self.ep_bias = None


def per_config(dev, sms, pk, steps, warmup):
    """Every configuration (and the supplement) at its automatic plan, under one
    clock sampler: kernel, degree, stage-1 and step times, and the roofline."""
    import torch
    out = {}
    sampler = ClockSampler(dev.index or 0)
    sampler.start()
    time.sleep(0.3)
    t_begin = time.time()
    sampler.mark(True)
    for name in PER_CONFIG:
        if name not in WORKLOADS:
            continue
        try:
            wl = Workload(name, dev, sms)
        except Exception as e:  # pragma: no cover - reported, not fatal
            out[name] = {"error": str(e)[:200]}
            continue
        kname = wl.plan["kernel_name"]
        if kname == "generic" and wl.p.flops() > 2e10:  # the direct kernel would take seconds per step
            out[name] = {"kernel": kname, "skipped": "generic kernel on a large problem"}
            wl.free()
            continue
        ms, s1, s2 = wl.time(steps, warmup)
        st1 = statistics.mean(s1)
        flops = wl.p.flops()
        roof = roofline_for(kname, wl.p, wl.direction, flops, wl.in_bytes, st1, pk, sms)
        entry = {"workload": wl.desc, "kernel": kname, "split_k": wl.plan["split_k"],
                 "fold_width": wl.plan.get("fold_width", 1), "ctas": wl.plan["ctas"],
                 "step_ms": round(ms, 5), "stage1_ms": round(st1, 5), "fold_ms": round(statistics.mean(s2), 5),
                 "tflops": round(flops / (ms * 1e-3) / 1e12, 3), "launches_per_step": wl.launches_per_step(),
                 "l2": "flushed" if wl.flush is not None else "inputs larger than L2",
                 "roofline": {k: roof[k] for k in ("bound", "achieved", "peak", "unit", "frac", "hbm_frac")
                              if k in roof}}
        if "useful_frac_of_fp32_pipe" in roof:
            entry["roofline"]["useful_frac_of_fp32_pipe"] = roof["useful_frac_of_fp32_pipe"]
        entry["roofline"]["traffic"] = recorded_traffic(kname, name)
        wl.free()
        for req in SWEEP.get(name, []):
            sw = Workload(name, dev, sms, split_k=req)
            ms_s, s1_s, _ = sw.time(steps, warmup)
            entry.setdefault("split_sweep", []).append(
                {"request": req, "split_k": sw.plan["split_k"], "step_ms": round(ms_s, 5),
                 "stage1_ms": round(statistics.mean(s1_s), 5)})
            sw.free()
        out[name] = entry
        torch.cuda.empty_cache()
    for name, deg in FOLD_HBM:
        wl = Workload(name, dev, sms, split_k=deg)
        _, _, s2 = wl.time(steps, warmup)
        f_ms = statistics.mean(s2)
        fb = fold_bytes(wl.plan["split_k"], wl.out, wl.db)
        gbs = fb / (f_ms * 1e-3) / 1e9
        out[f"fold:{name}@S{deg}"] = {
            "workload": f"stage 2 alone of {wl.desc}, degree {wl.plan['split_k']}: "
                        f"{wl.plan['split_k']} fp32 slabs of {wl.out.numel()} elements, larger than L2",
            "kernel": "fold", "fold_ms": round(f_ms, 5), "bytes": fb,
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": pk["hbm"], "unit": "GB/s",
                         "frac": round(gbs / pk["hbm"], 4)}}
        wl.free()
        torch.cuda.empty_cache()
    sampler.mark(False)
    out["clocks"] = sampler.stop()
    out["seconds"] = round(time.time() - t_begin, 1)
    out["timing"] = ("per workload: warm-up, then each step (one call through the public API) timed with CUDA "
                     "events on its stream; L2 flushed between steps when the inputs are smaller than 4x L2")
    return out


def run_ours(a, rank, world, local_rank):
    import torch
    import implicit_gemm_convolution_nhwc_gb300 as cig
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    cig.load(build_if_missing=True)
    if a.kernel != "auto":
        cig.set_kernel_override(a.kernel)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    wl = Workload(a.workload, dev, sms, split_k=a.split_k, fused=bool(a.bias_relu), batch=a.batch)
    p, direction, plan = wl.p, wl.direction, wl.plan
    in_bytes, flush = wl.in_bytes, wl.flush
    sampler = ClockSampler(local_rank)
    sampler.start()
    time.sleep(0.3)
    ms_step, s1, s2 = wl.time(a.steps, a.warmup, world, sampler)
    clocks = sampler.stop()
    flops = p.flops()
    value = flops * world / (ms_step * 1e-3) / 1e12
    pk = peaks()
    stage1_ms = statistics.mean(s1)
    kname = plan["kernel_name"]
    roof = roofline_for(kname, p, direction, flops, in_bytes, stage1_ms, pk, sms)
    roof["kernel"] = kname
    roof["traffic"] = recorded_traffic(kname, a.workload)
    roof["kernel_ms"] = round(stage1_ms, 5)
    roof["fold_ms"] = round(statistics.mean(s2), 5)

    # e2e: inputs from pinned host memory and the result back, every step
    e2e = None
    if not a.no_e2e:
        out, db = wl.out, wl.db
        wl.x = wl.b = None
        torch.cuda.empty_cache()
        xh_d, bh_d, hosts = make_inputs_on_device(p, direction, wl.dist, wl.args, wl.seed, dev, pinned_copy=True)
        out_h = torch.empty(out.shape, dtype=wl.odt, pin_memory=True)
        db_h = torch.empty(p.k, dtype=wl.odt, pin_memory=True) if db is not None else None
        h2d = hosts[0].numel() * hosts[0].element_size() + hosts[1].numel() * hosts[1].element_size()
        d2h = out.numel() * out.element_size() + (db.numel() * db.element_size() if db is not None else 0)

        def e2e_step():
            xh_d.copy_(hosts[0], non_blocking=True)
            bh_d.copy_(hosts[1], non_blocking=True)
            wl.call(xh_d, bh_d)
            out_h.copy_(out, non_blocking=True)
            if db_h is not None:
                db_h.copy_(db, non_blocking=True)

        e2e_step()
        torch.cuda.synchronize(dev)
        n_e2e = max(1, min(a.steps, 5))
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(wl.stream)
        for _ in range(n_e2e):
            e2e_step()
        t1.record(wl.stream)
        torch.cuda.synchronize(dev)
        e2e_ms = t0.elapsed_time(t1) / n_e2e
        e2e = {"value": round(flops * world / (e2e_ms * 1e-3) / 1e12, 4), "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4),
               "steps": n_e2e}
        del xh_d, bh_d, hosts
    launches = wl.launches_per_step()
    wl.free()
    torch.cuda.empty_cache()

    cpu = None
    if rank == 0 and world == 1 and not a.no_cpu_baseline:
        fps, secs, n_s, used = time_oracle(p, direction, wl.dist, wl.args, wl.seed, a.cpu_seconds)
        cpu = {"value": round(fps / 1e12, 6), "unit": "TFLOP/s", "cores": used, "kind": "oracle",
               "sample": f"first {n_s} of {p.n} batch samples, every output, fp64 oracle ({secs:.1f} s)"}

    configs = None
    if world == 1 and not a.no_per_config and a.kernel == "auto" and not a.batch:
        cig.set_kernel_override("auto")
        configs = per_config(dev, sms, pk, a.per_config_steps, a.warmup)

    line = {
        "metric": METRIC, "value": round(value, 4), "unit": "TFLOP/s", "n_gpus": world, "steps": a.steps,
        "warmup": a.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": DT_NAME[p.in_dtype], "data": "synthetic (seeded counter-based generator)",
        "config": {"workload": wl.desc + (" + fused bias/ReLU epilogue" if wl.fused else ""), "name": a.workload,
                   "kernel": kname, "split_k": plan["split_k"], "fold_width": plan.get("fold_width", 1),
                   "split_k_request": a.split_k, "ctas": plan["ctas"], "workspace_bytes": plan["workspace_bytes"],
                   "parallelism": f"replicas x{world}" if world > 1 else "1 GPU",
                   "l2": "flushed between steps (2x L2 buffer written)" if flush is not None
                   else f"inputs larger than L2 ({in_bytes / 1e9:.2f} GB)",
                   "algorithmic_bytes": in_bytes, "flops_per_step": flops},
        "roofline": roof, "e2e": e2e, "cpu_baseline": cpu, "clocks": clocks,
        "gpu_launches": a.steps * launches,
        "timing": "value: the timed steps through conv_wgrad_bias / conv_fwd / conv_dgrad; stage_ms: a second loop of "
                  "conv_stage1 + conv_stage2 with an event between them",
        "stage_ms": {"stage1_mean": round(stage1_ms, 5), "stage1_min": round(min(s1), 5),
                     "fold_mean": round(statistics.mean(s2), 5)},
    }
    if configs is not None:
        line["per_config"] = configs
    if rank == 0:
        print(json.dumps(line), flush=True)


# --------------------------------------------------------------- reference arm

def run_reference(a, rank, world):
    if rank != 0:
        return
    kw, direction, dist, args, seed, desc = WORKLOADS[a.workload]
    import implicit_gemm_convolution_nhwc_gb300 as cig
    p = cig.Problem(**kw)
    import oracle
    orc = oracle.get()
    threads = max(1, len(os.sched_getaffinity(0)))
    # calibrate a bounded sample so the whole run stays within a few minutes
    budget = min(8.0, max(0.5, 150.0 / max(1, a.steps + a.warmup)))  # seconds per step
    fps, secs, n_s, used = time_oracle(p, direction, dist, args, seed, budget)
    x, b = oracle_sample(p, direction, dist, args, seed, n_s)
    op = oracle.Problem(n=n_s, h=p.h, w=p.w, c=p.c, k=p.k, r=p.r, s=p.s, stride_h=p.stride_h,
                        stride_w=p.stride_w, pad_h=p.pad_h, pad_w=p.pad_w, dil_h=p.dil_h, dil_w=p.dil_w,
                        groups=p.groups)

    def step():
        if direction == "fwd":
            orc.fwd(op, x, b, threads)
        elif direction == "dgrad":
            orc.dgrad(op, x, b, threads)
        else:
            orc.wgrad(op, x, b, None, threads)
            orc.bgrad(op, b)

    for _ in range(a.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(a.steps):
        step()
    dt = (time.perf_counter() - t0) / a.steps
    flops = 2 * n_s * p.out_hw[0] * p.out_hw[1] * p.k * (p.c // p.groups) * p.r * p.s
    value = flops / dt / 1e12
    sample = f"first {n_s} of {p.n} batch samples per step, every output, fp64 CPU oracle"
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world,
        "steps": a.steps, "warmup": a.warmup, "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded counter-based generator)",
        "config": {"workload": desc, "name": a.workload},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": used, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default=DEFAULT)
    ap.add_argument("--split-k", type=int, default=-1)
    ap.add_argument("--kernel", default="auto")
    ap.add_argument("--bias-relu", action="store_true",
                    help="forward workloads: fuse a bias + ReLU epilogue (runs unsplit)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--batch", type=int, default=0, help="override N (small cases for profiling)")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the per-configuration block after the headline")
    ap.add_argument("--per-config-steps", type=int, default=20)
    a = ap.parse_args()
    if a.warmup < 3:
        a.warmup = 3
    rank, world, local_rank = rank_info()
    if a.impl == "reference":
        run_reference(a, rank, world)
        return
    if world > 1:
        import torch
        import torch.distributed as dist_
        torch.cuda.set_device(local_rank)
        dist_.init_process_group("nccl")
    run_ours(a, rank, world, local_rank)
    if world > 1:
        import torch.distributed as dist_
        dist_.destroy_process_group()


if __name__ == "__main__":
    main()
