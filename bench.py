#!/usr/bin/env python3
"""Benchmark of the fp32 normalization kernels on GB300: one JSON line.

Default workload (the one the headline metric is quoted on): LayerNorm of an
fp32 (16, 64, 256, 256) tensor over its last three dims (16 rows of 4,194,304),
x ~ N(0,1), gamma ~ N(1,0.1), beta ~ N(0,0.1), eps 1e-5.  A step is one call of
norm_layer_fwd over that batch.  K steps run back to back between one pair of
CUDA events; no step finds its inputs in L2 (a step's x and y are larger than
twice the L2, or the steps rotate through enough buffer sets to cover three
L2s).  cold_launch adds the median single launch after an L2 flush, and
same_size_copy a device copy of the same x/y bytes timed the same way (the
practical bandwidth ceiling at that transfer size).  For the smaller
workloads per_config also reports the steps replayed from a CUDA graph.

value  = algorithmic bytes per step (x read once + y written once + gamma and
         beta read once) / mean device time of a step, in GB/s, summed over
         ranks (each rank runs the full workload on its own GPU: weak scaling,
         no collective on the data path).
e2e    = the same metric with host buffers: pinned host -> device copy of
         x/gamma/beta, the call, device -> host copy of y, all inside the timed
         region (steps alternate between two streams so copies in the two
         directions overlap).
roofline.achieved / peak: the dominant kernel's algorithmic GB/s against the
         measured HBM copy bandwidth of this GPU pool.
cpu_baseline: the float64 CPU oracle (test infrastructure) on the host cores.
per_config: the other workloads (RMSNorm (2,64,32,32) and (112,64,512,512),
         GroupNorm+LeakyReLU+x2 (1024,8192)/512 groups, LayerNorm cancellation
         stress, and LayerNorm over (16384, 4096) rows) timed the same way, N=1
         only.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
       [--config ln|ln_stress|ln_rows|gn|rms|rms_small] [--no-extras] [--cold-steps N]
       [--rms-batch B] [--cpu-seconds S]
Under torchrun each rank drives one GPU (RANK/LOCAL_RANK/WORLD_SIZE from env).
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "achieved HBM GB/s and % of GB300 roofline per norm kernel (elements/s)"
FALLBACK_HBM_GBS = 6800.0
DATA = ("synthetic: seeded counter-based SplitMix64 + Box-Muller normals (seed 0; tensor ids x=0, "
        "gamma=1, beta=2), identical bytes for the GPU path and the CPU oracle")

# GB300's nominal HBM3e bandwidth (GB/s), reported beside the measured copy peak.
NOMINAL_HBM_GBS = 7900.0

CONFIGS = {
    "rms_small": dict(op="rms", B=2, C=64, S=32 * 32, x=(0.0, 1.0),
                      workload="RMSNorm over dim 1 of fp32 NCHW (2,64,32,32), x~N(0,1), eps 1e-5"),
    "ln": dict(op="ln", rows=16, L=64 * 256 * 256, x=(0.0, 1.0), gamma=(1.0, 0.1), beta=(0.0, 0.1),
               workload="LayerNorm fp32 (16,64,256,256) over the last 3 dims (4,194,304 per row), "
                        "x~N(0,1), gamma~N(1,0.1), beta~N(0,0.1) of (64,256,256), eps 1e-5"),
    "gn": dict(op="gn", N=1024, C=8192, G=512, x=(0.0, 1.0), gamma=(1.0, 0.1), beta=(0.0, 0.1),
               workload="GroupNorm+LeakyReLU(0.01)+x2 fp32 (1024,8192), 512 groups of 16 contiguous "
                        "channels, y~N(0,1), gamma~N(1,0.1), beta~N(0,0.1), eps 1e-5"),
    "rms": dict(op="rms", B=112, C=64, S=512 * 512, x=(0.0, 1.0),
                workload="RMSNorm over dim 1 of fp32 NCHW (112,64,512,512), x~N(0,1), eps 1e-5"),
    "ln_stress": dict(op="ln", rows=16, L=64 * 256 * 256, x=(1000.0, 1e-2), gamma="ones", beta="zeros",
                      workload="LayerNorm cancellation stress fp32 (16,64,256,256), x~N(1000,0.01^2), "
                               "gamma=1, beta=0 (passed as tensors), eps 1e-5"),
    # beyond the five workloads above: LayerNorm over many short rows (the row kernel),
    # and bfloat16 storage (fp32 arithmetic) of three workloads
    "ln_rows_bf16": dict(op="ln", rows=16384, L=4096, x=(0.0, 1.0), gamma=(1.0, 0.1), beta=(0.0, 0.1), bf16=True,
                         workload="LayerNorm bf16 (16384, 4096) over the last dim, fp32 arithmetic, x~N(0,1), "
                                  "gamma~N(1,0.1), beta~N(0,0.1) rounded to bf16, eps 1e-5"),
    "gn_bf16": dict(op="gn", N=1024, C=8192, G=512, x=(0.0, 1.0), gamma=(1.0, 0.1), beta=(0.0, 0.1), bf16=True,
                    workload="GroupNorm+LeakyReLU(0.01)+x2 bf16 (1024,8192), 512 groups of 16, fp32 arithmetic"),
    "rms_bf16": dict(op="rms", B=112, C=64, S=512 * 512, x=(0.0, 1.0), bf16=True,
                     workload="RMSNorm over dim 1 of bf16 NCHW (112,64,512,512), fp32 arithmetic, eps 1e-5"),
    "ln_mid": dict(op="ln", rows=256, L=262144, x=(0.0, 1.0), gamma=(1.0, 0.1), beta=(0.0, 0.1),
                   workload="LayerNorm fp32 (256, 262144) over the last dim, x~N(0,1), gamma~N(1,0.1), "
                            "beta~N(0,0.1), eps 1e-5 (rows of mid length: the persistent kernel in 15 row groups)"),
    "ln_rows": dict(op="ln", rows=16384, L=4096, x=(0.0, 1.0), gamma=(1.0, 0.1), beta=(0.0, 0.1),
                    workload="LayerNorm fp32 (16384, 4096) over the last dim, x~N(0,1), gamma~N(1,0.1), "
                             "beta~N(0,0.1), eps 1e-5 (many short rows)"),
    # GroupNorm with a spatial extent: a group is its channels at every position
    "gn_nchw": dict(op="gn_nchw", N=8, C=512, S=64 * 64, G=32, x=(0.0, 1.0), gamma=(1.0, 0.1), beta=(0.0, 0.1),
                    workload="GroupNorm+LeakyReLU(0.01)+x2 fp32 NCHW (8,512,64,64), 32 groups of 16 channels x "
                             "4096 positions (65,536 values), x~N(0,1), gamma~N(1,0.1), beta~N(0,0.1), eps 1e-5"),
    "gn_nchw_bf16": dict(op="gn_nchw", N=8, C=512, S=64 * 64, G=32, x=(0.0, 1.0), gamma=(1.0, 0.1),
                         beta=(0.0, 0.1), bf16=True,
                         workload="GroupNorm+LeakyReLU(0.01)+x2 bf16 NCHW (8,512,64,64), 32 groups, fp32 "
                                  "arithmetic"),
    "gn_m48": dict(op="gn", N=8192, C=1536, G=32, x=(0.0, 1.0), gamma=(1.0, 0.1), beta=(0.0, 0.1),
                   workload="GroupNorm+LeakyReLU(0.01)+x2 fp32 (8192,1536), 32 groups of 48 contiguous channels "
                            "(not a power of two: the team-per-group kernel), x~N(0,1), gamma~N(1,0.1), "
                            "beta~N(0,0.1), eps 1e-5"),
    "gn_nchw_long": dict(op="gn_nchw", N=1, C=128, S=512 * 512, G=32, x=(0.0, 1.0), gamma=(1.0, 0.1),
                         beta=(0.0, 0.1),
                         workload="GroupNorm+LeakyReLU(0.01)+x2 fp32 NCHW (1,128,512,512), 32 groups of 4 "
                                  "channels x 262144 positions (1,048,576 values: the persistent kernel)"),
    # the GroupNorm page's whole module: Linear(8192, 8192) on (1024, 8192), then the
    # normalization, one kernel (tensor-core GEMM, group statistics in its epilogue)
    "linear_gn": dict(op="linear_gn", M=1024, K=8192, N=8192, G=512, x=(0.0, 1.0), gamma=(1.0, 0.1),
                      beta=(0.0, 0.1),
                      workload="Linear(8192, 8192) + GroupNorm(512 groups of 16) + LeakyReLU(0.01) + x2 on x "
                               "(1024, 8192); x ~ N(0,1) and W ~ U(-1/sqrt(8192), 1/sqrt(8192)) in bf16, bias ~ "
                               "U(-1/sqrt(8192), 1/sqrt(8192)), gamma ~ N(1,0.1), beta ~ N(0,0.1) fp32; y fp32"),
}
EXTRA_ORDER = ["rms_small", "gn", "rms", "ln_stress", "ln_mid", "ln_rows", "ln_rows_bf16", "gn_bf16", "rms_bf16",
               "gn_nchw", "gn_nchw_bf16", "gn_nchw_long", "gn_m48", "linear_gn"]


# ---------------------------------------------------------------------------- sizes

def elements(cfg) -> int:
    """Output elements of a step."""
    if cfg["op"] == "linear_gn":
        return cfg["M"] * cfg["N"]
    if cfg["op"] == "ln":
        return cfg["rows"] * cfg["L"]
    if cfg["op"] == "gn":
        return cfg["N"] * cfg["C"]
    if cfg["op"] == "gn_nchw":
        return cfg["N"] * cfg["C"] * cfg["S"]
    return cfg["B"] * cfg["C"] * cfg["S"]


def param_elems(cfg) -> int:
    if cfg["op"] == "ln":
        return 2 * cfg["L"]
    if cfg["op"] in ("gn", "gn_nchw"):
        return 2 * cfg["C"]
    return 0


def elem_bytes(cfg) -> int:
    return 2 if cfg.get("bf16") else 4


def algorithmic_bytes(cfg) -> int:
    """x read once + y written once + gamma/beta read once (for the Linear: bf16 x and W read
    once, fp32 bias/gamma/beta read once, fp32 y written once)."""
    if cfg["op"] == "linear_gn":
        return 2 * (cfg["M"] * cfg["K"] + cfg["N"] * cfg["K"]) + 4 * (3 * cfg["N"] + cfg["M"] * cfg["N"])
    return elem_bytes(cfg) * (2 * elements(cfg) + param_elems(cfg))


def algorithmic_flops(cfg) -> int:
    """The Linear's multiply-adds (2 M N K); the epilogue's few operations per output are not counted."""
    return 2 * cfg["M"] * cfg["N"] * cfg["K"] if cfg["op"] == "linear_gn" else 0


def l2_note(cfg, l2_bytes=None) -> str:
    if cfg["op"] == "linear_gn":
        return ("inputs larger than L2: x (16 MiB) and W (128 MiB) of one step exceed the L2; K back-to-back "
                "steps between one pair of CUDA events")
    if l2_bytes is None:
        return "inputs larger than L2 (back-to-back steps rotate through enough buffer sets)"
    n = buffer_sets(cfg, l2_bytes)
    mb = 2 * elem_bytes(cfg) * elements(cfg) * n / 2**20
    if n == 1:
        return (f"inputs larger than L2: one step moves {mb:.0f} MiB of x and y, more than twice the "
                f"{l2_bytes / 2**20:.0f} MiB L2; K back-to-back steps between one pair of CUDA events")
    return (f"inputs larger than L2: back-to-back steps rotate through {n} x/y buffer sets ({mb:.0f} MiB, "
            f"at least 3x the {l2_bytes / 2**20:.0f} MiB L2); K steps between one pair of CUDA events")


def shape_config(name, cfg, l2_bytes=None):
    out = {"workload": cfg["workload"], "name": name, "elements": elements(cfg),
           "algorithmic_bytes_per_step": algorithmic_bytes(cfg), "l2": l2_note(cfg, l2_bytes)}
    for k in ("rows", "L", "M", "K", "N", "C", "G", "B", "S"):
        if k in cfg:
            out[{"L": "row_len"}.get(k, k)] = cfg[k]
    return out


# ---------------------------------------------------------------------------- inputs

def host_inputs(cfg, seed=0):
    import numpy as np
    import normgen
    if cfg["op"] == "linear_gn":
        # x and W as the GPU reads them (bf16), bias/gamma/beta fp32: returned as (x, (W, bias), (gamma, beta))
        M, K, N = cfg["M"], cfg["K"], cfg["N"]
        bound = K ** -0.5
        x = normgen.round_bf16(normgen.normal(M * K, cfg["x"][0], cfg["x"][1], seed=seed,
                                              tensor_id=normgen.TENSOR_X))
        w = normgen.round_bf16(normgen.uniform(N * K, -bound, bound, seed=seed, tensor_id=normgen.TENSOR_W))
        bias = normgen.uniform(N, -bound, bound, seed=seed, tensor_id=normgen.TENSOR_LIN_BIAS)
        g = normgen.normal(N, cfg["gamma"][0], cfg["gamma"][1], seed=seed, tensor_id=normgen.TENSOR_GAMMA)
        b = normgen.normal(N, cfg["beta"][0], cfg["beta"][1], seed=seed, tensor_id=normgen.TENSOR_BETA)
        return x, (w, bias), (g, b)
    n = elements(cfg)
    x = normgen.normal(n, cfg["x"][0], cfg["x"][1], seed=seed, tensor_id=normgen.TENSOR_X)
    g = b = None
    if cfg["op"] in ("ln", "gn", "gn_nchw"):
        pn = cfg["L"] if cfg["op"] == "ln" else cfg["C"]
        if cfg.get("gamma") == "ones":
            g = np.ones(pn, dtype=np.float32)
        else:
            g = normgen.normal(pn, cfg["gamma"][0], cfg["gamma"][1], seed=seed, tensor_id=normgen.TENSOR_GAMMA)
        if cfg.get("beta") == "zeros":
            b = np.zeros(pn, dtype=np.float32)
        else:
            b = normgen.normal(pn, cfg["beta"][0], cfg["beta"][1], seed=seed, tensor_id=normgen.TENSOR_BETA)
    if cfg.get("bf16"):  # the values the GPU stores, so the oracle sees the same
        x, g, b = (None if a is None else normgen.round_bf16(a) for a in (x, g, b))
    return x, g, b


def device_tensor(a, cfg, dev):
    """A host float32 array on the device in the workload's storage type (bf16: rounded to
    nearest even by the input generator's helper)."""
    import numpy as np
    import torch
    import normgen
    if cfg.get("bf16"):
        return torch.from_numpy(normgen.bf16_bits(a).view(np.int16)).to(dev).view(torch.bfloat16)
    return torch.from_numpy(a).to(dev)


def main_kernel_name(cfg) -> str:
    if cfg["op"] == "linear_gn":
        return "linear_gn_kernel"
    if cfg["op"] == "ln":
        L, bf16 = cfg["L"], bool(cfg.get("bf16"))
        if L <= (8192 if bf16 else 16384):
            return "ln_rows_kernel"
        big = cfg["rows"] * L * (2 if bf16 else 4) >= (96 << 20)
        if L <= 131072 and L % (8 if bf16 else 4) == 0 and not (L >= 32768 and big):
            return "gns_stream_kernel"
        return "ln_persistent_kernel" if L % (8 if bf16 else 4) == 0 else "ln_split_apply_kernel"
    if cfg["op"] == "gn":
        M, bf16 = cfg["C"] // cfg["G"], bool(cfg.get("bf16"))
        if 4 <= M <= 128 and M & (M - 1) == 0:
            # bench tensors are 16-byte aligned: bf16 groups of 8 or more take 8 channels a thread
            return "gn_vec8_bf16_kernel" if bf16 and M >= 8 else "gn_vec4_kernel"
        items = M // 4 if M % 4 == 0 else M // 2 if M % 2 == 0 else M
        return "gns_team_kernel" if items <= (128 if bf16 else 256) else "gns_reg_kernel"
    if cfg["op"] == "gn_nchw":
        L = cfg["C"] // cfg["G"] * cfg["S"]
        if L % 4 == 0 and L <= 131072:
            return "gns_stream_kernel"
        return "ln_persistent_kernel" if gn_nchw_persistent(cfg) else "gns_split_apply_kernel"
    # bf16 with even S and an exact channel count of at most 64 takes two positions a thread
    if cfg.get("bf16") and cfg["S"] % 2 == 0 and cfg["C"] in (4, 8, 16, 32, 64):
        return "rms_bf16x2_kernel"
    return "rms_reg_kernel"


def gn_nchw_persistent(cfg) -> bool:
    """Groups longer than 131,072 values with S a multiple of the 16-byte unit (4 fp32 or 8 bf16
    values), and x of 48 MiB or more, take the persistent kernel."""
    bf16 = bool(cfg.get("bf16"))
    L = cfg["C"] // cfg["G"] * cfg["S"]
    n = cfg["N"] * cfg["C"] * cfg["S"]
    return cfg["S"] % (8 if bf16 else 4) == 0 and L > 131072 and (2 if bf16 else 4) * n >= 48 << 20


def gn_nchw_one_launch(cfg) -> bool:
    """Groups of at most 131,072 values (a multiple of 4) take the one-launch cluster kernel, longer
    fp32 ones the persistent kernel; the rest two launches."""
    L = cfg["C"] // cfg["G"] * cfg["S"]
    return (L % 4 == 0 and L <= 131072) or gn_nchw_persistent(cfg)


def make_call(ng, cfg, x, g, b, y, ws=None, ws_bytes=0, stream=None):
    """The C-ABI call of one step (device pointers) and the number of our kernel launches it makes."""
    op = cfg["op"]
    bf16 = bool(cfg.get("bf16"))
    if op == "linear_gn":  # g = (W, bias), b = (gamma, beta) on the device
        (w, bias), (gm, bt) = g, b
        return (lambda: ng.norm_linear_group_lrelu_x2_fwd(x, w, bias, gm, bt, y, cfg["M"], cfg["K"], cfg["N"],
                                                          cfg["G"], 1e-5, 0.01, stream)), 1
    if op == "ln":
        rows, L = cfg["rows"], cfg["L"]
        # the persistent kernel's longest bf16 row is twice its fp32 one (8 values a 16-byte unit)
        one_launch = L % 4 == 0 and (L <= (8192 if bf16 else 16384) or (L <= 131072 and L % (8 if bf16 else 4) == 0) or
                                     (L % (8 if bf16 else 4) == 0
                                      and L <= (2 if bf16 else 1) * ng.norm_layer_max_resident_row_len()))
        fn = ng.norm_layer_fwd_bf16 if bf16 else ng.norm_layer_fwd
        return (lambda: fn(x, g, b, y, rows, L, 1e-5, ws, ws_bytes, stream)), (1 if one_launch else 2)
    if op == "gn":
        fn = ng.norm_group_lrelu_x2_fwd_bf16 if bf16 else ng.norm_group_lrelu_x2_fwd
        return (lambda: fn(x, g, b, y, cfg["N"], cfg["C"], cfg["G"], 1e-5, 0.01, stream)), 1
    if op == "gn_nchw":
        fn = ng.norm_group_lrelu_x2_nchw_fwd_bf16 if bf16 else ng.norm_group_lrelu_x2_nchw_fwd
        return ((lambda: fn(x, g, b, y, cfg["N"], cfg["C"], cfg["S"], cfg["G"], 1e-5, 0.01, ws, ws_bytes, stream)),
                1 if gn_nchw_one_launch(cfg) else 2)
    fn = ng.norm_rms_channel_fwd_bf16 if bf16 else ng.norm_rms_channel_fwd
    return (lambda: fn(x, y, cfg["B"], cfg["C"], cfg["S"], 1e-5, stream)), 1


# ---------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples (100 ms) of SM clock and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []
        self._t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", self.gpu_id], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self._t = threading.Thread(target=self._read, daemon=True)
        self._t.start()
        time.sleep(0.25)  # let the sampler start before the timed region

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line.strip()))

    def mark(self):
        return time.perf_counter()

    def stop(self, t0, t1):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "nvidia-smi unavailable"}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        window = [l for (t, l) in self.lines if t0 - 0.1 <= t <= t1 + 0.1] or [l for (_, l) in self.lines]
        for line in window:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(power) if power else None}


def gpu_id_for(local_rank: int) -> str:
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        ids = [v.strip() for v in vis.split(",") if v.strip()]
        if local_rank < len(ids):
            return ids[local_rank]
    return str(local_rank)


# ---------------------------------------------------------------------------- peaks / ncu traffic

def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured (MEASURED_PEAKS.json hbm_gbs: copy of 1 Gi bf16, read+write bytes)"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback 6.8 TB/s (no measured peak file)"


def bf16_peak():
    """Dense bf16 tensor peak (TFLOP/s): the burst figure, for a kernel timed alone in a short loop."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["bf16_tflops"])
        return v, "measured (MEASURED_PEAKS.json bf16_tflops: cuBLAS bf16 8192^3, burst)"
    except (OSError, KeyError, ValueError):
        return 1900.0, "fallback 1.9 PFLOP/s bf16 burst (no measured peak file)"


# the kernel source files each workload's counters depend on
KERNEL_SOURCES = {"ln": ("ln_kernels.cu", "gns_kernels.cu", "norm_internal.cuh"), "gn": ("gn_kernels.cu", "gns_kernels.cu", "norm_internal.cuh"),
                  "gn_nchw": ("gns_kernels.cu", "ln_kernels.cu", "norm_internal.cuh"),
                  "rms": ("rms_kernels.cu", "norm_internal.cuh"),
                  "linear_gn": ("linear_gn_kernels.cu", "norm_internal.cuh")}


def code_only(text: str) -> str:
    """C/C++/CUDA source with comments and blank-space runs removed: what the compiler sees of it
    (string literals here hold no comment markers)."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_hash(op: str) -> str:
    """Hash of the code (not the comments) of the sources a workload's kernels are built from."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "memory_bound_normalization_norm_gb300", "csrc")
    for name in KERNEL_SOURCES[op]:
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            h.update(name.encode() + code_only(f.read()).encode())
    return h.hexdigest()[:16]


def ncu_traffic(config_name: str, op: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the current kernels."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None, "no ncu DRAM counters committed"
    entry = rec.get(config_name)
    if not entry:
        return None, "no ncu DRAM counters for this workload"
    if entry.get("kernel_source_hash") != kernel_source_hash(op):
        return None, "kernels changed since the ncu DRAM counters were taken"
    return entry.get("dram_bytes_per_launch"), entry.get("note", "")


# ---------------------------------------------------------------------------- distributed

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return world, rank, local


def dist_init(world, backend):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend)


def dist_barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def dist_max(value: float, world: int, device=None) -> float:
    """Max of a per-rank scalar over all ranks (timing only: no data-path collective)."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_value(bytes_per_rank: int, world: int, max_seconds_per_step: float) -> float:
    """Whole-job GB/s: the bytes all ranks moved in one step over the slowest rank's step time."""
    return bytes_per_rank * world / max_seconds_per_step / 1e9


# ---------------------------------------------------------------------------- GPU timing

def time_steps(calls, steps, warmup, stream, world=1):
    """W untimed steps, then K back-to-back steps between one pair of CUDA events on
    `stream`; step i uses buffer set i % len(calls).  Returns (mean seconds per step, t0, t1)."""
    import torch
    nset = len(calls)
    with torch.cuda.stream(stream):
        for i in range(warmup):
            calls[i % nset]()
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    dist_barrier(world)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        start.record(stream)
        for i in range(steps):
            calls[i % nset]()
        end.record(stream)
    torch.cuda.synchronize()
    t1 = time.perf_counter()
    dist_barrier(world)
    return start.elapsed_time(end) / 1e3 / steps, t0, t1


def time_cold(call, steps, flush, stream):
    """Single launches from a cold L2: a flush (write of 2x L2 bytes) before each launch, CUDA
    events around each launch only.  Returns the median seconds per launch."""
    import torch
    for _ in range(3):
        flush()
        with torch.cuda.stream(stream):
            call()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for i in range(steps):
            flush()
            starts[i].record(stream)
            call()
            ends[i].record(stream)
    torch.cuda.synchronize()
    return statistics.median(s.elapsed_time(e) for s, e in zip(starts, ends)) / 1e3


def time_graph(calls, stream, launches_per_graph=64, replays=20):
    """The same back-to-back steps captured once in a CUDA graph and replayed: the per-step
    time without the host launch path.  Returns seconds per step."""
    import torch
    # every buffer set at least once per replay, so no step finds its inputs in L2
    launches_per_graph = max(launches_per_graph, len(calls))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for i in range(launches_per_graph):
            calls[i % len(calls)]()
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        start.record(stream)
        for _ in range(replays):
            graph.replay()
        end.record(stream)
    torch.cuda.synchronize()
    return start.elapsed_time(end) / 1e3 / (replays * launches_per_graph)


def time_same_size_copy(xs, ys, steps, stream):
    """A device copy of x into y (the same bytes as one step: x read, y written), back to
    back over the same buffer sets: the practical bandwidth ceiling at this transfer size."""
    import torch
    calls = [(lambda a=a, b=b: b.copy_(a)) for a, b in zip(xs, ys)]
    sec, _, _ = time_steps(calls, steps, 5, stream)
    return sec


def buffer_sets(cfg, l2_bytes: int) -> int:
    """Input/output sets to rotate through so that no step finds its data in L2: one set
    when a step's x + y exceed twice the L2, else enough sets to cover three L2s."""
    if cfg["op"] == "linear_gn":
        return 1  # its inputs (x 16 MiB + W 128 MiB) exceed the L2; the GEMM is bound by the tensor cores
    if "sets" in cfg:
        return cfg["sets"]
    set_bytes = 2 * elem_bytes(cfg) * elements(cfg)
    if set_bytes > 2 * l2_bytes:
        return 1
    return -(-3 * l2_bytes // set_bytes)


def check_status(ng):
    st = ng.norm_last_error()
    if st != 0:
        raise RuntimeError(f"device status {ng.norm_status_string(st)}")


def linear_gn_device(cfg, x, wb, gb, dev):
    """Device tensors of the Linear + GroupNorm workload: x, (W, bias), (gamma, beta) and y."""
    import torch
    import normgen
    import numpy as np
    bf = lambda a: torch.from_numpy(normgen.bf16_bits(a).view(np.int16)).to(dev).view(torch.bfloat16)  # noqa: E731
    f32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dev)  # noqa: E731
    y = torch.empty(cfg["M"] * cfg["N"], dtype=torch.float32, device=dev)
    return bf(x), (bf(wb[0]), f32(wb[1])), (f32(gb[0]), f32(gb[1])), y


def run_config(ng, name, cfg, steps, warmup, stream, flush, l2_bytes, sampler=None, world=1, want_e2e=False,
               cold_steps=100, want_graph=False, want_copy=False):
    import torch
    x, g, b = host_inputs(cfg)
    dev = torch.device("cuda")
    nset = buffer_sets(cfg, l2_bytes)
    if cfg["op"] == "linear_gn":
        xd, gd, bd, yd = linear_gn_device(cfg, x, g, b, dev)
        xs, ys = [xd], [yd]
        want_copy = False
    else:
        xd, gd, bd = (None if a is None else device_tensor(a, cfg, dev) for a in (x, g, b))
        xs = [xd] + [xd.clone() for _ in range(nset - 1)]
        ys = [torch.empty_like(xd) for _ in range(nset)]
    ws = None
    ws_bytes = 0
    if cfg["op"] == "ln":
        ws_bytes = ng.norm_layer_workspace_bytes(cfg["rows"], cfg["L"])
        ws = torch.zeros((ws_bytes + 3) // 4 + 64, dtype=torch.float32, device=dev)
    elif cfg["op"] == "gn_nchw":
        ws_bytes = ng.norm_group_lrelu_x2_nchw_workspace_bytes(cfg["N"], cfg["C"], cfg["S"], cfg["G"])
        ws = torch.zeros((ws_bytes + 3) // 4 + 64, dtype=torch.float32, device=dev)
    calls = []
    launches = 1
    for xk, yk in zip(xs, ys):
        call, launches = make_call(ng, cfg, xk, gd, bd, yk, ws, ws_bytes, stream.cuda_stream)
        calls.append(call)
    torch.cuda.synchronize()
    if sampler:
        sampler.start()
    sec, t0, t1 = time_steps(calls, steps, warmup, stream, world=world)
    clocks = sampler.stop(t0, t1) if sampler else None
    check_status(ng)
    cold = time_cold(calls[0], cold_steps, flush, stream) if cold_steps else None
    check_status(ng)
    graph = None
    if want_graph and nset > 1:
        graph = time_graph(calls, stream)
        check_status(ng)
    copy = time_same_size_copy(xs, ys, min(steps, 200), stream) if want_copy else None
    res = {"name": name, "seconds_per_step": sec, "launches_per_step": launches, "clocks": clocks,
           "t_region_s": t1 - t0, "buffer_sets": nset, "cold_seconds_per_launch": cold,
           "graph_seconds_per_step": graph, "copy_seconds_per_step": copy}
    if want_e2e and cfg["op"] != "linear_gn":
        res["e2e"] = run_e2e(ng, cfg, x, g, b, xd, gd, bd, ys[0], ws, ws_bytes, stream, min(steps, 20), world)
    del xs, ys, xd, gd, bd, ws
    torch.cuda.empty_cache()
    return res


def run_e2e(ng, cfg, x, g, b, xd, gd, bd, yd, ws, ws_bytes, stream, steps, world):
    """Host buffers in, host buffer out, through the C ABI: every step copies its inputs
    from pinned host memory (H2D), makes the call and copies y back (D2H).  Steps alternate
    between two streams with a device buffer set each, so one step's H2D overlaps the
    previous step's call and D2H (the copy engines run both directions at once)."""
    import torch
    cpu = torch.device("cpu")
    xh, gh, bh = (None if a is None else device_tensor(a, cfg, cpu).pin_memory() for a in (x, g, b))
    yh = [torch.empty(xh.shape, dtype=xh.dtype).pin_memory() for _ in range(2)]
    streams = [stream, torch.cuda.Stream()]
    sets = [(xd, gd, bd, yd, ws)]
    ws2 = None if ws is None else torch.zeros_like(ws)
    sets.append((torch.empty_like(xd), None if gd is None else torch.empty_like(gd),
                 None if bd is None else torch.empty_like(bd), torch.empty_like(yd), ws2))
    calls = [make_call(ng, cfg, xs, gs, bs, ys, wss, ws_bytes, st.cuda_stream)[0]
             for (xs, gs, bs, ys, wss), st in zip(sets, streams)]
    h2d = sum(0 if t is None else t.numel() * t.element_size() for t in (xh, gh, bh))
    d2h = yh[0].numel() * yh[0].element_size()

    def step(k):
        i = k % 2
        xs, gs, bs, ys, _ = sets[i]
        with torch.cuda.stream(streams[i]):
            xs.copy_(xh, non_blocking=True)
            if gh is not None:
                gs.copy_(gh, non_blocking=True)
                bs.copy_(bh, non_blocking=True)
            calls[i]()
            yh[i].copy_(ys, non_blocking=True)

    for k in range(4):
        step(k)
    torch.cuda.synchronize()
    dist_barrier(world)
    s = torch.cuda.Event(enable_timing=True)
    e = torch.cuda.Event(enable_timing=True)
    s.record(streams[0])
    streams[1].wait_event(s)
    for k in range(steps):
        step(k)
    streams[0].wait_stream(streams[1])
    e.record(streams[0])
    torch.cuda.synchronize()
    dist_barrier(world)
    sec = s.elapsed_time(e) / 1e3 / steps
    return {"seconds_per_step": sec, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "note": "steps alternate between two streams and two device buffer sets"}


# ---------------------------------------------------------------------------- CPU oracle timing

def time_oracle(cfg, min_seconds, max_reps=1000, rows_per_step=None, x=None, g=None, b=None):
    """Time the float64 oracle (as it stands) on the host cores; returns (GB/s, seconds, reps, threads, sample)."""
    import oracle
    threads = oracle.default_threads()
    o = oracle.get()
    if x is None:
        x, g, b = host_inputs(cfg)
    op = cfg["op"]
    if op == "linear_gn":
        # a bounded sample: the first rows of x through the whole module (float64 matmul + groups)
        rows = max(1, min(cfg["M"], rows_per_step or 16))
        (w, bias), (gm, bt) = g, b
        xs = x[: rows * cfg["K"]]
        fn = lambda: o.linear_group_lrelu_x2(xs, w, bias, gm, bt, rows, cfg["K"], cfg["N"], cfg["G"], 1e-5, 0.01,  # noqa
                                             threads=threads)
        nbytes = algorithmic_bytes(dict(cfg, M=rows))
        sample = f"{rows} of {cfg['M']} rows of the workload per repetition"
        used = min(threads, rows)
    elif op == "ln":
        rows = cfg["rows"] if rows_per_step is None else max(1, min(cfg["rows"], rows_per_step))
        xs = x[: rows * cfg["L"]]
        fn = lambda: o.layer_norm(xs, g, b, rows, cfg["L"], 1e-5, threads=threads)  # noqa: E731
        nbytes = 8 * rows * cfg["L"] + 8 * cfg["L"]
        sample = f"{rows} of {cfg['rows']} rows of the workload per repetition"
        used = min(threads, rows)
    elif op == "gn":
        fn = lambda: o.group_lrelu_x2(x, g, b, cfg["N"], cfg["C"], cfg["G"], 1e-5, 0.01, threads=threads)  # noqa
        nbytes = algorithmic_bytes(cfg)
        sample = "the full workload per repetition"
        used = min(threads, cfg["N"])
    elif op == "gn_nchw":
        fn = lambda: o.group_lrelu_x2_nchw(x, g, b, cfg["N"], cfg["C"], cfg["S"], cfg["G"], 1e-5, 0.01,  # noqa
                                           threads=threads)
        nbytes = algorithmic_bytes(cfg)
        sample = "the full workload per repetition"
        used = min(threads, cfg["N"])
    else:
        fn = lambda: o.rms_channel(x, cfg["B"], cfg["C"], cfg["S"], 1e-5, threads=threads)  # noqa: E731
        nbytes = algorithmic_bytes(cfg)
        sample = "the full workload per repetition"
        used = min(threads, cfg["B"])
    reps = 0
    t0 = time.perf_counter()
    while True:
        fn()
        reps += 1
        el = time.perf_counter() - t0
        if el >= min_seconds or reps >= max_reps:
            break
    return nbytes * reps / el / 1e9, el, reps, used, sample


# ---------------------------------------------------------------------------- main

def reference_arm(args, world, rank):
    """The reference arm: the float64 CPU oracle on this host's cores, same metric and workload."""
    if rank != 0:
        return 0
    cfg = CONFIGS[args.config]
    import oracle
    x, g, b = host_inputs(cfg)
    # the GPU arm's config names the L2 it rotated buffers against: the same text here
    l2 = None
    try:
        import torch
        if torch.cuda.is_available():
            l2 = torch.cuda.get_device_properties(0).L2_cache_size
    except Exception:  # pragma: no cover - CPU-only host
        l2 = None
    # size each step so that the whole run stays within a few minutes
    budget_s = 150.0
    gbs, el, reps, used, sample = time_oracle(cfg, 0.0, max_reps=1, x=x, g=g, b=b)
    per_step = el
    rows_per_step = None
    if cfg["op"] == "ln" and per_step * (args.steps + args.warmup) > budget_s:
        per_row = per_step / cfg["rows"] * max(1, min(oracle.default_threads(), cfg["rows"]))
        rows_per_step = max(1, int(budget_s / (args.steps + args.warmup) / max(per_row, 1e-9)))
    for _ in range(args.warmup):
        time_oracle(cfg, 0.0, max_reps=1, rows_per_step=rows_per_step, x=x, g=g, b=b)
    times = []
    nbytes_tot = 0.0
    for _ in range(args.steps):
        gbs, el, reps, used, sample = time_oracle(cfg, 0.0, max_reps=1, rows_per_step=rows_per_step, x=x, g=g,
                                                  b=b)
        times.append(el)
        nbytes_tot += gbs * el * 1e9
    total = sum(times)
    value = nbytes_tot / total / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total / args.steps * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": DATA,
        "config": shape_config(args.config, cfg, l2),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": used, "kind": "oracle",
                         "sample": sample + " (float64 two-pass C oracle, OpenMP over independent units)"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", choices=sorted(CONFIGS), default="ln")
    ap.add_argument("--no-extras", action="store_true", help="skip the per_config measurements")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="CPU time budget of cpu_baseline")
    ap.add_argument("--cold-steps", type=int, default=100,
                    help="single launches after an L2 flush for cold_launch (0: skip)")
    ap.add_argument("--rms-batch", type=int, default=None,
                    help="batch B of the rms workload (default 112; smaller for profiling captures)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world, rank, local = dist_env()
    if args.impl == "reference":
        return reference_arm(args, world, rank)

    import torch
    torch.cuda.set_device(local)
    dist_init(world, "nccl")
    import memory_bound_normalization_norm_gb300 as ng

    cfg = CONFIGS[args.config]
    if args.rms_batch is not None and cfg["op"] == "rms":
        cfg = dict(cfg, B=args.rms_batch,
                   workload=cfg["workload"].replace(f"({cfg['B']},", f"({args.rms_batch},"))
    stream = torch.cuda.Stream()
    l2 = torch.cuda.get_device_properties(local).L2_cache_size
    flush_buf = torch.empty(max(2 * l2, 64 << 20) // 4, dtype=torch.float32, device="cuda")

    def flush():
        with torch.cuda.stream(stream):
            flush_buf.fill_(1.0)

    sampler = ClockSampler(gpu_id_for(local))
    main_res = run_config(ng, args.config, cfg, args.steps, args.warmup, stream, flush, l2, sampler, world,
                          want_e2e=True, cold_steps=args.cold_steps, want_copy=world == 1 and not args.no_extras)
    sec = dist_max(main_res["seconds_per_step"], world, device="cuda")
    nbytes = algorithmic_bytes(cfg)
    value = weak_scaling_value(nbytes, world, sec)
    e2e_sec = dist_max(main_res["e2e"]["seconds_per_step"], world, device="cuda") if "e2e" in main_res else None
    peak, peak_note = hbm_peak()
    tflops_peak, tflops_note = bf16_peak()
    achieved = nbytes / main_res["seconds_per_step"] / 1e9
    traffic, traffic_note = ncu_traffic(args.config, cfg["op"])

    extras = []
    if world == 1 and not args.no_extras:
        for name in EXTRA_ORDER:
            if name == args.config:
                continue
            c = CONFIGS[name]
            big = c["op"] == "rms" and c["B"] > 8
            k = min(args.steps, 50 if big else 1000)
            r = run_config(ng, name, c, k, 5, stream, flush, l2, cold_steps=10 if big else 100,
                           want_graph=True, want_copy=not big)
            a = algorithmic_bytes(c) / r["seconds_per_step"] / 1e9
            cold = r["cold_seconds_per_launch"]
            more = {}
            if r["graph_seconds_per_step"]:
                gs = r["graph_seconds_per_step"]
                more["graph_us_per_step"] = round(gs * 1e6, 3)
                more["graph_frac_of_measured_peak"] = round(algorithmic_bytes(c) / gs / 1e9 / peak, 4)
            if r["copy_seconds_per_step"]:
                cs = r["copy_seconds_per_step"]
                more["same_size_copy_us"] = round(cs * 1e6, 3)
                more["same_size_copy_frac_of_measured_peak"] = round(2 * elem_bytes(c) * elements(c) / cs / 1e9 / peak, 4)
            if name == "rms_small":
                # the per-call floor: the same entry point on a (1, 64, 32) tensor (16 KiB moved)
                tiny = dict(c, B=1, S=32, sets=64, workload="RMSNorm over dim 1 of fp32 (1,64,32)")
                rt = run_config(ng, "rms_floor", tiny, k, 5, stream, flush, l2, cold_steps=0, want_graph=True)
                more["launch_floor"] = {
                    "us_per_step": round(rt["seconds_per_step"] * 1e6, 3),
                    "graph_us_per_step": (round(rt["graph_seconds_per_step"] * 1e6, 3)
                                          if rt["graph_seconds_per_step"] else None),
                    "note": "the same call on a (1, 64, 32) tensor (16 KiB moved), timed the same way: what any "
                            "call costs before its bytes"}
            fl = algorithmic_flops(c)
            if fl:
                tf = fl / r["seconds_per_step"] / 1e12
                more["achieved_tflops"] = round(tf, 2)
                more["tensor_roofline"] = {"bound": "tensor", "achieved": round(tf, 2), "peak": tflops_peak,
                                           "unit": "TFLOP/s", "frac": round(tf / tflops_peak, 4),
                                           "peak_source": tflops_note}
            extras.append({"config": name, "workload": c["workload"], "steps": k,
                           "us_per_step": round(r["seconds_per_step"] * 1e6, 3),
                           "algorithmic_bytes": algorithmic_bytes(c), "achieved_gbs": round(a, 2),
                           "frac_of_measured_peak": round(a / peak, 4),
                           "elements_per_s": round(elements(c) / r["seconds_per_step"], 1),
                           "launches_per_step": r["launches_per_step"], "l2": l2_note(c, l2),
                           "cold_launch_us": round(cold * 1e6, 3),
                           "cold_frac_of_measured_peak": round(algorithmic_bytes(c) / cold / 1e9 / peak, 4),
                           **more})

    cpu = None
    if rank == 0 and args.cpu_seconds > 0:
        gbs, el, reps, used, sample = time_oracle(cfg, args.cpu_seconds, max_reps=200)
        cpu = {"value": round(gbs, 4), "unit": "GB/s", "cores": used, "kind": "oracle",
               "sample": f"{sample}, {reps} repetitions in {el:.1f} s (float64 two-pass C oracle)"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(sec * 1e3, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if cfg.get("bf16") or cfg["op"] == "linear_gn" else "f32", "data": DATA,
            "config": shape_config(args.config, cfg, l2),
            "elements_per_s": round(elements(cfg) * world / sec, 1),
            "same_size_copy": None if not main_res["copy_seconds_per_step"] else {
                "us": round(main_res["copy_seconds_per_step"] * 1e6, 3),
                "frac_of_measured_peak": round(2 * elem_bytes(cfg) * elements(cfg) / main_res["copy_seconds_per_step"] / 1e9
                                               / peak, 4),
                "note": "device copy of x into y (same bytes as a step minus gamma/beta), timed the same way"},
            "cold_launch": None if not main_res["cold_seconds_per_launch"] else {
                "us": round(main_res["cold_seconds_per_launch"] * 1e6, 3),
                "frac_of_measured_peak": round(nbytes / main_res["cold_seconds_per_launch"] / 1e9 / peak, 4),
                "note": "median single launch after an L2 flush (2x L2 written), CUDA events around each launch"},
            "roofline": ({"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                          "frac": round(achieved / peak, 4), "traffic": traffic,
                          "nominal_peak": NOMINAL_HBM_GBS, "frac_of_nominal": round(achieved / NOMINAL_HBM_GBS, 4),
                          "peak_source": peak_note, "traffic_note": traffic_note,
                          "kernel": main_kernel_name(cfg)} if not algorithmic_flops(cfg) else
                         {"bound": "tensor", "achieved": round(algorithmic_flops(cfg) / sec / 1e12, 2),
                          "peak": tflops_peak, "unit": "TFLOP/s",
                          "frac": round(algorithmic_flops(cfg) / sec / 1e12 / tflops_peak, 4), "traffic": traffic,
                          "peak_source": tflops_note, "traffic_note": traffic_note, "kernel": main_kernel_name(cfg)}),
            "cpu_baseline": cpu,
            "e2e": None if e2e_sec is None else {
                "value": round(weak_scaling_value(nbytes, world, e2e_sec), 3), "unit": "GB/s",
                "h2d_bytes_per_step": main_res["e2e"]["h2d_bytes_per_step"],
                "d2h_bytes_per_step": main_res["e2e"]["d2h_bytes_per_step"],
                "ms_per_step": round(e2e_sec * 1e3, 4), "note": main_res["e2e"]["note"]},
            "gpu_launches": main_res["launches_per_step"] * args.steps,
            "clocks": main_res["clocks"],
            "per_config": extras,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
