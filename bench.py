#!/usr/bin/env python3
"""BF16 Tensor Core GEMM benchmark on GB300: TFLOP/s = 2MNK / device time.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME | --m M --n N --k K [--A row|col] [--B row|col]
                     [--C bf16|f32] [--split-k S] [--persistent 0|1]]
                    [--no-cpu-baseline] [--sustained-seconds S] [--no-e2e] [--all-workloads]
                    [--oracle-table]

A step is one GEMM C = A . B over one batch of synthetic input (the whole hot
path: plan, TMA-fed tcgen05 main loop, epilogue, and the split-K combine when
the workload uses it).  The default workload is the largest single-GPU one,
the rectangular 16384 x 8192 x 8192 GEMM with bf16 A (row-major), B
(column-major) and C, inputs N(0,1)/sqrt(K), on the persistent scheduler.
--m/--n/--k (with the layout, output and split flags, as a library profiler
takes them) time any other shape.  After the K timed steps the same GEMM runs
back to back for --sustained-seconds more (default 4 s) to report the rate
the part sustains under its power cap, beside the clocks it ran at.

Timing: W untimed warm-up steps, then K steps bracketed by a barrier and
torch.cuda.synchronize() on both sides, CUDA events on the launching stream
around the whole region and around each launch.  Operands rotate through
enough copies that the bytes touched between two uses of one copy exceed L2,
so every step reads its inputs from HBM.  Under torchrun each rank runs the
same GEMM on its own GPU (the GEMM does not shard: replicas only); the time
is the maximum over ranks and the value counts every rank's FLOPs.

Prints one JSON line on rank 0.  ``--impl reference`` times the CPU oracle
(binary64 triple loop) on the host cores instead, on bounded row samples of
the same workload.
"""
from __future__ import annotations

import argparse
import ctypes
import datetime as _dt
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "GEMM TFLOP/s (2MNK/device time) and % of GB300 dense BF16 peak, 1 GPU"
UNIT = "TFLOP/s"

WORKLOADS = {
    "square4096": dict(M=4096, N=4096, K=4096, out="bf16", dist="normal", scaled=True, split_k=0,
                       desc="gemm_bf16 M=N=K=4096, A bf16 row-major, B bf16 column-major, C bf16 row-major, "
                            "inputs N(0,1)/sqrt(K), fp32 accumulate"),
    "square256": dict(M=256, N=256, K=256, out="f32", dist="uniform", scaled=False, split_k=0,
                      desc="gemm_bf16 M=N=K=256, A row-major, B column-major, C fp32, inputs uniform[-1,1]"),
    "n4095": dict(M=4095, N=4096, K=4096, out="bf16", dist="normal", scaled=True, split_k=0,
                  desc="gemm_bf16 4095x4096x4096, bf16 row x col -> bf16, N(0,1)/sqrt(K)"),
    "n4097": dict(M=4097, N=4096, K=4096, out="bf16", dist="normal", scaled=True, split_k=0,
                  desc="gemm_bf16 4097x4096x4096, bf16 row x col -> bf16, N(0,1)/sqrt(K)"),
    "k4088": dict(M=4096, N=4096, K=4088, out="bf16", dist="normal", scaled=True, split_k=0,
                  desc="gemm_bf16 4096x4096x4088, bf16 row x col -> bf16, N(0,1)/sqrt(K)"),
    "n4104": dict(M=4096, N=4104, K=4096, out="bf16", dist="normal", scaled=True, split_k=0,
                  desc="gemm_bf16 4096x4104x4096, bf16 row x col -> bf16, N(0,1)/sqrt(K)"),
    "m3968": dict(M=3968, N=4096, K=4096, out="bf16", dist="normal", scaled=True, split_k=0,
                  desc="gemm_bf16 3968x4096x4096, bf16 row x col -> bf16, N(0,1)/sqrt(K)"),
    "square4096_b_row": dict(M=4096, N=4096, K=4096, out="bf16", dist="normal", scaled=True, split_k=0,
                             b_row=True,
                             desc="gemm_bf16 M=N=K=4096, A bf16 row-major, B bf16 row-major (A @ B with a "
                                  "contiguous K x N B), C bf16, N(0,1)/sqrt(K)"),
    "square4096_a_col_b_row": dict(M=4096, N=4096, K=4096, out="bf16", dist="normal", scaled=True, split_k=0,
                                   a_col=True, b_row=True,
                                   desc="gemm_bf16 M=N=K=4096, A bf16 column-major, B bf16 row-major, C bf16, "
                                        "N(0,1)/sqrt(K)"),
    "square4096_residual_bias_gelu": dict(
        M=4096, N=4096, K=4096, out="bf16", dist="normal", scaled=True, split_k=0,
        epilogue=dict(alpha=1.0, beta=1.0, bias=True, activation="gelu"),
        desc="gemm_bf16 M=N=K=4096, A row-major, B column-major, C bf16 := gelu(A.B + C + bias[n]) "
             "(fused epilogue), N(0,1)/sqrt(K)"),
    "large": dict(M=16384, N=8192, K=8192, out="bf16", dist="normal", scaled=True, split_k=0,
                  desc="gemm_bf16 16384x8192x8192, bf16 row x col -> bf16, N(0,1)/sqrt(K)"),
    "large_one_cta_per_tile": dict(M=16384, N=8192, K=8192, out="bf16", dist="normal", scaled=True, split_k=0,
                                   non_persistent=True,
                                   desc="gemm_bf16 16384x8192x8192, bf16 row x col -> bf16, one CTA per tile"),
}
# implicit-GEMM convolutions (NHWC x KRSC -> NPQK, bf16), inputs N(0,1), filters N(0,1)/sqrt(R S C)
WORKLOADS["conv3x3_n32_56x56_c256_k256"] = dict(
    conv=dict(N=32, H=56, W=56, C=256, K=256, R=3, S=3, pad=(1, 1), stride=(1, 1), dil=(1, 1)), out="bf16",
    dist="normal", scaled=True, desc="conv2d fprop as implicit GEMM, N32 H56 W56 C256 -> K256, 3x3, pad 1, stride 1, "
                                     "NHWC/KRSC bf16 -> bf16")
WORKLOADS["conv3x3_n32_28x28_c512_k512"] = dict(
    conv=dict(N=32, H=28, W=28, C=512, K=512, R=3, S=3, pad=(1, 1), stride=(1, 1), dil=(1, 1)), out="bf16",
    dist="normal", scaled=True, desc="conv2d fprop as implicit GEMM, N32 H28 W28 C512 -> K512, 3x3, pad 1, stride 1, "
                                     "NHWC/KRSC bf16 -> bf16")
for _s in (1, 8, 32, 74, 148):
    WORKLOADS[f"splitk{_s}"] = dict(M=128, N=256, K=65536, out="f32", dist="uniform", scaled=True, split_k=_s,
                                    desc=f"gemm_bf16 128x256x65536, bf16 row x col -> fp32, uniform[-1,1]/sqrt(K), "
                                         f"split_k={_s}")

KERNEL_NAME = "gemm_bf16_kernel"
DEFAULT_WORKLOAD = "large"
# How every timed region keeps its operands out of L2 (the same words on both arms).
L2_POLICY = ("inputs larger than L2: operand sets rotate so that the bytes touched between two uses of one set "
             "exceed twice the L2 size")


def custom_workload(m: int, n: int, k: int, a: str, b: str, c: str, split_k: int, persistent: int, dist: str):
    """A workload from profiler-style flags (--m --n --k --A --B --C --split-k --persistent)."""
    scaled = dist != "int4"
    return dict(M=m, N=n, K=k, out=c, dist=dist, scaled=scaled, split_k=split_k, a_col=a == "col", b_row=b == "row",
                non_persistent=not persistent,
                desc=f"gemm_bf16 {m}x{n}x{k}, A bf16 {a}-major, B bf16 {b}-major, C {c} row-major, "
                     f"inputs {dist}{'/sqrt(K)' if scaled else ''}, split_k={split_k}, "
                     f"{'persistent' if persistent else 'one cluster per tile'}")


def workload_data(w: dict, seed: int) -> str:
    """The bench line's ``data`` for a GEMM workload (both arms)."""
    return f"synthetic (seeded SplitMix64, {w['dist']}{'/sqrt(K)' if w['scaled'] else ''}, seed {seed})"


def workload_config(w: dict) -> dict:
    """The bench line's ``config`` for a GEMM workload: what is computed and
    how it is timed, the same on both arms (the GPU arm's plan goes under
    ``plan``)."""
    return {"workload": w["desc"], "M": w["M"], "N": w["N"], "K": w["K"], "out": w["out"],
            "layout_a": "column-major" if w.get("a_col") else "row-major",
            "layout_b": "row-major" if w.get("b_row") else "column-major",
            "epilogue": w.get("epilogue"), "split_k": w["split_k"],
            "launch": "one cluster per tile" if w.get("non_persistent") else "persistent",
            "l2": L2_POLICY, "parallelism": "replicas (one independent GEMM per GPU)"}


def conv_out_dims(cv: dict):
    P = (cv["H"] + 2 * cv["pad"][0] - cv["dil"][0] * (cv["R"] - 1) - 1) // cv["stride"][0] + 1
    Q = (cv["W"] + 2 * cv["pad"][1] - cv["dil"][1] * (cv["S"] - 1) - 1) // cv["stride"][1] + 1
    return P, Q


CONV_METRIC = "conv2d TFLOP/s (2 N P Q K R S C / device time) and % of GB300 dense BF16 peak, 1 GPU"


def conv_data(seed: int) -> str:
    return f"synthetic (seeded SplitMix64, N(0,1) input, N(0,1)/sqrt(RSC) filter, seed {seed})"


def conv_config(w: dict) -> dict:
    cv = w["conv"]
    P, Q = conv_out_dims(cv)
    return {"workload": w["desc"], **{k: v for k, v in cv.items()}, "P": P, "Q": Q, "out": w["out"],
            "gemm": {"M": cv["N"] * P * Q, "N": cv["K"], "K": cv["R"] * cv["S"] * cv["C"]},
            "l2": L2_POLICY, "parallelism": "replicas (one independent convolution per GPU)"}


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return dict(bf16_burst=float(d["bf16_tflops"]), bf16_sustained=float(d["bf16_tflops_sustained"]),
                    hbm_gbs=float(d["hbm_gbs"]), source="measured")
    return dict(bf16_burst=1900.0, bf16_sustained=1700.0, hbm_gbs=6800.0, source="fallback")


def roofline_entry(flops: float, alg_bytes: float, mean_ms: float, peaks: dict, peak_tflops: float, peak_kind: str):
    """The bound of a launch from its arithmetic intensity against the measured
    ridge point (bf16 peak / HBM bandwidth): below it the launch is judged in
    GB/s of algorithmic bytes against the measured HBM bandwidth, above it in
    TFLOP/s against the bf16 peak."""
    ridge = peak_tflops * 1e12 / (peaks["hbm_gbs"] * 1e9)
    ai = flops / alg_bytes
    if ai < ridge:
        achieved = alg_bytes / (mean_ms * 1e-3) / 1e9
        return {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(achieved / peaks["hbm_gbs"], 4), "peak_source": f"copy bandwidth, {peaks['source']}",
                "arithmetic_intensity": round(ai, 1), "ridge_flop_per_byte": round(ridge, 1),
                "algorithmic_bytes_per_launch": alg_bytes}
    achieved = flops / (mean_ms * 1e-3) / 1e12
    return {"bound": "tensor", "achieved": round(achieved, 3), "peak": peak_tflops, "unit": "TFLOP/s",
            "frac": round(achieved / peak_tflops, 4), "peak_source": peak_kind,
            "arithmetic_intensity": round(ai, 1), "ridge_flop_per_byte": round(ridge, 1),
            "algorithmic_flops_per_launch": flops}


def _code_only(text: str) -> str:
    """C/C++ source without its comments (none of the library's string
    literals holds a comment marker), its whitespace collapsed: a change to
    the prose or the layout alone leaves the hash as it was."""
    code = re.sub(r"//[^\n]*", "", re.sub(r"/\*.*?\*/", "", text, flags=re.S))
    return " ".join(code.split())


# The files that decide what the GEMM kernels do and how a problem is cut into
# launches; the host-batch pipeline (host_pipeline.cpp) only feeds them.
KERNEL_SOURCES = ("gemm_bf16.cu", "kernel_config.h", "plan.cpp", "plan_internal.h", "ptx.cuh")


def kernel_source_hash() -> str:
    """sha256 over the library's sources with comments removed: the code the
    recorded counters were taken on, not its prose."""
    h = hashlib.sha256()
    files = [os.path.join(ROOT, "dense_tensor_core_bf16_gb300", "csrc", f) for f in KERNEL_SOURCES]
    files.append(os.path.join(ROOT, "include", "gemm_bf16.h"))
    for fn in files:
        with open(fn, encoding="utf-8") as f:
            h.update(os.path.basename(fn).encode())
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()


def recorded_traffic(workload: str):
    """DRAM bytes per launch of the main kernel from a committed ncu summary,
    if it was taken on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", f"dram_traffic_{workload}.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    if d.get("kernel_source_sha256") != kernel_source_hash():
        return None
    return d.get("dram_bytes_per_launch")


# ---- clocks sampled during the timed region ------------------------------------------

class ClockSampler:
    FIELDS = ["timestamp", "clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, gpu_id: str, period_ms: int = 100):
        self.rows = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", gpu_id, f"--query-gpu={','.join(self.FIELDS)}", "--format=csv,noheader,nounits",
                 f"-lms={period_ms}"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != len(self.FIELDS):
                continue
            try:
                ts = _dt.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                self.rows.append((ts, float(parts[1]), float(parts[2]), parts[4:]))
            except ValueError:
                continue

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "nvidia-smi gave no samples"}
        inside = [r for r in self.rows if t0 <= r[0] <= t1]
        note = "samples inside the timed region"
        if not inside:
            mid = 0.5 * (t0 + t1)
            inside = sorted(self.rows, key=lambda r: abs(r[0] - mid))[:3]
            note = "timed region shorter than the sampling period: nearest samples"
        names = ["active_mask", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in inside:
            for n, v in zip(names[1:], r[3][1:]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(r[1] for r in inside), "sm_max_mhz": max(r[2] for r in inside),
                "reasons": sorted(reasons), "samples": len(inside), "note": note}


class NvmlPoller:
    """SM clock, its maximum and the clock-event reasons read through NVML
    (read-only queries) while the host waits for a timed region's end event.
    The region of a short step lasts a few milliseconds, shorter than
    nvidia-smi's sampling period; these samples fall inside it."""
    # nvmlClocksEventReasons bits (NVML's public header)
    REASON_BITS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
                   0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}
    CLOCK_SM = 1

    def __init__(self, uuid: str | None):
        self.lib = None
        if not uuid:
            return
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                return
            handle = ctypes.c_void_p()
            if lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(handle)) != 0:
                return
            reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                lib.nvmlDeviceGetCurrentClocksThrottleReasons
        except (OSError, AttributeError):
            return
        self.lib, self.handle, self.reasons = lib, handle, reasons

    def sample(self):
        clk, mx, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        if (self.lib.nvmlDeviceGetClockInfo(self.handle, self.CLOCK_SM, ctypes.byref(clk)) != 0 or
                self.lib.nvmlDeviceGetMaxClockInfo(self.handle, self.CLOCK_SM, ctypes.byref(mx)) != 0 or
                self.reasons(self.handle, ctypes.byref(rs)) != 0):
            return None
        return float(clk.value), float(mx.value), int(rs.value)

    def sample_in_background(self, period_s: float = 0.002):
        """(rows, stop): samples appended to ``rows`` by a thread every
        ``period_s`` until ``stop()`` is called (ctypes releases the GIL
        during each NVML call)."""
        rows, done = [], threading.Event()

        def run():
            while not done.is_set():
                if self.lib is not None:
                    r = self.sample()
                    if r is not None:
                        rows.append(r)
                time.sleep(period_s)

        t = threading.Thread(target=run, daemon=True)
        t.start()

        def stop():
            done.set()
            t.join(timeout=5)
        return rows, stop

    def poll_until(self, event) -> list:
        """Samples taken until ``event`` (a torch.cuda.Event) has completed."""
        rows = []
        while not event.query():
            if self.lib is not None:
                r = self.sample()
                if r is not None:
                    rows.append(r)
            time.sleep(0.0002)
        return rows


def clocks_summary(nvml_rows: list, smi: dict) -> dict:
    """The bench line's ``clocks``: from the NVML samples inside the timed
    region when there are any, else nvidia-smi's; nvidia-smi's summary is
    kept beside them."""
    if not nvml_rows:
        return dict(smi)
    reasons = sorted({name for _, _, bits in nvml_rows for bit, name in NvmlPoller.REASON_BITS.items() if bits & bit})
    return {"sm_mhz": statistics.median(r[0] for r in nvml_rows), "sm_max_mhz": max(r[1] for r in nvml_rows),
            "reasons": reasons, "samples": len(nvml_rows),
            "note": "NVML samples taken inside the timed region", "nvidia_smi": smi}


# ---- distributed plumbing (host-side only: barrier and max/sum of scalars) ------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def aggregate(ms_local: float, flops_local: float, group=None):
    """(max elapsed ms over ranks, total FLOPs over ranks)."""
    import torch
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized():
        return ms_local, flops_local
    dev = "cuda" if dist.get_backend(group) == "nccl" else "cpu"
    t = torch.tensor([ms_local], dtype=torch.float64, device=dev)
    f = torch.tensor([flops_local], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    dist.all_reduce(f, op=dist.ReduceOp.SUM, group=group)
    return float(t.item()), float(f.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# ---- the GPU arm ---------------------------------------------------------------------

def make_host_operands(w):
    from dense_tensor_core_bf16_gb300 import inputs
    seed = inputs.DEFAULT_SEED + 100
    return inputs.workload_operands(w["M"], w["N"], w["K"], dist=w["dist"], scaled=w["scaled"], seed=seed), seed


def run_gpu(args, wname: str, w: dict, cpu_baseline: bool):
    import numpy as np
    import torch

    import dense_tensor_core_bf16_gb300 as g

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    M, N, K = w["M"], w["N"], w["K"]
    out_dtype = torch.bfloat16 if w["out"] == "bf16" else torch.float32
    (A_h, Bt_h), seed = make_host_operands(w)

    kw = dict(split_k=w["split_k"], non_persistent=w.get("non_persistent", False), kernel_variant=args.variant,
              no_stream_k=args.no_stream_k, raster_group_m=args.raster_group)
    epi = w.get("epilogue")
    if epi:
        from dense_tensor_core_bf16_gb300 import inputs
        # the fused epilogue: a bias of N values (seeded, like the operands); C is read (beta != 0)
        bias_bits = inputs.matrix(1, N, dist="normal", seed=seed, stream=8)[0]
        kw.update(alpha=epi["alpha"], beta=epi["beta"], activation=epi["activation"],
                  bias=torch.from_numpy((bias_bits.astype(np.uint32) << 16).view(np.float32)).cuda()
                  if epi["bias"] else None)
    # operand storage: A row-major (M x K) or column-major (stored K x M); B
    # column-major (stored N x K) or row-major (stored K x N)
    a_col, b_row = w.get("a_col", False), w.get("b_row", False)
    layout_a = g.GEMM_COL_MAJOR if a_col else g.GEMM_ROW_MAJOR
    layout_b = g.GEMM_ROW_MAJOR if b_row else g.GEMM_COL_MAJOR
    a_view = (lambda t: t.t()) if a_col else (lambda t: t)
    b_view = (lambda t: t) if b_row else (lambda t: t.t())
    A_store = np.ascontiguousarray(A_h.T) if a_col else A_h
    B_store = np.ascontiguousarray(Bt_h.T) if b_row else Bt_h
    # the plan the timed call makes: the same options, epilogue included (a
    # long epilogue changes how a stream-K tail is dealt out)
    plan_epi = None
    if epi:
        plan_epi = g.gemm_epilogue_t(alpha=epi["alpha"], beta=epi["beta"], bias=None,
                                     activation=g.ACTIVATIONS[epi["activation"]])
    st, plan = g.gemm_plan(M, N, K, layout_a, layout_b,
                           g.GEMM_OUT_BF16 if w["out"] == "bf16" else g.GEMM_OUT_F32,
                           g.options(split_k=kw["split_k"], non_persistent=int(kw["non_persistent"]),
                                     kernel_variant=kw["kernel_variant"], no_stream_k=int(kw["no_stream_k"]),
                                     raster_group_m=kw["raster_group_m"] or 0,
                                     epilogue=ctypes.pointer(plan_epi) if plan_epi is not None else None))
    if st:
        raise g.GemmError(st, "gemm_plan")
    if plan.workspace_bytes:
        st = g.gemm_reserve_workspace(plan.workspace_bytes)
        if st:
            raise g.GemmError(st, "gemm_reserve_workspace")

    props = torch.cuda.get_device_properties(local)
    l2 = getattr(props, "L2_cache_size", 135_528_448) or 135_528_448
    esize = 2 if w["out"] == "bf16" else 4
    set_bytes = 2 * M * K + 2 * N * K + esize * M * N
    copies = max(2, math.ceil(2 * l2 / set_bytes) + 1)

    # device copies with every line padded to a whole 16 bytes, as the library
    # requires of lda, ldb and ldc (no padding for the named workloads)
    def dev_padded(X):
        rows, cols = X.shape
        base = torch.zeros((rows, -(-cols // 8) * 8), dtype=torch.int16, device="cuda")
        base[:, :cols] = torch.from_numpy(np.ascontiguousarray(X).view(np.int16)).cuda()
        return base

    def c_padded():
        q = 8 if out_dtype == torch.bfloat16 else 4
        return torch.zeros((M, -(-N // q) * q), dtype=out_dtype, device="cuda")[:, :N]

    A0 = dev_padded(A_store)
    B0 = dev_padded(B_store)
    sets = []
    for i in range(copies):
        a = A0 if i == 0 else A0.clone()
        b = B0 if i == 0 else B0.clone()
        a = a[:, :A_store.shape[1]].view(torch.bfloat16)
        b = b[:, :B_store.shape[1]].view(torch.bfloat16)
        sets.append((a_view(a), b_view(b), c_padded()))
    launches_per_step = 1 + (1 if plan.split_k > 1 else 0)

    def step(i, **extra):
        a, b, c = sets[i % copies]
        g.matmul(a, b, out=c, **kw, **extra)

    # The clock sampler starts before the warm-up, so that the GPU does not sit
    # idle between the warm-up and the timed region (after an idle gap the
    # first launches of a short step run slower).
    gpu_id = getattr(props, "uuid", None)
    gpu_id = f"GPU-{gpu_id}" if gpu_id is not None else str(local)
    sampler = ClockSampler(gpu_id)
    nvml = NvmlPoller(gpu_id if gpu_id.startswith("GPU-") else None)
    time.sleep(0.3)
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    st, where = g.gemm_get_device_status(None)
    if st:
        raise RuntimeError(f"device fault during warm-up: {where:#x}")

    # The K steps go back to back between two events (events between launches
    # would break the overlap of one launch's prologue with the previous one's
    # tail).  The main kernel's mean launch time is the region time over K,
    # gaps included.  With split-K a step is two kernels; a separate short
    # pass with an event between them (recorded by the library) gives the
    # combine kernel's share.
    stream = torch.cuda.current_stream()
    two_kernels = plan.split_k > 1
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    e0.record(stream)
    for i in range(args.steps):
        step(i)
    e1.record(stream)
    nvml_rows = nvml.poll_until(e1)
    torch.cuda.synchronize()
    barrier()
    t_wall1 = time.time()
    time.sleep(0.25)
    sampler.stop()
    st, where = g.gemm_get_device_status(None)
    if st:
        raise RuntimeError(f"device fault in the timed region: {where:#x}")
    total_ms = e0.elapsed_time(e1)

    main_ms = [total_ms / args.steps]
    combine_ms = None
    if two_kernels:
        n_split = min(args.steps, 20)
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(n_split)]
        mids = [torch.cuda.Event(enable_timing=True) for _ in range(n_split)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(n_split)]
        for ev in mids:
            ev.record(stream)   # torch creates the CUDA event on its first record; the library records it again
        torch.cuda.synchronize()
        for i in range(n_split):
            starts[i].record(stream)
            step(i, mainloop_done_event=mids[i])
            ends[i].record(stream)
        torch.cuda.synchronize()
        combine_ms = [m.elapsed_time(e) for m, e in zip(mids, ends)]
        main_ms = [s_.elapsed_time(m) for s_, m in zip(starts, mids)]

    flops = 2.0 * M * N * K
    max_ms, total_flops = aggregate(total_ms, flops * args.steps)
    value = total_flops / (max_ms * 1e-3) / 1e12

    peaks = load_peaks()
    long_region = (t_wall1 - t_wall0) > 1.0
    peak = peaks["bf16_sustained"] if long_region else peaks["bf16_burst"]
    peak_kind = ("sustained" if long_region else "burst") + f" bf16, {peaks['source']}"
    mean_main_ms = statistics.fmean(main_ms)
    achieved = flops / (mean_main_ms * 1e-3) / 1e12
    result = {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(max_ms / args.steps, 6), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": workload_data(w, seed),
        "config": workload_config(w),
        "plan": {
            "kernel_variant": g.KERNEL_VARIANTS[plan.kernel_variant], "cluster_size": plan.cluster_size,
            "tile": f"{plan.tile_m}x{plan.tile_n}x{plan.tile_k}", "stages": plan.stages,
            "split_k": plan.split_k, "persistent": bool(plan.persistent), "grid_G": plan.grid,
            "launch_ctas": plan.launch_ctas, "resident_ctas": plan.resident_ctas, "num_sms": plan.num_sms,
            "ctas_per_sm": plan.ctas_per_sm,
            "occupancy_limiter": g.LIMITERS[plan.occupancy_limiter],
            "eta_wave": round(plan.eta_wave, 5), "eta_pad": round(plan.eta_pad, 5),
            "stream_k_tiles": plan.stream_k_tiles, "dp_tiles": plan.dp_tiles,
            "eta_stream_k": round(plan.eta_stream_k, 5), "raster_group_m": plan.raster_group_m,
            "pct_of_peak": round(100.0 * value / world / peak, 2), "peak_tflops": peak, "peak_kind": peak_kind,
            "l2_sets": f"{copies} rotating operand sets of {set_bytes / 1e6:.1f} MB "
                       f"({copies * set_bytes / 1e6:.0f} MB) vs L2 {l2 / 1e6:.1f} MB",
        },
        "roofline": {
            "kernel": f"{KERNEL_NAME}<{plan.cluster_size},{plan.tile_n}>",
            **roofline_entry(flops, 2.0 * M * K + 2.0 * N * K + esize * M * N, mean_main_ms, peaks, peak, peak_kind),
            "traffic": recorded_traffic(wname), "mean_launch_ms": round(mean_main_ms, 6),
            "launch_time_from": "events around each main kernel (separate pass)" if two_kernels else
                                "timed region / steps, launches back to back",
        },
        "gpu_launches": launches_per_step * args.steps,
    }
    if combine_ms is not None:
        comb = statistics.fmean(combine_ms)
        comb_bytes = plan.split_k * M * N * 4 + esize * M * N   # algorithmic: every slice read once, C written once
        result["plan"]["mainloop_us"] = round(mean_main_ms * 1e3, 3)
        result["plan"]["combine_us"] = round(comb * 1e3, 3)
        result["plan"]["combine_gbs"] = round(comb_bytes / (comb * 1e-3) / 1e9, 1)
    clocks = clocks_summary(nvml_rows, sampler.summary(t_wall0, t_wall1))
    result["clocks"] = clocks
    if args.sustained_seconds > 0:
        result["sustained"] = sustained_region(args.sustained_seconds, max_ms / args.steps, step, flops, peaks,
                                               stream, nvml, gpu_id)
    if args.no_e2e:
        if cpu_baseline and rank == 0 and world == 1:
            result["cpu_baseline"] = cpu_oracle_baseline(A_h, Bt_h, M, N, K, target_s=args.cpu_seconds)
        return result, rank

    # End to end through the public API: every step copies its A and B from
    # pinned host memory and its C back, through gemm_bf16_host_batch, which
    # overlaps one step's copies with another step's product.  Two host sets
    # alternate so that consecutive steps never share a buffer.
    e2e_steps = max(min(args.steps, 20), 2)
    hA = [torch.from_numpy(A_store.view(np.int16)).view(torch.bfloat16).pin_memory() for _ in range(2)]
    hB = [torch.from_numpy(B_store.view(np.int16)).view(torch.bfloat16).pin_memory() for _ in range(2)]
    hC = [torch.zeros((M, N), dtype=out_dtype).pin_memory() for _ in range(2)]
    ha = [a_view(x) for x in hA]
    hb = [b_view(x) for x in hB]
    hkw = {k: v for k, v in kw.items() if k in ("split_k", "no_stream_k", "non_persistent", "kernel_variant",
                                                 "alpha", "beta", "bias", "activation")}

    def e2e_batch(n):
        idx = [i % 2 for i in range(n)]
        return g.matmul_host_batch([ha[i] for i in idx], [hb[i] for i in idx], outs=[hC[i] for i in idx],
                                   stream=stream, **hkw)

    e2e_batch(2)   # grows the staging slots outside the timed region
    torch.cuda.synchronize()
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    f0.record(stream)
    e2e_batch(e2e_steps)
    f1.record(stream)
    torch.cuda.synchronize()
    e2e_ms, e2e_flops = aggregate(f0.elapsed_time(f1), flops * e2e_steps)
    result["e2e"] = {"value": round(e2e_flops / (e2e_ms * 1e-3) / 1e12, 3), "unit": UNIT,
                     "h2d_bytes_per_step": int(hA[0].numel() * 2 + hB[0].numel() * 2),
                     "d2h_bytes_per_step": int(hC[0].numel() * hC[0].element_size()), "steps": e2e_steps,
                     "ms_per_step": round(e2e_ms / e2e_steps, 4),
                     "api": "gemm_bf16_host_batch (host operands; copies overlapped with the products)",
                     "copy_floor": host_link_floor(hA[0], hB[0], hC[0], torch.empty_like(hA[0], device="cuda"),
                                                   torch.empty_like(hB[0], device="cuda"),
                                                   torch.empty_like(hC[0], device="cuda"))}

    if cpu_baseline and rank == 0 and world == 1:
        result["cpu_baseline"] = cpu_oracle_baseline(A_h, Bt_h, M, N, K, target_s=args.cpu_seconds)
    return result, rank


def host_link_floor(hA, hB, hC, dA, dB, dC, reps: int = 5) -> dict:
    """What the host link alone allows per step: the step's operand bytes
    host -> device and its C device -> host, each timed alone and both at once
    on two streams (plain pinned copies, no product).  An end-to-end step can
    be no faster than the concurrent figure."""
    import torch
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    main = torch.cuda.current_stream()

    def timed(do_in: bool, do_out: bool) -> float:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        for r in range(reps + 2):
            if r == 2:
                e0.record(main)
            start = torch.cuda.Event()
            start.record(main)
            for s, on in ((s_in, do_in), (s_out, do_out)):
                if not on:
                    continue
                s.wait_event(start)
                with torch.cuda.stream(s):
                    if s is s_in:
                        dA.copy_(hA, non_blocking=True)
                        dB.copy_(hB, non_blocking=True)
                    else:
                        hC.copy_(dC, non_blocking=True)
                done = torch.cuda.Event()
                done.record(s)
                main.wait_event(done)
        e1.record(main)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps

    bin_, bout = hA.numel() * 2 + hB.numel() * 2, hC.numel() * hC.element_size()
    t_in, t_out, t_both = timed(True, False), timed(False, True), timed(True, True)
    return {"h2d_gbs": round(bin_ / (t_in * 1e-3) / 1e9, 1), "d2h_gbs": round(bout / (t_out * 1e-3) / 1e9, 1),
            "ms_per_step_both_directions": round(t_both, 4)}


def sustained_region(seconds: float, ms_per_step: float, step, flops: float, peaks: dict, stream, nvml,
                     smi_id: str) -> dict:
    """The same step back to back for about ``seconds``: the rate the part
    sustains under its power cap, against the measured sustained bf16 peak,
    with the SM clock and clock-event reasons sampled inside the region
    (NVML every 2 ms, nvidia-smi every 100 ms).  ``cycles_per_step`` is the
    step time times the median SM clock, and ``tflops_at_max_clock`` the rate
    those cycles would give at the maximum clock."""
    import torch
    n = max(10, int(math.ceil(seconds * 1e3 / max(ms_per_step, 1e-3))))
    sampler = ClockSampler(smi_id)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    rows, stop = nvml.sample_in_background()
    t0 = time.time()
    e0.record(stream)
    for i in range(n):
        step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    stop()
    sampler.stop()
    ms = e0.elapsed_time(e1)
    value = flops * n / (ms * 1e-3) / 1e12
    peak = peaks["bf16_sustained"]
    clocks = clocks_summary(rows, sampler.summary(t0, t1))
    out = {"value": round(value, 3), "unit": UNIT, "steps": n, "seconds": round(ms * 1e-3, 3),
           "ms_per_step": round(ms / n, 6), "peak": peak,
           "peak_source": f"sustained bf16, {peaks['source']}", "frac": round(value / peak, 4), "clocks": clocks}
    mhz, mx = clocks.get("sm_mhz"), clocks.get("sm_max_mhz")
    if mhz and mx:
        out["cycles_per_step"] = round(ms / n * 1e-3 * mhz * 1e6)
        out["tflops_at_max_clock"] = round(value * mx / mhz, 3)
    return out


# ---- the oracle on the host cores ---------------------------------------------------------

def host_cpu() -> dict:
    """Host core count (os.cpu_count) and the CPU model from lscpu, when it runs."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.split(":")[0].strip() == "Model name":
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    return {"host_cores": os.cpu_count(), "cpu_model": model}


def _time_oracle_rows(A_h, Bt_h, M, N, K, target_s: float, threads: int):
    """(rows, seconds) of the oracle on the first rows of C, sized for about target_s."""
    import oracle
    r0 = min(M, 4 * max(threads, 1))
    t = time.perf_counter()
    oracle.gemm(A_h[:r0], Bt_h, r0, N, K, with_abs=False, threads=threads)
    dt0 = max(time.perf_counter() - t, 1e-3)
    rows = int(min(M, max(1, math.floor(r0 * target_s / dt0))))
    t = time.perf_counter()
    oracle.gemm(A_h[:rows], Bt_h, rows, N, K, with_abs=False, threads=threads)
    return rows, time.perf_counter() - t


def cpu_oracle_baseline(A_h, Bt_h, M, N, K, target_s: float):
    """Time the oracle, as it stands, on the first R rows of C (R x N outputs at
    the workload's K), R sized for about target_s seconds of CPU work with all
    of OpenMP's threads, and again on one thread for about a third of that."""
    import oracle
    oracle.build()
    cores = oracle.max_threads()
    oracle.gemm(A_h[:cores], Bt_h, cores, N, K, with_abs=False, threads=cores)   # start the thread pool
    rows, dt = _time_oracle_rows(A_h, Bt_h, M, N, K, target_s, cores)
    rows1, dt1 = _time_oracle_rows(A_h, Bt_h, M, N, K, target_s / 3.0, 1)
    return {"value": round(2.0 * rows * N * K / dt / 1e12, 6), "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"rows 0..{rows - 1} of C ({rows}x{N} outputs, K={K}), binary64 triple loop, "
                      f"{cores} OpenMP threads, {dt:.1f} s",
            "single_thread": {"value": round(2.0 * rows1 * N * K / dt1 / 1e12, 6), "unit": UNIT,
                              "sample": f"rows 0..{rows1 - 1} of C, one thread, {dt1:.1f} s"},
            **host_cpu()}


def oracle_table(one_thread_budget_s: float = 4.0):
    """The oracle alone on the host cores, for the correctness and square,
    neighbour and split-K workloads: every output of C with all of OpenMP's
    threads, and one thread on the first rows of C (all of them when that
    takes at most about 10 s; otherwise a row sample, scaled to the whole C and
    marked as such).  Yields one dict per workload."""
    import oracle
    oracle.build()
    cores = oracle.max_threads()
    names = ["square256", "square4096", "n4095", "n4097", "k4088", "n4104", "m3968", "splitk148"]
    for name in names:
        w = WORKLOADS[name]
        (A_h, Bt_h), seed = make_host_operands(w)
        M, N, K = w["M"], w["N"], w["K"]
        # the thread count is passed every time: the OpenMP runtime keeps the
        # last count it was given, and the one-thread timing below sets 1
        oracle.gemm(A_h[:min(M, cores)], Bt_h, min(M, cores), N, K, with_abs=False, threads=cores)   # pool up
        t = time.perf_counter()
        oracle.gemm(A_h, Bt_h, M, N, K, with_abs=False, threads=cores)
        dt_all = time.perf_counter() - t
        rows1, dt1 = _time_oracle_rows(A_h, Bt_h, M, N, K, one_thread_budget_s, 1)
        full1 = dt1 * M / rows1
        if rows1 < M and full1 <= 10.0:
            t = time.perf_counter()
            oracle.gemm(A_h, Bt_h, M, N, K, with_abs=False, threads=1)
            dt1, rows1 = time.perf_counter() - t, M
            full1 = dt1
        flops = 2.0 * M * N * K
        yield {"oracle_table": name, "workload": w["desc"], "M": M, "N": N, "K": K, "flops": flops,
               "all_threads": {"threads": cores, "seconds": round(dt_all, 3), "tflops": round(flops / dt_all / 1e12, 6),
                               "outputs": "all of C"},
               "one_thread": {"seconds": round(full1, 3), "tflops": round(flops / full1 / 1e12, 6),
                              "outputs": "all of C" if rows1 == M else
                              f"rows 0..{rows1 - 1} of C in {dt1:.1f} s, scaled to all {M} rows (extrapolated)"},
               "kind": "oracle", **host_cpu()}


def run_reference_conv(args, w: dict, oracle, cores: int):
    """The direct-convolution oracle on a bounded sample: one image, cut to a
    band of input rows sized so the whole run stays within a few minutes."""
    from dense_tensor_core_bf16_gb300 import inputs
    cv = w["conv"]
    seed = inputs.DEFAULT_SEED + 400
    x_h, w_h = conv_host_operands(cv, seed)
    conv_kw = dict(pad=cv["pad"], stride=cv["stride"], dil=cv["dil"])
    budget_s = min(3.0, 150.0 / max(1, args.steps + args.warmup))
    rows = min(cv["H"], cv["R"] + 1)
    t = time.perf_counter()
    oracle.conv2d(x_h[:1, :rows], w_h, with_abs=False, **conv_kw)
    dt0 = max(time.perf_counter() - t, 1e-4)
    rows = int(min(cv["H"], max(cv["R"], math.floor(rows * budget_s / dt0))))

    def sample(i):
        n = i % cv["N"]
        return oracle.conv2d(x_h[n:n + 1, :rows], w_h, with_abs=False, **conv_kw)[0]

    y = sample(0)
    flops = 2.0 * y.size * cv["R"] * cv["S"] * cv["C"]
    for i in range(args.warmup):
        sample(i)
    t = time.perf_counter()
    for i in range(args.steps):
        sample(i)
    dt = time.perf_counter() - t
    value = flops * args.steps / dt / 1e12
    desc = (f"each step: one image cut to its first {rows} input rows ({y.shape[1]}x{y.shape[2]} output pixels x "
            f"K={cv['K']}), direct binary64 convolution, {cores} OpenMP threads")
    return {
        "impl": "reference", "metric": CONV_METRIC,
        "value": round(value, 6), "unit": UNIT, "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt * 1e3 / args.steps, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": conv_data(seed),
        "config": conv_config(w),
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc},
        "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_reference(args, wname: str, w: dict):
    """The oracle as the reference arm: each step is a bounded row sample."""
    import oracle
    world, rank, _ = dist_env()
    if rank != 0:
        return None, rank
    oracle.build()
    cores = oracle.max_threads()
    if w.get("conv"):
        return run_reference_conv(args, w, oracle, cores), rank
    (A_h, Bt_h), seed = make_host_operands(w)
    M, N, K = w["M"], w["N"], w["K"]
    budget_s = min(3.0, 150.0 / max(1, args.steps + args.warmup))
    r0 = min(M, 2)
    t = time.perf_counter()
    oracle.gemm(A_h[:r0], Bt_h, r0, N, K, with_abs=False)
    dt0 = max(time.perf_counter() - t, 1e-4)
    rows = int(min(M, max(1, math.floor(r0 * budget_s / dt0))))
    for i in range(args.warmup):
        s = (i * rows) % max(1, M - rows + 1)
        oracle.gemm(A_h[s:s + rows], Bt_h, rows, N, K, with_abs=False)
    t = time.perf_counter()
    for i in range(args.steps):
        s = (i * rows) % max(1, M - rows + 1)
        oracle.gemm(A_h[s:s + rows], Bt_h, rows, N, K, with_abs=False)
    dt = time.perf_counter() - t
    value = 2.0 * rows * N * K * args.steps / dt / 1e12
    sample = (f"each step: {rows} rows of C ({rows}x{N} outputs, K={K}) of the workload, binary64 triple loop, "
              f"{cores} OpenMP threads")
    result = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3 / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": workload_data(w, seed),
        "config": workload_config(w),
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    return result, rank


def conv_host_operands(cv: dict, seed: int):
    """x (N H W C) and w (K R S C) bf16 bit patterns from the seeded generator."""
    from dense_tensor_core_bf16_gb300 import inputs
    N, H, W, C, K, R, S = (cv[k] for k in "N H W C K R S".split())
    x = inputs.matrix(N * H * W, C, dist="normal", seed=seed, stream=0).reshape(N, H, W, C)
    w = inputs.matrix(K, R * S * C, dist="normal", seed=seed, stream=1,
                      scale=1.0 / math.sqrt(R * S * C)).reshape(K, R, S, C)
    return x, w


def run_gpu_conv(args, wname: str, w: dict):
    """A convolution workload: the same contract as run_gpu (W warm-ups, K
    steps back to back between events, barrier, max over ranks, clocks,
    roofline, end to end with host copies)."""
    import numpy as np
    import torch
    import dense_tensor_core_bf16_gb300 as g
    from dense_tensor_core_bf16_gb300 import inputs

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    cv = w["conv"]
    seed = inputs.DEFAULT_SEED + 400
    x_h, w_h = conv_host_operands(cv, seed)
    desc = g.gemm_conv2d_desc_t(N=cv["N"], H=cv["H"], W=cv["W"], C=cv["C"], K=cv["K"], R=cv["R"], S=cv["S"],
                                pad_h=cv["pad"][0], pad_w=cv["pad"][1], stride_h=cv["stride"][0],
                                stride_w=cv["stride"][1], dil_h=cv["dil"][0], dil_w=cv["dil"][1])
    st, P, Q = g.gemm_conv2d_out_dims(desc)
    if st:
        raise g.GemmError(st, "gemm_conv2d_out_dims")
    out_dtype = torch.bfloat16 if w["out"] == "bf16" else torch.float32
    odt = g.GEMM_OUT_BF16 if w["out"] == "bf16" else g.GEMM_OUT_F32
    opts = g.options(kernel_variant=args.variant, no_stream_k=int(args.no_stream_k))
    st, plan = g.gemm_conv2d_plan(desc, odt, opts)
    if st:
        raise g.GemmError(st, "gemm_conv2d_plan")
    if plan.workspace_bytes:
        g.gemm_reserve_workspace(plan.workspace_bytes)
    kw = dict(pad=cv["pad"], stride=cv["stride"], dil=cv["dil"], kernel_variant=args.variant,
              no_stream_k=args.no_stream_k)

    props = torch.cuda.get_device_properties(local)
    l2 = getattr(props, "L2_cache_size", 135_528_448) or 135_528_448
    esize = 2 if w["out"] == "bf16" else 4
    set_bytes = x_h.nbytes + w_h.nbytes + esize * cv["N"] * P * Q * cv["K"]
    copies = max(2, math.ceil(2 * l2 / set_bytes) + 1)
    x0 = torch.from_numpy(x_h.view(np.int16)).cuda().view(torch.bfloat16)
    w0 = torch.from_numpy(w_h.view(np.int16)).cuda().view(torch.bfloat16)
    sets = []
    for i in range(copies):
        sets.append((x0 if i == 0 else x0.clone(), w0 if i == 0 else w0.clone(),
                     torch.zeros((cv["N"], P, Q, cv["K"]), dtype=out_dtype, device="cuda")))

    def step(i):
        xx, ww, yy = sets[i % copies]
        g.conv2d(xx, ww, out=yy, **kw)

    gpu_id = getattr(props, "uuid", None)
    sampler = ClockSampler(f"GPU-{gpu_id}" if gpu_id is not None else str(local))
    nvml = NvmlPoller(f"GPU-{gpu_id}" if gpu_id is not None else None)
    time.sleep(0.3)   # before the warm-up: no idle gap before the timed region
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    st, where = g.gemm_get_device_status(None)
    if st:
        raise RuntimeError(f"device fault during warm-up: {where:#x}")
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    e0.record(stream)
    for i in range(args.steps):
        step(i)
    e1.record(stream)
    nvml_rows = nvml.poll_until(e1)
    torch.cuda.synchronize()
    barrier()
    t_wall1 = time.time()
    time.sleep(0.25)
    sampler.stop()
    st, where = g.gemm_get_device_status(None)
    if st:
        raise RuntimeError(f"device fault in the timed region: {where:#x}")
    total_ms = e0.elapsed_time(e1)
    flops = 2.0 * cv["N"] * P * Q * cv["K"] * cv["R"] * cv["S"] * cv["C"]
    max_ms, total_flops = aggregate(total_ms, flops * args.steps)
    value = total_flops / (max_ms * 1e-3) / 1e12
    peaks = load_peaks()
    long_region = (t_wall1 - t_wall0) > 1.0
    peak = peaks["bf16_sustained"] if long_region else peaks["bf16_burst"]
    peak_kind = ("sustained" if long_region else "burst") + f" bf16, {peaks['source']}"
    mean_ms = total_ms / args.steps
    achieved = flops / (mean_ms * 1e-3) / 1e12
    result = {
        "metric": CONV_METRIC,
        "value": round(value, 3), "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(max_ms / args.steps, 6), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16",
        "data": conv_data(seed),
        "config": conv_config(w),
        "plan": {
            "kernel_variant": g.KERNEL_VARIANTS[plan.kernel_variant], "cluster_size": plan.cluster_size,
            "tile": f"{plan.tile_m}x{plan.tile_n}x{plan.tile_k}", "split_k": plan.split_k,
            "stream_k_tiles": plan.stream_k_tiles, "pct_of_peak": round(100.0 * value / world / peak, 2),
            "peak_tflops": peak, "peak_kind": peak_kind,
            "l2_sets": f"{copies} rotating sets of {set_bytes / 1e6:.1f} MB vs L2 {l2 / 1e6:.1f} MB",
        },
        "roofline": {
            "kernel": f"{KERNEL_NAME}<{plan.cluster_size},{plan.tile_n}> (im2col A)",
            **roofline_entry(flops, float(set_bytes), mean_ms, peaks, peak, peak_kind),
            "traffic": recorded_traffic(wname), "mean_launch_ms": round(mean_ms, 6),
            "launch_time_from": "timed region / steps, launches back to back",
        },
        "gpu_launches": (1 + (1 if plan.split_k > 1 else 0)) * args.steps,
        "clocks": clocks_summary(nvml_rows, sampler.summary(t_wall0, t_wall1)),
    }
    if args.no_e2e:
        return result, rank
    e2e_steps = min(args.steps, 20)
    hx = torch.from_numpy(x_h.view(np.int16)).view(torch.bfloat16).pin_memory()
    hw = torch.from_numpy(w_h.view(np.int16)).view(torch.bfloat16).pin_memory()
    yy = sets[0][2]
    hy = torch.empty(tuple(yy.shape), dtype=out_dtype).pin_memory()
    for _ in range(2):
        x0.copy_(hx, non_blocking=True)
        w0.copy_(hw, non_blocking=True)
        g.conv2d(x0, w0, out=yy, **kw)
        hy.copy_(yy, non_blocking=True)
    torch.cuda.synchronize()
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    f0.record(stream)
    for _ in range(e2e_steps):
        x0.copy_(hx, non_blocking=True)
        w0.copy_(hw, non_blocking=True)
        g.conv2d(x0, w0, out=yy, **kw)
        hy.copy_(yy, non_blocking=True)
    f1.record(stream)
    torch.cuda.synchronize()
    e2e_ms, e2e_flops = aggregate(f0.elapsed_time(f1), flops * e2e_steps)
    result["e2e"] = {"value": round(e2e_flops / (e2e_ms * 1e-3) / 1e12, 3), "unit": UNIT,
                     "h2d_bytes_per_step": int(hx.numel() * 2 + hw.numel() * 2),
                     "d2h_bytes_per_step": int(hy.numel() * hy.element_size()), "steps": e2e_steps}
    return result, rank


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default=DEFAULT_WORKLOAD)
    # an ad-hoc GEMM, flags as a library profiler takes them (all of --m --n --k, or none)
    ap.add_argument("--m", type=int)
    ap.add_argument("--n", type=int)
    ap.add_argument("--k", type=int)
    ap.add_argument("--A", choices=["row", "col"], default="row", help="layout of A (with --m --n --k)")
    ap.add_argument("--B", choices=["row", "col"], default="col", help="layout of B (with --m --n --k)")
    ap.add_argument("--C", choices=["bf16", "f32"], default="bf16", help="type of C (with --m --n --k)")
    ap.add_argument("--split-k", type=int, default=0, help="0: the plan chooses (with --m --n --k)")
    ap.add_argument("--persistent", type=int, choices=[0, 1], default=1, help="0: one cluster per tile")
    ap.add_argument("--dist", choices=["normal", "uniform", "int4"], default="normal",
                    help="input values (with --m --n --k): N(0,1)/sqrt(K), uniform[-1,1)/sqrt(K) or integers")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--sustained-seconds", type=float, default=None,
                    help="seconds of back-to-back steps after the timed region (default 4; 0: none)")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end (host buffers) measurement")
    ap.add_argument("--oracle-table", action="store_true",
                    help="time the oracle alone on the host cores (configs 1-4 in full, all threads, and a "
                         "one-thread sample); one JSON line per configuration")
    ap.add_argument("--no-stream-k", action="store_true", help="never spread a tail of tiles over the clusters")
    ap.add_argument("--raster-group", type=int, default=0,
                    help="m-tiles per raster group of the tile order (0: the library's default)")
    ap.add_argument("--variant", type=int, default=0, choices=[0, 1, 2, 3, 4],
                    help="kernel variant: 0 auto, 1 one-SM 128x256, 2 two-SM 256x256, 3 two-SM 256x128, "
                         "4 one-SM 128x128")
    ap.add_argument("--all-workloads", action="store_true",
                    help="run every workload (one JSON line each, no CPU baseline)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    shape = (args.m, args.n, args.k)
    if any(v is not None for v in shape):
        if any(v is None or v < 1 for v in shape):
            ap.error("--m, --n and --k go together, each at least 1")
        name = f"custom_{args.m}x{args.n}x{args.k}"
        WORKLOADS[name] = custom_workload(args.m, args.n, args.k, args.A, args.B, args.C, args.split_k,
                                          args.persistent, args.dist)
        args.workload = name
    if args.sustained_seconds is None:
        args.sustained_seconds = 0.0 if args.all_workloads else 4.0
    if args.oracle_table:
        for line in oracle_table():
            print(json.dumps(line), flush=True)
        return 0

    world, rank, local = dist_env()
    if args.impl == "reference":
        res, rank = run_reference(args, args.workload, WORKLOADS[args.workload])
        if rank == 0 and res is not None:
            print(json.dumps(res), flush=True)
        return 0

    import torch
    import torch.distributed as dist
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    try:
        names = sorted(WORKLOADS) if args.all_workloads else [args.workload]
        for name in names:
            if WORKLOADS[name].get("conv"):
                res, rank = run_gpu_conv(args, name, WORKLOADS[name])
            else:
                res, rank = run_gpu(args, name, WORKLOADS[name],
                                    cpu_baseline=not args.no_cpu_baseline and not args.all_workloads)
            if rank == 0:
                if args.all_workloads:
                    res["config"]["name"] = name
                print(json.dumps(res), flush=True)
    finally:
        if world > 1 and dist.is_initialized():
            dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
