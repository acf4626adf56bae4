#!/usr/bin/env python3
"""Benchmark of the decode GEMV: achieved HBM GB/s, fraction of GB300 peak and
microseconds per call, printed as one JSON line.

A step is one call of the hot path on one batch of synthetic input: for the
default workload, y = W·x for the down projection of a Llama-3.1-8B-shaped
layer (W 4,096 x 14,336 BF16, x 14,336 BF16, batch 1) through gemv_bf16. The
weights rotate over enough copies that together exceed the L2 cache, so every
step streams W from HBM ("Decode GEMV at half of HBM bandwidth", "Common
mistakes": a matrix that sits in L2 reports more than the HBM can deliver).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...   # the CPU oracle, timed as the baseline arm

Under torchrun each rank runs its own replica (weak scaling); the time is the
maximum over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

FALLBACK_HBM_GBS = 6800.0
VENDOR_HBM_GBS = 8000.0
METRIC = "achieved HBM GB/s and % of GB300 peak for BF16 decode GEMV (batch 1), µs/call"
UNIT = "GB/s"


# ----------------------------------------------------------------------------- helpers

def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=500)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="down_proj",
                    help="down_proj | k_proj | qkv | gate_up | o_proj | lm_head | decode_step | "
                         "skinny:<N>x<K>:B<b> | tail:<N>x<K>")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-probe", action="store_true",
                    help="skip the read-only ceiling probe (keeps device memory small)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    return ap.parse_args(argv)


def load_peaks() -> tuple[float, str]:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            peaks = json.load(f)
        return float(peaks["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


KERNEL_FILES = {   # the sources that make up each kernel family's launches
    "fma": ("gemv_internal.h", "gemv_common.cuh", "gemv_kernel.cuh", "gemv_fma_instances.cu",
            "gemv_dispatch.cu"),
    "mma": ("gemv_internal.h", "gemv_common.cuh", "gemv_mma_kernel.cuh", "gemv_mma_instances_nb1.cu",
            "gemv_mma_instances_nb2.cu", "gemv_dispatch.cu"),
    "w4": ("gemv_internal.h", "gemv_common.cuh", "gemv_mma_kernel.cuh", "gemv_w4_kernel.cuh",
           "gemv_w4_instances.cu", "gemv_dispatch.cu"),
    "f8": ("gemv_internal.h", "gemv_common.cuh", "gemv_mma_kernel.cuh", "gemv_fp8_kernel.cuh",
           "gemv_fp8_instances.cu", "gemv_dispatch.cu"),
    "sk": ("gemv_internal.h", "gemv_common.cuh", "gemv_kernel.cuh", "gemv_streamk_kernel.cuh",
           "gemv_streamk_instances.cu", "gemv_dispatch.cu"),
}


def kernel_source_hash(family: str, launch: dict | None = None) -> str:
    """Hash of one kernel family's sources and of the launch configuration the
    planner picks for the workload (grid, splits, K slices, chunks): together
    they decide the bytes a launch moves. Without a launch configuration (fused
    and multi-launch workloads) the planner's source stands in for it."""
    csrc = os.path.join(ROOT, "memory_bound_decode_gb300", "csrc")
    h = hashlib.sha256()
    names = KERNEL_FILES[family] + (() if launch else ("planner.cpp",))
    for name in names:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    if launch:
        h.update(json.dumps(launch, sort_keys=True).encode())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str, src_hash: str):
    """DRAM bytes per launch of the dominant kernel from the committed ncu
    summary for this workload, if it was taken on the current kernel source."""
    safe = re.sub(r"[^A-Za-z0-9_]+", "_", workload)
    path = os.path.join(ROOT, "profiles", f"gemv_{safe}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    m_hash = re.search(r"kernel_source_hash:\s*([0-9a-f]+)", text)
    m_bytes = re.search(r"dram_bytes_per_launch:\s*([0-9_,]+)", text)
    if not m_hash or not m_bytes or m_hash.group(1) != src_hash:
        return None
    return int(m_bytes.group(1).replace(",", "").replace("_", ""))


class ClockSampler:
    """nvidia-smi clock and throttle-reason samples while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 20):
        self.gpu_index = gpu_index
        self.period_ms = period_ms
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", f"-lms={self.period_ms}"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(self.period_ms / 1000.0 * 2)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = [r.split(",") for r in self.file.read().strip().splitlines() if r.strip()]
        self.file.close()
        os.unlink(self.file.name)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [c.strip() for c in r]
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except ValueError:
                continue
            for name, val in zip(names, r[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        # the samples under load are the ones above idle clocks
        loaded = [c for c in sm if c >= 0.5 * max(sm)] if sm else []
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- workloads

RMS_EPS = 1e-5
RMS_SUFFIX = "+rmsnorm"


def split_norm(workload: str) -> tuple[str, float | None]:
    """A workload name may end in "+rmsnorm": the same projections with the
    RMSNorm prologue on x (eps 1e-5)."""
    if workload.endswith(RMS_SUFFIX):
        return workload[: -len(RMS_SUFFIX)], RMS_EPS
    return workload, None


W4_PREFIX = "w4:"


def split_w4(workload: str) -> tuple[str, bool]:
    """A workload name may start with "w4:": the same shapes with group-quantised
    INT4 weights (128-column groups, BF16 scales)."""
    if workload.startswith(W4_PREFIX):
        return workload[len(W4_PREFIX):], True
    return workload, False


SK_PREFIX = "sk:"
F8_PREFIX = "f8:"
CC_PREFIX = "cc:"


def split_cc(workload: str) -> tuple[str, bool]:
    """A workload name may start with "cc:": the same BF16 projections on the
    CUDA-core kernel at every batch size (GEMV_FLAG_CUDA_CORES)."""
    if workload.startswith(CC_PREFIX):
        return workload[len(CC_PREFIX):], True
    return workload, False



def split_f8(workload: str) -> tuple[str, bool]:
    """A workload name may start with "f8:": the same shapes with FP8 (E4M3)
    weights and FP32 row scales."""
    if workload.startswith(F8_PREFIX):
        return workload[len(F8_PREFIX):], True
    return workload, False



def split_sk(workload: str) -> tuple[str, bool]:
    """A workload name may start with "sk:": the same BF16 batch-1 projections
    through the stream-K kernel (GEMV_FLAG_STREAMK)."""
    if workload.startswith(SK_PREFIX):
        return workload[len(SK_PREFIX):], True
    return workload, False


def describe(workload: str):
    """(kind, N-list, K, B) of a named workload."""
    from memory_bound_decode_gb300 import workloads as wl
    workload, _ = split_norm(workload)
    workload, _ = split_sk(workload)
    workload, _ = split_cc(workload)
    workload, _ = split_f8(workload)
    workload, _ = split_w4(workload)
    if workload in ("down_proj", "k_proj", "o_proj", "lm_head"):
        N, K = wl.SHAPES[workload]
        return "single", [N], K, 1
    if workload == "qkv":
        return "fused", [4096, 1024, 1024], 4096, 1
    if workload == "gate_up":
        return "fused", [14336, 14336], 4096, 1
    if workload == "decode_step":
        return "step", None, None, 1
    m = re.fullmatch(r"skinny:(\d+)x(\d+):B(\d+)", workload)
    if m:
        return "single", [int(m.group(1))], int(m.group(2)), int(m.group(3))
    m = re.fullmatch(r"tail:(\d+)x(\d+)", workload)
    if m:
        return "single", [int(m.group(1))], int(m.group(2)), 1
    raise SystemExit(f"unknown workload {workload}")


class GemvWorkload:
    """Rotating device-resident weight copies for one (possibly fused) GEMV."""

    def __init__(self, kind, rows, K, B, device, l2_bytes, rms_eps=None, w4=False, streamk=False, fp8=False,
                 cuda_cores=False):
        import torch
        from memory_bound_decode_gb300 import inputs, roofline
        self.kind, self.rows, self.K, self.B = kind, rows, K, B
        self.rms_eps = rms_eps
        self.w4 = w4
        self.streamk = streamk
        self.fp8 = fp8
        self.cuda_cores = cuda_cores
        if cuda_cores and (w4 or fp8 or streamk):
            raise SystemExit("cc: BF16 workloads only")
        if streamk and (w4 or fp8 or B != 1):
            raise SystemExit("stream-K: BF16 batch-1 workloads only")
        if fp8 and kind != "single":
            raise SystemExit("FP8 weights: single-matrix workloads only")
        self.N = sum(rows)
        if w4:
            if kind != "single":
                raise SystemExit("INT4 weights: single-matrix workloads only")
            self.ldq = (K // 2 + 15) // 16 * 16
            self.lds = K // inputs.W4_GROUP
            self.bytes_per_step = roofline.algorithmic_bytes_w4(self.N, K, B)
            wbytes = self.N * (self.ldq + 2 * self.lds)
        elif fp8:
            self.ldq = (K + 15) // 16 * 16
            self.bytes_per_step = roofline.algorithmic_bytes_fp8(self.N, K, B)
            wbytes = self.N * (self.ldq + 4)
        else:
            self.ldw = inputs.padded_ldw(K)
            self.bytes_per_step = roofline.algorithmic_bytes(self.N, K, B)
            wbytes = 2 * self.N * self.ldw
        self.copies = max(1, min(64, math.ceil(3 * l2_bytes / wbytes)))
        if fp8:
            self.Ws = [[inputs.fp8_weight(self.N, K, self.ldq, seed=0, index=10 * c, device=device)]
                       for c in range(self.copies)]
        elif w4:
            self.Ws = [[inputs.w4_weight_device(self.N, K, self.ldq, self.lds, seed=0, index=10 * c,
                                                device=device)] for c in range(self.copies)]
        else:
            self.Ws = [[inputs.weight(n, K, self.ldw, seed=0, index=10 * c + i, device=device)
                        for i, n in enumerate(rows)] for c in range(self.copies)]
        self.x = inputs.activations(B, K, seed=0, index=1000, device=device)
        self.ys = [torch.empty((B, n), dtype=torch.float32, device=device) for n in rows]
        self.launches_per_step = 1
        self.rotating_bytes = wbytes * self.copies

    def step(self, i: int, stream, x=None) -> None:
        from memory_bound_decode_gb300 import binding
        Ws = self.Ws[i % self.copies]
        x = self.x if x is None else x
        if self.fp8:
            Wq, S = Ws[0]
            binding.gemv_fp8_bf16(Wq, S, x, self.ys[0], self.N, self.K, self.B, self.ldq,
                                  rms_eps=self.rms_eps, stream=stream)
        elif self.w4:
            Wq, S = Ws[0]
            binding.gemv_w4_bf16(Wq, S, x, self.ys[0], self.N, self.K, self.B, self.ldq, self.lds,
                                 rms_eps=self.rms_eps, stream=stream)
        elif self.kind == "single" and self.rms_eps is None and not self.streamk and not self.cuda_cores:
            binding.gemv_bf16(Ws[0], x, self.ys[0], self.N, self.K, self.B, self.ldw, stream)
        elif self.kind == "single":
            binding.gemv_bf16_ex(Ws[0], x, self.ys[0], self.N, self.K, self.B, self.ldw,
                                 rms_eps=self.rms_eps, stream=stream, streamk=self.streamk,
                                 cuda_cores=self.cuda_cores)
        elif self.rms_eps is None and not self.streamk and not self.cuda_cores:
            binding.gemv_bf16_multi([(W, y, n, self.ldw) for W, y, n in zip(Ws, self.ys, self.rows)],
                                    x, self.K, self.B, stream)
        else:
            binding.gemv_bf16_multi_ex([(W, y, n, self.ldw) for W, y, n in zip(Ws, self.ys, self.rows)],
                                       x, self.K, self.B, rms_eps=self.rms_eps, stream=stream,
                                       streamk=self.streamk, cuda_cores=self.cuda_cores)

    def config(self) -> dict:
        shape = "+".join(str(n) for n in self.rows)
        norm = f", RMSNorm prologue eps={self.rms_eps}" if self.rms_eps is not None else ""
        wt = ("INT4-weight (128-col groups, BF16 scales)" if self.w4 else
              "FP8-weight (E4M3, FP32 row scales)" if self.fp8 else "BF16")
        sk = (", stream-K one-wave grid" if self.streamk else
              ", CUDA-core kernel" if self.cuda_cores else "")
        return {"workload": f"{self.kind} {wt} GEMV N={shape} K={self.K} B={self.B}{norm}{sk}",
                "N": self.N, "K": self.K, "B": self.B,
                "ldw": self.ldq if (self.w4 or self.fp8) else self.ldw,
                "segments": len(self.rows),
                "l2": f"inputs larger than L2: {self.copies} rotating weight copies, "
                      f"{self.rotating_bytes / 1e6:.0f} MB"}


class StepWorkload:
    """The full decode-step projection set replayed as one CUDA graph."""

    def __init__(self, device, stream, rms_eps=None, streamk=False, weights="bf16"):
        from memory_bound_decode_gb300 import workloads as wl
        self.spec = wl.decode_step_spec()
        self.weights = weights
        self.data = wl.DecodeStep(self.spec, seed=0, device=device, weights=weights)
        self.rms_eps = rms_eps
        self.streamk = streamk
        self.w4, self.fp8 = weights == "int4", weights == "fp8"
        self.plan = self.data.plan(rms_eps=rms_eps, streamk=streamk)
        self.plan.capture(stream)
        self.bytes_per_step = (wl.step_bytes_formula(self.spec) if weights == "bf16"
                               else self.data.algorithmic_bytes())
        self.launches_per_step = self.plan.num_launches()
        self.x = None
        self.B = 1

    def step(self, i: int, stream, x=None) -> None:
        self.plan.launch(stream)

    def config(self) -> dict:
        norm = (f"; RMSNorm prologue (eps={self.rms_eps}) on QKV, gate_up and lm_head"
                if self.rms_eps is not None else "")
        wt = {"bf16": "BF16", "fp8": "FP8 (E4M3, FP32 row scales)",
              "int4": "INT4 (128-col groups, BF16 scales)"}[self.weights]
        return {"workload": "decode step: 32 x {QKV 6144x4096, o 4096x4096, gate_up 28672x4096, "
                            f"down 4096x14336}} + lm_head 128256x4096, {wt} weights, batch 1, one CUDA graph" + norm,
                "launches_per_step": self.launches_per_step,
                "l2": f"inputs larger than L2: {self.data.weight_bytes() / 1e9:.2f} GB of weights per step"}


# ----------------------------------------------------------------------------- our arm

def max_over_ranks(value: float, dist, device) -> float:
    """The largest value any rank holds (all ranks get it)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def read_ceiling_gbs(torch, binding, stream) -> float:
    """Best of 10 read-only streams of a 4 GiB buffer with the GEMV's loads."""
    nbytes = 4 << 30
    buf = torch.empty(nbytes // 2, dtype=torch.int16, device="cuda")
    buf.fill_(1)
    sink = torch.empty(binding.gemv_probe_sink_words(), device="cuda")
    best = float("inf")
    for _ in range(12):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        binding.gemv_probe_stream_read(buf, nbytes, sink, stream)
        b.record(stream)
        b.synchronize()
        best = min(best, a.elapsed_time(b) / 1e3)
    del buf
    return nbytes / best / 1e9


def run_ours(args, rank: int, world: int, dist) -> dict | None:
    import torch
    from memory_bound_decode_gb300 import binding, build_lib

    build_lib.build()
    binding.lib()
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    props = torch.cuda.get_device_properties(device)
    l2 = getattr(props, "L2_cache_size", 126 << 20)

    kind, rows, K, B = describe(args.workload)
    _, rms_eps = split_norm(args.workload)
    base, streamk = split_sk(split_norm(args.workload)[0])
    base, cuda_cores = split_cc(base)
    base, fp8 = split_f8(base)
    _, w4 = split_w4(base)
    wk = StepWorkload(device, torch.cuda.Stream(), rms_eps, streamk,
                      "int4" if w4 else "fp8" if fp8 else "bf16") if kind == "step" else \
        GemvWorkload(kind, rows, K, B, device, l2, rms_eps, w4, streamk, fp8, cuda_cores)
    torch.cuda.synchronize()

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    for i in range(max(3, args.warmup)):
        wk.step(i, stream)
    torch.cuda.synchronize()

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.05)
    barrier()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for i in range(args.steps):
        wk.step(i, stream)
    ev1.record(stream)
    barrier()
    clock_info = clocks.stop()
    seconds = max_over_ranks(ev0.elapsed_time(ev1) / 1e3, dist, device)

    steps = args.steps
    total_bytes = wk.bytes_per_step * steps * world
    value = total_bytes / seconds / 1e9
    per_launch_s = seconds / (steps * wk.launches_per_step)

    # end to end through the public call: pinned host x in, GEMV, host y out,
    # synchronized, every step (gemv_bf16_host_io for single BF16 matrices)
    e2e = None
    if not args.no_e2e and kind != "step":
        x_host = wk.x.cpu().pin_memory()
        y_host = [torch.empty(y.shape, dtype=y.dtype).pin_memory() for y in wk.ys]
        x_dev = torch.empty_like(wk.x)
        e2e_steps = max(10, min(steps, 2000))
        host_io = kind == "single" and not getattr(wk, "w4", False) and not getattr(wk, "fp8", False)
        sk = getattr(wk, "streamk", False)
        sh = stream.cuda_stream

        def e2e_step(i):
            if host_io:
                binding.gemv_bf16_host_io(wk.Ws[i % wk.copies][0], x_host, y_host[0], x_dev, wk.ys[0],
                                          wk.N, wk.K, wk.B, wk.ldw, rms_eps=wk.rms_eps, stream=sh,
                                          streamk=sk, cuda_cores=getattr(wk, "cuda_cores", False))
            else:
                x_dev.copy_(x_host, non_blocking=True)
                wk.step(i, stream, x_dev)
                for yh, yd in zip(y_host, wk.ys):
                    yh.copy_(yd, non_blocking=True)
                stream.synchronize()

        for i in range(5):
            e2e_step(i)
        barrier()
        t0 = time.perf_counter()
        for i in range(e2e_steps):
            e2e_step(i)
        e2e_s = max_over_ranks(time.perf_counter() - t0, dist, device)
        e2e = {"value": round(wk.bytes_per_step * e2e_steps * world / e2e_s / 1e9, 2), "unit": UNIT,
               "h2d_bytes_per_step": int(x_host.numel() * x_host.element_size()),
               "d2h_bytes_per_step": int(sum(y.numel() * y.element_size() for y in y_host)),
               "us_per_step": round(e2e_s / e2e_steps * 1e6, 3), "steps": e2e_steps}

    read_ceiling = None
    if rank == 0 and not args.no_probe:
        read_ceiling = read_ceiling_gbs(torch, binding, stream)

    if rank != 0:
        return None
    peak, peak_kind = load_peaks()
    achieved = wk.bytes_per_step / (seconds / steps) / 1e9 if kind == "step" else \
        wk.bytes_per_step / per_launch_s / 1e9
    family = ("w4" if getattr(wk, "w4", False) else "f8" if getattr(wk, "fp8", False)
              else "sk" if getattr(wk, "streamk", False)
              else "fma" if (wk.B == 1 or getattr(wk, "cuda_cores", False)) else "mma")
    launch = None
    if kind == "single":
        sms = torch.cuda.get_device_properties(device).multi_processor_count
        if family == "w4":
            launch = binding.gemv_w4_query_launch(wk.N, wk.K, wk.B, sms)
        elif family == "f8":
            launch = binding.gemv_fp8_query_launch(wk.N, wk.K, wk.B, sms)
        else:
            launch = binding.gemv_query_launch_ex(
                wk.N, wk.K, wk.B, sms,
                binding.GEMV_FLAG_STREAMK if family == "sk" else
                binding.GEMV_FLAG_CUDA_CORES if getattr(wk, "cuda_cores", False) else 0)
    src_hash = kernel_source_hash(family, launch)
    traffic = profiled_traffic(args.workload, src_hash)
    result = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": steps, "warmup": max(3, args.warmup),
        "ms_per_step": round(seconds / steps * 1e3, 6),
        "us_per_call": round(per_launch_s * 1e6, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": {"w4": "u4 weights (bf16 group scales), bf16 x, fp32 accumulate",
                  "f8": "e4m3 weights (fp32 row scales), bf16 x, fp32 accumulate"}.get(family, "bf16 in, fp32 accumulate"),
        "data": "synthetic (seeded N(0,0.02^2) weights, N(0,1) x)",
        "config": dict(wk.config(), parallelism=f"replicas x{world}" if world > 1 else "1 GPU",
                       pdl=os.environ.get("GEMV_PDL", "1") != "0"),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": UNIT,
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "peak_kind": f"{peak_kind} copy (MEASURED_PEAKS hbm_gbs, burst)"
                     if peak_kind == "measured" else "fallback 6.8 TB/s",
                     "kernel": ("gemv_w4_kernel (INT4 codes, BF16 tensor cores)" if family == "w4"
                                else "gemv_fp8_kernel (E4M3 codes, BF16 tensor cores)" if family == "f8"
                                else "gemv_streamk_kernel (CUDA cores, one-wave grid)" if family == "sk"
                                else "gemv_bf16_kernel (CUDA cores)" if wk.B == 1
                                else "gemv_bf16_mma_kernel (BF16 tensor cores)"),
                     "kernel_source_hash": src_hash},
        "ceilings": {"copy_gbs": peak,
                     "read_probe_gbs": round(read_ceiling, 1) if read_ceiling else None,
                     "vendor_gbs": VENDOR_HBM_GBS,
                     "frac_of_read_probe": round(achieved / read_ceiling, 4) if read_ceiling else None,
                     "frac_of_vendor": round(achieved / VENDOR_HBM_GBS, 4)},
        "gpu_launches": steps * wk.launches_per_step,
        "clocks": clock_info,
    }
    if e2e is not None:
        result["e2e"] = e2e
    return result


# ----------------------------------------------------------------------------- CPU oracle arms

def oracle_sample(workload: str, rows_cap: int | None = None):
    """Host inputs for the oracle: the workload's shape, generated on the CPU
    with the same recipe, optionally restricted to the first rows_cap rows."""
    from memory_bound_decode_gb300 import inputs, roofline
    kind, rows, K, B = describe(workload)
    if kind == "step":
        rows, K, B = [4096], 14336, 1      # the step's down projection stands in
    N = sum(rows)
    n = N if rows_cap is None else max(1, min(N, rows_cap))
    ldw = inputs.padded_ldw(K)
    W = inputs.bits(inputs.weight(n, K, ldw, seed=0, index=0))
    x = inputs.bits(inputs.activations(B, K, seed=0, index=1))
    return W, x, K, B, n, N, roofline.algorithmic_bytes(n, K, B)


def cpu_baseline(workload: str, seconds: float) -> dict:
    from oracle import oracle
    threads = oracle.default_threads()
    W, x, K, B, n, N, nbytes = oracle_sample(workload)
    lib = oracle.load()
    passes = 0
    t0 = time.perf_counter()
    while True:
        lib.gemv(W, x, K, threads=threads)
        passes += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    result = {"value": round(nbytes * passes / el / 1e9, 4), "unit": UNIT, "cores": threads,
              "kind": "oracle",
              "sample": f"{passes} full passes of the FP64 oracle over {n}x{K} (B={B}) in {el:.1f} s"}
    # the same oracle on one core, on a row sample of about a tenth of the time
    rows = max(1, min(N, int(n * (seconds / 10.0) / max(el / passes * threads, 1e-9))))
    W1, x1, K1, B1, n1, _, nbytes1 = oracle_sample(workload, rows_cap=rows)
    passes1 = 0
    t0 = time.perf_counter()
    while True:
        lib.gemv(W1, x1, K1, threads=1)
        passes1 += 1
        el1 = time.perf_counter() - t0
        if el1 >= seconds / 10.0:
            break
    result["single_thread"] = {"value": round(nbytes1 * passes1 / el1 / 1e9, 4), "unit": UNIT, "cores": 1,
                               "sample": f"{passes1} passes over {n1} of {N} rows x K={K1} (B={B1}) in {el1:.1f} s"}
    return result


def run_reference(args, rank: int) -> dict | None:
    if rank != 0:
        return None
    from oracle import oracle
    threads = oracle.default_threads()
    lib = oracle.load()
    # calibrate, then size each step so the whole run stays within ~2 minutes
    W, x, K, B, n, N, _ = oracle_sample(args.workload, rows_cap=64)
    t0 = time.perf_counter()
    lib.gemv(W, x, K, threads=threads)
    per_row = (time.perf_counter() - t0) / n
    total_steps = args.steps + max(3, args.warmup)
    rows_cap = max(1, min(N, int(120.0 / total_steps / max(per_row, 1e-9))))
    W, x, K, B, n, N, nbytes = oracle_sample(args.workload, rows_cap=rows_cap)
    for _ in range(max(3, args.warmup)):
        lib.gemv(W, x, K, threads=threads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        lib.gemv(W, x, K, threads=threads)
    el = time.perf_counter() - t0
    value = nbytes * args.steps / el / 1e9
    kind, rows, K_, B_ = describe(args.workload)
    sample = f"each step: FP64 oracle over {n} of {N} rows x K={K} (B={B}), {threads} threads"
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
        "n_gpus": 1, "steps": args.steps, "warmup": max(3, args.warmup),
        "ms_per_step": round(el / args.steps * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,0.02^2) weights, N(0,1) x)",
        "config": {"workload": f"{kind} BF16 GEMV N={N} K={K} B={B} (CPU oracle, row sample)",
                   "N": N, "K": K, "B": B},
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# ----------------------------------------------------------------------------- main

def main(argv=None) -> int:
    args = parse_args(argv)
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))

    if args.impl == "reference":
        out = run_reference(args, rank)
        if out is not None:
            print(json.dumps(out), flush=True)
        return 0

    dist = None
    if world > 1:
        import torch
        import torch.distributed as dist_mod
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        dist_mod.init_process_group("nccl")
        dist = dist_mod
    out = run_ours(args, rank, world, dist)
    if out is not None:
        if not args.no_cpu_baseline and world == 1:
            out["cpu_baseline"] = cpu_baseline(args.workload, args.cpu_seconds)
        print(json.dumps(out), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
