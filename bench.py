#!/usr/bin/env python3
"""Benchmark of the decode GEMV: achieved HBM GB/s, fraction of GB300 peak and
microseconds per call, printed as one JSON line.

A step is one call of the hot path on one batch of synthetic input: for the
default workload, y = W·x for the down projection of a Llama-3.1-8B-shaped
layer (W 4,096 x 14,336 BF16, x 14,336 BF16, batch 1) through gemv_bf16. The
weights rotate over enough copies that together exceed the L2 cache, so every
step streams W from HBM ("Decode GEMV at half of HBM bandwidth", "Common
mistakes": a matrix that sits in L2 reports more than the HBM can deliver).

    python bench.py [--gpus 1] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...   # the CPU oracle, timed as the baseline arm

Timing: the K timed steps are captured into CUDA graphs (up to --graph-steps
calls each, cycling over the weight copies) and replayed between two CUDA
events on one stream, after a short device-side delay kernel that lets the
host enqueue the replays before the first event fires: the window holds the
K steps' device time and nothing of the host's launch cost. A lone launch
(GPU idle before it) is reported beside it as us_isolated.

The default run also times the other two decode targets, the fused gate/up
projection and the graph-captured decode step, under "targets", and, under
"batched", the same weights with 16 rows of x: down_proj's shape and the whole
decode step.

One GPU only: the path has no multi-GPU form, and a multi-rank launch
(WORLD_SIZE > 1) exits with an error before any CUDA call. The reference arm
(the CPU oracle) runs on rank 0 alone; other ranks exit without work.
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
    ap.add_argument("--graph-steps", type=int, default=256,
                    help="most calls captured into one CUDA graph of the timed loop")
    ap.add_argument("--no-targets", action="store_true",
                    help="skip timing the gate/up and decode-step targets of the default run")
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
    "tc": ("gemv_internal.h", "gemv_common.cuh", "gemv_tc_kernel.cuh", "gemv_tc_instances.cu",
           "gemv_dispatch.cu"),
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
    m = re.fullmatch(r"(qkv|gate_up|decode_step)(?::B(\d+))?", workload)
    if m:
        B = int(m.group(2)) if m.group(2) else 1
        if m.group(1) == "qkv":
            return "fused", [4096, 1024, 1024], 4096, B
        if m.group(1) == "gate_up":
            return "fused", [14336, 14336], 4096, B
        return "step", None, None, B
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

    def __init__(self, device, stream, rms_eps=None, streamk=False, weights="bf16", data=None,
                 keep_waits=False, batch=1):
        from memory_bound_decode_gb300 import workloads as wl
        self.spec = wl.decode_step_spec()
        self.weights = weights
        self.data = data if data is not None else wl.DecodeStep(self.spec, seed=0, device=device, weights=weights,
                                                                batch=batch)
        batch = self.data.batch
        self.rms_eps = rms_eps
        self.streamk = streamk
        self.keep_waits = keep_waits
        self.w4, self.fp8 = weights == "int4", weights == "fp8"
        if keep_waits:
            # every launch waits for the preceding grid, as if each projection
            # read the previous one's output (the planner's planwait knob,
            # read when the plan is created)
            saved = os.environ.get("GEMV_FORCE_VARIANT")
            os.environ["GEMV_FORCE_VARIANT"] = (saved + "," if saved else "") + "planwait=1"
            try:
                self.plan = self.data.plan(rms_eps=rms_eps, streamk=streamk)
            finally:
                if saved is None:
                    del os.environ["GEMV_FORCE_VARIANT"]
                else:
                    os.environ["GEMV_FORCE_VARIANT"] = saved
        else:
            self.plan = self.data.plan(rms_eps=rms_eps, streamk=streamk)
        self.plan.capture(stream)
        self.bytes_per_step = (wl.step_bytes_formula(self.spec, batch) if weights == "bf16"
                               else self.data.algorithmic_bytes())
        self.launches_per_step = self.plan.num_launches()
        self.x = None
        self.B = batch

    def step(self, i: int, stream, x=None) -> None:
        self.plan.launch(stream)

    def config(self) -> dict:
        norm = (f"; RMSNorm prologue (eps={self.rms_eps}) on QKV, gate_up and lm_head"
                if self.rms_eps is not None else "")
        wt = {"bf16": "BF16", "fp8": "FP8 (E4M3, FP32 row scales)",
              "int4": "INT4 (128-col groups, BF16 scales)"}[self.weights]
        return {"workload": "decode step: 32 x {QKV 6144x4096, o 4096x4096, gate_up 28672x4096, "
                            f"down 4096x14336}} + lm_head 128256x4096, {wt} weights, batch {self.B}, "
                            "one CUDA graph" + norm,
                "launches_per_step": self.launches_per_step,
                "l2": f"inputs larger than L2: {self.data.weight_bytes() / 1e9:.2f} GB of weights per step"}


# ----------------------------------------------------------------------------- our arm

TARGETS = {"down_proj": 0.85, "gate_up": 0.85, "decode_step": 0.80}   # fraction of HBM peak
DELAY_CYCLES = 1_000_000   # device-side delay before the first event (about 0.5 ms at 2 GHz)


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


def device_delay(torch) -> None:
    """A short device-side delay on the current stream: what is enqueued after
    it is in the stream before the GPU reaches it."""
    sleep = getattr(torch.cuda, "_sleep", None)
    if sleep is not None:
        sleep(DELAY_CYCLES)


def graph_partition(steps: int, copies: int, graph_max: int) -> tuple[int, int, int]:
    """(a, q, r): graph A holds a calls (a multiple of the weight copies, at
    most max(graph_max, copies)) and is replayed q times, graph B holds the
    remaining r < a calls (or all of them when steps < copies); q * a + r ==
    steps. Call i of either graph reads copy i % copies, so the copy sequence
    over A ... A B never repeats a copy back to back when copies > 1."""
    a = (min(steps, max(graph_max, copies)) // copies) * copies
    q = steps // a if a else 0
    return a, q, steps - q * a


class TimedLoop:
    """The K steps of the timed region, replayable: for matrix workloads CUDA
    graphs of consecutive calls (graph A with a multiple of the weight copies,
    replayed q times, then graph B with the remaining r calls, so that no two
    neighbouring calls read the same copy), for the decode step K launches of
    its captured plan."""

    def __init__(self, torch, wk, steps: int, stream, graph_max: int):
        self.torch, self.wk, self.steps, self.stream = torch, wk, steps, stream
        self.graphs = []
        if isinstance(wk, StepWorkload):
            self.q, self.r = 0, 0
            return
        a, self.q, self.r = graph_partition(steps, wk.copies, graph_max)
        self.gA = self._capture(a) if self.q else None
        self.gB = self._capture(self.r) if self.r else None

    def _capture(self, n: int):
        torch = self.torch
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=self.stream, capture_error_mode="thread_local"):
            cs = torch.cuda.current_stream()
            for i in range(n):
                self.wk.step(i, cs)
        return g

    def run(self) -> None:
        if isinstance(self.wk, StepWorkload):
            for i in range(self.steps):
                self.wk.step(i, self.stream)
            return
        for _ in range(self.q):
            self.gA.replay()
        if self.gB is not None:
            self.gB.replay()


def time_workload(torch, wk, args, stream, gpu_index: int, isolated: int = 20) -> dict:
    """Warm up, time exactly args.steps steps on the device (clocks sampled
    around the region while the same loop keeps the GPU busy), then time
    single launches with the GPU idle before each."""
    with torch.cuda.stream(stream):
        for i in range(max(3, args.warmup)):
            wk.step(i, stream)
        loop = TimedLoop(torch, wk, args.steps, stream, args.graph_steps)
        loop.run()
        torch.cuda.synchronize()
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)

        def region() -> float:
            torch.cuda.synchronize()
            device_delay(torch)
            ev0.record(stream)
            loop.run()
            ev1.record(stream)
            torch.cuda.synchronize()
            return ev0.elapsed_time(ev1) / 1e3

        est = region()
        clocks = ClockSampler(gpu_index)
        clocks.start()
        soak = max(1, math.ceil(0.25 / max(est, 1e-6)))   # about 250 ms under the same load
        for _ in range(soak):
            loop.run()
        seconds = region()
        for _ in range(max(1, soak // 4)):
            loop.run()
        torch.cuda.synchronize()
        clock_info = clocks.stop()
        clock_info["soak_loops"] = soak

        iso = []
        for i in range(isolated):
            torch.cuda.synchronize()
            device_delay(torch)
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            wk.step(i, stream)
            b.record(stream)
            torch.cuda.synchronize()
            iso.append(a.elapsed_time(b) / 1e3)
    return {"seconds": seconds, "clocks": clock_info, "isolated_s": statistics.median(iso),
            "graphs": {"calls_per_graph": (args.steps - loop.r) // loop.q if loop.q else loop.r,
                       "replays": loop.q + (1 if loop.r else 0)}
            if not isinstance(wk, StepWorkload) else {"plan_launches": args.steps}}


def time_e2e(torch, binding, wk, steps: int, stream) -> dict | None:
    """The same workload end to end through the public C entry points with
    host buffers: every step copies its inputs in from pinned host memory,
    runs, copies its outputs back and waits (host wall clock): gemv_bf16_host_io,
    gemv_bf16_multi_host_io, or gemv_plan_launch_host_io (the decode step, and
    a one-projection plan for quantised weights)."""
    sh = stream.cuda_stream
    if isinstance(wk, StepWorkload):
        d = wk.data
        x_host = d.x_arena.cpu().pin_memory()
        y_host = torch.empty(d.y_arena.shape, dtype=d.y_arena.dtype).pin_memory()
        xb = x_host.numel() * x_host.element_size()
        yb = y_host.numel() * y_host.element_size()

        def e2e_step(i):
            wk.plan.launch_host_io(x_host, d.x_arena, xb, d.y_arena, y_host, yb, sh)
        h2d, d2h = xb, yb
        n = max(5, min(steps, 200))
    else:
        x_host = wk.x.cpu().pin_memory()
        y_host = [torch.empty(y.shape, dtype=y.dtype).pin_memory() for y in wk.ys]
        x_dev = torch.empty_like(wk.x)
        bf16 = not wk.w4 and not wk.fp8

        def e2e_step(i):
            Ws = wk.Ws[i % wk.copies]
            if bf16 and wk.kind == "single":
                binding.gemv_bf16_host_io(Ws[0], x_host, y_host[0], x_dev, wk.ys[0], wk.N, wk.K, wk.B, wk.ldw,
                                          rms_eps=wk.rms_eps, stream=sh, streamk=wk.streamk,
                                          cuda_cores=wk.cuda_cores)
            elif bf16:
                binding.gemv_bf16_multi_host_io([(W, y, n_, wk.ldw) for W, y, n_ in zip(Ws, wk.ys, wk.rows)],
                                                x_host, x_dev, y_host, wk.K, wk.B, rms_eps=wk.rms_eps,
                                                stream=sh, streamk=wk.streamk, cuda_cores=wk.cuda_cores)
            else:   # quantised weights: a one-projection plan per weight copy, host to host
                plans[i % wk.copies].launch_host_io(x_host, x_dev, h2d, wk.ys[0], y_host[0], d2h, sh)
        h2d = int(x_host.numel() * x_host.element_size())
        d2h = int(sum(y.numel() * y.element_size() for y in y_host))
        n = max(10, min(steps, 2000))
        plans = []
        if not bf16:
            kind = binding.GEMV_WEIGHT_INT4 if wk.w4 else binding.GEMV_WEIGHT_FP8
            for Ws in wk.Ws:
                Wq, S = Ws[0]
                plans.append(binding.Plan([(Wq, x_dev, wk.ys[0], wk.N, wk.K, wk.ldq, wk.B, 0, wk.rms_eps, False, kind,
                                            S, wk.lds if wk.w4 else 0)]))
                plans[-1].capture(torch.cuda.Stream())
    with torch.cuda.stream(stream):
        for i in range(5):
            e2e_step(i)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for i in range(n):
            e2e_step(i)
        el = time.perf_counter() - t0
    return {"value": round(wk.bytes_per_step * n / el / 1e9, 2), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "us_per_step": round(el / n * 1e6, 3), "steps": n}


def make_workload(torch, name: str, device, l2: int):
    kind, rows, K, B = describe(name)
    _, rms_eps = split_norm(name)
    base, streamk = split_sk(split_norm(name)[0])
    base, cuda_cores = split_cc(base)
    base, fp8 = split_f8(base)
    _, w4 = split_w4(base)
    if kind == "step":
        return StepWorkload(device, torch.cuda.Stream(), rms_eps, streamk,
                            "int4" if w4 else "fp8" if fp8 else "bf16", batch=B)
    return GemvWorkload(kind, rows, K, B, device, l2, rms_eps, w4, streamk, fp8, cuda_cores)


def family_of(wk) -> str:
    if isinstance(wk, StepWorkload):
        return "w4" if wk.w4 else "f8" if wk.fp8 else "fma"
    return ("w4" if wk.w4 else "f8" if wk.fp8 else "sk" if wk.streamk
            else "fma" if (wk.B == 1 or wk.cuda_cores) else "mma")


def target_entry(torch, binding, name: str, args, stream, device, l2, peak, read_ceiling, gpu_index) -> dict:
    """One of the decode targets (or, without a target fraction, another
    workload), timed like the headline."""
    wk = make_workload(torch, name, device, l2)
    target = TARGETS.get(name)
    t = time_workload(torch, wk, args, stream, gpu_index)
    per_step = t["seconds"] / args.steps
    gbs = wk.bytes_per_step / per_step / 1e9
    out = {"workload": wk.config()["workload"], "bytes_per_step": wk.bytes_per_step,
           "steps": args.steps, "us_per_step": round(per_step * 1e6, 3),
           "us_isolated": round(t["isolated_s"] * 1e6, 3),
           "gbs": round(gbs, 2), "frac": round(gbs / peak, 4),
           "frac_of_read_probe": round(gbs / read_ceiling, 4) if read_ceiling else None,
           "gpu_launches": args.steps * wk.launches_per_step,
           "clocks": t["clocks"]}
    if target is not None:
        out["target_frac"] = target
        out["met"] = gbs / peak >= target
        out["met_vs_max_of_copy_and_read_probe"] = gbs / max(peak, read_ceiling or 0) >= target
    if isinstance(wk, StepWorkload):
        out["launches_per_step"] = wk.launches_per_step
        out["independent_launches"] = wk.plan.independent()
    if not args.no_e2e:
        out["e2e"] = time_e2e(torch, binding, wk, args.steps, stream)
    if isinstance(wk, StepWorkload):
        # The same step with every launch waiting for the preceding grid (as
        # if the projections were chained), on the same weights.
        dep = StepWorkload(device, torch.cuda.Stream(), wk.rms_eps, wk.streamk, wk.weights, data=wk.data,
                           keep_waits=True, batch=wk.B)
        td = time_workload(torch, dep, args, stream, gpu_index)
        per = td["seconds"] / args.steps
        gd = dep.bytes_per_step / per / 1e9
        out["with_every_wait"] = {"us_per_step": round(per * 1e6, 3), "gbs": round(gd, 2), "frac": round(gd / peak, 4),
                                  "independent_launches": dep.plan.independent(), "clocks": td["clocks"]}
        if target is not None:
            out["with_every_wait"]["met"] = gd / peak >= target
        dep.plan.destroy()
        del dep
    del wk
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return out


def run_ours(args) -> dict:
    import torch
    from memory_bound_decode_gb300 import binding, build_lib

    build_lib.build()
    binding.lib()
    gpu_index = 0
    torch.cuda.set_device(gpu_index)
    device = torch.device("cuda", gpu_index)
    stream = torch.cuda.Stream()
    props = torch.cuda.get_device_properties(device)
    l2 = getattr(props, "L2_cache_size", 126 << 20)

    wk = make_workload(torch, args.workload, device, l2)
    kind = "step" if isinstance(wk, StepWorkload) else wk.kind
    torch.cuda.synchronize()
    t = time_workload(torch, wk, args, stream, gpu_index)
    seconds = t["seconds"]
    steps = args.steps
    value = wk.bytes_per_step * steps / seconds / 1e9
    per_launch_s = seconds / (steps * wk.launches_per_step)

    e2e = None if args.no_e2e else time_e2e(torch, binding, wk, steps, stream)

    read_ceiling = None if args.no_probe else read_ceiling_gbs(torch, binding, stream)

    peak, peak_kind = load_peaks()
    achieved = wk.bytes_per_step / (seconds / steps) / 1e9 if kind == "step" else \
        wk.bytes_per_step / per_launch_s / 1e9
    family = family_of(wk)
    launch = None
    if kind == "single":
        sms = props.multi_processor_count
        if family == "w4":
            launch = binding.gemv_w4_query_launch(wk.N, wk.K, wk.B, sms)
        elif family == "f8":
            launch = binding.gemv_fp8_query_launch(wk.N, wk.K, wk.B, sms)
        else:
            launch = binding.gemv_query_launch_ex(
                wk.N, wk.K, wk.B, sms,
                binding.GEMV_FLAG_STREAMK if family == "sk" else
                binding.GEMV_FLAG_CUDA_CORES if wk.cuda_cores else 0)
    if launch and launch.get("path") == 5:
        family = "tc"   # the planner chose the tcgen05 kernel for this shape
    src_hash = kernel_source_hash(family, launch)
    traffic = profiled_traffic(args.workload, src_hash)
    knobs = {k: v for k, v in os.environ.items() if k in ("GEMV_FORCE_SPLIT", "GEMV_FORCE_VARIANT", "GEMV_PDL")}
    result = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": 1,
        "steps": steps, "warmup": max(3, args.warmup),
        "ms_per_step": round(seconds / steps * 1e3, 6),
        "us_per_call": round(per_launch_s * 1e6, 3),
        "us_isolated": round(t["isolated_s"] * 1e6, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": {"w4": "u4 weights (bf16 group scales), bf16 x, fp32 accumulate",
                  "f8": "e4m3 weights (fp32 row scales), bf16 x, fp32 accumulate"}.get(family, "bf16 in, fp32 accumulate"),
        "data": "synthetic (seeded N(0,0.02^2) weights, N(0,1) x)",
        "config": dict(wk.config(), parallelism="1 GPU",
                       pdl=os.environ.get("GEMV_PDL", "1") != "0",
                       timing=("K steps as CUDA graph replays between two events, after a device-side "
                               "delay kernel; " + json.dumps(t["graphs"])),
                       **({"knobs": knobs} if knobs else {})),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": UNIT,
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "peak_kind": f"{peak_kind} copy (MEASURED_PEAKS hbm_gbs, burst)"
                     if peak_kind == "measured" else "fallback 6.8 TB/s",
                     "kernel": ("gemv_w4_kernel (INT4 codes, BF16 tensor cores)" if family == "w4"
                                else "gemv_fp8_kernel (E4M3 codes, BF16 tensor cores)" if family == "f8"
                                else "gemv_streamk_kernel (CUDA cores, one-wave grid)" if family == "sk"
                                else "gemv_tc_kernel (tcgen05, accumulator in tensor memory)" if family == "tc"
                                else "gemv_bf16_kernel (CUDA cores)" if wk.B == 1 or family == "fma"
                                else "gemv_bf16_mma_kernel (BF16 tensor cores)"),
                     "kernel_source_hash": src_hash},
        "ceilings": {"copy_gbs": peak,
                     "read_probe_gbs": round(read_ceiling, 1) if read_ceiling else None,
                     "vendor_gbs": VENDOR_HBM_GBS,
                     "frac_of_read_probe": round(achieved / read_ceiling, 4) if read_ceiling else None,
                     "frac_of_vendor": round(achieved / VENDOR_HBM_GBS, 4)},
        "gpu_launches": steps * wk.launches_per_step,
        "clocks": t["clocks"],
    }
    if e2e is not None:
        result["e2e"] = e2e
    del wk
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    if args.workload == "down_proj" and not args.no_targets:
        targets = {"down_proj": {"us_per_step": result["us_per_call"], "gbs": result["value"],
                                 "frac": result["roofline"]["frac"],
                                 "frac_of_read_probe": result["ceilings"]["frac_of_read_probe"],
                                 "target_frac": TARGETS["down_proj"],
                                 "met": result["roofline"]["frac"] >= TARGETS["down_proj"],
                                 "met_vs_max_of_copy_and_read_probe":
                                     achieved / max(peak, read_ceiling or 0) >= TARGETS["down_proj"]}}
        for name in ("gate_up", "decode_step"):
            targets[name] = target_entry(torch, binding, name, args, stream, device, l2, peak, read_ceiling,
                                         gpu_index)
        result["targets"] = targets
        result["batched"] = {name: target_entry(torch, binding, name, args, stream, device, l2, peak, read_ceiling,
                                                gpu_index)
                             for name in ("skinny:4096x14336:B16", "decode_step:B16")}
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

    if world > 1 or args.gpus != 1:
        # Checked before anything touches CUDA: the path runs on one GPU.
        print(f"bench.py: one GPU only (got --gpus {args.gpus}, WORLD_SIZE {world}); "
              "the decode GEMV has no multi-GPU form here", file=sys.stderr, flush=True)
        return 2
    out = run_ours(args)
    if not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(args.workload, args.cpu_seconds)
    print(json.dumps(out), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
