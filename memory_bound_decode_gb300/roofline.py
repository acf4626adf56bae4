"""Byte, FLOP and occupancy arithmetic for the decode GEMV and its measurement.

Plain host arithmetic used by the benchmark and the planner checks. Each helper
restates a rule from the pages; the worked numbers those pages print are the
golden values in tests/golden/pages_worked_numbers.json.
"""
from __future__ import annotations

import math

SECTOR_BYTES = 32


def algorithmic_bytes(N: int, K: int, B: int = 1) -> int:
    """Bytes a GEMV must move at minimum: W once (N*K BF16), x once (B*K BF16)
    and y once (B*N FP32). ldw padding, split-K partials and re-reads are not
    counted. ("Decode GEMV at half of HBM bandwidth", "How to approach it":
    at batch 1 the kernel is a byte stream and only bytes per second matter.)"""
    return 2 * N * K + 2 * B * K + 4 * B * N


def algorithmic_bytes_w4(N: int, K: int, B: int = 1, group: int = 128) -> int:
    """The same for INT4 weights: N*K/2 bytes of codes plus N*K/group BF16 scales
    ("Decode GEMV at half of HBM bandwidth", "What interviewers probe next": with
    INT4 weights the bytes fall four times)."""
    return N * K // 2 + 2 * N * (K // group) + 2 * B * K + 4 * B * N


def algorithmic_bytes_fp8(N: int, K: int, B: int = 1) -> int:
    """The same for FP8 weights: N*K bytes of E4M3 codes plus N FP32 row scales
    (the bytes fall two times against BF16)."""
    return N * K + 4 * N + 2 * B * K + 4 * B * N


def flops(N: int, K: int, B: int = 1) -> int:
    """One multiply and one add per weight element per batch row."""
    return 2 * B * N * K


def intensity(N: int, K: int, B: int = 1) -> float:
    """FLOP per algorithmic byte ("How to optimize an ML kernel that
    underutilizes the GPU", Step 1: arithmetic intensity)."""
    return flops(N, K, B) / algorithmic_bytes(N, K, B)


def bytes_in_flight(bandwidth_Bps: float, latency_s: float) -> float:
    """Little's law for memory: outstanding bytes = bandwidth x latency
    ("GPU performance chains", "Bytes in flight to reach bandwidth")."""
    return bandwidth_Bps * latency_s


def loads_in_flight_per_sm(bandwidth_Bps: float, latency_s: float, sms: int,
                           load_bytes: int = 16) -> float:
    return bytes_in_flight(bandwidth_Bps, latency_s) / sms / load_bytes


def stream_time_s(nbytes: float, bandwidth_Bps: float) -> float:
    return nbytes / bandwidth_Bps


def programs(N: int, rows_per_program: int, splits: int = 1) -> int:
    """Grid size of a row-tiled GEMV with optional split-K ("Decode GEMV at half
    of HBM bandwidth", "A strong answer", cause 1: grid = rows/tile x splits)."""
    return math.ceil(N / rows_per_program) * splits


def waves(tiles: int, sms: int, per_sm: int = 1) -> int:
    return math.ceil(tiles / (sms * per_sm))


def wave_efficiency(tiles: int, sms: int, per_sm: int = 1) -> float:
    """Fraction of SM-slots doing work over all waves ("GPU performance chains",
    "Wave quantization")."""
    return tiles / (waves(tiles, sms, per_sm) * sms * per_sm)


def mbu(nbytes: float, time_s: float, peak_Bps: float) -> float:
    """Memory-bandwidth utilisation: bytes over time over peak ("GPU performance
    chains", "Launch gaps in a decode step")."""
    return nbytes / time_s / peak_Bps


def ridge(flops_per_s: float, bandwidth_Bps: float) -> float:
    """FLOP per byte where a kernel turns from bandwidth- to compute-bound
    ("Take a GEMM from naive to 70% of peak", "A strong answer")."""
    return flops_per_s / bandwidth_Bps


def warp_load_sectors(lane_stride_bytes: int, bytes_per_lane: int, lanes: int = 32) -> tuple[int, float]:
    """32-byte sectors touched by one warp-wide load and the fraction of their
    bytes used ("GPU performance chains", "A coalesced warp load")."""
    sectors = set()
    for lane in range(lanes):
        a0 = lane * lane_stride_bytes
        for a in range(a0, a0 + bytes_per_lane):
            sectors.add(a // SECTOR_BYTES)
    used = lanes * bytes_per_lane
    return len(sectors), used / (len(sectors) * SECTOR_BYTES)


def occupancy_blocks(threads: int, regs_per_thread: int, smem_per_block: int, *,
                     sm_regs: int = 65536, sm_smem: int = 228 * 1024,
                     smem_reserved: int = 1024, sm_max_warps: int = 64,
                     sm_max_blocks: int = 32) -> dict:
    """Resident blocks per SM as the minimum of three limits ("GPU performance
    chains", "Occupancy from three limits"): registers, shared memory (with the
    per-block reservation) and warps."""
    warps = math.ceil(threads / 32)
    by_regs = sm_regs // (threads * regs_per_thread) if regs_per_thread else sm_max_blocks
    by_smem = sm_smem // (smem_per_block + smem_reserved)
    by_warps = sm_max_warps // warps
    blocks = min(by_regs, by_smem, by_warps, sm_max_blocks)
    return {"by_regs": by_regs, "by_smem": by_smem, "by_warps": by_warps,
            "blocks": blocks, "occupancy": blocks * warps / sm_max_warps}


def alu_time_s(N: int, K: int, B: int, sms: int, sm_clock_hz: float,
               ops_per_element: float | None = None, lanes_per_sm: int = 128) -> float:
    """Lower bound on the time of the FP32 multiply-adds on CUDA cores: one
    issue slot per lane per clock. ``ops_per_element`` defaults to B
    multiply-adds plus one BF16 widening per weight element."""
    ops = (B + 1) if ops_per_element is None else ops_per_element
    return N * K * ops / (sms * lanes_per_sm * sm_clock_hz)


def bytes_in_flight_per_sm(bandwidth_Bps: float, latency_s: float, sms: int) -> float:
    return bytes_in_flight(bandwidth_Bps, latency_s) / sms


def weight_bytes(N: int, K: int, elem_bytes: int = 2) -> int:
    return N * K * elem_bytes


def idle_sms(tiles: int, sms: int) -> int:
    """SMs that receive no tile in a grid of ``tiles`` one-SM tiles."""
    return max(0, sms - tiles)


def gap_time_s(step_s: float, kernel_s: float) -> float:
    """Time in a step not covered by kernels (launch gaps and stalls)."""
    return step_s - kernel_s


def quantized_time_s(ideal_s: float, tiles: int, sms: int, per_sm: int = 1) -> float:
    """Run time once the last partial wave is paid for in full."""
    return ideal_s / wave_efficiency(tiles, sms, per_sm)
