"""Host-side logic of bench.py and the workload definitions, on the CPU: the
JSON contract of the reference arm, the byte accounting of the decode step,
the split of the timed steps into CUDA graphs, and the refusal of multi-rank
launches."""
import json
import os
import subprocess
import sys

import pytest

import bench
from memory_bound_decode_gb300 import workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_defaults_and_workloads():
    a = bench.parse_args([])
    assert a.gpus == 1 and a.impl == "ours" and a.workload == "down_proj"
    assert a.warmup >= 3
    assert bench.describe("down_proj") == ("single", [4096], 14336, 1)
    assert bench.describe("qkv") == ("fused", [4096, 1024, 1024], 4096, 1)
    assert bench.describe("gate_up") == ("fused", [14336, 14336], 4096, 1)
    assert bench.describe("skinny:4096x14336:B16") == ("single", [4096], 14336, 16)
    assert bench.describe("tail:33x65537") == ("single", [33], 65537, 1)
    with pytest.raises(SystemExit):
        bench.describe("nonsense")


def test_decode_step_bytes():
    spec = workloads.decode_step_spec()
    assert workloads.step_bytes_formula(spec) == 15_017_047_040
    tiny = workloads.decode_step_spec(layers=2, hidden=64, intermediate=192, vocab=300,
                                      q_rows=64, kv_rows=16)
    step = workloads.DecodeStep(tiny, seed=0, device="cpu")
    assert step.algorithmic_bytes() == workloads.step_bytes_formula(tiny)
    assert len(step.projs) == 2 * 7 + 1
    groups = [p.group for p in step.projs]
    assert groups[:3] == [groups[0]] * 3 and groups[0] > 0      # q, k, v fused
    assert groups[3] == 0                                        # o_proj alone


def test_peaks_and_traffic_lookup(tmp_path, monkeypatch):
    peak, kind = bench.load_peaks()
    assert peak > 1000 and kind in ("measured", "fallback")
    from memory_bound_decode_gb300 import binding
    launch = binding.gemv_query_launch(4096, 14336, 1, 152)
    h = bench.kernel_source_hash("fma", launch)
    assert len(h) == 16
    # the launch configuration and the kernel family are part of the hash
    assert h != bench.kernel_source_hash("fma", binding.gemv_query_launch(1024, 4096, 1, 152))
    assert h != bench.kernel_source_hash("mma", launch)
    assert bench.kernel_source_hash("sk", None) != bench.kernel_source_hash("fma", None)
    assert bench.profiled_traffic("no_such_workload", h) is None
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "gemv_x_y.md").write_text(f"kernel_source_hash: {h}\ndram_bytes_per_launch: 1,234\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profiled_traffic("x:y", h) == 1234
    assert bench.profiled_traffic("x:y", "0" * 16) is None


def test_reference_arm_json_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "2", "--warmup", "3"],
                         capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr
    lines = [l for l in out.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference"
    for key in ["metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "config", "cpu_baseline", "e2e"]:
        assert key in rec
    assert rec["steps"] == 2 and rec["value"] > 0
    assert rec["cpu_baseline"]["kind"] == "oracle" and rec["cpu_baseline"]["cores"] >= 1
    assert rec["e2e"]["h2d_bytes_per_step"] == 0


def test_reference_arm_other_ranks_are_silent(monkeypatch):
    args = bench.parse_args(["--impl", "reference", "--steps", "1"])
    assert bench.run_reference(args, rank=1) is None


def test_clock_sampler_without_nvidia_smi(monkeypatch):
    monkeypatch.setenv("PATH", "/nonexistent")
    c = bench.ClockSampler(0)
    c.start()
    info = c.stop()
    assert info["samples"] == 0 and info["sm_mhz"] is None


def test_multi_rank_launch_exits_before_cuda():
    """The path runs on one GPU: a multi-rank launch (WORLD_SIZE > 1, as
    torchrun sets it) or --gpus > 1 stops with an error before torch or the
    library is imported."""
    code = ("import os, sys; sys.path.insert(0, %r); import bench; rc = bench.main(%s); "
            "print(rc, 'torch' in sys.modules, 'memory_bound_decode_gb300.binding' in sys.modules)")
    for env, argv in [({"WORLD_SIZE": "2", "RANK": "0"}, "[]"), ({"WORLD_SIZE": "2", "RANK": "1"}, "[]"),
                      ({}, "['--gpus', '2']")]:
        out = subprocess.run([sys.executable, "-c", code % (ROOT, argv)], capture_output=True, text=True,
                             timeout=120, cwd=ROOT, env=dict(os.environ, **env))
        assert out.returncode == 0, out.stderr
        assert out.stdout.split() == ["2", "False", "False"], out.stdout
        assert "one GPU only" in out.stderr
    # the same through the script's own exit status
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--steps", "1"], capture_output=True,
                         text=True, timeout=120, cwd=ROOT, env=dict(os.environ, WORLD_SIZE="2"))
    assert out.returncode != 0 and "one GPU only" in out.stderr


@pytest.mark.parametrize("steps", [1, 3, 4, 5, 20, 255, 256, 257, 1000, 20000])
@pytest.mark.parametrize("copies", [1, 2, 4, 7])
def test_graph_partition(steps, copies):
    a, q, r = bench.graph_partition(steps, copies, 256)
    assert q * a + r == steps and 0 <= r
    assert a % copies == 0 and a <= max(256, copies)
    if q:
        assert r < a
    seq = [i % copies for _ in range(q) for i in range(a)] + [i % copies for i in range(r)]
    assert len(seq) == steps
    if copies > 1:
        assert all(u != v for u, v in zip(seq, seq[1:]))


def test_no_collective_in_bench():
    src = open(os.path.join(ROOT, "bench.py")).read()
    for word in ("init_process_group", "torch.distributed", "all_reduce"):
        assert word not in src
