"""Fused multi-projection launches and the CUDA-graph decode-step plan, against
the CPU oracle."""
import numpy as np
import pytest
import torch

from memory_bound_decode_gb300 import binding, inputs, workloads
from oracle import oracle
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _segments(rows, K, seed):
    ldw = inputs.padded_ldw(K)
    Ws = [inputs.weight(n, K, ldw, seed=seed, index=i, device=DEV) for i, n in enumerate(rows)]
    return Ws, ldw


@pytest.mark.parametrize("rows,K,B", [
    ((4096, 1024, 1024), 4096, 1),      # Q, K, V
    ((4096, 1024, 1024), 4096, 4),      # Q, K, V at batch 4 (tensor cores, x by bulk copies)
    ((14336, 14336), 4096, 1),          # gate, up
    ((7, 33, 1, 100), 4103, 3),         # ragged segments
    ((5,) * 8, 129, 2),                 # the most segments one launch takes
    ((4096, 1024, 1024), 4096, 16),     # Q, K, V at batch 16 (the tcgen05 kernel, a tensor map per segment)
    ((14336, 14336), 4096, 12),         # gate, up at batch 12 (tcgen05)
    ((100, 257, 3000), 8192, 9),        # ragged segments (tcgen05)
    ((5,) * 8, 136, 16),                # the most segments, each one partial tile (tcgen05)
    ((20000, 20000, 77), 1024, 16),     # more row tiles than one wave (persistent tcgen05)
])
def test_fused_matches_oracle(rows, K, B):
    Ws, ldw = _segments(rows, K, seed=20)
    x = inputs.activations(B, K, seed=20, index=99, device=DEV)
    ys = [gu.guarded_y(B, n) for n in rows]
    binding.gemv_bf16_multi([(W, y, n, ldw) for W, (_, y), n in zip(Ws, ys, rows)], x, K, B)
    torch.cuda.synchronize()
    for W, (buf, y), n in zip(Ws, ys, rows):
        gu.check_guards(buf)
        y_ref, s = gu.reference(W, x, K)
        gu.assert_parity(y.cpu().numpy(), y_ref, s, f"segment N={n}")


def test_fused_equals_concatenated_single_call():
    """One fused launch over Q, K and V computes each row exactly as a single
    call over the concatenated 6,144-row matrix does (same plan, same order)."""
    rows, K = (4096, 1024, 1024), 4096
    Ws, ldw = _segments(rows, K, seed=21)
    x = inputs.activations(1, K, seed=21, index=99, device=DEV)
    ys = [torch.empty((1, n), device=DEV) for n in rows]
    binding.gemv_bf16_multi([(W, y, n, ldw) for W, y, n in zip(Ws, ys, rows)], x, K, 1)
    Wcat = torch.cat(Ws, 0)
    ycat = torch.empty((1, sum(rows)), device=DEV)
    binding.gemv_bf16(Wcat, x, ycat, sum(rows), K, 1, ldw)
    torch.cuda.synchronize()
    assert torch.equal(torch.cat(ys, 1), ycat)


def test_plan_replays_and_sees_updated_x():
    """A two-layer decode step at reduced width: capture once, replay, update x
    in place, replay again; every projection checked against the oracle."""
    spec = workloads.decode_step_spec(layers=2, hidden=512, intermediate=1536, vocab=2000,
                                      q_rows=512, kv_rows=128)
    step = workloads.DecodeStep(spec, seed=22, device=DEV)
    plan = step.plan()
    assert plan.num_launches() == 2 * 4 + 1
    s = torch.cuda.Stream()
    plan.capture(s)
    for round_ in range(2):
        if round_ == 1:
            step.refresh_x(seed=23)
        for y in step.outputs():
            y.fill_(float("nan"))
        torch.cuda.synchronize()
        plan.launch(s)
        s.synchronize()
        for name, W, x, y, K in step.checks():
            y_ref, sc = gu.reference(W, x, K)
            gu.assert_parity(y.cpu().numpy(), y_ref, sc, f"round {round_} {name}")
    plan.destroy()


def test_plan_errors():
    W = inputs.weight(64, 64, device=DEV)
    x = inputs.activations(1, 64, device=DEV)
    y = torch.empty((1, 64), device=DEV)
    plan = binding.Plan([(W, x, y, 64, 64, 64, 1, 0)])
    assert plan.launch(torch.cuda.current_stream(), check=False) == binding.GEMV_ERR_UNSUPPORTED
    assert binding.lib().gemv_plan_capture(plan._h, None) == binding.GEMV_ERR_INVALID
    s = torch.cuda.Stream()
    plan.capture(s)
    plan.capture(s)   # re-capture replaces the graph
    plan.launch(s)
    s.synchronize()
    y_ref, sc = gu.reference(W, x, 64)
    gu.assert_parity(y.cpu().numpy(), y_ref, sc)
    plan.destroy()


@pytest.mark.parametrize("batch", [16, 9])
def test_batched_decode_step_every_element(batch):
    """A decode step of two layers and the LM head at 16 (9) rows of x: the
    layers' projections take the tcgen05 kernel (fused QKV and gate/up with a
    tensor map per segment), the LM head, whose row tiles exceed one wave, the
    register-fed tensor-core kernel. One captured graph, run end to end through
    gemv_plan_launch_host_io; every output compared with the FP64 oracle."""
    spec = workloads.decode_step_spec(layers=2)
    step = workloads.DecodeStep(spec, seed=1, device=DEV, batch=batch)
    plan = step.plan()
    assert plan.num_launches() == 2 * 4 + 1
    s = torch.cuda.Stream()
    plan.capture(s)
    x_host = step.x_arena.cpu().pin_memory()
    y_host = torch.full(step.y_arena.shape, float("nan"), dtype=torch.float32).pin_memory()
    step.y_arena.fill_(float("nan"))
    torch.cuda.synchronize()
    plan.launch_host_io(x_host, step.x_arena, x_host.numel() * 2, step.y_arena, y_host, y_host.numel() * 4, s)
    assert torch.equal(y_host.view(torch.int32), step.y_arena.cpu().view(torch.int32))
    threads = oracle.default_threads()
    off = 0
    for name, W, x, y, K in step.checks():
        N = W.shape[0]
        assert x.shape == (batch, K) and y.shape == (batch, N)
        assert y.data_ptr() == step.y_arena.data_ptr() + 4 * off
        y_ref, sc = oracle.gemv(inputs.bits(W), inputs.bits(x), K, threads=threads)
        gu.assert_parity(y_host[off:off + batch * N].numpy().reshape(batch, N), y_ref, sc, name)
        off += batch * N
    assert off == step.y_arena.numel()
    assert binding.gemv_device_status(reset=True) == 0
    plan.destroy()
    del step
    torch.cuda.empty_cache()


def test_full_decode_step_every_element():
    """The full Llama-3.1-8B-shaped step (32 layers + LM head, 15 GB of BF16
    weights) in the launch configuration the benchmark times: one captured
    graph of 129 launches, run end to end through gemv_plan_launch_host_io
    (host x in, the graph, host y out). Every output of every projection is
    compared with the FP64 oracle (about 15 GB of weights through the oracle
    on all host cores: seconds)."""
    free, _ = torch.cuda.mem_get_info()
    if free < 40 << 30:
        pytest.skip("needs 40 GB of free device memory")
    spec = workloads.decode_step_spec()
    step = workloads.DecodeStep(spec, seed=0, device=DEV)
    plan = step.plan()
    assert plan.num_launches() == 32 * 4 + 1
    s = torch.cuda.Stream()
    plan.capture(s)
    x_host = step.x_arena.cpu().pin_memory()
    y_host = torch.full(step.y_arena.shape, float("nan"), dtype=torch.float32).pin_memory()
    step.y_arena.fill_(float("nan"))
    torch.cuda.synchronize()
    plan.launch_host_io(x_host, step.x_arena, x_host.numel() * 2, step.y_arena, y_host, y_host.numel() * 4, s)
    assert torch.equal(y_host.view(torch.int32), step.y_arena.cpu().view(torch.int32))
    threads = oracle.default_threads()
    off = 0
    checked = 0
    for name, W, x, y, K in step.checks():
        N = W.shape[0]
        assert y.data_ptr() == step.y_arena.data_ptr() + 4 * off
        y_ref, sc = oracle.gemv(inputs.bits(W), inputs.bits(x), K, threads=threads)
        gu.assert_parity(y_host[off:off + N].numpy()[None, :], y_ref, sc, name)
        off += N
        checked += N
    assert off == step.y_arena.numel() and checked == 1_504_512
    plan.destroy()
    del step
    torch.cuda.empty_cache()


def test_plan_launch_host_io_rejects():
    W = inputs.weight(64, 64, device=DEV)
    x = inputs.activations(1, 64, device=DEV)
    y = torch.empty((1, 64), device=DEV)
    plan = binding.Plan([(W, x, y, 64, 64, 64, 1, 0)])
    xh = x.cpu().pin_memory()
    yh = torch.empty((1, 64)).pin_memory()
    s = torch.cuda.Stream()
    # not captured yet
    assert plan.launch_host_io(xh, x, 128, y, yh, 256, s, check=False) == binding.GEMV_ERR_UNSUPPORTED
    plan.capture(s)
    assert plan.launch_host_io(None, x, 128, y, yh, 256, s, check=False) == binding.GEMV_ERR_INVALID
    assert plan.launch_host_io(xh, x, -1, y, yh, 256, s, check=False) == binding.GEMV_ERR_INVALID
    assert plan.launch_host_io(xh, x, 128, None, yh, 256, s, check=False) == binding.GEMV_ERR_INVALID
    # zero-byte copies leave the pointers unused
    plan.launch_host_io(None, None, 0, y, yh, 256, s)
    y_ref, sc = gu.reference(W, x, 64)
    gu.assert_parity(yh.numpy(), y_ref, sc)
    # a capturing stream cannot wait for itself
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s, capture_error_mode="thread_local"):
        rc = plan.launch_host_io(xh, x, 128, y, yh, 256, s, check=False)
    assert rc == binding.GEMV_ERR_CAPTURE
    plan.destroy()


def test_multi_host_io_matches_device_call():
    rows, K = (14336, 14336), 4096
    Ws, ldw = _segments(rows, K, seed=24)
    x = inputs.activations(1, K, seed=24, index=99, device=DEV)
    ys = [torch.full((1, n), float("nan"), device=DEV) for n in rows]
    x_host = x.cpu().pin_memory()
    x_dev = torch.empty_like(x)
    y_host = [torch.full((1, n), float("nan")).pin_memory() for n in rows]
    binding.gemv_bf16_multi_host_io([(W, y, n, ldw) for W, y, n in zip(Ws, ys, rows)], x_host, x_dev, y_host, K, 1)
    want = [torch.empty((1, n), device=DEV) for n in rows]
    binding.gemv_bf16_multi([(W, y, n, ldw) for W, y, n in zip(Ws, want, rows)], x, K, 1)
    torch.cuda.synchronize()
    for W, yh, yw in zip(Ws, y_host, want):
        assert torch.equal(yh.view(torch.int32), yw.cpu().view(torch.int32))
        y_ref, sc = gu.reference(W, x, K)
        gu.assert_parity(yh.numpy(), y_ref, sc, "multi host io")
    # bad arguments are refused before any copy
    segs = [(W, y, n, ldw) for W, y, n in zip(Ws, ys, rows)]
    assert binding.gemv_bf16_multi_host_io(segs, x_host, x_dev, [y_host[0], None], K, 1,
                                           check=False) == binding.GEMV_ERR_INVALID
    assert binding.gemv_bf16_multi_host_io(segs, None, x_dev, y_host, K, 1,
                                           check=False) == binding.GEMV_ERR_INVALID


def test_plan_independence_and_ordering(monkeypatch):
    """A plan whose launches touch disjoint outputs runs them without waiting
    for each other; a plan where one launch writes what another reads or
    writes keeps every wait, and its launches take effect in list order."""
    N, K = 4096, 4096
    W1 = inputs.weight(N, K, seed=30, device=DEV)
    W2 = inputs.weight(N, K, seed=31, device=DEV)
    x1 = inputs.activations(1, K, seed=30, index=5, device=DEV)
    x2 = inputs.activations(1, K, seed=31, index=5, device=DEV)
    ya = torch.empty((1, N), device=DEV)
    yb = torch.empty((1, N), device=DEV)
    s = torch.cuda.Stream()

    # disjoint: independent, both results right
    p = binding.Plan([(W1, x1, ya, N, K, K, 1, 0), (W2, x2, yb, N, K, K, 1, 0)])
    assert p.independent()
    p.capture(s)
    ya.fill_(float("nan"))
    yb.fill_(float("nan"))
    torch.cuda.synchronize()
    p.launch(s)
    s.synchronize()
    for W, x, y in ((W1, x1, ya), (W2, x2, yb)):
        y_ref, sc = gu.reference(W, x, K)
        gu.assert_parity(y.cpu().numpy(), y_ref, sc, "independent plan")
    p.destroy()

    # the same y written twice: dependent; the later launch's result stays
    p = binding.Plan([(W1, x1, ya, N, K, K, 1, 0), (W2, x2, ya, N, K, K, 1, 0)])
    assert not p.independent()
    p.capture(s)
    for _ in range(3):
        ya.fill_(float("nan"))
        torch.cuda.synchronize()
        p.launch(s)
        s.synchronize()
        y_ref, sc = gu.reference(W2, x2, K)
        gu.assert_parity(ya.cpu().numpy(), y_ref, sc, "write after write")
    p.destroy()

    # a launch whose output overlaps a later launch's x, or its weights
    buf = torch.empty(N, device=DEV)
    xs = buf.view(torch.bfloat16)[:K].view(1, K)
    p = binding.Plan([(W1, x1, buf.view(1, N), N, K, K, 1, 0), (W2, xs, yb, N, K, K, 1, 0)])
    assert not p.independent()
    p.destroy()
    Wbuf = torch.empty((N, K), dtype=torch.bfloat16, device=DEV)
    p = binding.Plan([(W1, x1, Wbuf.view(-1).view(torch.float32)[:N].view(1, N), N, K, K, 1, 0),
                      (Wbuf, x2, yb, N, K, K, 1, 0)])
    assert not p.independent()
    p.destroy()

    # the sweep knob keeps the waits in an independent plan
    monkeypatch.setenv("GEMV_FORCE_VARIANT", "planwait=1")
    p = binding.Plan([(W1, x1, ya, N, K, K, 1, 0), (W2, x2, yb, N, K, K, 1, 0)])
    assert not p.independent()
    p.destroy()
    monkeypatch.delenv("GEMV_FORCE_VARIANT")

    # the decode step's projections are independent (each reads its own x)
    spec = workloads.decode_step_spec(layers=2, hidden=512, intermediate=1536, vocab=2000, q_rows=512, kv_rows=128)
    step = workloads.DecodeStep(spec, seed=32, device=DEV)
    plan = step.plan()
    assert plan.independent()
    assert not step.plan(streamk=True).independent()   # stream-K launches share a workspace
    plan.destroy()
