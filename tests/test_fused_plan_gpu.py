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
    ((14336, 14336), 4096, 1),          # gate, up
    ((7, 33, 1, 100), 4103, 3),         # ragged segments
    ((5,) * 8, 129, 2),                 # the most segments one launch takes
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


def test_full_decode_step_sampled():
    """The full Llama-3.1-8B-shaped step (32 layers + LM head, 15 GB of BF16
    weights) in the launch configuration the benchmark times: one captured
    graph. Sampled rows of every projection are checked one by one against
    the oracle."""
    free, _ = torch.cuda.mem_get_info()
    if free < 40 << 30:
        pytest.skip("needs 40 GB of free device memory")
    spec = workloads.decode_step_spec()
    step = workloads.DecodeStep(spec, seed=0, device=DEV)
    plan = step.plan()
    assert plan.num_launches() == 32 * 4 + 1
    s = torch.cuda.Stream()
    plan.capture(s)
    for y in step.outputs():
        y.fill_(float("nan"))
    torch.cuda.synchronize()
    plan.launch(s)
    s.synchronize()
    rng = np.random.default_rng(0)
    for name, W, x, y, K in step.checks():
        N = W.shape[0]
        rows = np.unique(np.concatenate([[0, N - 1], rng.integers(0, N, 6)]))
        yh = y.cpu().numpy()
        assert np.isfinite(yh).all(), name
        xb = inputs.bits(x)
        Wr = inputs.bits(W[torch.as_tensor(rows, device=DEV)])
        for i, n in enumerate(rows):
            y_ref, sc = oracle.gemv_one(Wr, xb, 0, i, K)
            assert abs(float(yh[0, n]) - y_ref) <= 1e-5 * sc, (name, n)
    plan.destroy()
    del step
    torch.cuda.empty_cache()
