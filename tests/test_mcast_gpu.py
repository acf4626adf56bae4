"""Batch 1 with x multicast: CTAs in clusters of 2 along the rows share one
bulk copy of x (rank 0 copies it into both CTAs' shared memory, an
mbarrier counts the bytes in each). The result must be the same bits as the
per-CTA staging, which a call takes when x is not 16-byte aligned (same
values, 2 bytes further on in memory), and agree with the CPU oracle; the
device status must stay clear (no mbarrier wait ran out)."""
import numpy as np
import pytest
import torch

from memory_bound_decode_gb300 import binding, inputs
from oracle import oracle
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu
DEV = "cuda"


def sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def shifted(x):
    """The same values at a 2-byte offset from a 16-byte boundary."""
    B, K = x.shape
    buf = torch.empty(B * K + 8, dtype=x.dtype, device=x.device)
    out = buf[1:1 + B * K].view(B, K)
    out.copy_(x)
    assert out.data_ptr() % 16 == 2
    return out


def run(W, x, K, rms_eps=None, cuda_cores=False):
    N, ldw = W.shape
    buf, y = gu.guarded_y(1, N)
    binding.gemv_bf16_ex(W, x, y, N, K, 1, ldw, rms_eps=rms_eps, cuda_cores=cuda_cores)
    torch.cuda.synchronize()
    gu.check_guards(buf)
    return y.cpu().numpy()


@pytest.mark.parametrize("N,K,mcast", [(4096, 14336, 2), (4097, 8199, 2), (1024, 14336, 2), (17, 16384, 2),
                                       (4096, 4096, 1), (9, 40960, 1)])
def test_multicast_matches_per_cta_staging_and_oracle(N, K, mcast):
    q = binding.gemv_query_launch(N, K, 1, sms())
    assert q["mcast"] == mcast, q
    ldw = inputs.padded_ldw(K)
    W = inputs.weight(N, K, ldw, seed=N + K, device=DEV)
    x = inputs.activations(1, K, seed=K, device=DEV)
    assert x.data_ptr() % 16 == 0
    binding.gemv_device_status(reset=True)
    y = run(W, x, K)
    y_fallback = run(W, shifted(x), K)
    assert np.array_equal(y.view(np.uint32), y_fallback.view(np.uint32))
    y_ref, s = gu.reference(W, x, K)
    gu.assert_parity(y, y_ref, s, f"multicast={q['mcast']} N={N} K={K}")
    assert binding.gemv_device_status(reset=True) == 0


def test_multicast_is_planned_for_long_x_only():
    q = binding.gemv_query_launch(4096, 14336, 1, sms())          # down_proj: x of 28 KB
    assert q["mcast"] == 2 and q["grid"] % 2 == 0, q
    for N, K in [(4096, 4096), (1024, 4096), (6144, 4096), (28672, 4096), (128256, 4096)]:
        assert binding.gemv_query_launch(N, K, 1, sms())["mcast"] == 1, (N, K)


def test_multicast_with_rmsnorm_and_segments():
    K, rows, eps = 14336, [4096, 1024, 1024, 7], 1e-5
    Ws = [inputs.weight(n, K, seed=30 + i, device=DEV) for i, n in enumerate(rows)]
    x = inputs.activations(1, K, seed=31, device=DEV)
    for xx in (x, shifted(x)):
        ys = [torch.full((1, n), float("nan"), device=DEV) for n in rows]
        binding.gemv_bf16_multi_ex([(W, y, n, K) for W, y, n in zip(Ws, ys, rows)], xx, K, 1, rms_eps=eps)
        torch.cuda.synchronize()
        if xx is x:
            first = [y.cpu().numpy() for y in ys]
        else:
            for a, y in zip(first, ys):
                assert np.array_equal(a.view(np.uint32), y.cpu().numpy().view(np.uint32))
    for W, a in zip(Ws, first):
        y_ref, s, _ = oracle.gemv_rmsnorm(inputs.bits(W), inputs.bits(x), eps, K, threads=oracle.default_threads())
        gu.assert_parity(a, y_ref, s, "segment with RMSNorm")
    assert binding.gemv_device_status(reset=True) == 0


def test_multicast_back_to_back_in_a_captured_graph():
    # the decode-step use: the same calls replayed from a graph, x updated in place
    N, K = 4096, 14336
    ldw = inputs.padded_ldw(K)
    W = inputs.weight(N, K, ldw, seed=5, device=DEV)
    x = inputs.activations(1, K, seed=6, device=DEV)
    y = torch.full((1, N), float("nan"), device=DEV)
    plan = binding.Plan([(W, x, y, N, K, ldw, 1, 0)] * 3, keepalive=(W, x, y))
    s = torch.cuda.Stream()
    plan.capture(s)
    for seed in (7, 8):
        x.copy_(inputs.activations(1, K, seed=seed, device=DEV))
        torch.cuda.synchronize()
        plan.launch(s)
        s.synchronize()
        y_ref, sc = gu.reference(W, x, K)
        gu.assert_parity(y.cpu().numpy(), y_ref, sc, f"graph replay, x seed {seed}")
    assert binding.gemv_device_status(reset=True) == 0


def test_multicast_only_from_device_memory_and_under_capture():
    # x in pinned host memory (mapped, reachable by the GPU): the per-CTA
    # staging serves it, with the same bits as device-resident x
    N, K = 4096, 14336
    ldw = inputs.padded_ldw(K)
    W = inputs.weight(N, K, ldw, seed=9, device=DEV)
    x = inputs.activations(1, K, seed=10, device=DEV)
    y_dev = run(W, x, K)
    x_host = x.cpu().pin_memory()
    y_host = run(W, x_host, K)
    assert np.array_equal(y_dev.view(np.uint32), y_host.view(np.uint32))
    # a direct call captured into a CUDA graph (the pointer query runs during capture)
    y = torch.full((1, N), float("nan"), device=DEV)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        binding.gemv_bf16(W, x, y, N, K, 1, ldw, s.cuda_stream)
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(y.cpu().numpy().view(np.uint32), y_dev.view(np.uint32))
    assert binding.gemv_device_status(reset=True) == 0


@pytest.mark.parametrize("B", [2, 5, 8, 16])
@pytest.mark.parametrize("N,K", [(4096, 14336), (1000, 4096), (300, 12288)])
def test_tensor_core_bulk_x_copy(monkeypatch, N, K, B):
    """Batches of 2..16 on the register-fed tensor-core kernel copy x into
    shared memory with bulk copies (or tensor boxes) when x is 16-byte aligned
    device memory of this GPU and K is a multiple of 8; x in pinned host memory
    takes the per-thread staging. Same bits either way, both against the
    oracle, and no wait ran out. (The tcgen05 kernel, which would take the
    device-memory call at B = 16, is switched off here.)"""
    monkeypatch.setenv("GEMV_FORCE_VARIANT", "tc=0")
    ldw = inputs.padded_ldw(K)
    W = inputs.weight(N, K, ldw, seed=N + B, device=DEV)
    x = inputs.activations(B, K, seed=K + B, device=DEV)

    def run_b(xx):
        buf, y = gu.guarded_y(B, N)
        binding.gemv_bf16(W, xx, y, N, K, B, ldw)
        torch.cuda.synchronize()
        gu.check_guards(buf)
        return y.cpu().numpy()

    y_dev = run_b(x)
    y_host = run_b(x.cpu().pin_memory())
    assert np.array_equal(y_dev.view(np.uint32), y_host.view(np.uint32))
    y_ref, sc = gu.reference(W, x, K)
    gu.assert_parity(y_dev, y_ref, sc, f"bulk x N={N} K={K} B={B}")
    assert binding.gemv_device_status(reset=True) == 0
