"""The stream-K batch-1 kernel (GEMV_FLAG_STREAMK) through the C ABI against the
CPU oracle, element by element within 1e-5 * sum_k |W x|; integer-valued
inputs bit for bit. Shapes cover rows wholly inside one warp's range, rows cut
between two or more warps (one row of 8191 columns over four warps), ragged K,
fused segments, the RMSNorm prologue, plans, and back-to-back calls that reuse
the per-row counters (zero after every launch). The SM count is read from the
device, so the row counts that fill whole rounds of warps exactly assume a
152-SM GB300 (on another part they are ordinary shapes)."""
import numpy as np
import pytest
import torch

from memory_bound_decode_gb300 import binding, inputs
from oracle import oracle
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu
DEV = "cuda"

SMALL = [(7, 129), (1, 1), (3, 8), (1, 8191), (3, 2049), (5, 24576), (65, 300), (300, 2056),
         (4097, 4103), (17, 10000), (1024, 4096),
         # whole rounds of rows exactly (no split part), and one row more, for the
         # whole-unit (4 CTAs per SM) and the ragged (3 per SM) instances
         (4864, 4096), (4865, 4096), (3648, 4103), (3649, 4103), (9729, 2048)]
FULL = [("k_proj", 1024, 4096), ("down_proj", 4096, 14336), ("qkv", 6144, 4096),
        ("o_proj", 4096, 4096), ("gate_up", 28672, 4096), ("lm_head", 128256, 4096)]


def run_sk(W, x, K, rms_eps=None, stream=None):
    N, ldw = W.shape
    buf, y = gu.guarded_y(1, N)
    binding.gemv_bf16_ex(W, x, y, N, K, 1, ldw, rms_eps=rms_eps, stream=stream, streamk=True)
    torch.cuda.synchronize()
    gu.check_guards(buf)
    return y.cpu().numpy()


def make(N, K, seed):
    ldw = inputs.padded_ldw(K)
    return inputs.weight(N, K, ldw, seed=seed, device=DEV), inputs.activations(1, K, seed=seed, device=DEV)


@pytest.mark.parametrize("N,K", SMALL)
def test_streamk_parity_small(N, K):
    W, x = make(N, K, N + K)
    y = run_sk(W, x, K)
    y_ref, s = gu.reference(W, x, K)
    gu.assert_parity(y, y_ref, s, f"stream-K N={N} K={K}")


@pytest.mark.parametrize("name,N,K", FULL, ids=[f[0] for f in FULL])
def test_streamk_parity_full_size(name, N, K):
    W, x = make(N, K, 1)
    y = run_sk(W, x, K)
    y_ref, s = gu.reference(W, x, K)
    gu.assert_parity(y, y_ref, s, name)


@pytest.mark.parametrize("N,K", [(1, 8191), (4097, 4103), (6144, 4096), (128256, 4096)])
def test_streamk_integer_inputs_exact(N, K):
    ldw = inputs.padded_ldw(K)
    W = inputs.int_weight(N, K, ldw, seed=3, device=DEV)
    x = inputs.int_activations(1, K, seed=3, device=DEV)
    y = run_sk(W, x, K)
    y_ref, _ = gu.reference(W, x, K)
    assert np.array_equal(y.astype(np.float64), y_ref)


def test_streamk_one_hot_and_determinism():
    N, K = 4097, 4103
    W, x = make(N, K, 4)
    Wh = inputs.bits(W)
    for j in (0, 2047, 2048, K - 1):
        xo = torch.zeros((1, K), dtype=torch.bfloat16, device=DEV)
        xo[0, j] = 1.0
        col = inputs.from_bits(Wh[:, j]).float().numpy()
        assert np.array_equal(run_sk(W, xo, K)[0], col), j
    y1 = run_sk(W, x, K)
    y2 = run_sk(W, x, K)
    assert np.array_equal(y1.view(np.uint32), y2.view(np.uint32))


def test_streamk_back_to_back_shapes_reuse_counters():
    """Calls of different shapes in a row, without synchronizing, share the
    device workspace; every launch leaves its counters at zero."""
    shapes = [(4096, 14336), (1, 8191), (6144, 4096), (1, 8191), (4096, 14336)]
    data = [make(N, K, 10 + i) for i, (N, K) in enumerate(shapes)]
    ys = []
    for (N, K), (W, x) in zip(shapes, data):
        y = torch.full((1, N), float("nan"), device=DEV)
        binding.gemv_bf16_ex(W, x, y, N, K, 1, W.shape[1], streamk=True)
        ys.append(y)
    torch.cuda.synchronize()
    for (N, K), (W, x), y in zip(shapes, data, ys):
        y_ref, s = gu.reference(W, x, K)
        gu.assert_parity(y.cpu().numpy(), y_ref, s, f"N={N} K={K}")


def test_streamk_segments():
    K = 4096
    rows = [4096, 1024, 1024]
    Ws = [inputs.weight(n, K, seed=20 + i, device=DEV) for i, n in enumerate(rows)]
    x = inputs.activations(1, K, seed=21, device=DEV)
    ys = [torch.full((1, n), float("nan"), device=DEV) for n in rows]
    binding.gemv_bf16_multi_ex([(W, y, n, K) for W, y, n in zip(Ws, ys, rows)], x, K, 1, streamk=True)
    torch.cuda.synchronize()
    for W, y in zip(Ws, ys):
        y_ref, s = gu.reference(W, x, K)
        gu.assert_parity(y.cpu().numpy(), y_ref, s, "segment")


def test_streamk_ragged_segments():
    K = 4103
    ldw = inputs.padded_ldw(K)
    rows = [5, 4097, 1, 300]
    Ws = [inputs.weight(n, K, ldw, seed=30 + i, device=DEV) for i, n in enumerate(rows)]
    x = inputs.activations(1, K, seed=31, device=DEV)
    ys = [torch.full((1, n), float("nan"), device=DEV) for n in rows]
    binding.gemv_bf16_multi_ex([(W, y, n, ldw) for W, y, n in zip(Ws, ys, rows)], x, K, 1, streamk=True)
    torch.cuda.synchronize()
    for W, y in zip(Ws, ys):
        y_ref, s = gu.reference(W, x, K)
        gu.assert_parity(y.cpu().numpy(), y_ref, s, "ragged segment")


@pytest.mark.parametrize("N,K", [(1, 8191), (4096, 14336), (6144, 4096)])
def test_streamk_rmsnorm(N, K):
    W, x = make(N, K, 40)
    y = run_sk(W, x, K, rms_eps=1e-5)
    y_ref, s, _ = oracle.gemv_rmsnorm(inputs.bits(W), inputs.bits(x), 1e-5, K, threads=oracle.default_threads())
    gu.assert_parity(y, y_ref, s, "stream-K rmsnorm")


def test_streamk_plan_mixed_with_default_launches():
    K = 4096
    W1, x1 = make(6144, K, 50)
    W2, _ = make(4096, K, 51)
    W3, x3 = make(4096, 14336, 52)
    y1 = torch.full((1, 6144), float("nan"), device=DEV)
    y2 = torch.full((1, 4096), float("nan"), device=DEV)
    y3 = torch.full((1, 4096), float("nan"), device=DEV)
    plan = binding.Plan([(W1, x1, y1, 6144, K, K, 1, 0, None, True),
                         (W2, x1, y2, 4096, K, K, 1, 0, None, False),
                         (W3, x3, y3, 4096, 14336, 14336, 1, 0, 1e-5, True)])
    s = torch.cuda.Stream()
    plan.capture(s)
    for _ in range(3):
        y1.fill_(float("nan")); y2.fill_(float("nan")); y3.fill_(float("nan"))
        torch.cuda.synchronize()
        plan.launch(s)
        s.synchronize()
        for W, x, y in ((W1, x1, y1), (W2, x1, y2)):
            y_ref, sc = gu.reference(W, x, K)
            gu.assert_parity(y.cpu().numpy(), y_ref, sc, "plan")
        y_ref, sc, _ = oracle.gemv_rmsnorm(inputs.bits(W3), inputs.bits(x3), 1e-5, 14336,
                                           threads=oracle.default_threads())
        gu.assert_parity(y3.cpu().numpy(), y_ref, sc, "plan rmsnorm")
    plan.destroy()


def test_streamk_workspace_release_and_capture_refusal():
    N, K = 4096, 4096
    W, x = make(N, K, 60)
    torch.cuda.synchronize()
    binding.gemv_workspace_release()
    y = torch.full((1, N), float("nan"), device=DEV)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        y.add_(0.0)
        rc = binding.gemv_bf16_ex(W, x, y, N, K, 1, K, streamk=True, stream=s, check=False)
    assert rc == binding.GEMV_ERR_CAPTURE
    del g
    # outside capture the workspace is allocated again
    y2 = run_sk(W, x, K)
    y_ref, sc = gu.reference(W, x, K)
    gu.assert_parity(y2, y_ref, sc, "after release")


@pytest.mark.parametrize("N,K,B", [(100, 4096, 2), (10, 65537, 1)])
def test_streamk_unsupported_shapes(N, K, B):
    ldw = inputs.padded_ldw(K)
    W = inputs.weight(N, K, ldw, seed=1, device=DEV)
    x = inputs.activations(B, K, seed=1, device=DEV)
    y = torch.empty((B, N), device=DEV)
    rc = binding.gemv_bf16_ex(W, x, y, N, K, B, ldw, streamk=True, check=False)
    assert rc == binding.GEMV_ERR_UNSUPPORTED


def test_streamk_host_io():
    N, K = 4096, 14336
    W, x = make(N, K, 70)
    x_host = x.cpu().pin_memory()
    y_host = torch.full((1, N), float("nan")).pin_memory()
    binding.gemv_bf16_host_io(W, x_host, y_host, torch.empty_like(x), torch.empty((1, N), device=DEV),
                              N, K, 1, K, streamk=True)
    y_ref, sc = gu.reference(W, x, K)
    gu.assert_parity(y_host.numpy(), y_ref, sc, "host io")
