"""The CUDA-core kernel at every batch size (GEMV_FLAG_CUDA_CORES: lanes along
K, FP32 multiply-adds, B accumulators per row), against the CPU oracle element
by element; integer inputs bit for bit; fused segments and the RMSNorm
prologue on the same path."""
import numpy as np
import pytest
import torch

from memory_bound_decode_gb300 import binding, inputs
from oracle import oracle
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu
DEV = "cuda"


def run_cc(W, x, K, rms_eps=None):
    N, ldw = W.shape
    B = x.shape[0]
    buf, y = gu.guarded_y(B, N)
    binding.gemv_bf16_ex(W, x, y, N, K, B, ldw, rms_eps=rms_eps, cuda_cores=True)
    torch.cuda.synchronize()
    gu.check_guards(buf)
    return y.cpu().numpy()


def make(N, K, B, seed):
    ldw = inputs.padded_ldw(K)
    return inputs.weight(N, K, ldw, seed=seed, device=DEV), inputs.activations(B, K, seed=seed, device=DEV)


@pytest.mark.parametrize("B", [2, 3, 4, 8, 9, 16])
@pytest.mark.parametrize("N,K", [(7, 129), (3, 8), (65, 300), (300, 2056), (1, 8191), (4097, 4103),
                                 (33, 65537), (1024, 4096)])
def test_cuda_cores_parity(N, K, B):
    W, x = make(N, K, B, seed=N + K + B)
    y = run_cc(W, x, K)
    y_ref, s = gu.reference(W, x, K)
    gu.assert_parity(y, y_ref, s, f"cuda cores N={N} K={K} B={B}")


@pytest.mark.parametrize("B", [4, 16])
def test_cuda_cores_full_size(B):
    W, x = make(4096, 14336, B, seed=3)
    y = run_cc(W, x, 14336)
    y_ref, s = gu.reference(W, x, 14336)
    gu.assert_parity(y, y_ref, s, f"4096x14336 B={B}")


@pytest.mark.parametrize("N,K,B", [(4097, 4103, 5), (33, 65537, 16), (128256, 4096, 2)])
def test_cuda_cores_integer_exact(N, K, B):
    ldw = inputs.padded_ldw(K)
    W = inputs.int_weight(N, K, ldw, seed=4, device=DEV)
    x = inputs.int_activations(B, K, seed=4, device=DEV)
    y = run_cc(W, x, K)
    y_ref, _ = gu.reference(W, x, K)
    assert np.array_equal(y.astype(np.float64), y_ref)


def test_cuda_cores_segments_and_rmsnorm():
    K, rows, B = 4096, [4096, 1024, 1024], 4
    Ws = [inputs.weight(n, K, seed=10 + i, device=DEV) for i, n in enumerate(rows)]
    x = inputs.activations(B, K, seed=11, device=DEV)
    ys = [torch.full((B, n), float("nan"), device=DEV) for n in rows]
    binding.gemv_bf16_multi_ex([(W, y, n, K) for W, y, n in zip(Ws, ys, rows)], x, K, B, rms_eps=1e-5,
                               cuda_cores=True)
    torch.cuda.synchronize()
    for W, y in zip(Ws, ys):
        y_ref, s, _ = oracle.gemv_rmsnorm(inputs.bits(W), inputs.bits(x), 1e-5, K, threads=oracle.default_threads())
        gu.assert_parity(y.cpu().numpy(), y_ref, s, "segment")


def test_cuda_cores_match_tensor_cores_within_tolerance():
    N, K, B = 2048, 5000, 8
    W, x = make(N, K, B, seed=12)
    y_cc = run_cc(W, x, K)
    y_tc = gu.gemv(W, x, K)
    _, s = gu.reference(W, x, K)
    assert np.all(np.abs(y_cc.astype(np.float64) - y_tc) <= 2e-5 * s)
