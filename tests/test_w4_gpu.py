"""INT4-weight GEMV (gemv_w4_bf16) against the CPU oracle, element by element:
|y - y_ref| <= 1e-5 * sum_k |(u - 8) * scale * x|, y finite, guard bands intact.
Power-of-two scales with integer x make every partial sum exact, so those cases
are compared bit for bit."""
import numpy as np
import pytest
import torch

from memory_bound_decode_gb300 import binding, inputs
from oracle import oracle
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu
DEV = "cuda"


def run_w4(Wq, S, x, N, K, rms_eps=None):
    B = x.shape[0]
    buf, y = gu.guarded_y(B, N)
    binding.gemv_w4_bf16(Wq, S, x, y, N, K, B, Wq.shape[1], S.shape[1], rms_eps=rms_eps)
    torch.cuda.synchronize()
    gu.check_guards(buf)
    return y.cpu().numpy()


def host_case(N, K, B, seed, ldq=None, lds=None, scales=None, int_x=False):
    Wq, S, u = inputs.w4_weight(N, K, ldq, lds, seed=seed, scales=scales)
    x = inputs.int_activations(B, K, lo=-3, hi=3, seed=seed) if int_x else inputs.activations(B, K, seed=seed)
    return torch.from_numpy(Wq).to(DEV), S.to(DEV), x.to(DEV), Wq, inputs.bits(S), inputs.bits(x)


@pytest.mark.parametrize("B", [1, 2, 3, 8, 16])
@pytest.mark.parametrize("N,K", [(7, 128), (300, 1280), (4097, 4096), (33, 65536), (1024, 4096), (1, 8192)])
def test_w4_parity(N, K, B):
    Wq, S, x, Wq_h, S_h, x_h = host_case(N, K, B, seed=N + K + B)
    y = run_w4(Wq, S, x, N, K)
    y_ref, s = oracle.gemv_w4(Wq_h, S_h, x_h, K, threads=oracle.default_threads())
    gu.assert_parity(y, y_ref, s, f"w4 N={N} K={K} B={B}")


@pytest.mark.parametrize("N,K,B,ldq,lds", [(64, 1024, 2, 528, 9), (17, 256, 16, 256, 4)])
def test_w4_wide_strides(N, K, B, ldq, lds):
    Wq, S, x, Wq_h, S_h, x_h = host_case(N, K, B, seed=5, ldq=ldq, lds=lds)
    y = run_w4(Wq, S, x, N, K)
    y_ref, s = oracle.gemv_w4(Wq_h, S_h, x_h, K)
    gu.assert_parity(y, y_ref, s)


@pytest.mark.parametrize("N,K,B", [(4096, 14336, 1), (28672, 4096, 1), (4096, 14336, 16), (33, 65536, 3)])
def test_w4_exact_with_power_of_two_scales(N, K, B):
    G = K // inputs.W4_GROUP
    scales = 2.0 ** (np.add.outer(np.arange(N), np.arange(G)) % 4 - 2)
    Wq, S, x, Wq_h, S_h, x_h = host_case(N, K, B, seed=6, scales=scales, int_x=True)
    y = run_w4(Wq, S, x, N, K)
    y_ref, _ = oracle.gemv_w4(Wq_h, S_h, x_h, K, threads=oracle.default_threads())
    assert np.array_equal(y.astype(np.float64), y_ref)


def test_w4_full_size_down_proj():
    N, K = 4096, 14336
    Wq, S, x, Wq_h, S_h, x_h = host_case(N, K, 1, seed=7)
    y = run_w4(Wq, S, x, N, K)
    y_ref, s = oracle.gemv_w4(Wq_h, S_h, x_h, K, threads=oracle.default_threads())
    gu.assert_parity(y, y_ref, s, "w4 down_proj")
    y2 = run_w4(Wq, S, x, N, K)
    assert np.array_equal(y.view(np.uint32), y2.view(np.uint32))


def test_w4_rmsnorm():
    N, K, B = 2048, 4096, 4
    Wq, S, x, Wq_h, S_h, x_h = host_case(N, K, B, seed=8)
    eps = 1e-5
    y = run_w4(Wq, S, x, N, K, rms_eps=eps)
    y_ref, s = oracle.gemv_w4(Wq_h, S_h, x_h, K, threads=oracle.default_threads())
    xd = inputs.from_bits(x_h).double().numpy()
    r = 1.0 / np.sqrt(np.mean(xd * xd, axis=1) + eps)
    gu.assert_parity(y, y_ref * r[:, None], s * r[:, None], "w4 rmsnorm")


def test_w4_device_packer_matches_layout():
    """The device-side generator produces the documented layout (checked through
    the oracle on a slice)."""
    N, K = 64, 1024
    Wq, S = inputs.w4_weight_device(N, K, seed=9, device=DEV)
    x = inputs.activations(2, K, seed=9, device=DEV)
    y = run_w4(Wq, S, x, N, K)
    y_ref, s = oracle.gemv_w4(Wq.cpu().numpy(), inputs.bits(S), inputs.bits(x), K)
    gu.assert_parity(y, y_ref, s)
