"""FP8-weight GEMV (gemv_fp8_bf16) against the CPU oracle, element by element:
|y - y_ref| <= 1e-5 * sum_k |e4m3(code) * S[n] * x|, y finite, guard bands
intact. The padding columns of every W hold the E4M3 NaN code and must never be
read. Integer-valued codes with power-of-two row scales and integer x make
every partial sum exact, so those cases, and one-hot x over all 254 finite
codes (normal and subnormal), are compared bit for bit."""
import numpy as np
import pytest
import torch

from memory_bound_decode_gb300 import binding, inputs
from oracle import oracle
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu
DEV = "cuda"


def run_fp8(Wq, S, x, N, K, rms_eps=None):
    B = x.shape[0]
    buf, y = gu.guarded_y(B, N)
    binding.gemv_fp8_bf16(Wq, S, x, y, N, K, B, Wq.shape[1], rms_eps=rms_eps)
    torch.cuda.synchronize()
    gu.check_guards(buf)
    return y.cpu().numpy()


def case(N, K, B, seed, ldq=None, device=DEV):
    Wq, S = inputs.fp8_weight(N, K, ldq, seed=seed, index=0, device=device)
    x = inputs.activations(B, K, seed=seed, index=1, device=device)
    return Wq, S, x


def reference(Wq, S, x, K):
    return oracle.gemv_fp8(Wq.cpu().numpy(), S.cpu().numpy(), inputs.bits(x), K,
                           threads=oracle.default_threads())


@pytest.mark.parametrize("B", [1, 2, 3, 8, 9, 16])
@pytest.mark.parametrize("N,K", [(7, 64), (1, 64), (17, 192), (5, 320), (300, 1280), (4097, 4096),
                                 (33, 65536), (1024, 4096)])
def test_fp8_parity(N, K, B):
    Wq, S, x = case(N, K, B, seed=N + K + B)
    y = run_fp8(Wq, S, x, N, K)
    y_ref, s = reference(Wq, S, x, K)
    gu.assert_parity(y, y_ref, s, f"fp8 N={N} K={K} B={B}")


@pytest.mark.parametrize("N,K,B,ldq", [(64, 1024, 2, 1536), (17, 256, 16, 272), (9, 640, 1, 656)])
def test_fp8_wide_row_stride(N, K, B, ldq):
    Wq, S, x = case(N, K, B, seed=5, ldq=ldq)
    assert torch.all(Wq[:, K:] == inputs.FP8_PAD)
    y = run_fp8(Wq, S, x, N, K)
    y_ref, s = reference(Wq, S, x, K)
    gu.assert_parity(y, y_ref, s)


@pytest.mark.parametrize("name,N,K,B", [("down_proj", 4096, 14336, 1), ("gate_up", 28672, 4096, 1),
                                        ("lm_head", 128256, 4096, 1), ("down_B8", 4096, 14336, 8),
                                        ("down_B16", 4096, 14336, 16)])
def test_fp8_full_size(name, N, K, B):
    Wq, S, x = case(N, K, B, seed=7)
    y = run_fp8(Wq, S, x, N, K)
    y_ref, s = reference(Wq, S, x, K)
    gu.assert_parity(y, y_ref, s, name)


@pytest.mark.parametrize("N,K,B", [(4096, 14336, 1), (300, 1280, 16), (33, 65536, 3), (28672, 4096, 1)])
def test_fp8_integer_codes_exact(N, K, B):
    g = torch.Generator().manual_seed(N + K)
    wi = torch.randint(-8, 9, (N, K), generator=g).to(torch.float32)     # exact in E4M3
    codes = wi.to(torch.float8_e4m3fn).view(torch.uint8)
    ldq = (K + 15) // 16 * 16
    Wq = torch.full((N, ldq), inputs.FP8_PAD, dtype=torch.uint8)
    Wq[:, :K] = codes
    S = (2.0 ** ((torch.arange(N) % 4) - 1)).to(torch.float32)
    x = inputs.int_activations(B, K, lo=-3, hi=3, seed=N)
    Wq, S, x = Wq.to(DEV), S.to(DEV), x.to(DEV)
    y = run_fp8(Wq, S, x, N, K)
    y_ref, _ = reference(Wq, S, x, K)
    assert np.array_equal(y.astype(np.float64), y_ref)


def test_fp8_every_finite_code_one_hot():
    """Row n holds code c_n in column j, so a one-hot x at column j gives
    e4m3(c_n) * S[n] exactly: all 254 finite codes, subnormals included."""
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    N, K = codes.size, 128
    rng = np.random.default_rng(3)
    Wq = np.full((N, K), inputs.FP8_PAD, dtype=np.uint8)
    for j in (0, 5, 77, 127):
        Wq[:, j] = rng.permutation(codes)
    S = (2.0 ** rng.integers(-3, 3, size=N)).astype(np.float32)
    Wq_d, S_d = torch.from_numpy(Wq).to(DEV), torch.from_numpy(S).to(DEV)
    for j in (0, 5, 77, 127):
        x = torch.zeros((1, K), dtype=torch.bfloat16, device=DEV)
        x[0, j] = 1.0
        Wj = Wq.copy()
        Wj[:, [c for c in range(K) if c != j]] = 0       # code 0 is +0: the rest of each row adds nothing
        y = run_fp8(torch.from_numpy(Wj).to(DEV), S_d, x, N, K)
        want = inputs.fp8_decode(Wq[:, j]) * S.astype(np.float64)
        assert np.array_equal(y[0].astype(np.float64), want), j
    del Wq_d


def test_fp8_rmsnorm():
    N, K, B = 4096, 14336, 2
    Wq, S, x = case(N, K, B, seed=9)
    y = run_fp8(Wq, S, x, N, K, rms_eps=1e-5)
    y_ref, s = reference(Wq, S, x, K)
    xd = x.double().cpu().numpy()
    r = 1.0 / np.sqrt(np.mean(xd * xd, axis=1) + 1e-5)
    gu.assert_parity(y, y_ref * r[:, None], s * r[:, None], "fp8 rmsnorm")


def test_fp8_deterministic():
    N, K, B = 4096, 14336, 1
    Wq, S, x = case(N, K, B, seed=10)
    y1 = run_fp8(Wq, S, x, N, K)
    y2 = run_fp8(Wq, S, x, N, K)
    assert np.array_equal(y1.view(np.uint32), y2.view(np.uint32))


def test_fp8_rejects_streamk_and_bad_k():
    Wq, S, x = case(64, 128, 1, seed=1)
    y = torch.empty((1, 64), device=DEV)
    opt = binding.gemv_options(binding.GEMV_FLAG_STREAMK, 0.0)
    assert binding.gemv_fp8_bf16(Wq, S, x, y, 64, 128, 1, 128, options=opt, check=False) == \
        binding.GEMV_ERR_UNSUPPORTED
    assert binding.gemv_fp8_bf16(Wq, S, x, y, 64, 96, 1, 128, check=False) == binding.GEMV_ERR_INVALID


@pytest.mark.parametrize("N,K,B", [(4096, 14336, 1), (1000, 4096, 4), (300, 12288, 16)])
def test_fp8_bulk_x_copy(N, K, B):
    """x in this GPU's memory, 16-byte aligned, is copied into shared memory by
    bulk copies; x in pinned host memory by per-thread copies. Same bits, both
    against the oracle, and no wait ran out."""
    Wq, S = inputs.fp8_weight(N, K, seed=N + B, device=DEV)
    x = inputs.activations(B, K, seed=K + B, device=DEV)

    def run_x(xx):
        buf, y = gu.guarded_y(B, N)
        binding.gemv_fp8_bf16(Wq, S, xx, y, N, K, B, Wq.shape[1])
        torch.cuda.synchronize()
        gu.check_guards(buf)
        return y.cpu().numpy()

    y_dev = run_x(x)
    y_host = run_x(x.cpu().pin_memory())
    assert np.array_equal(y_dev.view(np.uint32), y_host.view(np.uint32))
    y_ref, sc = oracle.gemv_fp8(Wq.cpu().numpy(), S.cpu().numpy(), inputs.bits(x), K,
                                threads=oracle.default_threads())
    gu.assert_parity(y_dev, y_ref, sc, f"fp8 bulk x N={N} K={K} B={B}")
    assert binding.gemv_device_status(reset=True) == 0
