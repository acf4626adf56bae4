"""The RMSNorm prologue (gemv_bf16_ex / gemv_bf16_multi_ex / plans with
GEMV_FLAG_RMSNORM) against the CPU oracle: y[b][n] = r_b * sum_k W[n][k] x[b][k],
r_b = (mean_k x[b][k]^2 + eps)^(-1/2), compared element by element within
1e-5 * r_b * sum_k |W[n][k] x[b][k]|."""
import numpy as np
import pytest
import torch

from memory_bound_decode_gb300 import binding, inputs
from oracle import oracle
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu
DEV = "cuda"
EPS = 1e-5


def run_ex(W, x, K, eps, stream=None):
    N, ldw = W.shape
    B = x.shape[0]
    buf, y = gu.guarded_y(B, N)
    binding.gemv_bf16_ex(W, x, y, N, K, B, ldw, rms_eps=eps, stream=stream)
    torch.cuda.synchronize()
    gu.check_guards(buf)
    return y.cpu().numpy()


def reference(W, x, K, eps):
    y, s, _ = oracle.gemv_rmsnorm(inputs.bits(W), inputs.bits(x), eps, K, threads=oracle.default_threads())
    return y, s


@pytest.mark.parametrize("B", [1, 2, 5, 16])
@pytest.mark.parametrize("N,K", [(7, 129), (4097, 4103), (33, 65537), (1024, 4096), (4096, 14336), (3, 8)])
def test_rmsnorm_parity(N, K, B):
    """Single-chunk, chunked (B = 16 with long K) and cluster-split (33 x 65537) instances."""
    ldw = inputs.padded_ldw(K)
    W = inputs.weight(N, K, ldw, seed=N + B, device=DEV)
    x = inputs.activations(B, K, seed=K + B, device=DEV)
    y = run_ex(W, x, K, EPS)
    y_ref, s = reference(W, x, K, EPS)
    gu.assert_parity(y, y_ref, s, f"rmsnorm N={N} K={K} B={B}")


def test_rmsnorm_is_the_plain_gemv_times_r():
    N, K, B = 2048, 5000, 3
    W = inputs.weight(N, K, seed=1, device=DEV)
    x = (inputs.activations(B, K, seed=2, device=DEV).float() * 3.0).to(torch.bfloat16)
    y_plain = gu.gemv(W, x, K).astype(np.float64)
    y_norm = run_ex(W, x, K, 0.5).astype(np.float64)
    xd = x.double().cpu().numpy()
    r = 1.0 / np.sqrt(np.mean(xd * xd, axis=1) + 0.5)
    assert np.allclose(y_norm, y_plain * r[:, None], rtol=1e-5, atol=1e-6)


def test_rmsnorm_deterministic_and_scale_free():
    N, K, B = 4096, 14336, 2
    W = inputs.weight(N, K, seed=3, device=DEV)
    x = inputs.activations(B, K, seed=3, device=DEV)
    y1 = run_ex(W, x, K, 0.0)
    y2 = run_ex(W, x, K, 0.0)
    assert np.array_equal(y1.view(np.uint32), y2.view(np.uint32))
    # eps = 0: RMSNorm removes any power-of-two scale of x, bit for bit
    y4 = run_ex(W, (x.float() * 4.0).to(torch.bfloat16), K, 0.0)
    assert np.array_equal(y4, y1)


def test_rmsnorm_fused_segments():
    rows, K, B = (4096, 1024, 1024), 4096, 1
    ldw = inputs.padded_ldw(K)
    Ws = [inputs.weight(n, K, ldw, seed=30, index=i, device=DEV) for i, n in enumerate(rows)]
    x = inputs.activations(B, K, seed=31, device=DEV)
    ys = [gu.guarded_y(B, n) for n in rows]
    binding.gemv_bf16_multi_ex([(W, y, n, ldw) for W, (_, y), n in zip(Ws, ys, rows)], x, K, B, rms_eps=EPS)
    torch.cuda.synchronize()
    for W, (buf, y), n in zip(Ws, ys, rows):
        gu.check_guards(buf)
        y_ref, s = reference(W, x, K, EPS)
        gu.assert_parity(y.cpu().numpy(), y_ref, s, f"segment {n}")


def test_rmsnorm_in_a_plan():
    """QKV and gate/up read the normalised x, o_proj the raw one: three launches."""
    K = 512
    ldw = K
    x = inputs.activations(1, K, seed=40, device=DEV)
    Wq, Wk, Wo, Wg = (inputs.weight(n, K, ldw, seed=41, index=i, device=DEV)
                      for i, n in enumerate((512, 128, 512, 1536)))
    ys = [torch.empty((1, W.shape[0]), device=DEV) for W in (Wq, Wk, Wo, Wg)]
    projs = [(Wq, x, ys[0], 512, K, ldw, 1, 1, EPS), (Wk, x, ys[1], 128, K, ldw, 1, 1, EPS),
             (Wo, x, ys[2], 512, K, ldw, 1, 0), (Wg, x, ys[3], 1536, K, ldw, 1, 2, EPS)]
    plan = binding.Plan(projs)
    assert plan.num_launches() == 3
    s = torch.cuda.Stream()
    plan.capture(s)
    plan.launch(s)
    s.synchronize()
    for (W, _, y, *_rest), norm in zip(projs, (True, True, False, True)):
        if norm:
            y_ref, sc = reference(W, x, K, EPS)
        else:
            y_ref, sc = gu.reference(W, x, K)
        gu.assert_parity(y.cpu().numpy(), y_ref, sc)
    plan.destroy()
