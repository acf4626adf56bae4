"""The planner's sweep knobs (GEMV_FORCE_SPLIT, GEMV_FORCE_VARIANT) force
launch shapes the rules never pick; every forced shape must still match the
FP64 oracle element by element, with y's guard bands intact."""
import numpy as np
import pytest
import torch

from memory_bound_decode_gb300 import binding, inputs
from oracle import oracle
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


@pytest.mark.parametrize("knobs", [
    {"GEMV_FORCE_SPLIT": "1x1"}, {"GEMV_FORCE_SPLIT": "8x1"}, {"GEMV_FORCE_SPLIT": "2x4"},
    {"GEMV_FORCE_SPLIT": "1x8"}, {"GEMV_FORCE_VARIANT": "mcast=1"}, {"GEMV_FORCE_VARIANT": "mcast=4"},
    {"GEMV_FORCE_VARIANT": "mcast=8"}, {"GEMV_FORCE_VARIANT": "streamk=1"},
    {"GEMV_FORCE_SPLIT": "4x1", "GEMV_FORCE_VARIANT": "mcast=2"},
])
@pytest.mark.parametrize("N,K,B", [(4096, 14336, 1), (4097, 8200, 1), (1000, 4096, 3), (300, 12288, 16)])
def test_forced_bf16_launches(monkeypatch, knobs, N, K, B):
    for k, v in knobs.items():
        monkeypatch.setenv(k, v)
    W = inputs.weight(N, K, seed=N + K, device=DEV)
    x = inputs.activations(B, K, seed=B, device=DEV)
    y = gu.gemv(W, x, K)
    y_ref, s = gu.reference(W, x, K)
    q = binding.gemv_query_launch_ex(N, K, B, _sms(), 0)
    gu.assert_parity(y, y_ref, s, f"{knobs} N={N} K={K} B={B} launch={q}")
    assert binding.gemv_device_status(reset=True) == 0


@pytest.mark.parametrize("knobs", [{"GEMV_FORCE_SPLIT": "1x1"}, {"GEMV_FORCE_SPLIT": "4x2"},
                                   {"GEMV_FORCE_VARIANT": "unroll=4"}, {"GEMV_FORCE_VARIANT": "unroll=8"}])
@pytest.mark.parametrize("kind", ["w4", "fp8"])
@pytest.mark.parametrize("N,K,B", [(4096, 14336, 1), (1000, 4096, 4)])
def test_forced_quantised_launches(monkeypatch, knobs, kind, N, K, B):
    for k, v in knobs.items():
        monkeypatch.setenv(k, v)
    x = inputs.activations(B, K, seed=K, device=DEV)
    y = torch.full((B, N), float("nan"), device=DEV)
    if kind == "w4":
        Wq, S = inputs.w4_weight_device(N, K, seed=N, device=DEV)
        binding.gemv_w4_bf16(Wq, S, x, y, N, K, B, Wq.shape[1], S.shape[1])
        y_ref, s = oracle.gemv_w4(Wq.cpu().numpy(), inputs.bits(S), inputs.bits(x), K,
                                  threads=oracle.default_threads())
    else:
        Wq, S = inputs.fp8_weight(N, K, seed=N, device=DEV)
        binding.gemv_fp8_bf16(Wq, S, x, y, N, K, B, Wq.shape[1])
        y_ref, s = oracle.gemv_fp8(Wq.cpu().numpy(), S.cpu().numpy(), inputs.bits(x), K,
                                   threads=oracle.default_threads())
    torch.cuda.synchronize()
    gu.assert_parity(y.cpu().numpy(), y_ref, s, f"{kind} {knobs} N={N} K={K} B={B}")
