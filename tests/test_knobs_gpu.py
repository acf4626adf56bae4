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
    {"GEMV_FORCE_VARIANT": "l2pf=0"}, {"GEMV_FORCE_VARIANT": "l2pf=4"},
    {"GEMV_FORCE_SPLIT": "2x2", "GEMV_FORCE_VARIANT": "l2pf=2"},
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
                                   {"GEMV_FORCE_VARIANT": "unroll=4"}, {"GEMV_FORCE_VARIANT": "unroll=8"},
                                   {"GEMV_FORCE_VARIANT": "l2pf=4"}, {"GEMV_FORCE_VARIANT": "unroll=8,l2pf=1"}])
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


@pytest.mark.parametrize("variant", ["tc=0", "tc=0,xbox=1", "tc=0,xbox=2", "tc=0,xbox=0", "tc=0,xpieces=1",
                                     "tc=0,xpieces=2", "tc=0,xpieces=3", "tc=0,xbox=2,xpieces=2"])
@pytest.mark.parametrize("N,K,B", [(4096, 14336, 16), (1000, 4096, 9), (333, 8192, 13), (4097, 4128, 16),
                                   (2048, 14368, 11), (64, 65536, 16)])
def test_x_as_tensor_boxes(monkeypatch, variant, N, K, B):
    """More than 8 rows of x on the tensor cores: x copied as narrow or wide
    tensor boxes in any number of pieces (or by row copies) gives the oracle's
    result; shapes with ragged rows, K a multiple of 32 but not of 256, K-slices
    of unequal length and odd batch sizes."""
    monkeypatch.setenv("GEMV_FORCE_VARIANT", variant)
    W = inputs.weight(N, K, seed=N + B, device=DEV)
    x = inputs.activations(B, K, seed=K + B, device=DEV)
    q = binding.gemv_query_launch(N, K, B, _sms())
    y = gu.gemv(W, x, K)
    y_ref, s = gu.reference(W, x, K)
    gu.assert_parity(y, y_ref, s, f"{variant} N={N} K={K} B={B} launch={q}")
    assert binding.gemv_device_status(reset=True) == 0
