"""The tcgen05 kernel (path 5: W streamed by tensor copies through a
shared-memory ring, tcgen05.mma with the accumulator in tensor memory),
selected with GEMV_FORCE_VARIANT=tc=1, against the FP64 oracle element by
element: ragged rows and columns, K-slices of unequal length, every batch
size it serves, padded W rows (NaN padding must never enter a sum), and a
CUDA-graph plan."""
import pytest
import torch

from memory_bound_decode_gb300 import binding, inputs
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


@pytest.mark.parametrize("stages", ["2", "3", "4", "5", "2,tccols=64", "3,tccols=64", "4,tccols=64", "8,tccols=64",
                                    "10,tccols=64", "2,l2pf=2", "4,tccols=64,l2pf=4"])
@pytest.mark.parametrize("N,K,B", [
    (4096, 14336, 16), (4096, 14336, 2), (4096, 4096, 16), (6144, 4096, 16), (1024, 4096, 8),
    (4097, 4104, 9), (333, 8192, 13), (64, 65536, 16), (129, 136, 3), (7, 8, 2), (2000, 12288, 5),
    (4096, 14336, 11),
])
def test_tc_parity(monkeypatch, N, K, B, stages):
    monkeypatch.setenv("GEMV_FORCE_VARIANT", f"tc=1,tcstages={stages}")
    q = binding.gemv_query_launch(N, K, B, _sms())
    assert q["path"] == 5, q
    W = inputs.weight(N, K, seed=N + K + B, device=DEV)
    x = inputs.activations(B, K, seed=B + 7, device=DEV)
    y = gu.gemv(W, x, K)
    y_ref, s = gu.reference(W, x, K)
    gu.assert_parity(y, y_ref, s, f"tc N={N} K={K} B={B} launch={q}")
    assert binding.gemv_device_status(reset=True) == 0


@pytest.mark.parametrize("split", ["1x1", "1x2", "1x8"])
def test_tc_forced_splits(monkeypatch, split):
    monkeypatch.setenv("GEMV_FORCE_VARIANT", "tc=1")
    monkeypatch.setenv("GEMV_FORCE_SPLIT", split)
    N, K, B = 2048, 8192, 16
    q = binding.gemv_query_launch(N, K, B, _sms())
    assert q["path"] == 5 and q["splits"] == int(split.split("x")[1]), q
    W = inputs.weight(N, K, seed=3, device=DEV)
    x = inputs.activations(B, K, seed=4, device=DEV)
    y = gu.gemv(W, x, K)
    y_ref, s = gu.reference(W, x, K)
    gu.assert_parity(y, y_ref, s, f"tc {split}")


def test_tc_integer_inputs_exact(monkeypatch):
    """Small integers: every product and partial sum is exact in FP32, so the
    tensor-core result must equal the oracle's exactly."""
    monkeypatch.setenv("GEMV_FORCE_VARIANT", "tc=1")
    N, K, B = 1000, 4096, 16
    W = inputs.int_weight(N, K, seed=5, device=DEV)
    x = inputs.int_activations(B, K, seed=6, device=DEV)
    y = gu.gemv(W, x, K)
    y_ref, _ = gu.reference(W, x, K)
    assert (y == y_ref).all()


def test_tc_host_x_falls_back():
    """x in pinned host memory: the tcgen05 kernel's tensor copies read this
    GPU's memory only, so the call takes the register-fed kernel; both results
    match the oracle."""
    N, K, B = 4096, 14336, 16
    assert binding.gemv_query_launch(N, K, B, _sms())["path"] == 5
    W = inputs.weight(N, K, seed=8, device=DEV)
    x = inputs.activations(B, K, seed=9, device=DEV)
    y_ref, s = gu.reference(W, x, K)
    gu.assert_parity(gu.gemv(W, x, K), y_ref, s, "device x")
    gu.assert_parity(gu.gemv(W, x.cpu().pin_memory(), K), y_ref, s, "host x")
    assert binding.gemv_device_status(reset=True) == 0


@pytest.mark.parametrize("stages", ["", "tcstages=3", "tcstages=4,tc=1"])
@pytest.mark.parametrize("N,K,B", [(128256, 4096, 16), (60000, 1024, 9), (58600, 520, 16), (58369, 136, 12)])
def test_tc_persistent_parity(monkeypatch, N, K, B, stages):
    """More row tiles than one wave: the persistent grid (each CTA an equal
    share of the tiles, the accumulator alternating between two halves of
    tensor memory) against the oracle, ragged rows and columns included, for
    each ring the persistent form has."""
    monkeypatch.setenv("GEMV_FORCE_VARIANT", stages)
    q = binding.gemv_query_launch(N, K, B, _sms())
    assert q["path"] == 5 and q["persistent"] == 1, q
    W = inputs.weight(N, K, seed=N + B, device=DEV)
    x = inputs.activations(B, K, seed=B + 1, device=DEV)
    y = gu.gemv(W, x, K)
    y_ref, s = gu.reference(W, x, K)
    gu.assert_parity(y, y_ref, s, f"tc persistent N={N} K={K} B={B} launch={q}")
    assert binding.gemv_device_status(reset=True) == 0
