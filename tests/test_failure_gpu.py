"""The failure path of the tcgen05 kernels, made to run on purpose without a
fault: a test build (GEMV_DEBUG_DROP_X) never issues the copies of x, so every
stage's mbarrier waits for bytes that never come; the bounded waits run out
(2^14 try_wait rounds in that build), and the kernel stores NaN, sets the
status bit the host reads with gemv_device_status, waits for the copies it did
issue and frees its tensor memory. The context stays usable: the regular
library computes correct results right after, in the same process."""
import numpy as np
import pytest
import torch

from memory_bound_decode_gb300 import binding, build_lib, inputs
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def drop_x_lib():
    return build_lib.build_debug_drop_x()


@pytest.mark.parametrize("N,K,B", [(1000, 4096, 16), (128256, 512, 9)])
def test_tc_wait_runs_out_and_reports(drop_x_lib, monkeypatch, N, K, B):
    monkeypatch.setenv("GEMV_FORCE_VARIANT", "tc=1")
    W = inputs.weight(N, K, seed=1, device=DEV)
    x = inputs.activations(B, K, seed=2, device=DEV)
    binding.gemv_device_status(reset=True)
    with binding.use_library(drop_x_lib):
        binding.gemv_device_status(reset=True)
        q = binding.gemv_query_launch(N, K, B, torch.cuda.get_device_properties(0).multi_processor_count)
        assert q["path"] == 5, q
        y = torch.zeros((B, N), device=DEV)
        binding.gemv_bf16(W, x, y, N, K, B, W.shape[1])   # returns GEMV_OK: the launch itself is fine
        torch.cuda.synchronize()
        assert torch.isnan(y).all(), "a CTA whose wait ran out must not store a plausible number"
        assert binding.gemv_device_status(reset=True) & binding.GEMV_STATUS_WAIT_TIMEOUT
        assert binding.gemv_device_status(reset=True) == 0   # cleared by the read
    # the same context, the regular library: correct results
    y2 = gu.gemv(W, x, K)
    y_ref, s = gu.reference(W, x, K)
    gu.assert_parity(y2, y_ref, s, "after a timed-out launch")
    assert binding.gemv_device_status(reset=True) == 0
