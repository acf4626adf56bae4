"""gemv_bf16_streamk_noalloc (the stream-K GEMV on the library's fixed scratch)
against the FP64 oracle and against the existing entry point it mirrors,
gemv_bf16_ex with GEMV_FLAG_STREAMK, through the C ABI. Collected last (file name), and written
to pass alone as well: it depends on no state left by other tests (the fixed
scratch's counters are zero at load and after every launch)."""
import numpy as np
import pytest
import torch

from memory_bound_decode_gb300 import binding, inputs
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu
DEV = "cuda"
TICKETS, PART_FLOATS = 4096, 2 * 8192   # capacity stated in include/gemv.h


def fits(N, K):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    q = binding.gemv_query_launch_ex(N, K, 1, sms, binding.GEMV_FLAG_STREAMK)
    rest_rows = q["units"] // q["chunks"]
    return rest_rows <= TICKETS and 2 * q["warps"] <= PART_FLOATS


@pytest.mark.parametrize("N,K,eps", [(4096, 14336, None), (6144, 4096, None), (4097, 4103, None),
                                     (1, 8191, None), (4096, 4096, 1e-5), (128256, 4096, None)])
def test_noalloc_matches_streamk_entry_point_twice(N, K, eps):
    assert fits(N, K)
    ldw = inputs.padded_ldw(K)
    W = inputs.weight(N, K, ldw, seed=N, device=DEV)
    x = inputs.activations(1, K, seed=K, device=DEV)
    y_ref = torch.full((1, N), float("nan"), device=DEV)
    binding.gemv_bf16_ex(W, x, y_ref, N, K, 1, ldw, rms_eps=eps, streamk=True)
    bufs = [gu.guarded_y(1, N) for _ in range(2)]
    # two calls in a row on the same stream, no synchronization in between
    for _, y in bufs:
        binding.gemv_bf16_streamk_noalloc(W, x, y, N, K, ldw, rms_eps=eps)
    torch.cuda.synchronize()
    want = y_ref.cpu().numpy()
    y_or, scale = gu.reference(W, x, K)
    if eps is not None:
        xd = x.double().cpu().numpy()
        r = 1.0 / np.sqrt(np.mean(xd * xd) + eps)
        y_or, scale = y_or * r, scale * r
    for buf, y in bufs:
        gu.check_guards(buf)
        got = y.cpu().numpy()
        # against the FP64 oracle directly, element by element
        gu.assert_parity(got, y_or, scale, f"no-alloc N={N} K={K} against the oracle")
        assert np.all(np.abs(got.astype(np.float64) - want) <= 1e-5 * scale)
        # same kernel, same partition: the same bits
        assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


def test_noalloc_rejects_oversize_and_unsupported():
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    # a split part of more than 4,096 rows (N below one round of warps on a GB300)
    N, K = 4500, 4096
    W = inputs.weight(N, K, seed=1, device=DEV)
    x = inputs.activations(1, K, seed=1, device=DEV)
    y = torch.full((1, N), float("nan"), device=DEV)
    rc = binding.gemv_bf16_streamk_noalloc(W, x, y, N, K, K, check=False)
    if fits(N, K):
        assert rc == binding.GEMV_OK, sms
    else:
        assert rc == binding.GEMV_ERR_UNSUPPORTED
        torch.cuda.synchronize()
        assert torch.isnan(y).all()          # nothing was launched
    # x row too long for the stream-K kernel
    K2 = 24584
    W2 = inputs.weight(8, K2, seed=2, device=DEV)
    x2 = inputs.activations(1, K2, seed=2, device=DEV)
    rc = binding.gemv_bf16_streamk_noalloc(W2, x2, torch.empty((1, 8), device=DEV), 8, K2, W2.shape[1],
                                           check=False)
    assert rc == binding.GEMV_ERR_UNSUPPORTED
