"""Every output element is written exactly once and nothing else is written:
the test build of the library (GEMV_DEBUG_WRITECOUNT) adds 1 per store to a
counter per element of y (one more counter for stores outside y), on every
kernel family and launch shape: the CUDA-core kernel (every batch size) with
warps and cluster CTAs along K and chunked x, the tensor-core kernel, fused segments, the
RMSNorm prologue, INT4 and FP8 weights, the stream-K kernel with rows cut
between warps, its fixed-scratch entry point, and a captured plan."""
import numpy as np
import pytest
import torch

from memory_bound_decode_gb300 import binding, build_lib, inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def debug_lib():
    path = build_lib.build_debug()
    with binding.use_library(path):
        yield path


def counted(total: int):
    """A y buffer of `total` floats and its n + 1 zeroed counters, registered."""
    y = torch.full((total,), float("nan"), device=DEV)
    counts = torch.zeros(total + 1, dtype=torch.int32, device=DEV)
    binding.gemv_debug_write_count(counts, y, total)
    return y, counts


def assert_once(counts: torch.Tensor, what: str):
    torch.cuda.synchronize()
    c = counts.cpu().numpy()
    assert c[-1] == 0, f"{what}: {c[-1]} stores outside y"
    bad = np.flatnonzero(c[:-1] != 1)
    assert bad.size == 0, f"{what}: {bad.size} elements not written exactly once, e.g. {bad[:5]} -> {c[bad[:5]]}"


@pytest.mark.parametrize("N,K,B", [(4096, 14336, 1), (33, 65537, 1), (1024, 4096, 1), (4097, 4103, 1), (7, 129, 3),
                                   (4097, 4103, 8), (4096, 14336, 16), (1, 8191, 16), (300, 2056, 5)])
def test_bf16_written_once(debug_lib, N, K, B):
    ldw = inputs.padded_ldw(K)
    W = inputs.weight(N, K, ldw, seed=1, device=DEV)
    x = inputs.activations(B, K, seed=2, device=DEV)
    for eps in (None, 1e-5):
        for cc in ((False, True) if B > 1 else (False,)):
            y, counts = counted(B * N)
            binding.gemv_bf16_ex(W, x, y, N, K, B, ldw, rms_eps=eps, cuda_cores=cc)
            assert_once(counts, f"N={N} K={K} B={B} eps={eps} cuda_cores={cc}")
            assert torch.isfinite(y).all()
    binding.gemv_debug_write_count(None, None, 0)


def test_fused_segments_written_once(debug_lib):
    K, rows = 4096, [4096, 1024, 1024, 7]
    Ws = [inputs.weight(n, K, seed=i, device=DEV) for i, n in enumerate(rows)]
    for B in (1, 8):
        x = inputs.activations(B, K, seed=3, device=DEV)
        y, counts = counted(B * sum(rows))
        views, off = [], 0
        for n in rows:
            views.append(y[off:off + B * n].view(B, n))
            off += B * n
        binding.gemv_bf16_multi([(W, v, n, K) for W, v, n in zip(Ws, views, rows)], x, K, B)
        assert_once(counts, f"fused B={B}")
    binding.gemv_debug_write_count(None, None, 0)


@pytest.mark.parametrize("N,K,B", [(4096, 14336, 1), (300, 1280, 16), (33, 65536, 3)])
def test_int4_written_once(debug_lib, N, K, B):
    Wq, S = inputs.w4_weight_device(N, K, seed=4)
    x = inputs.activations(B, K, seed=5, device=DEV)
    y, counts = counted(B * N)
    binding.gemv_w4_bf16(Wq, S, x, y, N, K, B, Wq.shape[1], S.shape[1])
    assert_once(counts, f"int4 N={N} K={K} B={B}")
    binding.gemv_debug_write_count(None, None, 0)


@pytest.mark.parametrize("N,K,B", [(4096, 14336, 1), (128256, 4096, 1), (300, 1280, 16), (7, 64, 9)])
def test_fp8_written_once(debug_lib, N, K, B):
    Wq, S = inputs.fp8_weight(N, K, seed=6, device=DEV)
    x = inputs.activations(B, K, seed=7, device=DEV)
    y, counts = counted(B * N)
    binding.gemv_fp8_bf16(Wq, S, x, y, N, K, B, Wq.shape[1])
    assert_once(counts, f"fp8 N={N} K={K} B={B}")
    binding.gemv_debug_write_count(None, None, 0)


@pytest.mark.parametrize("N,K", [(1, 8191), (4096, 14336), (6144, 4096), (4097, 4103), (4864, 4096)])
def test_streamk_written_once(debug_lib, N, K):
    ldw = inputs.padded_ldw(K)
    W = inputs.weight(N, K, ldw, seed=8, device=DEV)
    x = inputs.activations(1, K, seed=9, device=DEV)
    y, counts = counted(N)
    binding.gemv_bf16_ex(W, x, y, N, K, 1, ldw, streamk=True)
    assert_once(counts, f"stream-K N={N} K={K}")
    y, counts = counted(N)
    binding.gemv_bf16_streamk_noalloc(W, x, y, N, K, ldw)
    assert_once(counts, f"stream-K no-alloc N={N} K={K}")
    binding.gemv_debug_write_count(None, None, 0)


def test_plan_written_once(debug_lib):
    K = 4096
    shapes = [(6144, 1, 1), (4096, 1, 0), (1024, 4, 0)]
    Ws = [inputs.weight(n, K, seed=10 + i, device=DEV) for i, (n, _, _) in enumerate(shapes)]
    xs = [inputs.activations(b, K, seed=20 + i, device=DEV) for i, (_, b, _) in enumerate(shapes)]
    total = sum(n * b for n, b, _ in shapes)
    y, counts = counted(total)
    views, off = [], 0
    for n, b, _ in shapes:
        views.append(y[off:off + b * n].view(b, n))
        off += b * n
    plan = binding.Plan([(W, x, v, n, K, K, b, 0, None, bool(sk))
                         for W, x, v, (n, b, sk) in zip(Ws, xs, views, shapes)])
    binding.gemv_debug_write_count(None, None, 0)   # the plan kept the counters it was created with
    s = torch.cuda.Stream()
    plan.capture(s)
    counts.zero_()
    torch.cuda.synchronize()
    plan.launch(s)
    s.synchronize()
    assert_once(counts, "plan")
    plan.destroy()
