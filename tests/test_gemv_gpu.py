"""Parity of the CUDA GEMV (through the C ABI) with the CPU oracle.

Every comparison is element by element: |y_gpu - y_ref| <= 1e-5 * sum_k |W x|
and y_gpu finite, y surrounded by sentinel guard bands that must survive and
prefilled with NaN so that every element must be written. Integer-valued and
one-hot inputs, for which every FP32 summation order is exact, are compared
bitwise.
"""
import numpy as np
import pytest
import torch

from memory_bound_decode_gb300 import binding, inputs
from oracle import oracle
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

DEV = "cuda"

SMALL = [  # (N, K): ragged tails, split-K, tiny and degenerate shapes
    (7, 129), (1, 1), (3, 8), (5, 9), (65, 300), (300, 2056), (1, 8191),
    (4097, 4103), (33, 65537), (1024, 4096), (17, 100000),
]


def make(N, K, B, seed=0, device=DEV):
    ldw = inputs.padded_ldw(K)
    W = inputs.weight(N, K, ldw, seed=seed, index=0, device=device)
    x = inputs.activations(B, K, seed=seed, index=1, device=device)
    return W, x, ldw


@pytest.mark.parametrize("B", [1, 2, 3, 4, 8, 16])
@pytest.mark.parametrize("N,K", SMALL)
def test_parity_small(N, K, B):
    W, x, _ = make(N, K, B, seed=N + K + B)
    y = gu.gemv(W, x, K)
    y_ref, s = gu.reference(W, x, K)
    gu.assert_parity(y, y_ref, s, f"N={N} K={K} B={B}")


@pytest.mark.parametrize("N,K,ldw", [(64, 1000, 1024), (9, 129, 256), (100, 4096, 4104)])
def test_wide_row_stride(N, K, ldw):
    """ldw well beyond K: the padding (NaN) is never part of a sum."""
    W, x, _ = make(N, K, 2)
    W2 = torch.full((N, ldw), float("nan"), dtype=torch.bfloat16, device=DEV)
    W2[:, :K] = W[:, :K]
    y = gu.gemv(W2, x, K)
    y_ref, s = gu.reference(W2, x, K)
    gu.assert_parity(y, y_ref, s)


FULL = [  # the decode projections of a Llama-3.1-8B-shaped layer, and the LM head
    ("k_proj", 1024, 4096), ("down_proj", 4096, 14336), ("qkv", 6144, 4096),
    ("o_proj", 4096, 4096), ("gate_up", 28672, 4096), ("lm_head", 128256, 4096),
]


@pytest.mark.parametrize("name,N,K", FULL, ids=[f[0] for f in FULL])
def test_parity_full_size(name, N, K):
    W, x, _ = make(N, K, 1, seed=1)
    y = gu.gemv(W, x, K)
    y_ref, s = gu.reference(W, x, K)
    gu.assert_parity(y, y_ref, s, name)


@pytest.mark.parametrize("B", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("N,K", [(4096, 4096), (4096, 14336), (4864, 14336), (28672, 4096)])
def test_parity_skinny_batch(N, K, B):
    W, x, _ = make(N, K, B, seed=2)
    y = gu.gemv(W, x, K)
    y_ref, s = gu.reference(W, x, K)
    gu.assert_parity(y, y_ref, s, f"B={B}")


@pytest.mark.parametrize("B", [2, 3, 4, 8, 9, 12, 16])
@pytest.mark.parametrize("N,K", [(4096, 14336), (1000, 4096), (33, 65537)])
def test_tensor_core_wide_dynamic_range(N, K, B):
    """The batch 2..16 path runs on the tensor cores, whose internal addition
    order and rounding the PTX ISA leaves open. Rows mixing columns scaled by
    1e4 and by 1e-4 (and weight rows scaled by 1e3 or 1e-3) put products of
    very different magnitude into one dot product; every element must still be
    within 1e-5 of the sum of the products' magnitudes."""
    W, x, ldw = make(N, K, B, seed=N + K + 7 * B)
    g = inputs.generator(N + K, 5, DEV)
    col = torch.where(torch.rand(K, generator=g, device=DEV) < 0.5, 1e4, 1e-4)
    row = torch.where(torch.rand(N, generator=g, device=DEV) < 0.5, 1e3, 1e-3)
    x = (x.float() * col[None, :]).to(torch.bfloat16)
    W2 = W.clone()
    W2[:, :K] = (W[:, :K].float() * row[:, None]).to(torch.bfloat16)
    y = gu.gemv(W2, x, K)
    y_ref, s = gu.reference(W2, x, K)
    gu.assert_parity(y, y_ref, s, f"dynamic range N={N} K={K} B={B}")


@pytest.mark.parametrize("N,K,B", [(7, 129, 1), (4097, 4103, 3), (33, 65537, 1), (1, 8191, 16),
                                   (128256, 4096, 1), (4096, 14336, 16)])
def test_integer_inputs_are_exact(N, K, B):
    """Small integers: every partial sum is an integer below 2^24, so any FP32
    order gives the exact result, bit for bit."""
    ldw = inputs.padded_ldw(K)
    W = inputs.int_weight(N, K, ldw, seed=3, device=DEV)
    x = inputs.int_activations(B, K, seed=3, device=DEV)
    y = gu.gemv(W, x, K)
    y_ref, _ = gu.reference(W, x, K)
    assert np.array_equal(y.astype(np.float64), y_ref)


@pytest.mark.parametrize("N,K", [(4097, 4103), (33, 65537), (1024, 4096)])
def test_one_hot_selects_a_column(N, K):
    W, _, _ = make(N, K, 1, seed=4)
    Wh = inputs.bits(W)
    for j in (0, 7, 8, 255, 256, K - 1):
        x = torch.zeros((1, K), dtype=torch.bfloat16, device=DEV)
        x[0, j] = 1.0
        y = gu.gemv(W, x, K)
        col = inputs.from_bits(Wh[:, j]).float().numpy()
        assert np.array_equal(y[0], col), j


def test_identity_padded():
    N, K = 300, 129
    ldw = inputs.padded_ldw(K)
    W = torch.zeros((N, ldw), dtype=torch.bfloat16, device=DEV)
    W[:, K:] = float("nan")
    idx = torch.arange(min(N, K), device=DEV)
    W[idx, idx] = 1.0
    x = inputs.activations(1, K, seed=5, device=DEV)
    y = gu.gemv(W, x, K)
    want = np.zeros(N, dtype=np.float32)
    want[:K] = x[0].float().cpu().numpy()
    assert np.array_equal(y[0], want)


@pytest.mark.parametrize("N,K,B", [(4096, 14336, 1), (33, 65537, 1), (1000, 3000, 4)])
def test_deterministic_and_scale_exact(N, K, B):
    W, x, _ = make(N, K, B, seed=6)
    y1 = gu.gemv(W, x, K)
    y2 = gu.gemv(W, x, K)
    assert np.array_equal(y1.view(np.uint32), y2.view(np.uint32))
    y4 = gu.gemv(W, (x.float() * 4.0).to(torch.bfloat16), K)
    assert np.array_equal(y4, y1 * np.float32(4.0))


def test_row_permutation_permutes_y():
    N, K, B = 4097, 4103, 2
    W, x, _ = make(N, K, B, seed=7)
    perm = torch.randperm(N, generator=torch.Generator().manual_seed(0)).to(DEV)
    y = gu.gemv(W, x, K)
    yp = gu.gemv(W[perm].contiguous(), x, K)
    assert np.array_equal(yp, y[:, perm.cpu().numpy()])


def test_batch_rows_match_single_calls():
    N, K, B = 2048, 5000, 8
    W, x, _ = make(N, K, B, seed=8)
    y = gu.gemv(W, x, K)
    y_ref, s = gu.reference(W, x, K)
    for b in range(B):
        yb = gu.gemv(W, x[b:b + 1].contiguous(), K)
        assert np.all(np.abs(yb[0].astype(np.float64) - y[b]) <= 2e-5 * s[b])


def test_linearity():
    N, K = 1024, 4096
    W, _, _ = make(N, K, 1, seed=9)
    xa = inputs.int_activations(1, K, lo=-8, hi=8, seed=1, device=DEV)
    xb = inputs.int_activations(1, K, lo=-8, hi=8, seed=2, device=DEV)
    ya = gu.gemv(W, xa, K).astype(np.float64)
    yb = gu.gemv(W, xb, K).astype(np.float64)
    ys = gu.gemv(W, (xa.float() + xb.float()).to(torch.bfloat16), K).astype(np.float64)
    _, sa = gu.reference(W, xa, K)
    _, sb = gu.reference(W, xb, K)
    assert np.all(np.abs(ys - (ya + yb)) <= 2e-5 * (sa + sb))


def test_misaligned_x_rows():
    """x rows start at odd 2-byte offsets when K % 8 != 0; x itself may start at
    any even address."""
    N, K, B = 500, 1001, 5
    W, x, _ = make(N, K, B, seed=10)
    xbuf = torch.zeros(B * K + 3, dtype=torch.bfloat16, device=DEV)
    xbuf[3:] = x.reshape(-1)
    xs = xbuf[3:].view(B, K)
    buf, y = gu.guarded_y(B, N)
    binding.gemv_bf16(W, xs, y, N, K, B, W.shape[1])
    torch.cuda.synchronize()
    gu.check_guards(buf)
    y_ref, s = gu.reference(W, x, K)
    gu.assert_parity(y.cpu().numpy(), y_ref, s)


def test_side_stream_and_no_sync():
    N, K = 4096, 4096
    W, x, _ = make(N, K, 1, seed=11)
    s = torch.cuda.Stream()
    buf, y = gu.guarded_y(1, N)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        binding.gemv_bf16(W, x, y, N, K, 1, W.shape[1], s)
    s.synchronize()
    gu.check_guards(buf)
    y_ref, sc = gu.reference(W, x, K)
    gu.assert_parity(y.cpu().numpy(), y_ref, sc)


def test_probe_stream_read_runs():
    nbytes = 64 << 20
    src = torch.randint(-1000, 1000, (nbytes // 2,), dtype=torch.int16, device=DEV)
    sink = torch.full((binding.gemv_probe_sink_words(),), -1.0, device=DEV)
    binding.gemv_probe_stream_read(src, nbytes, sink)
    torch.cuda.synchronize()
    assert torch.isfinite(sink[:152]).all()


def test_host_io_round_trip():
    N, K, B = 4096, 14336, 2
    W, x, ldw = make(N, K, B, seed=12)
    x_host = x.cpu().pin_memory()
    y_host = torch.full((B, N), float("nan")).pin_memory()
    x_dev = torch.empty_like(x)
    y_dev = torch.empty((B, N), device=DEV)
    s = torch.cuda.Stream()
    binding.gemv_bf16_host_io(W, x_host, y_host, x_dev, y_dev, N, K, B, ldw, stream=s)
    # synchronous: the host buffer already holds the result
    y_ref, sc = gu.reference(W, x, K)
    gu.assert_parity(y_host.numpy(), y_ref, sc)
    binding.gemv_bf16_host_io(W, x_host, y_host, x_dev, y_dev, N, K, B, ldw, rms_eps=1e-5, stream=s)
    assert np.isfinite(y_host.numpy()).all()


@pytest.mark.parametrize("pinned", [True, False])
def test_host_io_pinned_and_pageable(pinned):
    """Pinned (device-mapped) y_host takes the kernel's stores directly; pageable
    y_host goes through y_dev and a copy. Both hold the result on return."""
    N, K, B = 4097, 4103, 3
    W, x, ldw = make(N, K, B, seed=13)
    x_host = x.cpu()
    y_host = torch.full((B, N), float("nan"))
    if pinned:
        x_host, y_host = x_host.pin_memory(), y_host.pin_memory()
    y_dev = torch.full((B, N), float("nan"), device=DEV)
    binding.gemv_bf16_host_io(W, x_host, y_host, torch.empty_like(x), y_dev, N, K, B, ldw)
    y_ref, sc = gu.reference(W, x, K)
    gu.assert_parity(y_host.numpy(), y_ref, sc, f"pinned={pinned}")
    for _ in range(3):   # repeated calls, no stale results
        y_host.fill_(float("nan"))
        binding.gemv_bf16_host_io(W, x_host, y_host, torch.empty_like(x), y_dev, N, K, B, ldw)
        gu.assert_parity(y_host.numpy(), y_ref, sc, f"pinned={pinned} repeat")


@pytest.mark.parametrize("xkind", ["pinned", "pageable", "pinned_unaligned"])
@pytest.mark.parametrize("N,K,B", [(4096, 14336, 1), (1000, 4096, 4), (4097, 4103, 3), (70000, 4096, 1)])
def test_host_io_matches_device_call(N, K, B, xkind):
    """gemv_bf16_host_io (host x in, GEMV, host y out, synchronized) gives the
    bits of the device-resident call on the same inputs, whichever way x comes
    in (a copy kernel from 16-byte aligned mapped pinned memory, else a DMA
    copy) and y goes out (stored straight into mapped memory up to 256 KB, else
    copied back)."""
    W, x, ldw = make(N, K, B, seed=N + K)
    y_ref = torch.empty((B, N), device=DEV)
    binding.gemv_bf16(W, x, y_ref, N, K, B, ldw)
    if xkind == "pinned":
        xh = x.cpu().pin_memory()
    elif xkind == "pageable":
        xh = x.cpu()
    else:
        raw = torch.empty(B * K + 1, dtype=torch.bfloat16).pin_memory()
        raw[1:] = x.cpu().reshape(-1)
        xh = raw[1:].view(B, K)           # 2 bytes past a 16-byte boundary
    yh = torch.full((B, N), float("nan")).pin_memory()
    x_dev = torch.empty_like(x)
    y_dev = torch.empty((B, N), device=DEV)
    s = torch.cuda.Stream()
    for _ in range(2):                    # twice in a row: the same bits
        yh.fill_(float("nan"))
        binding.gemv_bf16_host_io(W, xh, yh, x_dev, y_dev, N, K, B, ldw, stream=s)
        assert torch.equal(yh.view(torch.int32), y_ref.cpu().view(torch.int32))
    y_o, sc = gu.reference(W, x, K)
    gu.assert_parity(yh.numpy(), y_o, sc, f"host io {xkind}")
