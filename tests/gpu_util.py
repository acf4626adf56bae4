"""Helpers for the GPU parity tests: run the C-ABI GEMV with guard bands around
y and compare with the CPU oracle."""
from __future__ import annotations

import numpy as np
import torch

from memory_bound_decode_gb300 import binding, inputs
from oracle import oracle

GUARD = 64
SENTINEL = np.uint32(0x7F800001)   # a signalling-NaN pattern no kernel writes


def guarded_y(B: int, N: int, device="cuda"):
    """A y buffer with GUARD sentinel words on both sides; y itself is NaN."""
    buf = torch.empty(B * N + 2 * GUARD, dtype=torch.float32, device=device)
    buf.view(torch.int32).fill_(int(SENTINEL.view(np.int32)))
    y = buf[GUARD:GUARD + B * N].view(B, N)
    y.fill_(float("nan"))
    return buf, y


def check_guards(buf: torch.Tensor) -> None:
    raw = buf.view(torch.int32).cpu().numpy().view(np.uint32)
    assert np.all(raw[:GUARD] == SENTINEL), "write before y"
    assert np.all(raw[-GUARD:] == SENTINEL), "write after y"


def gemv(W: torch.Tensor, x: torch.Tensor, K: int, stream=None) -> np.ndarray:
    N, ldw = W.shape
    B = x.shape[0]
    buf, y = guarded_y(B, N, W.device)
    binding.gemv_bf16(W, x, y, N, K, B, ldw, stream)
    torch.cuda.synchronize()
    check_guards(buf)
    return y.cpu().numpy()


def reference(W: torch.Tensor, x: torch.Tensor, K: int):
    return oracle.gemv(inputs.bits(W), inputs.bits(x), K, threads=oracle.default_threads())


def assert_parity(y_gpu: np.ndarray, y_ref: np.ndarray, scale: np.ndarray, what="") -> None:
    ok = oracle.accept(y_gpu, y_ref, scale)
    if not ok.all():
        idx = np.argwhere(~ok)[:5]
        detail = [(tuple(i), float(y_gpu[tuple(i)]), float(y_ref[tuple(i)]), float(scale[tuple(i)]))
                  for i in idx]
        raise AssertionError(f"{what}: {int((~ok).sum())} of {ok.size} outside tolerance: {detail}")
