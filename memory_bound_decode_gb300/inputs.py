"""Seeded synthetic inputs for the decode GEMV.

This module draws numbers and lays them out; it holds none of the GEMV's
arithmetic. Tests, the benchmark and the oracle checks all take their inputs
from here, so the CUDA path and the CPU oracle see the same bits.

Recipe (the shapes and value distributions of the decode projections of a
Llama-3.1-8B-shaped model; random init, no trained weights):
  - weights  W ~ N(0, 0.02^2) drawn in FP32, rounded to BF16 (round to nearest
    even), row-major [N, ldw] with ldw = K rounded up to a multiple of 8 and
    the padding columns k in [K, ldw) filled with a BF16 NaN (0x7FC0), so that
    any use of padding, even a multiply by zero, shows up as a NaN;
  - activations x ~ N(0, 1) drawn in FP32, rounded to BF16, [B, K] row-major
    with row stride K;
  - every tensor draws from its own generator, seeded seed * 1_000_003 + index,
    where index numbers the tensors of one workload in a fixed order.
Device-side draws (``device="cuda"``) and host-side draws give different bits
for the same seed; parity always copies the exact device bits to the host.
"""
from __future__ import annotations

import numpy as np
import torch

BF16_NAN = 0x7FC0


def padded_ldw(K: int) -> int:
    """K rounded up to a multiple of 8 BF16 elements (16 bytes)."""
    return (int(K) + 7) // 8 * 8


def generator(seed: int, index: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) * 1_000_003 + int(index))
    return g


def _fill_padding(W: torch.Tensor, K: int, pad: int | None) -> None:
    if pad is not None and W.shape[1] > K:
        W.view(torch.int16)[:, K:] = np.int16(np.uint16(pad).view(np.int16))


def weight(N: int, K: int, ldw: int | None = None, *, seed: int = 0, index: int = 0,
           std: float = 0.02, device="cpu", pad: int | None = BF16_NAN) -> torch.Tensor:
    """BF16 [N, ldw] with W[:, :K] ~ N(0, std^2) and NaN padding."""
    ldw = padded_ldw(K) if ldw is None else int(ldw)
    g = generator(seed, index, device)
    W = torch.empty((N, ldw), dtype=torch.bfloat16, device=device)
    rows = max(1, (1 << 26) // max(K, 1))  # bounded FP32 staging
    for r0 in range(0, N, rows):
        r1 = min(N, r0 + rows)
        part = torch.randn((r1 - r0, K), generator=g, dtype=torch.float32, device=device)
        part.mul_(std)
        W[r0:r1, :K] = part.to(torch.bfloat16)
    _fill_padding(W, K, pad)
    return W


def activations(B: int, K: int, *, seed: int = 0, index: int = 1, device="cpu") -> torch.Tensor:
    """BF16 [B, K] with entries N(0, 1), row stride K."""
    g = generator(seed, index, device)
    return torch.randn((B, K), generator=g, dtype=torch.float32, device=device).to(torch.bfloat16)


def int_weight(N: int, K: int, ldw: int | None = None, *, lo: int = -3, hi: int = 3,
               seed: int = 0, index: int = 0, device="cpu",
               pad: int | None = BF16_NAN) -> torch.Tensor:
    """BF16 [N, ldw] of small integers in [lo, hi] (exact in BF16)."""
    ldw = padded_ldw(K) if ldw is None else int(ldw)
    g = generator(seed, index, device)
    W = torch.empty((N, ldw), dtype=torch.bfloat16, device=device)
    W[:, :K] = torch.randint(lo, hi + 1, (N, K), generator=g, device=device).to(torch.bfloat16)
    _fill_padding(W, K, pad)
    return W


def int_activations(B: int, K: int, *, lo: int = -2, hi: int = 2, seed: int = 0,
                    index: int = 1, device="cpu") -> torch.Tensor:
    g = generator(seed, index, device)
    return torch.randint(lo, hi + 1, (B, K), generator=g, device=device).to(torch.bfloat16)


def bits(t: torch.Tensor) -> np.ndarray:
    """The BF16 bit patterns of a tensor as a host uint16 array (a copy)."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def from_bits(a: np.ndarray, device="cpu") -> torch.Tensor:
    """A BF16 tensor holding the given uint16 bit patterns."""
    a = np.ascontiguousarray(a, dtype=np.uint16)
    return torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16).to(device)


# ----------------------------------------------------------------------------- INT4 weights
#
# Layout of a group-quantised INT4 weight (group of W4_GROUP consecutive k per
# row, one BF16 scale each; the value of an element is (u - 8) * scale with u
# its 4-bit code):
#   Wq : uint8 [N, ldq], ldq >= K / 2, ldq % 16 == 0. Row n, 32-bit word w
#        (bytes 4w .. 4w+3, little endian) holds k = 8w .. 8w+7: the code of
#        k = 8w + 2j sits in bits 4j .. 4j+3 and that of k = 8w + 2j + 1 in bits
#        16 + 4j .. 16 + 4j + 3 (j = 0..3): even k in the low half-word, odd k in
#        the high half-word.
#   S  : BF16 [N, lds], lds >= K / W4_GROUP; S[n][g] scales k in [g*W4_GROUP, (g+1)*W4_GROUP).
W4_GROUP = 128


def w4_pack(u: np.ndarray, ldq: int | None = None) -> np.ndarray:
    """Pack 4-bit codes u (uint8 in [0, 15], [N, K], K % 8 == 0) into the layout above."""
    u = np.asarray(u, dtype=np.uint32)
    N, K = u.shape
    assert K % 8 == 0 and u.max(initial=0) < 16
    ldq = K // 2 if ldq is None else int(ldq)
    g = u.reshape(N, K // 8, 4, 2)               # [n, word, j, parity]
    shifts = (4 * np.arange(4, dtype=np.uint32))[None, None, :]
    words = ((g[..., 0] << shifts) | (g[..., 1] << (shifts + 16))).sum(axis=2, dtype=np.uint64).astype(np.uint32)
    out = np.zeros((N, ldq), dtype=np.uint8)
    out[:, : K // 2] = words.view(np.uint8).reshape(N, K // 2)
    return out


def w4_weight(N: int, K: int, ldq: int | None = None, lds: int | None = None, *, seed: int = 0,
              index: int = 0, scale_lo: float = 0.002, scale_hi: float = 0.006, codes=None,
              scales=None):
    """(Wq uint8 [N, ldq], S bf16 [N, lds], u uint8 [N, K]) on the host: random codes
    (or ``codes``) and scales uniform in [scale_lo, scale_hi] rounded to BF16 (or
    ``scales``, float [N, K / W4_GROUP])."""
    assert K % W4_GROUP == 0
    ldq = (K // 2 + 15) // 16 * 16 if ldq is None else int(ldq)
    G = K // W4_GROUP
    lds = G if lds is None else int(lds)
    g = generator(seed, index, "cpu")
    if codes is None:
        codes = torch.randint(0, 16, (N, K), generator=g, dtype=torch.int32).numpy().astype(np.uint8)
    if scales is None:
        scales = (torch.rand((N, G), generator=g, dtype=torch.float32) * (scale_hi - scale_lo) + scale_lo)
    S = torch.zeros((N, lds), dtype=torch.bfloat16)
    S[:, :G] = torch.as_tensor(scales, dtype=torch.float32).to(torch.bfloat16)
    return w4_pack(codes, ldq), S, np.asarray(codes, dtype=np.uint8)


def w4_weight_device(N: int, K: int, ldq: int | None = None, lds: int | None = None, *, seed: int = 0,
                     index: int = 0, device="cuda", scale_lo: float = 0.002, scale_hi: float = 0.006):
    """Random INT4 weight in the layout above, drawn and packed on the device
    (for workloads too large to pack on the host): (Wq uint8 [N, ldq], S bf16 [N, lds])."""
    assert K % W4_GROUP == 0
    ldq = (K // 2 + 15) // 16 * 16 if ldq is None else int(ldq)
    G = K // W4_GROUP
    lds = G if lds is None else int(lds)
    g = generator(seed, index, device)
    Wq = torch.zeros((N, ldq), dtype=torch.uint8, device=device)
    rows = max(1, (1 << 26) // K)
    for r0 in range(0, N, rows):
        r1 = min(N, r0 + rows)
        u = torch.randint(0, 16, (r1 - r0, K // 8, 4, 2), generator=g, device=device, dtype=torch.int64)
        shifts = 4 * torch.arange(4, device=device, dtype=torch.int64)
        words = ((u[..., 0] << shifts) | (u[..., 1] << (shifts + 16))).sum(dim=2)
        words = torch.where(words >= 2 ** 31, words - 2 ** 32, words).to(torch.int32)
        Wq[r0:r1, : K // 2] = words.contiguous().view(torch.uint8).view(r1 - r0, K // 2)
    S = torch.zeros((N, lds), dtype=torch.bfloat16, device=device)
    sc = torch.rand((N, G), generator=g, device=device, dtype=torch.float32) * (scale_hi - scale_lo) + scale_lo
    S[:, :G] = sc.to(torch.bfloat16)
    return Wq, S


# ----------------------------------------------------------------------------- FP8 weights
#
# Layout of an FP8 weight: Wq uint8 [N, ldq], ldq >= K, ldq % 16 == 0, holding
# E4M3 codes (sign, 4 exponent bits with bias 7, 3 mantissa bits; no infinities,
# S.1111.111 is NaN), and S float32 [N], one scale per output row: element
# (n, k) is e4m3(Wq[n][k]) * S[n]. Columns k in [K, ldq) are padding.
FP8_PAD = 0x7F   # an E4M3 NaN: any use of padding shows up


def fp8_quantize(Wf: torch.Tensor):
    """Row-scaled E4M3 codes of a float weight: S[n] = max_k |W[n][k]| / 448 (1
    for an all-zero row), codes = W / S rounded to E4M3 (round to nearest even,
    by torch's conversion). Returns (codes uint8 [N, K], S float32 [N])."""
    amax = Wf.abs().amax(dim=1)
    S = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax)).to(torch.float32)
    codes = (Wf / S[:, None]).to(torch.float8_e4m3fn).view(torch.uint8)
    return codes, S


def fp8_weight(N: int, K: int, ldq: int | None = None, *, seed: int = 0, index: int = 0,
               std: float = 0.02, device="cpu", pad: int | None = FP8_PAD):
    """(Wq uint8 [N, ldq], S float32 [N]): W ~ N(0, std^2) drawn in FP32, then
    quantised per row with fp8_quantize; padding columns hold an E4M3 NaN."""
    ldq = (int(K) + 15) // 16 * 16 if ldq is None else int(ldq)
    g = generator(seed, index, device)
    Wq = torch.empty((N, ldq), dtype=torch.uint8, device=device)
    S = torch.empty((N,), dtype=torch.float32, device=device)
    rows = max(1, (1 << 26) // max(K, 1))
    for r0 in range(0, N, rows):
        r1 = min(N, r0 + rows)
        part = torch.randn((r1 - r0, K), generator=g, dtype=torch.float32, device=device).mul_(std)
        codes, sc = fp8_quantize(part)
        Wq[r0:r1, :K] = codes
        S[r0:r1] = sc
    if pad is not None and ldq > K:
        Wq[:, K:] = pad
    return Wq, S


def fp8_decode(codes) -> np.ndarray:
    """E4M3 codes (uint8 array or tensor) to float64 by torch's float8_e4m3fn type."""
    t = torch.as_tensor(np.ascontiguousarray(codes) if isinstance(codes, np.ndarray) else codes)
    return t.cpu().view(torch.float8_e4m3fn).to(torch.float64).numpy()
