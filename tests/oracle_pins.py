"""Pins for the CPU oracle: checks against facts fixed by mathematics, not by the
oracle itself. Each function takes an oracle handle (``oracle.OracleLib``) and
raises AssertionError on a violation, so the same pins run against the real
oracle and against deliberately broken copies of it (see test_oracle_pins.py).

What pins what:
  exact_rational      every output and scale on tiny inputs, against an exact
                      rational sum (fractions.Fraction) of values decoded by
                      torch, an independent BF16 decoder
  integer_matmul      all outputs on integer data, against numpy int64 matmul
  ones_row_sums       x = ones gives the row sums of W
  one_hot_column      one-hot x at column j selects column j, exactly
  identity_padded     W = [I | 0] returns x itself
  scaling_exact       y(2^e x) = 2^e y(x) bitwise
  linearity           y(x1 + x2) = y(x1) + y(x2) within FP64 rounding
  row_permutation     permuting rows of W permutes y, bitwise
  batch_rows          row b of a batch equals a single-row call on x[b]
  padding_unread      NaN in the ldw padding never reaches y
  float64_matmul      random BF16 data against numpy float64 matmul
  single_element      the one-element entry point equals the full computation
  rms_constant_x      RMSNorm prologue: x = c gives r = (c^2 + eps)^(-1/2), y = r*c*rowsum
  rms_scale_free      RMSNorm prologue with eps = 0: y(4x) = y(x) bitwise
  rms_independent     r from numpy's own mean and sqrt; y and scale = r * the plain GEMV
  w4_integer_exact    INT4 weights, power-of-two group scales, integer x: y exact
                      against numpy int64 arithmetic on the codes the packer was given
  w4_one_hot          INT4: one-hot x at every position of a word and across a group
                      boundary selects (u - 8) * scale
  w4_dense            INT4 against numpy float64 on weights dequantised from the codes
  fp8_decode_table    FP8: every one of the 256 E4M3 codes against torch's float8_e4m3fn
                      decode (NaN codes NaN) and closed forms (1, 448, 2^-6, 2^-9, -0)
  fp8_integer_exact   FP8 codes of small integers, power-of-two row scales, integer x:
                      y exact against numpy int64 arithmetic
  fp8_dense           FP8 against numpy float64 on torch-decoded weights times row scales,
                      with NaN codes in the ldq padding that must not reach y
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np
import torch

from memory_bound_decode_gb300 import inputs

EPS64 = 2.0 ** -53


def _decode(bits: np.ndarray) -> np.ndarray:
    """BF16 bits -> float64 via torch's own conversion (independent of the oracle)."""
    return inputs.from_bits(bits).to(torch.float64).numpy()


def _rand_case(N, K, B, ldw, seed):
    W = inputs.bits(inputs.weight(N, K, ldw, seed=seed, index=0, std=1.0))
    x = inputs.bits(inputs.activations(B, K, seed=seed, index=1))
    return W, x


def exact_rational(lib):
    cases = [(7, 129, 1, 136), (3, 17, 2, 24), (1, 8, 1, 8), (2, 1, 3, 8),
             (5, 33, 16, 40), (4, 9, 5, 16)]
    for i, (N, K, B, ldw) in enumerate(cases):
        W, x = _rand_case(N, K, B, ldw, seed=100 + i)
        y, s = lib.gemv(W, x)
        Wd = _decode(W[:, :K])
        xd = _decode(x)
        for b in range(B):
            for n in range(N):
                terms = [Fraction(float(Wd[n, k])) * Fraction(float(xd[b, k])) for k in range(K)]
                exact = sum(terms, Fraction(0))
                mag = sum((abs(t) for t in terms), Fraction(0))
                bound = 4 * K * EPS64 * float(mag)
                assert abs(y[b, n] - float(exact)) <= bound, (N, K, B, b, n)
                assert abs(s[b, n] - float(mag)) <= bound, (N, K, B, b, n)


def integer_matmul(lib):
    for (N, K, B, ldw) in [(7, 129, 1, 136), (33, 1000, 3, 1000), (16, 4103, 2, 4104)]:
        W = inputs.bits(inputs.int_weight(N, K, ldw, seed=7))
        x = inputs.bits(inputs.int_activations(B, K, seed=7))
        Wi = _decode(W[:, :K]).astype(np.int64)
        xi = _decode(x).astype(np.int64)
        y, s = lib.gemv(W, x)
        assert np.array_equal(y, (xi @ Wi.T).astype(np.float64))
        assert np.array_equal(s, (np.abs(xi) @ np.abs(Wi).T).astype(np.float64))


def ones_row_sums(lib):
    N, K, ldw = 9, 300, 304
    W = inputs.bits(inputs.int_weight(N, K, ldw, lo=-100, hi=100, seed=3))
    ones = np.full((1, K), 0x3F80, dtype=np.uint16)  # BF16 1.0
    y, s = lib.gemv(W, ones)
    Wd = _decode(W[:, :K])
    assert np.array_equal(y[0], Wd.sum(axis=1))
    assert np.array_equal(s[0], np.abs(Wd).sum(axis=1))


def one_hot_column(lib):
    N, K, ldw = 11, 77, 80
    W, _ = _rand_case(N, K, 1, ldw, seed=5)
    Wd = _decode(W[:, :K])
    for j in (0, 7, 8, K - 1):
        x = np.zeros((1, K), dtype=np.uint16)
        x[0, j] = 0x3F80
        y, _ = lib.gemv(W, x)
        assert np.array_equal(y[0], Wd[:, j]), j


def identity_padded(lib):
    for N, K in [(5, 9), (12, 8), (8, 8)]:
        ldw = inputs.padded_ldw(K)
        W = np.zeros((N, ldw), dtype=np.uint16)
        for n in range(min(N, K)):
            W[n, n] = 0x3F80
        W[:, K:] = inputs.BF16_NAN
        x = inputs.bits(inputs.activations(1, K, seed=9))
        y, _ = lib.gemv(W, x)
        xd = _decode(x)[0]
        want = np.zeros(N)
        want[:min(N, K)] = xd[:min(N, K)]
        assert np.array_equal(y[0], want), (N, K)


def scaling_exact(lib):
    N, K, ldw = 6, 129, 136
    W, x = _rand_case(N, K, 1, ldw, seed=11)
    y1, _ = lib.gemv(W, x)
    x4 = inputs.bits(inputs.from_bits(x).float().mul(4.0).to(torch.bfloat16))
    y4, _ = lib.gemv(W, x4)
    assert np.array_equal(y4, 4.0 * y1)


def linearity(lib):
    N, K, ldw = 6, 200, 200
    W, _ = _rand_case(N, K, 1, ldw, seed=12)
    xa = inputs.int_activations(1, K, lo=-8, hi=8, seed=1)
    xb = inputs.int_activations(1, K, lo=-8, hi=8, seed=2)
    xs = (xa.float() + xb.float()).to(torch.bfloat16)  # exact: small integers
    ya, sa = lib.gemv(W, inputs.bits(xa))
    yb, sb = lib.gemv(W, inputs.bits(xb))
    ys, _ = lib.gemv(W, inputs.bits(xs))
    assert np.all(np.abs(ys - (ya + yb)) <= 4 * K * EPS64 * (sa + sb))
    assert not np.allclose(ya, 0.0)


def row_permutation(lib):
    N, K, ldw = 10, 129, 136
    W, x = _rand_case(N, K, 2, ldw, seed=13)
    perm = np.random.default_rng(0).permutation(N)
    y, s = lib.gemv(W, x)
    yp, sp = lib.gemv(np.ascontiguousarray(W[perm]), x)
    assert np.array_equal(yp, y[:, perm])
    assert np.array_equal(sp, s[:, perm])


def batch_rows(lib):
    N, K, ldw, B = 6, 131, 136, 5
    W, x = _rand_case(N, K, B, ldw, seed=14)
    y, _ = lib.gemv(W, x)
    for b in range(B):
        yb, _ = lib.gemv(W, x[b:b + 1])
        assert np.array_equal(yb[0], y[b]), b


def padding_unread(lib):
    N, K, ldw = 4, 13, 24
    W, x = _rand_case(N, K, 2, ldw, seed=15)
    W[:, K:] = inputs.BF16_NAN
    y, s = lib.gemv(W, x)
    assert np.all(np.isfinite(y)) and np.all(np.isfinite(s))
    W2 = W.copy()
    W2[:, K:] = 0x3F80
    y2, _ = lib.gemv(W2, x)
    assert np.array_equal(y, y2)


def float64_matmul(lib):
    N, K, B, ldw = 64, 1000, 3, 1000
    W, x = _rand_case(N, K, B, ldw, seed=16)
    y, s = lib.gemv(W, x)
    Wd = _decode(W[:, :K])
    xd = _decode(x)
    ref = xd @ Wd.T
    assert np.all(np.abs(y - ref) <= 4 * K * EPS64 * s)
    assert np.allclose(s, np.abs(xd) @ np.abs(Wd).T, rtol=1e-12, atol=0)


def single_element(lib):
    N, K, B, ldw = 9, 70, 3, 72
    W, x = _rand_case(N, K, B, ldw, seed=17)
    y, s = lib.gemv(W, x)
    for b, n in [(0, 0), (2, 8), (1, 4)]:
        yo, so = lib.gemv_one(W, x, b, n)
        assert yo == y[b, n] and so == s[b, n]


def rms_constant_x(lib):
    N, K, ldw = 6, 40, 48
    W = inputs.bits(inputs.int_weight(N, K, ldw, lo=-5, hi=5, seed=21))
    Wd = _decode(W[:, :K])
    for c_bits, c in [(0x3F00, 0.5), (0xC040, -3.0)]:
        x = np.full((2, K), c_bits, dtype=np.uint16)
        for eps in (0.0, 1e-5, 0.25):
            y, sc, r = lib.gemv_rmsnorm(W, x, eps)
            r_want = 1.0 / np.sqrt(c * c + eps)
            assert np.allclose(r, r_want, rtol=1e-15, atol=0), (c, eps, r)
            want = r_want * c * Wd.sum(axis=1)
            assert np.allclose(y[0], want, rtol=1e-14, atol=0) and np.array_equal(y[0], y[1])
            assert np.allclose(sc[0], r_want * abs(c) * np.abs(Wd).sum(axis=1), rtol=1e-14, atol=0)


def rms_scale_free(lib):
    N, K, ldw, B = 7, 129, 136, 3
    W, x = _rand_case(N, K, B, ldw, seed=22)
    x4 = inputs.bits(inputs.from_bits(x).float().mul(4.0).to(torch.bfloat16))
    y1, s1, r1 = lib.gemv_rmsnorm(W, x, 0.0)
    y4, s4, r4 = lib.gemv_rmsnorm(W, x4, 0.0)
    assert np.array_equal(y1, y4) and np.array_equal(s1, s4)
    assert np.array_equal(r4 * 4.0, r1)


def rms_independent(lib):
    N, K, ldw, B = 33, 1000, 1008, 4
    W, x = _rand_case(N, K, B, ldw, seed=23)
    eps = 1e-6
    y0, s0 = lib.gemv(W, x)
    y, sc, r = lib.gemv_rmsnorm(W, x, eps)
    xd = _decode(x)
    r_np = 1.0 / np.sqrt(np.mean(xd * xd, axis=1) + eps)
    assert np.allclose(r, r_np, rtol=1e-13, atol=0)
    assert np.allclose(y, y0 * r_np[:, None], rtol=1e-12, atol=1e-300)
    assert np.allclose(sc, s0 * r_np[:, None], rtol=1e-12, atol=0)
    try:
        lib.gemv_rmsnorm(W, x, -1.0)
    except ValueError:
        pass
    else:
        raise AssertionError("negative eps accepted")


def _w4_case(N, K, B, seed, ldq=None, lds=None, pow2_scales=False):
    G = K // inputs.W4_GROUP
    scales = None
    if pow2_scales:
        scales = np.array([[2.0 ** ((n + g) % 5 - 2) for g in range(G)] for n in range(N)])
    Wq, S, u = inputs.w4_weight(N, K, ldq, lds, seed=seed, scales=scales)
    return Wq, inputs.bits(S), u


def w4_integer_exact(lib):
    for (N, K, B, ldq, lds) in [(5, 256, 2, 144, 3), (9, 1024, 3, 512, 8), (3, 128, 1, 64, 1)]:
        Wq, S, u = _w4_case(N, K, B, seed=N + K, ldq=ldq, lds=lds, pow2_scales=True)
        x = inputs.bits(inputs.int_activations(B, K, lo=-3, hi=3, seed=N))
        y, sc = lib.gemv_w4(Wq, S, x, K)
        G = K // inputs.W4_GROUP
        s4 = (_decode(S[:, :G]) * 4).astype(np.int64)                 # 4 * scale is an integer
        w4 = (u.astype(np.int64) - 8) * np.repeat(s4, inputs.W4_GROUP, axis=1)
        xi = _decode(x).astype(np.int64)
        assert np.array_equal(y * 4, (xi @ w4.T).astype(np.float64)), (N, K)
        assert np.array_equal(sc * 4, (np.abs(xi) @ np.abs(w4).T).astype(np.float64))


def w4_one_hot(lib):
    N, K = 6, 384
    Wq, S, u = _w4_case(N, K, 1, seed=31)
    Sd = _decode(S)
    for k in list(range(8)) + [127, 128, 129, 255, 383]:
        x = np.zeros((1, K), dtype=np.uint16)
        x[0, k] = 0x3F80
        y, _ = lib.gemv_w4(Wq, S, x, K)
        want = (u[:, k].astype(np.float64) - 8) * Sd[:, k // inputs.W4_GROUP]
        assert np.array_equal(y[0], want), k


def w4_dense(lib):
    N, K, B = 40, 1024, 4
    Wq, S, u = _w4_case(N, K, B, seed=32)
    x = inputs.bits(inputs.activations(B, K, seed=33))
    y, sc = lib.gemv_w4(Wq, S, x, K)
    Wd = (u.astype(np.float64) - 8) * np.repeat(_decode(S), inputs.W4_GROUP, axis=1)
    xd = _decode(x)
    assert np.all(np.abs(y - xd @ Wd.T) <= 4 * K * EPS64 * sc)
    assert np.allclose(sc, np.abs(xd) @ np.abs(Wd).T, rtol=1e-12, atol=0)
    zero = inputs.w4_pack(np.full((N, K), 8, dtype=np.uint8))
    y0, s0 = lib.gemv_w4(zero, S, x, K)
    assert np.array_equal(y0, np.zeros_like(y0)) and np.array_equal(s0, np.zeros_like(s0))


def fp8_decode_table(lib):
    N, K = 256, 1
    Wq = np.arange(256, dtype=np.uint8).reshape(N, K)
    S = np.ones(N, dtype=np.float32)
    x = np.array([[0x3F80]], dtype=np.uint16)          # 1.0
    y, sc = lib.gemv_fp8(Wq, S, x, K)
    want = inputs.fp8_decode(Wq[:, 0])
    nan = np.isnan(want)
    assert set(np.flatnonzero(nan)) == {0x7F, 0xFF}
    assert np.all(np.isnan(y[0, nan]))
    assert np.array_equal(y[0, ~nan], want[~nan])
    for code, value in ((0x38, 1.0), (0x7E, 448.0), (0x08, 2.0 ** -6), (0x01, 2.0 ** -9),
                        (0x07, 7 * 2.0 ** -9), (0xB8, -1.0), (0x3C, 1.5), (0x00, 0.0)):
        assert y[0, code] == value, hex(code)
    assert y[0, 0x80] == 0.0 and sc[0, 0x80] == 0.0      # -0 (a sum from +0 loses its sign)


def _fp8_codes_of(values: np.ndarray) -> np.ndarray:
    return torch.as_tensor(values, dtype=torch.float32).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def fp8_integer_exact(lib):
    rng = np.random.default_rng(5)
    for (N, K, B, ldq) in [(7, 64, 2, 64), (9, 300, 3, 304), (3, 17, 1, 32)]:
        wi = rng.integers(-8, 9, size=(N, K))               # |w| <= 8: exact in E4M3
        codes = np.zeros((N, ldq), dtype=np.uint8)
        codes[:, :K] = _fp8_codes_of(wi.astype(np.float32))
        shifts = (np.arange(N) % 4) - 1                       # row scales 2^-1 .. 2^2
        S = (2.0 ** shifts).astype(np.float32)
        x = inputs.bits(inputs.int_activations(B, K, lo=-3, hi=3, seed=N))
        y, sc = lib.gemv_fp8(codes, S, x, K)
        xi = _decode(x).astype(np.int64)
        w2 = wi * (2 ** (shifts + 1))[:, None]                # 2 * w * S, an integer
        assert np.array_equal(y * 2, (xi @ w2.T).astype(np.float64)), (N, K)
        assert np.array_equal(sc * 2, (np.abs(xi) @ np.abs(w2).T).astype(np.float64))


def fp8_dense(lib):
    N, K, B, ldq = 33, 1000, 3, 1024
    Wq, S = inputs.fp8_weight(N, K, ldq, seed=44)
    Wq, S = Wq.numpy(), S.numpy()
    assert np.all(Wq[:, K:] == inputs.FP8_PAD)
    x = inputs.bits(inputs.activations(B, K, seed=45))
    y, sc = lib.gemv_fp8(Wq, S, x, K)
    Wd = inputs.fp8_decode(Wq[:, :K]) * S.astype(np.float64)[:, None]
    xd = _decode(x)
    assert np.all(np.isfinite(y))
    assert np.all(np.abs(y - xd @ Wd.T) <= 4 * K * EPS64 * sc)
    assert np.allclose(sc, np.abs(xd) @ np.abs(Wd).T, rtol=1e-12, atol=0)
    # a sign flip of every code negates y
    yn, _ = lib.gemv_fp8(Wq ^ np.uint8(0x80), S, x, K)
    assert np.array_equal(yn, -y)


ALL_PINS = [exact_rational, integer_matmul, ones_row_sums, one_hot_column,
            identity_padded, scaling_exact, linearity, row_permutation,
            batch_rows, padding_unread, float64_matmul, single_element,
            rms_constant_x, rms_scale_free, rms_independent,
            w4_integer_exact, w4_one_hot, w4_dense,
            fp8_decode_table, fp8_integer_exact, fp8_dense]


def failures(lib) -> list[str]:
    out = []
    for pin in ALL_PINS:
        try:
            pin(lib)
        except AssertionError as e:
            out.append(f"{pin.__name__}: {e}")
        except Exception as e:  # a broken oracle may also crash a pin
            out.append(f"{pin.__name__}: {type(e).__name__}: {e}")
    return out
