"""Python front end of the CPU oracle for y = W·x (BF16 in, FP64 accumulate).

TEST INFRASTRUCTURE ONLY. The product path never imports this module: only the
tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg do. It
shares no code with the CUDA library; both sides see the same input bits, which
come from the seeded generators, never from the CUDA path.

The arithmetic lives in ``gemv_oracle.c`` (plain C, FP64, k ascending); this
file compiles it with the host C compiler, loads it with ctypes and splits the
rows over threads (ctypes releases the GIL during the call, so the threads run
in parallel; each thread owns a disjoint range of output rows, so threading does
not change any result).

The acceptance rule for the decode GEMV: an FP32
result may differ from the exact value only by summation rounding, so each
element is accepted when |y_gpu - y_ref| <= rtol * sum_k |W[n,k] * x[b,k]|
and y_gpu is finite ("Decode GEMV at half of HBM bandwidth", "A strong answer":
the kernel accumulates in FP32 and only the order of additions differs).
"""
from __future__ import annotations

import ctypes
import os
import platform
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "gemv_oracle.c")
BUILD_DIR = os.path.join(_HERE, "_build")

RTOL = 1e-5

_lock = threading.Lock()
_cache: dict[str, "OracleLib"] = {}


def lib_path(tag: str = "") -> str:
    name = f"liboracle_{platform.machine()}{tag}.so"
    return os.path.join(BUILD_DIR, name)


def build(source: str = SOURCE, out: str | None = None, force: bool = False) -> str:
    """Compile the C oracle into a shared library and return its path.

    Plain ``-O2`` with contraction off, so every product and sum is the single
    IEEE operation the C source writes.
    """
    out = out or lib_path()
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(source)):
        return out
    tmp = f"{out}.{os.getpid()}.tmp"
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
           "-shared", "-fPIC", "-o", tmp, source, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


class OracleLib:
    """ctypes handle on one compiled oracle library."""

    def __init__(self, path: str):
        self.path = path
        self._lib = ctypes.CDLL(path)
        i64 = ctypes.c_int64
        vp = ctypes.c_void_p
        f = self._lib.oracle_gemv_f64
        f.restype = ctypes.c_int
        f.argtypes = [vp, vp, i64, i64, i64, i64, i64, i64, vp, vp]
        g = self._lib.oracle_gemv_f64_one
        g.restype = ctypes.c_int
        g.argtypes = [vp, vp, i64, i64, i64, i64, i64, i64, vp, vp]
        h = self._lib.oracle_gemv_rmsnorm_f64
        h.restype = ctypes.c_int
        h.argtypes = [vp, vp, i64, i64, i64, i64, ctypes.c_double, i64, i64, vp, vp, vp]
        q = self._lib.oracle_gemv_w4_f64
        q.restype = ctypes.c_int
        q.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, i64, i64, i64, vp, vp]
        f8 = self._lib.oracle_gemv_fp8_f64
        f8.restype = ctypes.c_int
        f8.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, i64, vp, vp]

    def gemv(self, W: np.ndarray, x: np.ndarray, K: int | None = None,
             threads: int | None = None) -> tuple[np.ndarray, np.ndarray]:
        """Return (y_ref, scale), both float64 of shape [B, N].

        ``W`` is uint16 [N, ldw] (BF16 bits), ``x`` is uint16 [B, K] or [K].
        """
        W, x, N, K, B, ldw = _check(W, x, K)
        y = np.empty((B, N), dtype=np.float64)
        s = np.empty((B, N), dtype=np.float64)
        threads = max(1, min(threads or 1, N))
        bounds = np.linspace(0, N, threads + 1).astype(np.int64)

        def run(i: int) -> int:
            return self._lib.oracle_gemv_f64(
                W.ctypes.data, x.ctypes.data, N, K, B, ldw,
                int(bounds[i]), int(bounds[i + 1]), y.ctypes.data, s.ctypes.data)

        if threads == 1:
            rcs = [run(0)]
        else:
            with ThreadPoolExecutor(max_workers=threads) as ex:
                rcs = list(ex.map(run, range(threads)))
        if any(rc != 0 for rc in rcs):
            raise ValueError("oracle rejected its arguments")
        return y, s

    def gemv_rmsnorm(self, W: np.ndarray, x: np.ndarray, eps: float, K: int | None = None,
                     threads: int | None = None) -> tuple[np.ndarray, np.ndarray, np.ndarray]:
        """Return (y_ref, scale, r): the GEMV of the RMS-normalised x.

        r[b] = (mean_k x[b][k]^2 + eps)^(-1/2); y_ref and scale as for gemv, times r[b].
        """
        W, x, N, K, B, ldw = _check(W, x, K)
        y = np.empty((B, N), dtype=np.float64)
        s = np.empty((B, N), dtype=np.float64)
        r = np.empty((B,), dtype=np.float64)
        threads = max(1, min(threads or 1, N))
        bounds = np.linspace(0, N, threads + 1).astype(np.int64)
        rs = [np.empty((B,), dtype=np.float64) for _ in range(threads)]

        def run(i: int) -> int:
            return self._lib.oracle_gemv_rmsnorm_f64(
                W.ctypes.data, x.ctypes.data, N, K, B, ldw, float(eps),
                int(bounds[i]), int(bounds[i + 1]), y.ctypes.data, s.ctypes.data, rs[i].ctypes.data)

        if threads == 1:
            rcs = [run(0)]
        else:
            with ThreadPoolExecutor(max_workers=threads) as ex:
                rcs = list(ex.map(run, range(threads)))
        if any(rc != 0 for rc in rcs):
            raise ValueError("oracle rejected its arguments")
        r[:] = rs[0]
        return y, s, r

    def gemv_w4(self, Wq: np.ndarray, S: np.ndarray, x: np.ndarray, K: int, group: int = 128,
                threads: int | None = None) -> tuple[np.ndarray, np.ndarray]:
        """(y_ref, scale) of the INT4 GEMV. Wq uint8 [N, ldq], S uint16 [N, lds]
        (BF16 bits), x uint16 [B, K]."""
        if Wq.dtype != np.uint8 or S.dtype != np.uint16 or x.dtype != np.uint16:
            raise TypeError("Wq uint8, S and x BF16 bits as uint16")
        if x.ndim == 1:
            x = x[None, :]
        Wq = np.ascontiguousarray(Wq)
        S = np.ascontiguousarray(S)
        x = np.ascontiguousarray(x)
        N, ldq = Wq.shape
        lds = S.shape[1]
        B = x.shape[0]
        if x.shape[1] != K or S.shape[0] != N:
            raise ValueError("shapes disagree")
        y = np.empty((B, N), dtype=np.float64)
        s = np.empty((B, N), dtype=np.float64)
        threads = max(1, min(threads or 1, N))
        bounds = np.linspace(0, N, threads + 1).astype(np.int64)

        def run(i: int) -> int:
            return self._lib.oracle_gemv_w4_f64(
                Wq.ctypes.data, S.ctypes.data, x.ctypes.data, N, K, B, ldq, lds, group,
                int(bounds[i]), int(bounds[i + 1]), y.ctypes.data, s.ctypes.data)

        if threads == 1:
            rcs = [run(0)]
        else:
            with ThreadPoolExecutor(max_workers=threads) as ex:
                rcs = list(ex.map(run, range(threads)))
        if any(rc != 0 for rc in rcs):
            raise ValueError("oracle rejected its arguments")
        return y, s

    def gemv_fp8(self, Wq: np.ndarray, S: np.ndarray, x: np.ndarray, K: int,
                 threads: int | None = None) -> tuple[np.ndarray, np.ndarray]:
        """(y_ref, scale) of the FP8 (E4M3) GEMV. Wq uint8 [N, ldq] codes,
        S float32 [N] row scales, x uint16 [B, K] (BF16 bits)."""
        if Wq.dtype != np.uint8 or S.dtype != np.float32 or x.dtype != np.uint16:
            raise TypeError("Wq uint8 codes, S float32, x BF16 bits as uint16")
        if x.ndim == 1:
            x = x[None, :]
        Wq = np.ascontiguousarray(Wq)
        S = np.ascontiguousarray(S.reshape(-1))
        x = np.ascontiguousarray(x)
        N, ldq = Wq.shape
        B = x.shape[0]
        if x.shape[1] != K or S.shape[0] != N:
            raise ValueError("shapes disagree")
        y = np.empty((B, N), dtype=np.float64)
        s = np.empty((B, N), dtype=np.float64)
        threads = max(1, min(threads or 1, N))
        bounds = np.linspace(0, N, threads + 1).astype(np.int64)

        def run(i: int) -> int:
            return self._lib.oracle_gemv_fp8_f64(
                Wq.ctypes.data, S.ctypes.data, x.ctypes.data, N, K, B, ldq,
                int(bounds[i]), int(bounds[i + 1]), y.ctypes.data, s.ctypes.data)

        if threads == 1:
            rcs = [run(0)]
        else:
            with ThreadPoolExecutor(max_workers=threads) as ex:
                rcs = list(ex.map(run, range(threads)))
        if any(rc != 0 for rc in rcs):
            raise ValueError("oracle rejected its arguments")
        return y, s

    def gemv_one(self, W: np.ndarray, x: np.ndarray, b: int, n: int,
                 K: int | None = None) -> tuple[float, float]:
        """Return (y_ref[b, n], scale[b, n]) for a single output element."""
        W, x, N, K, B, ldw = _check(W, x, K)
        yo = ctypes.c_double()
        so = ctypes.c_double()
        rc = self._lib.oracle_gemv_f64_one(
            W.ctypes.data, x.ctypes.data, N, K, B, ldw, b, n,
            ctypes.addressof(yo), ctypes.addressof(so))
        if rc != 0:
            raise ValueError("oracle rejected its arguments")
        return yo.value, so.value


def _check(W: np.ndarray, x: np.ndarray, K: int | None):
    if W.dtype != np.uint16 or x.dtype != np.uint16:
        raise TypeError("oracle inputs are BF16 bit patterns as uint16 arrays")
    if W.ndim != 2:
        raise ValueError("W must be [N, ldw]")
    if x.ndim == 1:
        x = x[None, :]
    N, ldw = W.shape
    B, kx = x.shape
    K = kx if K is None else int(K)
    if kx != K or K > ldw:
        raise ValueError("x must be [B, K] with K <= ldw")
    W = np.ascontiguousarray(W)
    x = np.ascontiguousarray(x)
    return W, x, int(N), int(K), int(B), int(ldw)


def load(path: str | None = None) -> OracleLib:
    """Build (if needed) and load the oracle library; cached per path."""
    with _lock:
        path = path or build()
        if path not in _cache:
            _cache[path] = OracleLib(path)
        return _cache[path]


def gemv(W: np.ndarray, x: np.ndarray, K: int | None = None,
         threads: int | None = None) -> tuple[np.ndarray, np.ndarray]:
    return load().gemv(W, x, K, threads)


def gemv_rmsnorm(W: np.ndarray, x: np.ndarray, eps: float, K: int | None = None,
                 threads: int | None = None):
    return load().gemv_rmsnorm(W, x, eps, K, threads)


def gemv_w4(Wq: np.ndarray, S: np.ndarray, x: np.ndarray, K: int, group: int = 128,
            threads: int | None = None):
    return load().gemv_w4(Wq, S, x, K, group, threads)


def gemv_fp8(Wq: np.ndarray, S: np.ndarray, x: np.ndarray, K: int, threads: int | None = None):
    return load().gemv_fp8(Wq, S, x, K, threads)


def gemv_one(W: np.ndarray, x: np.ndarray, b: int, n: int, K: int | None = None):
    return load().gemv_one(W, x, b, n, K)


def accept(y_gpu: np.ndarray, y_ref: np.ndarray, scale: np.ndarray,
           rtol: float = RTOL) -> np.ndarray:
    """Boolean mask of accepted elements: finite and within rtol * scale.

    Where scale is 0 every term is zero, so the result must be exactly zero
    (either sign).
    """
    y_gpu = np.asarray(y_gpu, dtype=np.float64)
    return np.isfinite(y_gpu) & (np.abs(y_gpu - y_ref) <= rtol * scale)


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1
