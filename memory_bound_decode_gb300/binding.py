"""Python binding of libgemv.so: argument marshalling only.

Every function here has the name of the C entry point it calls (include/gemv.h)
and does nothing but turn tensors into pointers and streams into handles. There
is no fallback: if the library is not built, the first call raises.

Pointers may be given as integers or as tensors (their ``data_ptr()``);
``stream`` may be an integer handle, a ``torch.cuda.Stream`` or None (the
current PyTorch stream).
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "_lib", "libgemv.so")

GEMV_OK = 0
GEMV_ERR_INVALID = -1
GEMV_ERR_ALIGN = -2
GEMV_ERR_CUDA = -3
GEMV_ERR_NOMEM = -4
GEMV_ERR_CAPTURE = -5
GEMV_ERR_UNSUPPORTED = -6
GEMV_MAX_BATCH = 16
GEMV_MAX_SEGMENTS = 8

GEMV_FLAG_RMSNORM = 1
GEMV_FLAG_STREAMK = 2
GEMV_FLAG_CUDA_CORES = 4

GEMV_WEIGHT_BF16 = 0
GEMV_WEIGHT_INT4 = 1
GEMV_WEIGHT_FP8 = 2

EXPORTED = [
    "gemv_bf16", "gemv_bf16_ex", "gemv_bf16_host_io", "gemv_bf16_multi", "gemv_bf16_multi_ex",
    "gemv_bf16_multi_host_io",
    "gemv_plan_create", "gemv_plan_capture",
    "gemv_plan_launch", "gemv_plan_launch_host_io", "gemv_plan_num_launches", "gemv_plan_independent",
    "gemv_plan_destroy",
    "gemv_query_launch", "gemv_query_launch_ex", "gemv_workspace_release", "gemv_device_status",
    "gemv_bf16_streamk_noalloc",
    "gemv_debug_write_count",
    "gemv_w4_bf16", "gemv_w4_query_launch", "gemv_fp8_bf16", "gemv_fp8_query_launch",
    "gemv_probe_stream_read", "gemv_probe_sink_words",
    "gemv_status_string", "gemv_last_cuda_error",
]

i64 = ctypes.c_int64
vp = ctypes.c_void_p


class gemv_segment(ctypes.Structure):
    _fields_ = [("W", vp), ("y", vp), ("N", i64), ("ldw", i64)]


class gemv_proj(ctypes.Structure):
    _fields_ = [("W", vp), ("x", vp), ("y", vp), ("N", i64), ("K", i64), ("ldw", i64),
                ("B", ctypes.c_int), ("fuse_group", ctypes.c_int), ("flags", ctypes.c_int),
                ("rms_eps", ctypes.c_float), ("weight_kind", ctypes.c_int), ("S", vp), ("lds", i64)]


class gemv_options(ctypes.Structure):
    _fields_ = [("flags", ctypes.c_int), ("rms_eps", ctypes.c_float)]


class gemv_launch_info(ctypes.Structure):
    _fields_ = [("rows_per_cta", i64), ("row_tiles", i64), ("grid", i64), ("kslice", i64),
                ("kchunk", i64), ("warps_per_cta", ctypes.c_int32), ("warps_per_row", ctypes.c_int32),
                ("splits", ctypes.c_int32), ("rows_per_warp", ctypes.c_int32),
                ("unroll", ctypes.c_int32), ("smem_bytes", ctypes.c_int32), ("path", ctypes.c_int32),
                ("xstride", ctypes.c_int32), ("nbuf", ctypes.c_int32),
                ("units", i64), ("warps", i64), ("chunks", ctypes.c_int32), ("ctas_per_sm", ctypes.c_int32),
                ("dp_rounds", ctypes.c_int32), ("mcast", ctypes.c_int32), ("xbox", ctypes.c_int32),
                ("xpieces", ctypes.c_int32), ("xboxes_per_piece", ctypes.c_int32), ("persistent", ctypes.c_int32),
                ("l2_prefetch", ctypes.c_int32)]

    def as_dict(self) -> dict:
        return {name: getattr(self, name) for name, _ in self._fields_}


class GemvError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = gemv_status_string(status)
        if status == GEMV_ERR_CUDA:
            msg += f" (cudaError {gemv_last_cuda_error()})"
        super().__init__(f"{where}: {msg}")


_lock = threading.Lock()
_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            _lib = _load(LIB_PATH)
        return _lib


@contextlib.contextmanager
def use_library(path: str):
    """Route every call in the block to another build of the library (the
    store-counting test build); the default library is restored afterwards."""
    global _lib
    other = _load(path)
    with _lock:
        saved = _lib
        _lib = other
    try:
        yield other
    finally:
        with _lock:
            _lib = saved


def _load(path: str) -> ctypes.CDLL:
    """Load one build of the library and declare its signatures."""
    if not os.path.exists(path):
        raise RuntimeError(f"libgemv.so is not built ({path}); "
                           "run memory_bound_decode_gb300.build_lib.build()")
    L = ctypes.CDLL(path)
    L.gemv_bf16.argtypes = [vp, vp, vp, i64, i64, ctypes.c_int, i64, vp]
    L.gemv_bf16_multi.argtypes = [ctypes.POINTER(gemv_segment), ctypes.c_int, vp, i64,
                                  ctypes.c_int, vp]
    L.gemv_bf16_ex.argtypes = [vp, vp, vp, i64, i64, ctypes.c_int, i64,
                               ctypes.POINTER(gemv_options), vp]
    L.gemv_bf16_multi_ex.argtypes = [ctypes.POINTER(gemv_segment), ctypes.c_int, vp, i64,
                                     ctypes.c_int, ctypes.POINTER(gemv_options), vp]
    L.gemv_bf16_host_io.argtypes = [vp, vp, vp, vp, vp, i64, i64, ctypes.c_int, i64,
                                    ctypes.POINTER(gemv_options), vp]
    L.gemv_plan_create.argtypes = [ctypes.POINTER(gemv_proj), ctypes.c_int,
                                   ctypes.POINTER(vp)]
    L.gemv_plan_capture.argtypes = [vp, vp]
    L.gemv_plan_launch.argtypes = [vp, vp]
    L.gemv_plan_launch_host_io.argtypes = [vp, vp, vp, i64, vp, vp, i64, vp]
    L.gemv_bf16_multi_host_io.argtypes = [ctypes.POINTER(gemv_segment), ctypes.c_int, vp, vp,
                                          ctypes.POINTER(vp), i64, ctypes.c_int,
                                          ctypes.POINTER(gemv_options), vp]
    L.gemv_plan_num_launches.argtypes = [vp]
    L.gemv_plan_independent.argtypes = [vp]
    L.gemv_plan_destroy.argtypes = [vp]
    L.gemv_plan_destroy.restype = None
    L.gemv_query_launch.argtypes = [i64, i64, ctypes.c_int, ctypes.c_int,
                                    ctypes.POINTER(gemv_launch_info)]
    L.gemv_query_launch_ex.argtypes = [i64, i64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                       ctypes.POINTER(gemv_launch_info)]
    L.gemv_workspace_release.argtypes = []
    L.gemv_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint), ctypes.c_int]
    L.gemv_debug_write_count.argtypes = [vp, vp, i64]
    L.gemv_bf16_streamk_noalloc.argtypes = [vp, vp, vp, i64, i64, i64, ctypes.POINTER(gemv_options), vp]
    L.gemv_w4_bf16.argtypes = [vp, vp, vp, vp, i64, i64, ctypes.c_int, i64, i64,
                               ctypes.POINTER(gemv_options), vp]
    L.gemv_w4_query_launch.argtypes = [i64, i64, ctypes.c_int, ctypes.c_int,
                                       ctypes.POINTER(gemv_launch_info)]
    L.gemv_fp8_bf16.argtypes = [vp, vp, vp, vp, i64, i64, ctypes.c_int, i64,
                                ctypes.POINTER(gemv_options), vp]
    L.gemv_fp8_query_launch.argtypes = [i64, i64, ctypes.c_int, ctypes.c_int,
                                        ctypes.POINTER(gemv_launch_info)]
    L.gemv_probe_stream_read.argtypes = [vp, i64, vp, vp]
    L.gemv_probe_sink_words.argtypes = []
    L.gemv_status_string.argtypes = [ctypes.c_int]
    L.gemv_status_string.restype = ctypes.c_char_p
    L.gemv_last_cuda_error.argtypes = []
    for name in EXPORTED:
        f = getattr(L, name)
        if name not in ("gemv_plan_destroy", "gemv_status_string"):
            f.restype = ctypes.c_int
    return L


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(s) -> int | None:
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else None
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(rc: int, where: str) -> int:
    if rc != GEMV_OK:
        raise GemvError(rc, where)
    return rc


def gemv_status_string(status: int) -> str:
    return lib().gemv_status_string(int(status)).decode()


def gemv_last_cuda_error() -> int:
    return lib().gemv_last_cuda_error()


def gemv_bf16(W, x, y, N: int, K: int, B: int, ldw: int, stream=None, check: bool = True) -> int:
    rc = lib().gemv_bf16(_ptr(W), _ptr(x), _ptr(y), N, K, B, ldw, _stream(stream))
    return _check(rc, "gemv_bf16") if check else rc


def _options(rms_eps, streamk: bool = False, cuda_cores: bool = False):
    if rms_eps is None and not streamk and not cuda_cores:
        return None
    flags = ((GEMV_FLAG_RMSNORM if rms_eps is not None else 0) | (GEMV_FLAG_STREAMK if streamk else 0)
             | (GEMV_FLAG_CUDA_CORES if cuda_cores else 0))
    return ctypes.byref(gemv_options(flags, float(rms_eps) if rms_eps is not None else 0.0))


def gemv_bf16_ex(W, x, y, N: int, K: int, B: int, ldw: int, rms_eps=None, stream=None,
                 check: bool = True, options=None, streamk: bool = False, cuda_cores: bool = False) -> int:
    """gemv_bf16 with options; ``rms_eps`` (not None) turns on the RMSNorm prologue,
    ``streamk`` the stream-K kernel, ``cuda_cores`` the CUDA-core kernel at every
    batch size. ``options`` (a gemv_options) overrides them."""
    opt = ctypes.byref(options) if options is not None else _options(rms_eps, streamk, cuda_cores)
    rc = lib().gemv_bf16_ex(_ptr(W), _ptr(x), _ptr(y), N, K, B, ldw, opt, _stream(stream))
    return _check(rc, "gemv_bf16_ex") if check else rc


def gemv_bf16_host_io(W, x_host, y_host, x_dev, y_dev, N: int, K: int, B: int, ldw: int, rms_eps=None,
                      stream=None, check: bool = True, streamk: bool = False, cuda_cores: bool = False) -> int:
    """Host x in, host y out, synchronous (see gemv.h)."""
    rc = lib().gemv_bf16_host_io(_ptr(W), _ptr(x_host), _ptr(y_host), _ptr(x_dev), _ptr(y_dev), N, K, B, ldw,
                                 _options(rms_eps, streamk, cuda_cores), _stream(stream))
    return _check(rc, "gemv_bf16_host_io") if check else rc


def gemv_bf16_multi_ex(segments, x, K: int, B: int, rms_eps=None, stream=None, check: bool = True,
                       options=None, streamk: bool = False, cuda_cores: bool = False) -> int:
    arr = (gemv_segment * max(1, len(segments)))()
    for i, (W, y, N, ldw) in enumerate(segments):
        arr[i] = gemv_segment(_ptr(W), _ptr(y), N, ldw)
    opt = ctypes.byref(options) if options is not None else _options(rms_eps, streamk, cuda_cores)
    rc = lib().gemv_bf16_multi_ex(arr, len(segments), _ptr(x), K, B, opt, _stream(stream))
    return _check(rc, "gemv_bf16_multi_ex") if check else rc


def gemv_bf16_multi_host_io(segments, x_host, x_dev, y_host, K: int, B: int, rms_eps=None, stream=None,
                            check: bool = True, streamk: bool = False, cuda_cores: bool = False) -> int:
    """Host x in, fused launch over ``segments`` (W, y_dev, N, ldw), each
    segment's y copied to ``y_host[i]``, synchronous (see gemv.h)."""
    n = len(segments)
    arr = (gemv_segment * max(1, n))()
    for i, (W, y, N, ldw) in enumerate(segments):
        arr[i] = gemv_segment(_ptr(W), _ptr(y), N, ldw)
    yh = (vp * max(1, n))(*[_ptr(t) for t in y_host])
    rc = lib().gemv_bf16_multi_host_io(arr, n, _ptr(x_host), _ptr(x_dev), yh, K, B,
                                       _options(rms_eps, streamk, cuda_cores), _stream(stream))
    return _check(rc, "gemv_bf16_multi_host_io") if check else rc


def gemv_bf16_multi(segments, x, K: int, B: int, stream=None, check: bool = True) -> int:
    """``segments``: sequence of (W, y, N, ldw)."""
    arr = (gemv_segment * max(1, len(segments)))()
    for i, (W, y, N, ldw) in enumerate(segments):
        arr[i] = gemv_segment(_ptr(W), _ptr(y), N, ldw)
    rc = lib().gemv_bf16_multi(arr, len(segments), _ptr(x), K, B, _stream(stream))
    return _check(rc, "gemv_bf16_multi") if check else rc


def gemv_query_launch(N: int, K: int, B: int, sm_count: int) -> dict:
    info = gemv_launch_info()
    _check(lib().gemv_query_launch(N, K, B, sm_count, ctypes.byref(info)), "gemv_query_launch")
    return info.as_dict()


def gemv_query_launch_ex(N: int, K: int, B: int, sm_count: int, flags: int) -> dict:
    info = gemv_launch_info()
    _check(lib().gemv_query_launch_ex(N, K, B, sm_count, flags, ctypes.byref(info)), "gemv_query_launch_ex")
    return info.as_dict()


def gemv_bf16_streamk_noalloc(W, x, y, N: int, K: int, ldw: int, rms_eps=None, stream=None,
                              check: bool = True) -> int:
    """The stream-K GEMV (batch 1) with the library's fixed scratch: no allocation (see gemv.h)."""
    rc = lib().gemv_bf16_streamk_noalloc(_ptr(W), _ptr(x), _ptr(y), N, K, ldw, _options(rms_eps),
                                         _stream(stream))
    return _check(rc, "gemv_bf16_streamk_noalloc") if check else rc


def gemv_debug_write_count(counts, y_base, n: int, check: bool = True) -> int:
    """Test support (a GEMV_DEBUG_WRITECOUNT build only): count output stores."""
    rc = lib().gemv_debug_write_count(_ptr(counts), _ptr(y_base), n)
    return _check(rc, "gemv_debug_write_count") if check else rc


def gemv_workspace_release() -> int:
    return _check(lib().gemv_workspace_release(), "gemv_workspace_release")


GEMV_STATUS_WAIT_TIMEOUT = 1


def gemv_device_status(reset: bool = True) -> int:
    """Status bits the kernels recorded on the current device (GEMV_STATUS_*),
    cleared when ``reset``."""
    bits = ctypes.c_uint(0)
    _check(lib().gemv_device_status(ctypes.byref(bits), 1 if reset else 0), "gemv_device_status")
    return bits.value


def gemv_w4_bf16(Wq, S, x, y, N: int, K: int, B: int, ldq: int, lds: int, rms_eps=None,
                 stream=None, check: bool = True, options=None) -> int:
    opt = ctypes.byref(options) if options is not None else _options(rms_eps)
    rc = lib().gemv_w4_bf16(_ptr(Wq), _ptr(S), _ptr(x), _ptr(y), N, K, B, ldq, lds, opt, _stream(stream))
    return _check(rc, "gemv_w4_bf16") if check else rc


def gemv_w4_query_launch(N: int, K: int, B: int, sm_count: int) -> dict:
    info = gemv_launch_info()
    _check(lib().gemv_w4_query_launch(N, K, B, sm_count, ctypes.byref(info)), "gemv_w4_query_launch")
    return info.as_dict()


def gemv_fp8_bf16(Wq, S, x, y, N: int, K: int, B: int, ldq: int, rms_eps=None,
                  stream=None, check: bool = True, options=None) -> int:
    """FP8 (E4M3) weights with FP32 row scales S (see gemv.h)."""
    opt = ctypes.byref(options) if options is not None else _options(rms_eps)
    rc = lib().gemv_fp8_bf16(_ptr(Wq), _ptr(S), _ptr(x), _ptr(y), N, K, B, ldq, opt, _stream(stream))
    return _check(rc, "gemv_fp8_bf16") if check else rc


def gemv_fp8_query_launch(N: int, K: int, B: int, sm_count: int) -> dict:
    info = gemv_launch_info()
    _check(lib().gemv_fp8_query_launch(N, K, B, sm_count, ctypes.byref(info)), "gemv_fp8_query_launch")
    return info.as_dict()


def gemv_probe_sink_words() -> int:
    return lib().gemv_probe_sink_words()


def gemv_probe_stream_read(src, nbytes: int, sink, stream=None) -> int:
    return _check(lib().gemv_probe_stream_read(_ptr(src), nbytes, _ptr(sink), _stream(stream)),
                  "gemv_probe_stream_read")


class Plan:
    """Owner of a gemv_plan handle (gemv_plan_create / capture / launch / destroy).

    ``projections``: sequence of (W, x, y, N, K, ldw, B, fuse_group),
    (W, x, y, N, K, ldw, B, fuse_group, rms_eps) with rms_eps None for no
    RMSNorm prologue, (..., rms_eps, streamk) with streamk a bool, or
    (..., rms_eps, streamk, weight_kind, S, lds) for INT4 / FP8 weights (W the
    codes, ldw their row stride in bytes, S the scales). The tensors behind the
    pointers must outlive the plan; keep them referenced.
    """

    def __init__(self, projections, keepalive=None):
        n = len(projections)
        arr = (gemv_proj * max(1, n))()
        for i, pr in enumerate(projections):
            W, x, y, N, K, ldw, B, grp = pr[:8]
            eps = pr[8] if len(pr) > 8 else None
            sk = bool(pr[9]) if len(pr) > 9 else False
            kind = int(pr[10]) if len(pr) > 10 else GEMV_WEIGHT_BF16
            S = pr[11] if len(pr) > 11 else None
            lds = int(pr[12]) if len(pr) > 12 else 0
            flags = (GEMV_FLAG_RMSNORM if eps is not None else 0) | (GEMV_FLAG_STREAMK if sk else 0)
            arr[i] = gemv_proj(_ptr(W), _ptr(x), _ptr(y), N, K, ldw, B, grp, flags,
                               float(eps) if eps is not None else 0.0, kind, _ptr(S), lds)
        handle = vp()
        _check(lib().gemv_plan_create(arr, n, ctypes.byref(handle)), "gemv_plan_create")
        self._h = handle
        self._keepalive = keepalive

    @property
    def handle(self) -> int:
        return self._h.value or 0

    def capture(self, stream) -> None:
        _check(lib().gemv_plan_capture(self._h, _stream(stream)), "gemv_plan_capture")

    def launch(self, stream=None, check: bool = True) -> int:
        rc = lib().gemv_plan_launch(self._h, _stream(stream))
        return _check(rc, "gemv_plan_launch") if check else rc

    def launch_host_io(self, x_host, x_dev, x_bytes: int, y_dev, y_host, y_bytes: int, stream=None,
                       check: bool = True) -> int:
        """gemv_plan_launch_host_io: host x in, the captured step, host y out, synchronous."""
        rc = lib().gemv_plan_launch_host_io(self._h, _ptr(x_host), _ptr(x_dev), int(x_bytes), _ptr(y_dev),
                                            _ptr(y_host), int(y_bytes), _stream(stream))
        return _check(rc, "gemv_plan_launch_host_io") if check else rc

    def num_launches(self) -> int:
        return lib().gemv_plan_num_launches(self._h)

    def independent(self) -> bool:
        """Whether the plan's launches run without waiting for each other (see gemv.h)."""
        return bool(lib().gemv_plan_independent(self._h))

    def destroy(self) -> None:
        if self._h is not None and self._h.value:
            lib().gemv_plan_destroy(self._h)
        self._h = None

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass


def gemv_plan_create(projections, keepalive=None) -> Plan:
    return Plan(projections, keepalive)
