"""The C-ABI library on a machine without a GPU: it loads, exports every entry
point include/gemv.h declares, rejects bad arguments before touching the
device, and plans launches by the stated rules."""
import ctypes
import os
import re

import pytest

from memory_bound_decode_gb300 import binding, build_lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gemv.h")
GB300_SMS = 152


@pytest.fixture(scope="module")
def L():
    build_lib.build()
    return binding.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*[A-Za-z_][\w\s\*]*?\b(gemv_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ["gemv_bf16", "gemv_bf16_multi", "gemv_plan_create", "gemv_plan_capture",
                     "gemv_plan_launch", "gemv_plan_destroy", "gemv_status_string",
                     "gemv_last_cuda_error"]:
        assert required in names
    assert sorted(names) == sorted(binding.EXPORTED)


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), name
        assert ctypes.cast(getattr(L, name), ctypes.c_void_p).value


def test_status_strings(L):
    for s in [0, -1, -2, -3, -4, -5, -6]:
        assert binding.gemv_status_string(s).startswith("GEMV_")
    assert binding.gemv_status_string(12345) == "unknown gemv status"
    assert binding.gemv_last_cuda_error() == 0


A16 = 1 << 20   # a fake, 16-byte aligned address: never dereferenced by validation


@pytest.mark.parametrize("args,status", [
    ((0, A16, A16, 8, 8, 1, 8), binding.GEMV_ERR_INVALID),          # W NULL
    ((A16, 0, A16, 8, 8, 1, 8), binding.GEMV_ERR_INVALID),          # x NULL
    ((A16, A16, 0, 8, 8, 1, 8), binding.GEMV_ERR_INVALID),          # y NULL
    ((A16, A16, A16, 0, 8, 1, 8), binding.GEMV_ERR_INVALID),        # N = 0
    ((A16, A16, A16, 8, 0, 1, 8), binding.GEMV_ERR_INVALID),        # K = 0
    ((A16, A16, A16, 8, 8, 0, 8), binding.GEMV_ERR_INVALID),        # B = 0
    ((A16, A16, A16, 8, 8, 17, 8), binding.GEMV_ERR_INVALID),       # B > 16
    ((A16, A16, A16, 8, 9, 1, 8), binding.GEMV_ERR_INVALID),        # ldw < K
    ((A16, A16, A16, 8, 9, 1, 12), binding.GEMV_ERR_ALIGN),         # ldw % 8
    ((A16 + 8, A16, A16, 8, 8, 1, 8), binding.GEMV_ERR_ALIGN),      # W not 16-B aligned
    ((A16, A16 + 1, A16, 8, 8, 1, 8), binding.GEMV_ERR_ALIGN),      # x odd address
    ((A16, A16, A16 + 2, 8, 8, 1, 8), binding.GEMV_ERR_ALIGN),      # y not 4-B aligned
    ((A16, A16, A16, 1 << 31, 8, 1, 8), binding.GEMV_ERR_INVALID),  # N too large
])
def test_gemv_bf16_rejects_before_launch(L, args, status):
    assert binding.gemv_bf16(*args, stream=0, check=False) == status


def test_multi_rejects(L):
    seg = (A16, A16, 8, 8)
    assert binding.gemv_bf16_multi([], A16, 8, 1, stream=0, check=False) == binding.GEMV_ERR_INVALID
    assert binding.gemv_bf16_multi([seg] * 9, A16, 8, 1, stream=0, check=False) == binding.GEMV_ERR_INVALID
    assert binding.gemv_bf16_multi([seg, (A16 + 8, A16, 8, 8)], A16, 8, 1, stream=0,
                                   check=False) == binding.GEMV_ERR_ALIGN
    assert binding.gemv_bf16_multi([seg, (A16, A16, 8, 4)], A16, 8, 1, stream=0,
                                   check=False) == binding.GEMV_ERR_INVALID


def test_plan_rejects(L):
    good = (A16, A16, A16, 8, 8, 8, 1, 0)
    with pytest.raises(binding.GemvError) as e:
        binding.Plan([good, (A16, A16, A16, 8, 8, 8, 17, 0)])
    assert e.value.status == binding.GEMV_ERR_INVALID
    with pytest.raises(binding.GemvError) as e:
        binding.Plan([(A16, A16, A16, 8, 8, 8, 1, -1)])
    assert e.value.status == binding.GEMV_ERR_INVALID
    assert L.gemv_plan_create(None, 1, None) == binding.GEMV_ERR_INVALID
    assert L.gemv_plan_launch(None, None) == binding.GEMV_ERR_INVALID
    assert L.gemv_plan_capture(None, None) == binding.GEMV_ERR_INVALID
    assert L.gemv_plan_num_launches(None) == 0
    L.gemv_plan_destroy(None)


def test_probe_rejects(L):
    assert L.gemv_probe_stream_read(A16, 15, A16, None) == binding.GEMV_ERR_INVALID
    assert L.gemv_probe_stream_read(A16 + 4, 64, A16, None) == binding.GEMV_ERR_ALIGN
    assert binding.gemv_probe_sink_words() >= GB300_SMS * 8


SHAPES = [  # (N, K) of the decode projections and the ragged cases
    (1024, 4096), (4096, 14336), (6144, 4096), (28672, 4096), (4096, 4096), (128256, 4096),
    (7, 129), (4097, 4103), (1, 8191), (33, 65537), (1, 1), (3, 8), (100000, 300),
]


@pytest.mark.parametrize("B", [1, 2, 3, 4, 8, 16])
@pytest.mark.parametrize("N,K", SHAPES)
def test_plan_covers_the_problem(L, N, K, B):
    q = binding.gemv_query_launch(N, K, B, GB300_SMS)
    assert q["warps_per_cta"] * 32 == 256
    assert q["warps_per_row"] in (1, 2, 4, 8)
    assert 1 <= q["splits"] <= 8
    if q["path"] == 5:
        # the tcgen05 kernel: more than 8 rows of x, 128-row tiles, a grid of one wave that
        # fills the SMs; a power-of-two cluster along K, slices of whole 128-column stages;
        # or, with more tiles than one wave, a persistent grid taking equal shares of them
        assert (B > 8 or (B == 8 and N >= 16384)) and q["rows_per_cta"] == 128 and q["warps_per_row"] == 1
        assert q["row_tiles"] * 128 >= N > (q["row_tiles"] - 1) * 128
        assert GB300_SMS <= q["grid"] <= (3 if q["persistent"] else 2) * GB300_SMS
        if q["persistent"]:
            each = -(-q["row_tiles"] // q["grid"])
            assert q["splits"] == 1 and q["row_tiles"] > 2 * GB300_SMS
            assert (q["grid"] - 1) * each < q["row_tiles"] <= q["grid"] * each
        else:
            assert q["grid"] == q["row_tiles"] * q["splits"]
        assert q["splits"] in (1, 2, 4, 8) and q["kslice"] % 128 == 0
        assert q["splits"] * q["kslice"] >= K > (q["splits"] - 1) * q["kslice"]
        assert q["smem_bytes"] <= 227 * 1024
        assert q["l2_prefetch"] == 0
        return
    # L2 prefetch one batch ahead: batch 1 on the CUDA cores in grids of at most 8 CTAs per SM
    assert q["l2_prefetch"] == (1 if B == 1 and q["grid"] <= 8 * GB300_SMS else 0)
    # batch 1 on the CUDA cores, batches 2..16 on the BF16 tensor cores (16-row tiles)
    assert q["path"] == (0 if B == 1 else 1)
    assert q["rows_per_warp"] == (1 if B == 1 else 16)
    assert q["rows_per_cta"] == (8 // q["warps_per_row"]) * q["rows_per_warp"]
    assert q["row_tiles"] * q["rows_per_cta"] >= N > (q["row_tiles"] - 1) * q["rows_per_cta"]
    # x multicast: batch 1, no K split, one x chunk, x of at least 1,024 vectors; the
    # grid is then whole clusters of mcast CTAs along the rows
    if q["mcast"] > 1:
        assert B == 1 and q["splits"] == 1 and q["nbuf"] == 1 and K // 8 >= 1024 and q["mcast"] == 2
        assert q["grid"] == -(-q["row_tiles"] // q["mcast"]) * q["mcast"]
    else:
        assert q["mcast"] == 1
        assert not (B == 1 and q["splits"] == 1 and q["nbuf"] == 1 and K // 8 >= 1024 and q["row_tiles"] >= 2)
        assert q["grid"] == q["row_tiles"] * q["splits"]
    # K-slices are whole 256-column steps, cover K, and none is empty
    assert q["kslice"] % 256 == 0 and q["kchunk"] % 256 == 0
    assert q["splits"] * q["kslice"] >= K > (q["splits"] - 1) * q["kslice"]
    assert q["kchunk"] <= q["kslice"]
    # x fits its budget, double-buffered exactly when the slice takes several chunks
    assert q["xstride"] >= q["kchunk"]
    assert q["nbuf"] == (1 if q["kchunk"] == q["kslice"] else 2)
    assert q["nbuf"] * B * q["xstride"] * 2 <= 80 * 1024 or q["kchunk"] == 256
    assert q["smem_bytes"] <= 112 * 1024


def test_no_split_when_rows_fill_the_gpu(L):
    # "Splitting K on every shape, including those that already fill the
    # machine many times over" is the mistake to avoid: large-N projections
    # stream whole rows per warp with no split at all.
    for N, K in [(4096, 14336), (6144, 4096), (28672, 4096), (4096, 4096), (128256, 4096)]:
        q = binding.gemv_query_launch(N, K, 1, GB300_SMS)
        assert q["splits"] == 1 and q["warps_per_row"] == 1, (N, K, q)
        assert q["grid"] * 8 >= GB300_SMS * 16


def test_split_when_rows_do_not_fill_the_gpu(L):
    # few rows, long K: K is split until the GPU is covered
    q = binding.gemv_query_launch(33, 65537, 1, GB300_SMS)
    assert q["warps_per_row"] * q["splits"] > 1
    assert q["grid"] * 8 >= 33 * 8
    small = binding.gemv_query_launch(1024, 4096, 1, GB300_SMS)
    assert small["warps_per_row"] * small["splits"] > 1


def test_planner_rejects(L):
    with pytest.raises(binding.GemvError):
        binding.gemv_query_launch(0, 8, 1, GB300_SMS)
    with pytest.raises(binding.GemvError):
        binding.gemv_query_launch(8, 8, 17, GB300_SMS)
    with pytest.raises(binding.GemvError):
        binding.gemv_query_launch(8, 8, 1, 0)


def test_options_rejected_before_launch(L):
    ok = dict(stream=0, check=False)
    for flags in (8, 16, binding.GEMV_FLAG_STREAMK | binding.GEMV_FLAG_CUDA_CORES):   # unknown, conflicting
        bad_flags = binding.gemv_options(flags, 0.0)
        assert binding.gemv_bf16_ex(A16, A16, A16, 8, 8, 1, 8, options=bad_flags, **ok) == binding.GEMV_ERR_INVALID
    for eps in (-1.0, float("nan"), float("inf")):
        assert binding.gemv_bf16_ex(A16, A16, A16, 8, 8, 1, 8, rms_eps=eps, **ok) == binding.GEMV_ERR_INVALID
        assert binding.gemv_bf16_multi_ex([(A16, A16, 8, 8)], A16, 8, 1, rms_eps=eps, **ok) == binding.GEMV_ERR_INVALID
    with pytest.raises(binding.GemvError) as e:
        binding.Plan([(A16, A16, A16, 8, 8, 8, 1, 0, -1.0)])
    assert e.value.status == binding.GEMV_ERR_INVALID
    # argument checks still come first
    assert binding.gemv_bf16_ex(0, A16, A16, 8, 8, 1, 8, rms_eps=1e-5, **ok) == binding.GEMV_ERR_INVALID


def test_w4_rejects_before_launch(L):
    ok = dict(stream=0, check=False)
    f = binding.gemv_w4_bf16
    assert f(0, A16, A16, A16, 8, 128, 1, 64, 1, **ok) == binding.GEMV_ERR_INVALID          # Wq NULL
    assert f(A16, 0, A16, A16, 8, 128, 1, 64, 1, **ok) == binding.GEMV_ERR_INVALID          # S NULL
    assert f(A16, A16, A16, A16, 8, 100, 1, 64, 1, **ok) == binding.GEMV_ERR_INVALID        # K % 128
    assert f(A16, A16, A16, A16, 8, 256, 1, 64, 2, **ok) == binding.GEMV_ERR_INVALID        # ldq < K/2
    assert f(A16, A16, A16, A16, 8, 256, 1, 128, 1, **ok) == binding.GEMV_ERR_INVALID       # lds < K/128
    assert f(A16, A16, A16, A16, 8, 256, 17, 128, 2, **ok) == binding.GEMV_ERR_INVALID      # B > 16
    assert f(A16, A16, A16, A16, 8, 256, 1, 136, 2, **ok) == binding.GEMV_ERR_ALIGN         # ldq % 16
    assert f(A16 + 8, A16, A16, A16, 8, 256, 1, 128, 2, **ok) == binding.GEMV_ERR_ALIGN     # Wq alignment
    assert f(A16, A16 + 1, A16, A16, 8, 256, 1, 128, 2, **ok) == binding.GEMV_ERR_ALIGN     # S alignment
    assert f(A16, A16, A16, A16, 8, 256, 1, 128, 2, rms_eps=-1.0, **ok) == binding.GEMV_ERR_INVALID


@pytest.mark.parametrize("B", [1, 8, 16])
@pytest.mark.parametrize("N,K", [(4096, 14336), (128256, 4096), (7, 128), (33, 65536)])
def test_w4_plan_covers_the_problem(L, N, K, B):
    q = binding.gemv_w4_query_launch(N, K, B, GB300_SMS)
    assert q["path"] == 2 and q["rows_per_warp"] == 16
    assert q["row_tiles"] * q["rows_per_cta"] >= N
    assert q["splits"] * q["kslice"] >= K > (q["splits"] - 1) * q["kslice"]
    assert q["kslice"] % 128 == 0 and q["kchunk"] % 128 == 0      # groups never straddle
    with pytest.raises(binding.GemvError):
        binding.gemv_w4_query_launch(N, 100, B, GB300_SMS)


def test_host_io_rejects(L):
    ok = dict(stream=0, check=False)
    f = binding.gemv_bf16_host_io
    assert f(A16, 0, A16, A16, A16, 8, 8, 1, 8, **ok) == binding.GEMV_ERR_INVALID        # x_host NULL
    assert f(A16, A16, 0, A16, A16, 8, 8, 1, 8, **ok) == binding.GEMV_ERR_INVALID        # y_host NULL
    assert f(A16, A16, A16, 0, A16, 8, 8, 1, 8, **ok) == binding.GEMV_ERR_INVALID        # x_dev NULL
    assert f(A16, A16, A16, A16, A16 + 2, 8, 8, 1, 8, **ok) == binding.GEMV_ERR_ALIGN    # y_dev


def test_streamk_noalloc_rejects(L):
    f = lambda *a: binding.gemv_bf16_streamk_noalloc(*a, stream=0, check=False)
    assert f(0, A16, A16, 8, 8, 8) == binding.GEMV_ERR_INVALID            # W NULL
    assert f(A16, A16, A16, 0, 8, 8) == binding.GEMV_ERR_INVALID          # N = 0
    assert f(A16, A16, A16, 8, 8, 4) == binding.GEMV_ERR_INVALID          # ldw < K
    assert f(A16, A16, A16 + 2, 8, 8, 8) == binding.GEMV_ERR_ALIGN        # y misaligned
    assert f(A16 + 8, A16, A16, 8, 8, 8) == binding.GEMV_ERR_ALIGN        # W not 16-byte aligned


def test_fp8_argument_checks(L):
    f = lambda Wq, S, x, y, N, K, B, ldq: binding.gemv_fp8_bf16(Wq, S, x, y, N, K, B, ldq, stream=0, check=False)
    assert f(0, A16, A16, A16, 8, 64, 1, 64) == binding.GEMV_ERR_INVALID          # Wq NULL
    assert f(A16, 0, A16, A16, 8, 64, 1, 64) == binding.GEMV_ERR_INVALID          # S NULL
    assert f(A16, A16, A16, A16, 8, 96, 1, 96) == binding.GEMV_ERR_INVALID        # K % 64
    assert f(A16, A16, A16, A16, 8, 64, 1, 48) == binding.GEMV_ERR_INVALID        # ldq < K
    assert f(A16, A16, A16, A16, 8, 64, 17, 64) == binding.GEMV_ERR_INVALID       # B > 16
    assert f(A16, A16, A16, A16, 8, 64, 1, 72) == binding.GEMV_ERR_ALIGN          # ldq % 16
    assert f(A16 + 8, A16, A16, A16, 8, 64, 1, 64) == binding.GEMV_ERR_ALIGN      # Wq alignment
    assert f(A16, A16 + 2, A16, A16, 8, 64, 1, 64) == binding.GEMV_ERR_ALIGN      # S alignment


@pytest.mark.parametrize("N,K,B", [(4096, 14336, 1), (128256, 4096, 1), (4096, 14336, 16), (7, 64, 3)])
def test_fp8_query(L, N, K, B):
    q = binding.gemv_fp8_query_launch(N, K, B, 152)
    assert q["path"] == 4 and q["rows_per_warp"] == 16
    assert q["grid"] == q["row_tiles"] * q["splits"]
    assert q["kslice"] % 64 == 0 and q["xstride"] >= q["kchunk"]
    with pytest.raises(binding.GemvError):
        binding.gemv_fp8_query_launch(N, 100, B, 152)


def test_write_count_is_debug_only(L):
    # the product build never counts stores
    assert binding.gemv_debug_write_count(A16, A16, 8, check=False) == binding.GEMV_ERR_UNSUPPORTED


@pytest.mark.parametrize("B", [1, 2, 3, 8, 9, 16])
def test_cuda_core_plans(L, B):
    for N, K in [(4096, 14336), (7, 129), (33, 65537), (128256, 4096)]:
        q = binding.gemv_query_launch_ex(N, K, B, GB300_SMS, binding.GEMV_FLAG_CUDA_CORES)
        assert q["path"] == 0 and q["rows_per_warp"] == 1
        assert q["grid"] == q["row_tiles"] * q["splits"]
        assert q["smem_bytes"] <= 112 * 1024
    with pytest.raises(binding.GemvError):
        binding.gemv_query_launch_ex(8, 8, 1, GB300_SMS, binding.GEMV_FLAG_CUDA_CORES | binding.GEMV_FLAG_STREAMK)


@pytest.mark.parametrize("N,K", [(4096, 14336), (4097, 8199), (17, 16384), (1024, 14336), (9, 40960),
                                 (3000, 40960), (5, 8192), (2, 8200)])
def test_multicast_copy_geometry(L, N, K):
    # the multicast instance copies the whole vectors of x in one or more bulk
    # copies of at most 32 KB (sizes multiples of 16 bytes) into the staged x
    # area, and writes the partial vector at column K itself
    q = binding.gemv_query_launch(N, K, 1, GB300_SMS)
    if q["mcast"] == 1:
        assert q["splits"] > 1 or q["nbuf"] > 1 or K // 8 < 1024 or q["row_tiles"] < 2
        return
    nfull = K // 8
    nbytes = 16 * nfull
    pieces = [min(32768, nbytes - off) for off in range(0, nbytes, 32768)]
    assert sum(pieces) == nbytes and all(p % 16 == 0 and 0 < p <= 32768 for p in pieces)
    tail = 1 if K % 8 else 0
    assert 8 * (nfull + tail) <= q["xstride"]                  # x area holds every vector
    assert q["smem_bytes"] >= 16 + 2 * q["xstride"]            # mbarrier head + x
    assert q["grid"] % q["mcast"] == 0 and q["grid"] - q["row_tiles"] < q["mcast"]


def test_device_status_rejects_null(L):
    assert L.gemv_device_status(None, 0) == binding.GEMV_ERR_INVALID


# ---- sweep knobs (GEMV_FORCE_SPLIT, GEMV_FORCE_VARIANT): read on every plan


@pytest.mark.parametrize("kw,S", [(1, 1), (2, 1), (1, 2), (4, 2), (2, 4), (8, 8)])
def test_force_split(L, monkeypatch, kw, S):
    default = binding.gemv_query_launch(4096, 14336, 1, GB300_SMS)
    monkeypatch.setenv("GEMV_FORCE_SPLIT", f"{kw}x{S}")
    q = binding.gemv_query_launch(4096, 14336, 1, GB300_SMS)
    assert q["warps_per_row"] == kw and q["splits"] == S
    assert q["rows_per_cta"] == 8 // kw
    assert q["kslice"] * q["splits"] >= 14336 and q["kslice"] % 256 == 0
    assert q["mcast"] == (2 if S == 1 else 1)
    # the tensor-core path and the quantised kernels take it as well
    t = binding.gemv_query_launch(4096, 14336, 16, GB300_SMS)
    assert t["warps_per_row"] == kw and t["splits"] == S
    f = binding.gemv_fp8_query_launch(4096, 14336, 1, GB300_SMS)
    assert f["warps_per_row"] == kw and f["splits"] == S
    monkeypatch.delenv("GEMV_FORCE_SPLIT")
    assert binding.gemv_query_launch(4096, 14336, 1, GB300_SMS) == default


@pytest.mark.parametrize("bad", ["3x1", "2x16", "2", "x2", "2x", "2x2x", "a"])
def test_force_split_rejects(L, monkeypatch, bad):
    monkeypatch.setenv("GEMV_FORCE_SPLIT", bad)
    info = binding.gemv_launch_info()
    assert L.gemv_query_launch(4096, 14336, 1, GB300_SMS, ctypes.byref(info)) == binding.GEMV_ERR_INVALID


def test_force_variant(L, monkeypatch):
    assert binding.gemv_query_launch(4096, 14336, 1, GB300_SMS)["mcast"] == 2
    assert binding.gemv_query_launch(1024, 4096, 1, GB300_SMS)["mcast"] == 1
    monkeypatch.setenv("GEMV_FORCE_VARIANT", "mcast=1")
    assert binding.gemv_query_launch(4096, 14336, 1, GB300_SMS)["mcast"] == 1
    monkeypatch.setenv("GEMV_FORCE_VARIANT", "mcast=4")
    q = binding.gemv_query_launch(4096, 14336, 1, GB300_SMS)
    assert q["mcast"] == 4 and q["grid"] % 4 == 0
    assert binding.gemv_query_launch(1024, 4096, 1, GB300_SMS)["mcast"] == 4   # below the size rule
    assert binding.gemv_query_launch(4096, 14336, 2, GB300_SMS)["mcast"] == 1  # batch 2: no multicast
    # the quantised kernels' deep and standard instances
    monkeypatch.setenv("GEMV_FORCE_VARIANT", "unroll=4")
    assert binding.gemv_fp8_query_launch(4096, 14336, 1, GB300_SMS)["unroll"] == 4
    assert binding.gemv_w4_query_launch(4096, 14336, 1, GB300_SMS)["unroll"] == 4
    monkeypatch.setenv("GEMV_FORCE_VARIANT", "unroll=8")
    assert binding.gemv_fp8_query_launch(128256, 4096, 1, GB300_SMS)["unroll"] == 8
    assert binding.gemv_w4_query_launch(128256, 4096, 4, GB300_SMS)["unroll"] == 8
    assert binding.gemv_w4_query_launch(128256, 4096, 16, GB300_SMS)["unroll"] == 4   # no deep instance
    # stream-K for batch-1 BF16 calls
    assert binding.gemv_query_launch_ex(4096, 4096, 1, GB300_SMS, 0)["path"] == 0
    monkeypatch.setenv("GEMV_FORCE_VARIANT", "streamk=1,mcast=2")
    assert binding.gemv_query_launch_ex(4096, 4096, 1, GB300_SMS, 0)["path"] == 3
    assert binding.gemv_query_launch_ex(4096, 4096, 2, GB300_SMS, 0)["path"] == 1
    assert binding.gemv_query_launch_ex(16, 65536, 1, GB300_SMS, 0)["path"] == 0      # x too long for it
    # more than 8 rows of x: the tcgen05 kernel where its one-wave grid fills the SMs
    monkeypatch.setenv("GEMV_FORCE_VARIANT", "")
    q = binding.gemv_query_launch(4096, 14336, 16, GB300_SMS)
    assert (q["path"], q["splits"], q["unroll"]) == (5, 8, 2)
    assert binding.gemv_query_launch(4096, 14336, 8, GB300_SMS)["path"] == 1     # 8 rows
    assert binding.gemv_query_launch(28672, 4096, 8, GB300_SMS)["path"] == 5     # 8 rows, a wide matrix
    assert binding.gemv_query_launch(1024, 4096, 16, GB300_SMS)["path"] == 1     # 64 CTAs only
    q = binding.gemv_query_launch(128256, 4096, 16, GB300_SMS)                  # several waves:
    assert (q["path"], q["persistent"], q["grid"], q["splits"]) == (5, 1, 334, 1)  # 3 tiles per CTA
    monkeypatch.setenv("GEMV_FORCE_VARIANT", "tc=1")
    q = binding.gemv_query_launch(4096, 14336, 2, GB300_SMS)
    assert q["path"] == 5
    monkeypatch.setenv("GEMV_FORCE_VARIANT", "tc=1,tcstages=5")
    q = binding.gemv_query_launch(4096, 14336, 16, GB300_SMS)
    assert (q["path"], q["splits"], q["unroll"]) == (5, 4, 5)                     # one CTA per SM
    # on the register-fed tensor-core path: x of more than 8 rows as tensor boxes
    # (narrow by default), pieces capped by xpieces
    monkeypatch.setenv("GEMV_FORCE_VARIANT", "tc=0")
    q = binding.gemv_query_launch(4096, 14336, 16, GB300_SMS)
    assert (q["path"], q["xbox"], q["xpieces"], q["xboxes_per_piece"]) == (1, 1, 7, 1)
    assert binding.gemv_query_launch(4096, 14336, 8, GB300_SMS)["xbox"] == 0   # 8 rows: row copies
    assert binding.gemv_query_launch(4096, 14352, 16, GB300_SMS)["xbox"] == 0  # K % 32 != 0
    monkeypatch.setenv("GEMV_FORCE_VARIANT", "tc=0,xbox=2")
    assert binding.gemv_query_launch(4096, 14336, 16, GB300_SMS)["xbox"] == 2
    assert binding.gemv_query_launch(4096, 14368, 16, GB300_SMS)["xbox"] == 0  # wide needs K % 256 == 0
    monkeypatch.setenv("GEMV_FORCE_VARIANT", "tc=0,xbox=0")
    assert binding.gemv_query_launch(4096, 14336, 16, GB300_SMS)["xbox"] == 0
    monkeypatch.setenv("GEMV_FORCE_VARIANT", "tc=0,xpieces=2")
    q = binding.gemv_query_launch(4096, 14336, 16, GB300_SMS)
    assert (q["xbox"], q["xpieces"], q["xboxes_per_piece"]) == (1, 2, 4)
    # L2 prefetch ahead of the register batch: batch 1 on the CUDA cores in
    # grids of at most 8 CTAs per SM by default, any depth on request (also INT4)
    monkeypatch.setenv("GEMV_FORCE_VARIANT", "")
    for (N, K), pf in [((4096, 14336), 1), ((6144, 4096), 1), ((4096, 4096), 1), ((1024, 4096), 1),
                       ((28672, 4096), 0), ((128256, 4096), 0)]:
        assert binding.gemv_query_launch(N, K, 1, GB300_SMS)["l2_prefetch"] == pf, (N, K)
    assert binding.gemv_query_launch(4096, 14336, 2, GB300_SMS)["l2_prefetch"] == 0
    assert binding.gemv_w4_query_launch(4096, 14336, 1, GB300_SMS)["l2_prefetch"] == 0
    assert binding.gemv_fp8_query_launch(4096, 14336, 1, GB300_SMS)["l2_prefetch"] == 0
    monkeypatch.setenv("GEMV_FORCE_VARIANT", "l2pf=3")
    assert binding.gemv_query_launch(28672, 4096, 1, GB300_SMS)["l2_prefetch"] == 3
    assert binding.gemv_w4_query_launch(4096, 14336, 1, GB300_SMS)["l2_prefetch"] == 3
    assert binding.gemv_query_launch(4096, 14336, 16, GB300_SMS)["l2_prefetch"] == 3   # tcgen05, one wave
    assert binding.gemv_query_launch(128256, 4096, 16, GB300_SMS)["l2_prefetch"] == 0  # its persistent form
    monkeypatch.setenv("GEMV_FORCE_VARIANT", "l2pf=0")
    assert binding.gemv_query_launch(4096, 14336, 1, GB300_SMS)["l2_prefetch"] == 0
    for bad in ["mcast=3", "unroll=2", "streamk=2", "foo=1", "mcast", "mcast=", "mcast=2,,x=1", "xbox=3",
                "xpieces=0", "xpieces=9", "tc=2", "tcstages=1", "tcstages=11", "tccols=96", "l2pf=5", "l2pf=-1"]:
        monkeypatch.setenv("GEMV_FORCE_VARIANT", bad)
        info = binding.gemv_launch_info()
        assert L.gemv_query_launch(4096, 14336, 1, GB300_SMS, ctypes.byref(info)) == binding.GEMV_ERR_INVALID, bad


@pytest.mark.parametrize("stages,cols,exists", [
    (2, 128, True), (3, 128, True), (4, 128, True), (5, 128, True), (2, 64, True), (3, 64, True),
    (4, 64, True), (8, 64, True), (10, 64, True), (6, 128, False), (5, 64, False), (9, 64, False)])
def test_tc_ring_instances(monkeypatch, stages, cols, exists):
    """Every ring the tcgen05 knobs name is planned where an instance of it is
    compiled (one wave: the stage count comes back as `unroll`); a ring with
    no instance leaves the call to the register-fed kernel."""
    monkeypatch.setenv("GEMV_FORCE_VARIANT", f"tc=1,tcstages={stages},tccols={cols}")
    q = binding.gemv_query_launch(4096, 14336, 16, GB300_SMS)
    if exists:
        assert (q["path"], q["unroll"], q["persistent"]) == (5, stages, 0), q
    else:
        assert q["path"] == 1, q


def test_host_io_calls_reject_before_any_copy(L):
    """The host-to-host entry points validate their arguments before touching
    the device (checked here without a GPU)."""
    seg = binding.gemv_segment(A16, A16, 8, 8)
    segs = (binding.gemv_segment * 1)(seg)
    yh = (ctypes.c_void_p * 1)(A16)
    ynull = (ctypes.c_void_p * 1)(None)
    # NULL host buffers, too many segments, a NULL segment destination
    assert L.gemv_bf16_multi_host_io(segs, 1, None, A16, yh, 8, 1, None, None) == binding.GEMV_ERR_INVALID
    assert L.gemv_bf16_multi_host_io(segs, 1, A16, A16, None, 8, 1, None, None) == binding.GEMV_ERR_INVALID
    assert L.gemv_bf16_multi_host_io(segs, 1, A16, A16, ynull, 8, 1, None, None) == binding.GEMV_ERR_INVALID
    assert L.gemv_bf16_multi_host_io(segs, 9, A16, A16, yh, 8, 1, None, None) == binding.GEMV_ERR_INVALID
    # device-side arguments follow the gemv_bf16_multi rules
    assert L.gemv_bf16_multi_host_io(segs, 1, A16, A16 + 1, yh, 8, 1, None, None) == binding.GEMV_ERR_ALIGN
    assert L.gemv_bf16_multi_host_io(segs, 1, A16, A16, yh, 8, 17, None, None) == binding.GEMV_ERR_INVALID
    # plans: a NULL plan, negative sizes
    assert L.gemv_plan_launch_host_io(None, A16, A16, 16, A16, A16, 16, None) == binding.GEMV_ERR_INVALID
    assert L.gemv_plan_independent(None) == 0
    # the single-matrix host-io call
    assert L.gemv_bf16_host_io(A16, None, A16, A16, A16, 8, 8, 1, 8, None, None) == binding.GEMV_ERR_INVALID
    assert L.gemv_bf16_host_io(A16, A16, A16, A16, A16, 8, 8, 1, 12, None, None) == binding.GEMV_ERR_ALIGN
