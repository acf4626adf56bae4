"""Host-side checks of the stream-K launch (no GPU): the planner's grid through
the C ABI, and the work partition the kernel derives from it, restated here.

The kernel gives warp w the units [w*U/NW, (w+1)*U/NW) and finds the warps of
a row as the owners of its first and last unit, owner(u) = ((u+1)*NW - 1) // U;
a warp keeps the partial of its first row in slot 2w and of its last row in
slot 2w+1. These tests check on the planner's own numbers that every unit has
exactly one warp, that the owners match the ranges, that every warp between the
first and the last owner of a row holds part of the row (so the row's counter
reaches the count the kernel expects), and that no two partials share a slot.
"""
import pytest

from memory_bound_decode_gb300 import binding

SK = binding.GEMV_FLAG_STREAMK
SHAPES = [(1024, 4096), (4096, 14336), (6144, 4096), (4096, 4096), (28672, 4096), (128256, 4096),
          (4864, 4096), (9728, 2048), (4865, 4096),
          (7, 129), (4097, 4103), (1, 8191), (1, 1), (3, 2049), (5, 24576), (300, 2056), (17, 10000)]


def partition_ok(U, NW, C):
    begin = lambda w: w * U // NW
    owner = lambda u: ((u + 1) * NW - 1) // U
    assert 1 <= NW <= U
    for w in range(NW):
        assert begin(w + 1) > begin(w)                       # every warp takes a unit
    slots = set()
    rows = (U + C - 1) // C
    for n in range(rows):
        wa, wb = owner(n * C), owner(n * C + C - 1)
        assert begin(wa) <= n * C < begin(wa + 1)
        assert begin(wb) <= n * C + C - 1 < begin(wb + 1)
        covered = 0
        for q in range(wa, wb + 1):
            lo, hi = max(begin(q), n * C), min(begin(q + 1), (n + 1) * C)
            assert hi > lo                                    # the warp arrives at the counter
            covered += hi - lo
            if wa != wb:
                side = 0 if begin(q) // C == n else 1
                assert (q, side) not in slots
                slots.add((q, side))
                if side == 1:
                    assert (begin(q + 1) - 1) // C == n       # slot 1 only for the warp's last row
        assert covered == C


@pytest.mark.parametrize("N,K", SHAPES)
def test_streamk_plan_and_partition(N, K):
    q = binding.gemv_query_launch_ex(N, K, 1, 152, SK)
    assert q["path"] == 3
    C = (K + 2047) // 2048
    GW = 152 * q["ctas_per_sm"] * 8                           # warps of one wave
    R = N // GW
    assert q["dp_rounds"] == R
    rest = N - R * GW                                          # rows of the split part
    assert q["chunks"] == C and q["units"] == rest * C
    assert q["warps"] == min(q["units"], GW)
    assert q["grid"] == (GW // 8 if R > 0 else (q["warps"] + 7) // 8)
    assert q["grid"] <= 152 * q["ctas_per_sm"]                 # one wave
    assert q["xstride"] == 8 * ((K + 7) // 8)
    assert q["smem_bytes"] >= 2 * q["xstride"]
    # whole rows: round r, warp w -> row r * GW + w covers rows [0, R * GW) once each
    assert sorted(r * GW + w for r in range(R) for w in range(GW)) == list(range(R * GW))
    if 0 < rest * C <= 300_000:
        partition_ok(q["units"], q["warps"], C)


def test_streamk_partition_small_grids():
    for U in range(1, 60):
        for NW in range(1, U + 1):
            for C in (1, 2, 3, 7):
                if U % C == 0:
                    partition_ok(U, NW, C)


@pytest.mark.parametrize("N,K,B", [(100, 24577, 1), (10, 65537, 1), (100, 4096, 2), (8, 512, 16)])
def test_streamk_unsupported(N, K, B):
    with pytest.raises(binding.GemvError) as e:
        binding.gemv_query_launch_ex(N, K, B, 152, SK)
    assert e.value.status == binding.GEMV_ERR_UNSUPPORTED


def test_query_ex_without_flag_matches_default():
    for N, K, B in [(4096, 14336, 1), (6144, 4096, 8)]:
        a = binding.gemv_query_launch(N, K, B, 152)
        b = binding.gemv_query_launch_ex(N, K, B, 152, 0)
        assert a == b


def test_query_ex_rejects_unknown_flags():
    with pytest.raises(binding.GemvError) as e:
        binding.gemv_query_launch_ex(64, 64, 1, 152, 8)
    assert e.value.status == binding.GEMV_ERR_INVALID
