"""The split-K cluster combine's index arithmetic, restated in Python and
checked on the launches the planner makes (no GPU): rank r of a cluster of S
owns outputs [r * chunk, (r + 1) * chunk) of the tile's rows_per_cta * B
outputs; every rank stores its partial of output i into slot
[rank][i - owner * chunk] of the owner's shared memory; the owner adds the S
slots in rank order. Outputs are mapped to (row, batch row) with a multiply-high
by ceil(2^32 / B) instead of a division."""
import pytest

from memory_bound_decode_gb300 import binding

GB300_SMS = 152
K_MAX_SPLITS = 8
K_MAX_BATCH = 16
K_WARPS = 8
SHAPES = [(1024, 4096), (4096, 14336), (6144, 4096), (28672, 4096), (4096, 4096), (128256, 4096),
          (7, 129), (4097, 4103), (1, 8191), (33, 65537), (1, 1), (3, 8), (100000, 300)]


def div_by_batch(i, B):
    if B == 1:
        return i
    magic = 0xFFFFFFFF // B + 1
    return (i * magic) >> 32


@pytest.mark.parametrize("B", range(1, 17))
def test_division_free_output_index(B):
    # every output index a tile can have: rows_per_cta * B <= 128 * 16
    for i in range(128 * 16 + 1):
        assert div_by_batch(i, B) == i // B
    # and far beyond, up to the bound the kernel relies on (i < 2^16)
    for i in range(0, 1 << 16, 97):
        assert div_by_batch(i, B) == i // B


def launches():
    for N, K in SHAPES:
        for B in (1, 2, 3, 4, 8, 9, 16):
            yield "bf16", N, K, B, binding.gemv_query_launch(N, K, B, GB300_SMS)
            yield "cc", N, K, B, binding.gemv_query_launch_ex(N, K, B, GB300_SMS, binding.GEMV_FLAG_CUDA_CORES)
            if K % 128 == 0:
                yield "w4", N, K, B, binding.gemv_w4_query_launch(N, K, B, GB300_SMS)
            if K % 64 == 0:
                yield "f8", N, K, B, binding.gemv_fp8_query_launch(N, K, B, GB300_SMS)


def test_reduce_scatter_slots_cover_every_output_once():
    seen_split = 0
    for kind, N, K, B, q in launches():
        S = q["splits"]
        if S == 1:
            continue
        seen_split += 1
        nout = q["rows_per_cta"] * B
        chunk = -(-nout // S)
        # the receive area the kernels reserve: rows_per_cta * B + kMaxSplits floats
        assert S * chunk <= nout + K_MAX_SPLITS, (kind, N, K, B, q)
        owned = []
        for r in range(S):
            i0, i1 = r * chunk, min((r + 1) * chunk, nout)
            owned += list(range(i0, i1)) if i1 > i0 else []
        assert owned == list(range(nout)), (kind, N, K, B)
        # every (writer rank, output) pair has its own slot in the owner's area
        slots = set()
        for rank in range(S):
            for i in range(nout):
                owner = i // chunk
                slot = (owner, rank * chunk + (i - owner * chunk))
                assert slot not in slots
                assert 0 <= slot[1] < S * chunk
                slots.add(slot)
    assert seen_split > 10   # the shapes do exercise clusters


def test_shared_memory_holds_the_combine_areas():
    # x buffers + warp partials [kw][rows][B + 1] + cluster slots (rows * B + kMaxSplits)
    # + misc floats (per-warp and CTA sums of squares, row scales, every rank's sums)
    misc = K_WARPS * K_MAX_BATCH + 2 * K_MAX_BATCH + K_MAX_SPLITS * K_MAX_BATCH
    for kind, N, K, B, q in launches():
        rows, kw = q["rows_per_cta"], q["warps_per_row"]
        if kind in ("bf16", "cc") and q["path"] in (0, 1):
            if q["xbox"]:
                # x as tensor boxes: kw groups x pieces x boxes of 8 blocks x B rows x 32 columns
                xbytes = kw * q["xpieces"] * q["xboxes_per_piece"] * 8 * B * 32 * 2
                assert q["nbuf"] == 1 and q["xpieces"] * kw <= 8, (kind, N, K, B, q)
                # every warp group's blocks fit its pieces
                nblk = q["kslice"] // 32
                span = -(-nblk // kw)
                assert q["xpieces"] * q["xboxes_per_piece"] * 8 >= span, (kind, N, K, B, q)
            else:
                xbytes = q["nbuf"] * B * q["xstride"] * 2
            need = (xbytes + rows * (B + 1) * kw * 4
                    + (rows * B + K_MAX_SPLITS) * 4 + misc * 4)
            assert q["smem_bytes"] >= need, (kind, N, K, B, q)
        assert q["smem_bytes"] <= 112 * 1024
