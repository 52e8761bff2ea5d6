"""Host check of the prefill V transposer's lane map (prefill_tc.cuh, V transposer role).

The transposer rewrites each TMA-staged V tile (rows = keys, 128-byte swizzle: 16-byte chunk
index = (d quad ^ key) & 7) in place as V^T (rows = d, chunk index = (key quad ^ d) & 7), one
4x4 block (key quad aa, d quad dq) per thread and iteration, with four 16-byte loads and four
16-byte stores.  A 16-byte shared access is served a quarter-warp at a time, so the map must
give the eight lanes of every quarter-warp eight distinct chunks, on the loads and on the
stores, and must cover every block of the tile exactly once.  The map is restated here from
the kernel source (lane q = lane & 7 of a quarter-warp gets key quad 8*ah + q and d quad
8*dh + (q ^ s), with c = it*16 + warp*4 + lane/8 giving s = c & 7 and (ah, dh) = c >> 3) and
checked exhaustively for every head dimension that uses it.
"""
import pytest


def block_of(D, BN, wv, lane, it):
    q = lane & 7
    c = it * 16 + wv * 4 + (lane >> 3)
    rest = c >> 3
    return 8 * (rest % (BN // 32)) + q, 8 * (rest // (BN // 32)) + (q ^ (c & 7))


def staged_chunk(key, dq):          # V tile as the TMA box leaves it
    return (dq & 7) ^ (key & 7)


def vt_chunk(aa, d):                # V^T row d, key quad aa
    return (aa & 7) ^ (d & 7)


@pytest.mark.parametrize("D,BN", [(32, 128), (64, 128), (128, 64)])
def test_diagonal_map_covers_tile_once(D, BN):
    per = (BN // 4) * (D // 4) // 128
    seen = {}
    for wv in range(4):
        for lane in range(32):
            for it in range(per):
                aa, dq = block_of(D, BN, wv, lane, it)
                assert 0 <= aa < BN // 4 and 0 <= dq < D // 4
                seen[(aa, dq)] = seen.get((aa, dq), 0) + 1
    assert len(seen) == (BN // 4) * (D // 4)
    assert set(seen.values()) == {1}


@pytest.mark.parametrize("D,BN", [(32, 128), (64, 128), (128, 64)])
def test_diagonal_map_is_conflict_free(D, BN):
    per = (BN // 4) * (D // 4) // 128
    for wv in range(4):
        for it in range(per):
            for qw in range(4):
                blocks = [block_of(D, BN, wv, qw * 8 + q, it) for q in range(8)]
                for rr in range(4):
                    loads = {staged_chunk(4 * aa + rr, dq) for aa, dq in blocks}
                    stores = {vt_chunk(aa, 4 * dq + rr) for aa, dq in blocks}
                    assert len(loads) == 8 and len(stores) == 8


def test_row_major_map_would_conflict():
    """The map is needed: four key quads x two d quads per quarter-warp (the obvious
    row-major lane order) puts two lanes on one chunk for every load."""
    worst = 0
    for rr in range(4):
        chunks = [staged_chunk(4 * (q % 4) + rr, q // 4) for q in range(8)]
        worst = max(worst, max(chunks.count(c) for c in chunks))
    assert worst == 2
