"""A model of the SM-pair GEMM's tile indexing, written out in Python, and what the kernel relies on:
the banded walk (column tiles in bands of 8, row tiles running fastest within a band) visits every
256 x 256 output tile exactly once; for the fused QKV projection, the two 128-row halves of a
tile's B operand come from the right weight segment (W_Q, W_K or W_V) at the right row, so the
output columns [0, n_q hd), [n_q hd, n_q hd + n_kv hd) and the rest are each read once from their
own matrix, and each half's output columns follow on from the previous segment's.  This checks
the scheme; the GPU parity tests check the kernel."""
import pytest

BAND = 8


def tile_coords(m_tiles, n_tiles, t):
    band_tiles = m_tiles * BAND
    band = t // band_tiles
    rem = t - band * band_tiles
    gw = min(BAND, n_tiles - band * BAND)
    return rem // gw, band * BAND + rem % gw          # (mb, nb)


def half_source(seg_half_end, nb, hh):
    """Segment and first row of half hh (0, 1) of column tile nb, from the cumulative half counts."""
    gh = 2 * nb + hh
    seg, start = 0, 0
    while seg < len(seg_half_end) - 1 and gh >= seg_half_end[seg]:
        start = seg_half_end[seg]
        seg += 1
    return seg, (gh - start) * 128


@pytest.mark.parametrize("m_tiles,n_tiles", [(32, 24), (32, 16), (32, 112), (8, 10), (1, 1), (3, 9), (2, 17)])
def test_banded_walk_visits_every_tile_once(m_tiles, n_tiles):
    seen = [tile_coords(m_tiles, n_tiles, t) for t in range(m_tiles * n_tiles)]
    assert sorted(seen) == [(mb, nb) for mb in range(m_tiles) for nb in range(n_tiles)]


@pytest.mark.parametrize("n_q,n_kv,hd", [(32, 8, 128), (32, 32, 128), (8, 2, 64), (8, 8, 128), (40, 8, 128)])
def test_qkv_halves_read_each_weight_row_once(n_q, n_kv, hd):
    rows = [n_q * hd, n_kv * hd, n_kv * hd]                 # W_Q, W_K, W_V
    if any(r % 128 for r in rows) or sum(r // 128 for r in rows) % 2:
        pytest.skip("not an SM-pair shape (the one-SM kernel takes it)")
    ends, acc = [], 0
    for r in rows:
        acc += r // 128
        ends.append(acc)
    n_tiles = acc // 2
    read = {s: [] for s in range(3)}
    for nb in range(n_tiles):
        for hh in range(2):
            seg, row = half_source(ends, nb, hh)
            read[seg].append(row)
            # the epilogue's output column of this half is where the segment's rows land in [q | k | v]
            col = 256 * nb + 128 * hh
            assert col == sum(rows[:seg]) + row
    for s in range(3):
        assert sorted(read[s]) == list(range(0, rows[s], 128))
