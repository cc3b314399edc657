"""Host test of the wide-tile schedule of the tensor-core GEMM (no GPU).

The GEMM runs the store, bias + GeLU and GeLU' products on 256 x 512 tiles of a
CTA pair; the last partial wave of such tiles is split into half-width slots.
This restates, in Python, the slot order (wide_coords over tile_coords), the
columns each CTA's B copy brings, the columns each pair MMA half covers and the
output columns each epilogue warp writes, and checks for many shapes and unit
counts that
- every 256-row x 512-column tile's columns are written exactly once, by the
  slot that computed them, with the B columns that slot loaded;
- the slots a launch runs are exactly the tiles of the output (nothing skipped,
  nothing twice), and the split tail fits in one wave.
"""
import itertools

import pytest

TILE_M, TILE_N, HALF = 256, 512, 256


def tile_coords(tile, m_tiles, n_tiles, group, raster_n):
    per_batch = m_tiles * n_tiles
    zb, tile = divmod(tile, per_batch)
    fast_tiles, slow_tiles = (n_tiles, m_tiles) if raster_n else (m_tiles, n_tiles)
    per_group = group * slow_tiles
    g = tile // per_group
    first = g * group
    gsize = min(fast_tiles - first, group)
    local = tile - g * per_group
    fast, slow = first + local % gsize, local // gsize
    return (slow, fast, zb) if raster_n else (fast, slow, zb)


def wide_tail(tiles, resident):
    r = tiles % resident
    return r if 2 * r <= resident else 0


def wide_coords(tile, m_tiles, n_tiles, batch, tail, group, raster_n):
    full = m_tiles * n_tiles * batch - tail
    wt, hm = tile, 3
    if tile >= full:
        j = tile - full
        wt, hm = full + (j >> 1), 1 << (j & 1)
    return tile_coords(wt, m_tiles, n_tiles, group, raster_n) + (hm,)


def b_columns_loaded(nb, rank, hm):
    """B columns CTA `rank` copies into its stage, by the stage's half slot."""
    hs = 1 if hm == 2 else 0
    n0 = nb * TILE_N + 256 * rank + 128 * hs
    count = 256 if hm == 3 else 128
    cols = list(range(n0, n0 + count))
    # slot s of the stage holds columns [n0_s, n0_s + 128) for half s
    return {hs + i: cols[128 * i:128 * (i + 1)] for i in range(count // 128)}


def mma_half_columns(nb, hh, loaded0, loaded1):
    """Output column of each TMEM column of accumulator half hh: the pair MMA
    takes 128 B columns from each CTA's half-hh slot (even CTA first)."""
    return loaded0[hh] + loaded1[hh]


def epilogue_columns(nb, half, q):
    col0 = nb * TILE_N + half * (TILE_N // 2)
    return list(range(col0 + 32 * q, col0 + 32 * q + 32))


def epilogue_tmem(half, q):
    base = (q >> 2) * 256 + half * 128 + (q & 3) * 32
    return list(range(base, base + 32))


@pytest.mark.parametrize("m_tiles,n_tiles,batch,resident,group,raster_n", [
    (16, 64, 1, 76, 8, False),   # fc1 / dY at h8192 (1024 tiles: 13 waves + 36 split)
    (129, 16, 1, 76, 16, True),  # dB at h8192 with the ones tile row
    (32, 64, 1, 76, 24, False),  # dA at h8192
    (8, 96, 1, 76, 8, False),    # fc1 at h12288, b = 1 (768 tiles)
    (2, 3, 1, 76, 2, False),     # a small problem: every tile split
    (2, 3, 1, 4, 1, True),       # forced 4 units: wide tiles and a split tail in one launch
    (2, 3, 1, 3, 2, False),      # 3 units: 6 % 3 = 0, no split
    (5, 7, 2, 11, 3, False),     # batched problems
    (65, 8, 1, 76, 8, False),    # dB at h4096: 520 tiles, 64 left over, not split (2 * 64 > 76)
])
def test_wide_schedule_covers_every_column_once(m_tiles, n_tiles, batch, resident, group, raster_n):
    tiles = m_tiles * n_tiles * batch
    tail = wide_tail(tiles, resident)
    slots = tiles + tail
    units = min(slots, resident)
    assert 2 * tail <= units or tail == 0
    written = {}
    for unit in range(units):
        for slot in range(unit, slots, units):
            mb, nb, zb, hm = wide_coords(slot, m_tiles, n_tiles, batch, tail, min(group, n_tiles if raster_n else m_tiles), raster_n)
            assert 0 <= mb < m_tiles and 0 <= nb < n_tiles and 0 <= zb < batch
            loaded = [b_columns_loaded(nb, r, hm) for r in (0, 1)]
            halves = [h for h in (0, 1) if hm & (1 << h)]
            tmem_to_col = {}
            for hh in halves:
                cols = mma_half_columns(nb, hh, loaded[0], loaded[1])
                assert len(cols) == 256
                for c, col in enumerate(cols):
                    tmem_to_col[256 * hh + c] = col
            qa, qb = (4 if hm == 2 else 0), (4 if hm == 1 else 8)
            for half in (0, 1):
                for q in range(qa, qb):
                    # the epilogue's column formula agrees with the MMA's placement
                    assert [tmem_to_col[c] for c in epilogue_tmem(half, q)] == epilogue_columns(nb, half, q)
                    for col in epilogue_columns(nb, half, q):
                        key = (zb, mb, col)
                        assert key not in written, key
                        written[key] = slot
    assert len(written) == tiles * TILE_N
    # the split tail is the last partial wave only
    assert tail == 0 or (tiles - tail) % resident == 0 or tiles < resident


def test_split_tail_halves_the_last_wave():
    """1024 wide tiles on 76 pairs: 13 full waves, then 36 tiles as 72 halves."""
    tiles, resident = 16 * 64, 76
    tail = wide_tail(tiles, resident)
    assert tail == 36
    slots = tiles + tail
    work = [0.0] * resident
    for unit in range(resident):
        for slot in range(unit, slots, resident):
            work[unit] += 1.0 if slot < tiles - tail else 0.5
    assert max(work) == 13.5 and min(work) == 13.0
