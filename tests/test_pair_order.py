"""Host test of the tile order of the causal per-head products (no GPU).

The products against P or dS (P V, dS K: k below the end of the M-tile; P^T dO,
dS^T Q: k from the start of the M-tile on) have one N-tile per problem, and
M-tile i costs i + 1 (or m_tiles - i) k-blocks.  The GEMM hands each unit the
M-tiles of a problem in complementary pairs (i, m_tiles - 1 - i).  This
restates, in Python, the slot -> (problem, M-tile) map of tile_coords and checks
that
- it is a bijection onto the tiles of the launch, for many shapes and unit
  counts;
- in the full double rounds, the two slots a unit runs back to back are one
  pair of one problem;
- at the attention workload's size (128 problems of 8 M-tiles on 76 units) the
  busiest unit does at most 1/0.96 of the mean work, where the earlier order
  (odd problems reversed) left it at 1/0.905.
"""
import pytest


def pair_coords(tile, m_tiles, batch, units):
    half = m_tiles // 2
    n = m_tiles * batch
    R = n // (2 * units)
    s = n - 2 * R * units
    k, u = divmod(tile, units)
    twice = s - units if s > units else 0
    if k < 2 * R:
        pair, member = u + (k >> 1) * units, k & 1
    elif u < twice:
        pair, member = R * units + u, k - 2 * R
    else:
        v = u - twice
        pair, member = R * units + twice + (v >> 1), v & 1
    z, i = divmod(pair, half)
    return z, (i if member else m_tiles - 1 - i)


def flip_coords(tile, m_tiles):
    z, m = divmod(tile, m_tiles)
    return z, (m_tiles - 1 - m if z % 2 else m)


def loads(coords, n, units, cost):
    load = [0] * units
    for u in range(units):
        for t in range(u, n, units):
            load[u] += cost(coords(t)[1])
    return load


@pytest.mark.parametrize("m_tiles,batch,units", [
    (8, 128, 76), (8, 128, 75), (8, 64, 76), (16, 128, 76), (2, 2, 76), (2, 5, 3),
    (8, 3, 4), (4, 7, 5), (6, 13, 11), (8, 1, 76), (8, 19, 76), (8, 20, 76),
])
def test_pair_order_is_a_bijection(m_tiles, batch, units):
    n = m_tiles * batch
    units = min(units, n)
    seen = set()
    for t in range(n):
        z, mb = pair_coords(t, m_tiles, batch, units)
        assert 0 <= z < batch and 0 <= mb < m_tiles
        seen.add((z, mb))
    assert len(seen) == n
    # full double rounds: back-to-back slots of a unit are one complementary pair
    R = n // (2 * units)
    for u in range(units):
        for j in range(R):
            a = pair_coords(u + 2 * j * units, m_tiles, batch, units)
            b = pair_coords(u + (2 * j + 1) * units, m_tiles, batch, units)
            assert a[0] == b[0] and a[1] + b[1] == m_tiles - 1


@pytest.mark.parametrize("cost", [lambda i: i + 1, lambda i: 8 - i])
def test_pair_order_balances_the_attention_workload(cost):
    m_tiles, batch, units = 8, 128, 76
    n = m_tiles * batch
    pair = loads(lambda t: pair_coords(t, m_tiles, batch, units), n, units, cost)
    flip = loads(lambda t: flip_coords(t, m_tiles), n, units, cost)
    mean = sum(pair) / units
    assert sum(pair) == sum(flip)
    assert mean / max(pair) >= 0.96
    assert mean / max(flip) < 0.91
