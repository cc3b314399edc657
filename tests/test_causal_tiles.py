"""Host-side check of the causal tile arithmetic of the per-head attention GEMMs,
for every sequence length up to 4096 (multiples of 8) and both tile heights.

The kernels skip work by tile: the score and dS GEMMs skip every tile whose
first column lies past its last row, and the products against P or dS run only
part of K (keys below the end of the M-tile for P V and dS K, queries from the
start of the M-tile on for P^T dO and dS^T Q).  With TPMLP_ATTN_P_UPPER_ZERO
the softmax writes row s of P only in columns [0, min(seq, (s // 256 + 1) * 256)).

This test restates those rules (the GEMM's k_range and tile_active, with
BK = 64, 256-column N-tiles for the scores and dS, and M-tiles of 256 rows on
CTA pairs or 128 on single CTAs) and checks, for every tile, that each element
of P (or dS) a GEMM reads lies where the softmax (or the dS GEMM) has written.
The GPU test test_p_upper_tiles_flag plants a sentinel in the unwritten tiles
and finds every output bit-identical, at one length; this covers all lengths."""
import numpy as np
import pytest

BK, BN, WTILE = 64, 256, 256


def written_end(S):
    """[S]: end (exclusive) of the written columns of each row of P."""
    s = np.arange(S)
    return np.minimum(S, (s // WTILE + 1) * WTILE)


def ds_written_end(S, TM):
    """[S]: end of the columns of each row of dS that the dS GEMM writes: the
    active 256-column tiles of the row's M-tile (first column not past its last
    row), clipped to S."""
    s = np.arange(S)
    mb = s // TM
    last_row = mb * TM + TM - 1
    n_active = last_row // BN + 1          # tiles nb with nb * BN <= last_row
    return np.minimum(S, n_active * BN)


def ranges(S, TM):
    m_tiles = -(-S // TM)
    k_blocks = -(-S // BK)
    for mb in range(m_tiles):
        rows = np.arange(mb * TM, min(S, (mb + 1) * TM))
        # causal_k = 1: k < (mb + 1) * TM;  causal_k = 2: k >= mb * TM
        k1 = min(k_blocks, (mb + 1) * (TM // BK)) * BK
        k0 = mb * (TM // BK) * BK
        yield mb, rows, k0, k1


@pytest.mark.parametrize("TM", [256, 128])
def test_every_read_of_p_and_ds_lies_in_a_written_region(TM):
    for S in range(8, 4097, 8):
        wp = written_end(S)
        wd = ds_written_end(S, TM)
        for mb, rows, k0, k1 in ranges(S, TM):
            hi = min(S, k1)  # columns past S are zero-filled by the TMA unit, not read
            # P V and dS K (A = P or dS, K-major): rows of the M-tile, columns [0, k1)
            assert np.all(hi <= wp[rows]), (S, TM, mb, "P V")
            assert np.all(hi <= wd[rows]), (S, TM, mb, "dS K")
            # P^T dO and dS^T Q (A = P^T or dS^T): keys of the M-tile as columns of P,
            # queries [k0, S) as rows
            cols_hi = rows[-1] + 1
            queries = np.arange(k0, S)
            assert np.all(cols_hi <= wp[queries]), (S, TM, mb, "P^T dO")
            assert np.all(cols_hi <= wd[queries]), (S, TM, mb, "dS^T Q")
            # dS reads P on its active 256-column tiles
            n_active = (mb * TM + TM - 1) // BN + 1
            assert np.all(min(S, n_active * BN) <= wp[rows]), (S, TM, mb, "dS epilogue")


@pytest.mark.parametrize("TM", [256, 128])
def test_skipped_tiles_lie_above_the_diagonal(TM):
    """A skipped score or dS tile holds no element on or below the diagonal, so
    the softmax (which reads up to the diagonal) never meets one."""
    for S in range(8, 4097, 8):
        for mb in range(-(-S // TM)):
            for nb in range(-(-S // BN)):
                if nb * BN <= mb * TM + TM - 1:
                    continue  # computed
                first_col, last_row = nb * BN, min(S, mb * TM + TM) - 1
                assert first_col > last_row, (S, TM, mb, nb)


def test_written_region_covers_the_diagonal():
    for S in range(8, 4097, 8):
        assert np.all(written_end(S) > np.arange(S))
