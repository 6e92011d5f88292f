"""Pins for the oracle's integer tile rules against the pages' printed tables."""
import os

import pytest

from oracle import tiles

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield line.split()


def test_seed_rule_reproduces_printed_tiles_and_grids():
    rows = list(_rows("tile_rule_96cu.txt"))
    assert len(rows) == 10
    for size, tile, _bk, _warps, grid in rows:
        n = int(size)
        assert tiles.seed_tile(n, n, 96) == tile, size
        bm, bn = (int(v) for v in tile.split("x"))
        gx, gy = (int(v) for v in grid.split("x"))
        assert tiles.grid(n, n, bm, bn) == (gx, gy), size


def test_workgroup_counts():
    for m, n, bm, bn, wg in _rows("workgroup_counts.txt"):
        gx, gy = tiles.grid(int(m), int(n), int(bm), int(bn))
        assert gx * gy == int(wg)


def test_seed_rule_thresholds_at_96():
    # exactly at the printed thresholds
    assert tiles.seed_tile(128 * 12, 128 * 8, 96) == "128x128"   # 96 blocks
    assert tiles.seed_tile(128 * 8, 128 * 8, 96) == "64x128"     # 64 blocks
    assert tiles.seed_tile(128 * 9, 128 * 7, 96) == "64x64"      # 63 blocks


TILE = dict(BM=128, BN=128, BK=64, smem_bytes=100_000, tmem_cols=128)


def test_feasible_rules():
    lim = 232_448
    assert tiles.feasible(256, 256, 256, TILE, lim)
    assert not tiles.feasible(256 + 64, 256, 256, TILE, lim)        # (i) M
    assert not tiles.feasible(256, 192, 256, TILE, lim)             # (i) N
    assert not tiles.feasible(256, 256, 96, TILE, lim)              # (i) K
    assert not tiles.feasible(256, 256, 64, TILE, lim)              # (ii) one k-tile
    assert not tiles.feasible(256, 256, 256, dict(TILE, smem_bytes=lim + 1), lim)  # (iii)
    assert not tiles.feasible(256, 256, 256, dict(TILE, tmem_cols=1024), lim)
    assert not tiles.feasible(0, 256, 256, TILE, lim)


@pytest.mark.parametrize("n_k", [1, 2, 4, 32, 64])
def test_kloop_order_is_rotation_permutation(n_k):
    for cta in range(0, 70, 7):
        order = tiles.kloop_order(cta, n_k)
        assert sorted(order) == list(range(n_k))
        assert order[0] == cta % n_k
        assert all((order[i + 1] - order[i]) % n_k == 1 for i in range(n_k - 1))


@pytest.mark.parametrize("n_k", [3, 30, 31, 33, 34, 36])
def test_kloop_order_off_when_not_pow2(n_k):
    # the K-scan counts 1920..2304 / 64 = 30..36: only 32 is a power of two
    assert tiles.kloop_order(5, n_k) == list(range(n_k))
