"""The two-CTA tile's last-round plan (sdt_pair_tail_plan: the host logic of gemm_f16_ws
and gemm_ex_ws), with no GPU: hand-worked cases on a 152-SM part and the invariants
every plan keeps."""
import itertools

import pytest

import shape_driven_tile_gb300 as sdt
from shape_driven_tile_gb300._lib import SdtError

SMEM = 232448  # opt-in shared memory per block on GB300


def tid(name):
    return sdt.tile_id(name)


def plan(M, N, K, tile="2cta_256x256", sm=152, **kw):
    return sdt.pair_tail_plan(M, N, K, tid(tile), sm, SMEM, **kw)


def test_workspace_bytes():
    # the 1 MiB counter region, then one 256 x 256 fp32 slot per SM pair
    assert sdt.gemm_workspace_bytes(152) == (1 << 20) + 76 * 256 * 256 * 4 == 20 * (1 << 20)
    assert sdt.gemm_workspace_bytes(2) == (1 << 20) + 256 * 256 * 4
    assert sdt.gemm_workspace_bytes(0) == 0


def test_hand_worked_cases():
    # 4096^3: 256 tiles on 76 pairs -> 3 whole rounds (228) and 28 left.  The estimate: half-width
    # items 64 x 0.272 + 2.4 = 19.8 us; two k-ranges (76 // 28 = 2 at most), split 0 of
    # (64 + 12) / 2 = 38 k-tiles: 38 x 0.366 + 4.1 = 18.0 us -> two k-ranges given a workspace
    assert plan(4096, 4096, 4096) == (228, 284, 2, 38)
    assert plan(4096, 4096, 4096, workspace=False) == (228, 284, 0, 0)
    assert plan(4096, 4096, 4096, tail_splits=0) == (228, 284, 0, 0)
    assert plan(4096, 4096, 4096, tail_splits=2) == (228, 284, 2, 38)
    assert plan(4096, 4096, 4096, tail_splits=8) == (228, 284, 2, 38)
    # 8192^3: 1024 tiles -> 13 rounds (988) and 36 left; halves 128 x 0.272 + 2.4 = 37.2 us
    # against split 0 of 70 k-tiles: 70 x 0.366 + 4.1 = 29.7 us
    assert plan(8192, 8192, 8192) == (988, 1060, 2, 70)
    assert plan(8192, 8192, 8192, tail_splits=0) == (988, 1060, 0, 0)
    # 12288^3: 2304 tiles -> 30 rounds (2280) and 24 left; three k-ranges, split 0 of
    # (192 + 24 + 2) // 3 = 72 k-tiles: 26.4 + 9.7 + 2.5 = 38.6 us beats two (102 k-tiles:
    # 37.3 + 4.1 = 41.4 us) and half-width items (54.6 us)
    assert plan(12288, 12288, 12288) == (2280, 2352, 3, 72)
    # 2560^3: 100 tiles -> 76 + 24: halves 40 x 0.272 + 2.4 = 13.3 us beat two k-ranges
    # (26 x 0.366 + 4.1 = 13.6 us)
    assert plan(2560, 2560, 2560) == (76, 124, 0, 0)
    # 3072^3: 144 tiles -> 76 + 68: neither halves (136 > 76) nor a split (76 // 68 = 1)
    assert plan(3072, 3072, 3072) == (144, 144, 0, 0)
    # tiles that fill every pair leave no last round
    assert plan(256 * 76, 256, 4096) == (76, 76, 0, 0)
    # a short contraction: 8 k-tiles (halves 4.6 us against 7 x 0.366 + 4.1 = 6.7 us)
    assert plan(4096, 4096, 512) == (228, 284, 0, 0)
    # fewer tiles than pairs: all of them are in the last round.  Eight k-ranges would need
    # 7 x 8 KB of copy buffers per epilogue warp, more than its 48 KB quarter of the ring: seven
    # (4 tiles x 7 items; split 0 of (33 + 6 x 12 + 6) // 7 = 15 k-tiles, the other six share 18)
    assert plan(512, 512, 2112, tail_splits=8) == (0, 28, 7, 15)
    assert plan(512, 512, 2112, tail_splits=5)[:3] == (0, 20, 5)
    # ... and a split count is never above the k-tile count
    assert plan(512, 512, 128, tail_splits=8) == (0, 8, 2, 1)


def test_narrow_pair_tiles_never_halve():
    # half-width items exist for BN = 256 only; the 224- and 128-wide pair tiles split in K or not at all
    for tile in ("2cta_256x224", "2cta_256x128"):
        ts, items, sp, _ = plan(4096, 4096, 4096, tile, workspace=False)
        assert ts == items and sp == 0
        ts, items, sp, _ = plan(512, 448, 2112, tile, tail_splits=3)
        assert (ts, sp) == (0, 3)


@pytest.mark.parametrize("tile", ["2cta_256x256", "2cta_256x224", "2cta_256x128"])
def test_invariants(tile):
    bm, bn = 256, {"2cta_256x256": 256, "2cta_256x224": 224, "2cta_256x128": 128}[tile]
    for sm, M, N, K, ws, req in itertools.product(
            (152, 148, 132, 16), (256, 1000, 2560, 4096, 9000), (256, 1504, 4096, 6144), (64, 1000, 4096, 12288),
            (True, False), (-1, 0, 2, 5, 8)):
        ts, items, sp, long_k = sdt.pair_tail_plan(M, N, K, tid(tile), sm, SMEM, workspace=ws, tail_splits=req)
        pairs = sm // 2
        tiles = -(-M // bm) * -(-N // bn)
        nk = -(-K // 64)
        last = tiles % pairs
        case = (sm, M, N, K, ws, req)
        assert 0 <= ts <= tiles and items >= ts, case
        if items == ts:  # whole tiles throughout
            assert ts == tiles and sp == 0 and long_k == 0, case
            continue
        assert ts == tiles - last and ts % pairs == 0, case  # only the last round changes
        assert items - ts <= pairs, case                        # at most one item per pair
        if sp == 0:  # half-width items
            assert bn == 256 and items - ts == 2 * last and long_k == 0, case
        else:
            assert ws and req != 0, case
            assert 2 <= sp <= min(7, nk) and items - ts == last * sp, case
            # split 0 at least an even share, every other split at least one k-tile
            assert -(-nk // sp) <= long_k <= nk - (sp - 1), case
            if req >= 2:
                assert sp <= req, case


def test_argument_errors():
    with pytest.raises(SdtError) as e:
        sdt.pair_tail_plan(4096, 4096, 4096, tid("p128x256"), 152, SMEM)
    assert e.value.status == "SDT_ERR_TILE"
    for bad in ((0, 4096, 4096, 152), (4096, 4096, 4096, 1)):
        with pytest.raises(SdtError) as e:
            sdt.pair_tail_plan(*bad[:3], tid("2cta_256x256"), bad[3], SMEM)
        assert e.value.status == "SDT_ERR_ARG"
    with pytest.raises(SdtError) as e:
        plan(4096, 4096, 4096, tail_splits=1)
    assert e.value.status == "SDT_ERR_ARG"
