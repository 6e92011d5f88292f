"""Host-side tile logic of libsdt against the oracle's plain rules (no GPU).

feasible_tiles is integer work, so it must agree with the oracle's three
feasibility rules exactly; pick_tile must only return feasible tiles and keep
the widest tile on deep grids; the seed rule must reproduce the pages' table.
"""
import itertools
import os

import pytest

import shape_driven_tile_gb300 as sdt
from oracle import tiles as otiles

SMEM = 232448
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

SIZES = [0, 64, 128, 192, 256, 320, 512, 768, 1000, 1024, 1536, 1984, 2048, 2304, 4096, 8192]


def ladder():
    return [t for t in sdt.tiles() if not t["skinny"]]  # the skinny tiles are gemm_ex-only


@pytest.mark.parametrize("smem", [SMEM, 150_000, 100_000, 50_000])
def test_feasible_tiles_match_oracle_rules(smem):
    ts = ladder()
    for M, N, K in itertools.product(SIZES, SIZES[:8], [0, 64, 128, 192, 1920, 2048]):
        want = [t["id"] for t in ts if otiles.feasible(M, N, K, t, smem)]
        assert sdt.feasible_tiles(M, N, K, smem_limit=smem) == want, (M, N, K, smem)


def test_feasible_count_beyond_cap():
    n = sdt.lib().sdt_feasible_tiles_for(256, 256, 256, SMEM, None, 0)
    assert n == len(sdt.feasible_tiles(256, 256, 256, smem_limit=SMEM)) > 0


@pytest.mark.parametrize("sm", [96, 148, 152])
def test_pick_tile_is_always_feasible(sm):
    for M, N, K in itertools.product(SIZES[1:], SIZES[1:], [128, 256, 2048, 4096]):
        feas = sdt.feasible_tiles(M, N, K, smem_limit=SMEM)
        if not feas:
            with pytest.raises(sdt.SdtError):
                sdt.pick_tile(M, N, K, sm_count=sm)
            continue
        assert sdt.pick_tile(M, N, K, sm_count=sm) in feas


@pytest.mark.parametrize("sm", [148, 152])
def test_pick_tile_keeps_wide_tile_on_deep_grids(sm):
    # Once even the widest single-CTA tile cuts several waves of CTAs, there is no
    # occupancy reason to move to a narrower one (the FlyDSL pull request's second
    # safety property, restated for this ladder).
    big = [t for t in ladder() if t["cta_group"] == 1 and t["BM"] * t["BN"] >= 128 * 256]
    for n in (6144, 8192, 12288, 16384):
        ctas = (n // 128) * (n // 256)
        assert ctas >= 4 * sm
        pick = sdt.tile_info(sdt.pick_tile(n, n, n, sm_count=sm))
        assert pick["BM"] * pick["BN"] >= 128 * 128, (n, pick["name"])
        assert big


def test_pick_tile_uses_small_tiles_on_small_grids():
    # 256^3 cuts only 4 CTAs of 128x128 (the pages' "cuts only 4 workgroups"): the pick
    # must cut at least as many CTAs as 128x128 would, and more when it can.
    t = sdt.tile_info(sdt.pick_tile(256, 256, 256, sm_count=148))
    assert (256 // t["BM"]) * (256 // t["BN"]) >= 4


def test_seed_rule_matches_oracle_and_golden():
    for M, N in itertools.product(range(128, 4097, 128), [128, 512, 1024, 2048, 4096]):
        for units in (96, 148, 152):
            want = otiles.seed_tile(M, N, units)
            assert sdt.tile_info(sdt.seed_tile(M, N, units))["name"] == want
    with open(os.path.join(GOLDEN, "tile_rule_96cu.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                size, tile = line.split()[:2]
                assert sdt.tile_info(sdt.seed_tile(int(size), int(size), 96))["name"] == tile


def test_pick_tile_errors():
    with pytest.raises(sdt.SdtError) as e:
        sdt.pick_tile(100, 256, 256, sm_count=148)
    assert e.value.status == "SDT_ERR_SHAPE"
    with pytest.raises(sdt.SdtError):
        sdt.pick_tile(256, 256, 256, sm_count=0)


# ---- tune table ----------------------------------------------------------------------


def test_tune_table_roundtrip(tmp_path):
    p = tmp_path / "table.txt"
    p.write_text("# frozen sweep\n256 256 256 64x64\n\n4096 4096 4096 128x256 1  # staggered\n")
    sdt.load_tune_table(str(p))
    try:
        assert sdt.lib().sdt_tune_table_size() == 2
        assert sdt.tile_info(sdt.tune_table_lookup(256, 256, 256))["name"] == "64x64"
        assert sdt.tile_info(sdt.tune_table_lookup(4096, 4096, 4096))["name"] == "128x256"
        assert sdt.tune_table_lookup(512, 512, 512) == -1
    finally:
        sdt.clear_tune_table()
    assert sdt.lib().sdt_tune_table_size() == 0


def test_tune_table_takes_raster_and_depth(tmp_path):
    # the coordinate-descent tuner freezes tile, stagger, raster band and ring depth
    p = tmp_path / "table.txt"
    p.write_text("4096 4096 4096 2cta_256x256 0 1 6  # tuned\n2048 2048 2048 p128x256 -1 0 0\n")
    sdt.load_tune_table(str(p))
    try:
        assert sdt.lib().sdt_tune_table_size() == 2
        assert sdt.tile_info(sdt.tune_table_lookup(4096, 4096, 4096))["name"] == "2cta_256x256"
    finally:
        sdt.clear_tune_table()


@pytest.mark.parametrize("body,needle", [
    ("256 256 256 99x99\n", "unknown tile"),
    ("192 256 256 128x128\n", "infeasible"),
    ("256 256\n", "expected"),
    ("256 256 256 64x64 7\n", "stagger"),
    ("256 256 256 64x64 0 -2\n", "raster"),
    ("256 256 256 64x64 0 4 1\n", "stages"),
    ("256 256 256 64x64 0 4 99\n", "stages"),
    ("256 256 256 64x64" + " " * 600 + "0\n", "longer than"),
])
def test_tune_table_rejects_bad_entries(tmp_path, body, needle):
    p = tmp_path / "bad.txt"
    p.write_text("512 512 512 64x64\n" + body)
    good = tmp_path / "good.txt"
    good.write_text("1024 1024 1024 128x128\n")
    sdt.load_tune_table(str(good))
    try:
        with pytest.raises(sdt.SdtError) as e:
            sdt.load_tune_table(str(p))
        assert e.value.status == "SDT_ERR_TABLE"
        assert needle in str(e.value)
        # a rejected table leaves the previous one in place
        assert sdt.lib().sdt_tune_table_size() == 1
    finally:
        sdt.clear_tune_table()


def test_tune_table_long_comment_is_not_read_as_entries(tmp_path):
    # a comment longer than the loader's line buffer: its tail (which here looks like an
    # entry for another shape) must not be parsed
    p = tmp_path / "table.txt"
    p.write_text("256 256 256 64x64  # " + "x" * 600 + " 1024 1024 1024 128x128\n512 512 512 64x64\n")
    sdt.load_tune_table(str(p))
    try:
        assert sdt.lib().sdt_tune_table_size() == 2
        assert sdt.tune_table_lookup(1024, 1024, 1024) == -1
        assert sdt.tile_info(sdt.tune_table_lookup(512, 512, 512))["name"] == "64x64"
    finally:
        sdt.clear_tune_table()


def test_tune_table_missing_file():
    with pytest.raises(sdt.SdtError):
        sdt.load_tune_table("/nonexistent/table.txt")


def test_skinny_tiles_are_never_feasible_for_gemm_f16():
    skinny = [t["id"] for t in sdt.tiles() if t["skinny"]]
    assert len(skinny) == 2
    for M, N, K in [(128, 16, 128), (256, 32, 4096), (256, 64, 4096), (4096, 4096, 4096)]:
        feas = sdt.feasible_tiles(M, N, K, smem_limit=232448)
        assert not set(skinny) & set(feas)
        if feas:
            assert sdt.pick_tile(M, N, K, sm_count=152) not in skinny
    for t in skinny:
        assert sdt.splitk_workspace_bytes(256, 32, 4096, t, 2) == 0        # not gemm_f16_splitk
        assert sdt.splitk_ex_workspace_bytes(16, 4096, 4096, t, 2) > 0     # gemm_ex_splitk


def test_pick_tile_any_matches_pick_tile_where_the_tiles_divide():
    # gemm_ex's picker lets tiles overhang ragged edges; on the measured configurations,
    # where the tiles divide the shape, it must make gemm_f16's choice
    shapes = [(n, n, n) for n in (256, 512, 768, 1024, 1536, 2048, 2560, 3072, 3584, 4096, 8192)]
    shapes += [(2048, 2048, k) for k in (1920, 1984, 2048, 2112, 2176, 2304)]
    for M, N, K in shapes:
        assert sdt.pick_tile_any(M, N, K, sm_count=152, smem_limit=SMEM) == \
            sdt.pick_tile(M, N, K, sm_count=152, smem_limit=SMEM), (M, N, K)


def test_pick_tile_any_on_ragged_shapes():
    candidates = {t["id"] for t in ladder() if t["name"] not in ("128x256", "2cta_256x128")}
    for M, N, K in itertools.product([1, 7, 100, 1000, 4097], [8, 136, 1000, 16384], [1, 9, 70, 4096]):
        tid = sdt.pick_tile_any(M, N, K, sm_count=152, smem_limit=SMEM)
        assert tid in candidates, (M, N, K, tid)
        assert sdt.tile_info(tid)["smem_bytes"] <= SMEM
    for bad in [(0, 8, 8), (8, -1, 8), (8, 8, 0)]:
        with pytest.raises(sdt.SdtError):
            sdt.pick_tile_any(*bad, sm_count=152, smem_limit=SMEM)
    with pytest.raises(sdt.SdtError):
        sdt.pick_tile_any(8, 8, 8, sm_count=0, smem_limit=SMEM)
