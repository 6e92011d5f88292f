"""Split-K host logic without a GPU: workspace arithmetic, the picker, argument checks."""
import pytest

import shape_driven_tile_gb300 as sdt

SPLIT_TILES = ["64x64", "64x128", "128x64", "128x128", "128x256"]


@pytest.mark.parametrize("name", SPLIT_TILES)
def test_workspace_bytes(name):
    t = sdt.tile_info(sdt.tile_id(name))
    M, N, K = 512, 768, 4096
    for splits in (1, 2, 3, 7, 64):
        nk = K // 64
        kps = -(-nk // splits)
        eff = -(-nk // kps)
        want = -(-((M // t["BM"]) * (N // t["BN"]) * 4) // 256) * 256 + eff * M * N * 4
        assert sdt.splitk_workspace_bytes(M, N, K, name, splits) == want


def test_workspace_bytes_invalid():
    assert sdt.splitk_workspace_bytes(512, 512, 4096, "p128x256", 2) == 0      # no split form
    assert sdt.splitk_workspace_bytes(500, 512, 4096, "64x64", 2) == 0         # does not divide
    assert sdt.splitk_workspace_bytes(512, 512, 4096, "64x64", 65) == 0        # more splits than k-tiles
    assert sdt.splitk_workspace_bytes(512, 512, 4096, "64x64", 0) == 0


def test_pick_splitk_prefers_splitting_small_deep_shapes():
    tid, sp = sdt.pick_splitk(256, 256, 8192)
    assert sdt.tile_info(tid)["name"] in SPLIT_TILES
    assert sp > 1                       # 4 to 16 output tiles for 152 SMs: splitting pays
    tid, sp = sdt.pick_splitk(8192, 8192, 1024)
    assert sp == 1                      # already many waves of tiles


def test_pick_splitk_only_valid_choices():
    for M, N, K in [(256, 256, 256), (512, 2048, 8192), (1024, 1024, 1024), (4096, 256, 4096)]:
        tid, sp = sdt.pick_splitk(M, N, K)
        assert sdt.splitk_workspace_bytes(M, N, K, tid, sp) > 0


def test_splitk_argument_errors_without_gpu():
    L = sdt.lib()
    # null workspace / bad algorithm are rejected before anything touches a device
    assert L.gemm_f16_splitk(256, 256, 256, 0x1000, 0x2000, 0x3000, None, 0, 0, 2, 9, None) == -10
    assert L.gemm_f16_splitk(256, 256, 256, 0x1000, 0x2008, 0x3000, 0x4000, 1 << 20, 0, 2, 1, None) == -2
    assert L.gemm_f16_splitk(0, 256, 256, None, None, None, None, 0, 0, 2, 1, None) == 0


@pytest.mark.parametrize("name", SPLIT_TILES)
def test_ex_workspace_bytes_cover_whole_tiles(name):
    # gemm_ex_splitk: partial planes are whole tiles, so ragged shapes round up
    t = sdt.tile_info(sdt.tile_id(name))
    for M, N, K in [(16, 4096, 4096), (300, 136, 1000), (512, 768, 4096), (1, 8, 65)]:
        Mp, Np = -(-M // t["BM"]) * t["BM"], -(-N // t["BN"]) * t["BN"]
        nk = -(-K // 64)
        for splits in (1, 2, 3, 7):
            if splits > nk:
                assert sdt.splitk_ex_workspace_bytes(M, N, K, name, splits) == 0
                continue
            kps = -(-nk // splits)
            eff = -(-nk // kps)
            tiles = (Mp // t["BM"]) * (Np // t["BN"])
            want = -(-(tiles * 4) // 256) * 256 + eff * Mp * Np * 4
            assert sdt.splitk_ex_workspace_bytes(M, N, K, name, splits) == want
        # on shapes the tile divides, the same bytes as gemm_f16_splitk's workspace
        if M % t["BM"] == 0 and N % t["BN"] == 0 and K % 64 == 0:
            assert sdt.splitk_ex_workspace_bytes(M, N, K, name, 3) == sdt.splitk_workspace_bytes(M, N, K, name, 3)


def test_ex_workspace_bytes_invalid_and_pick():
    assert sdt.splitk_ex_workspace_bytes(512, 512, 4096, "p128x256", 2) == 0    # no split form
    assert sdt.splitk_ex_workspace_bytes(0, 512, 4096, "64x64", 2) == 0
    tid, sp = sdt.pick_splitk_any(16, 16384, 4096)
    assert sdt.tile_info(tid)["name"] in SPLIT_TILES and sdt.splitk_ex_workspace_bytes(16, 16384, 4096, tid, sp) > 0
    tid, sp = sdt.pick_splitk_any(16, 16, 4096)
    assert sp > 1                       # one output tile, 64 k-tiles: splitting pays
