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
        want = -(-(eff * M * N * 4) // 256) * 256 + (M // t["BM"]) * (N // t["BN"]) * 4
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
