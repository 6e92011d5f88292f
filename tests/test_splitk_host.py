"""Split-K host logic without a GPU: workspace arithmetic, the picker, argument checks."""
import pytest

import shape_driven_tile_gb300 as sdt

SPLIT_TILES = ["64x64", "64x128", "128x64", "128x128", "128x256"]
COUNTER_REGION = 1 << 20  # u32 counters at the start of every split-K / stream-K workspace


@pytest.mark.parametrize("name", SPLIT_TILES)
def test_workspace_bytes(name):
    t = sdt.tile_info(sdt.tile_id(name))
    M, N, K = 512, 768, 4096
    for splits in (1, 2, 3, 7, 64):
        nk = K // 64
        kps = -(-nk // splits)
        eff = -(-nk // kps)
        want = COUNTER_REGION + eff * M * N * 4
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
            want = COUNTER_REGION + eff * Mp * Np * 4
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


def test_counter_region_is_shared_by_every_configuration():
    # partials always start past the same 1 MiB: a configuration with many tiles never
    # finds another configuration's partials on its counters
    for M, N, K in [(4096, 4096, 4096), (64, 64, 64), (16, 16384, 4096)]:
        for name in SPLIT_TILES:
            t = sdt.tile_info(sdt.tile_id(name))
            Mp, Np = -(-M // t["BM"]) * t["BM"], -(-N // t["BN"]) * t["BN"]
            assert sdt.splitk_ex_workspace_bytes(M, N, K, name, 1) == COUNTER_REGION + Mp * Np * 4


# ---- stream-K ------------------------------------------------------------------------

STREAM_TILES = SPLIT_TILES + ["s128x16", "s128x32"]


def sk_first_unit(g, G, U):
    return g * U // G


def sk_segments(g, G, U, nk):
    """(tile, kb, ke) segments of CTA g, as the kernel walks them."""
    u, end, out = sk_first_unit(g, G, U), sk_first_unit(g + 1, G, U), []
    while u < end:
        tile, kb = divmod(u, nk)
        ke = min(nk, kb + (end - u))
        out.append((tile, kb, ke))
        u += ke - kb
    return out


def sk_owner(u, G, U):
    return ((u + 1) * G - 1) // U


@pytest.mark.parametrize("tiles,nk,G", [(1, 64, 16), (1, 3, 3), (32, 256, 152), (128, 128, 152), (7, 5, 3),
                                        (16, 1, 152), (512, 64, 152), (3, 100, 7), (152, 8, 152), (5, 9, 45)])
def test_streamk_unit_split(tiles, nk, G):
    """The kernel's unit split, restated: every (tile, k-tile) unit belongs to exactly one
    CTA; CTAs get floor or ceil of U/G units; a CTA's middle tiles are whole; and the
    fix-up's view of a tile's contributors (owner of its first and last unit, slot 2g
    when the tile is g's first else 2g+1) matches the slots the CTAs write."""
    U = tiles * nk
    G = min(G, U)
    seen = [0] * U
    written = {}  # tile -> list of (g, slot, kb, ke)
    for g in range(G):
        segs = sk_segments(g, G, U, nk)
        n = sum(ke - kb for _, kb, ke in segs)
        assert n in (U // G, -(-U // G))
        for j, (tile, kb, ke) in enumerate(segs):
            for k in range(kb, ke):
                seen[tile * nk + k] += 1
            whole = kb == 0 and ke == nk
            if 0 < j < len(segs) - 1:
                assert whole
            if not whole:
                written.setdefault(tile, []).append((g, 2 * g + (0 if j == 0 else 1), kb, ke))
    assert seen == [1] * U
    for tile in range(tiles):
        lo, hi = sk_owner(tile * nk, G, U), sk_owner(tile * nk + nk - 1, G, U)
        if lo == hi:
            assert tile not in written          # one CTA holds the whole tile
            continue
        slots = [2 * lo + (0 if sk_first_unit(lo, G, U) // nk == tile else 1)] + [2 * g for g in range(lo + 1, hi + 1)]
        got = sorted(written[tile])
        assert [g for g, *_ in got] == list(range(lo, hi + 1))
        assert [s for _, s, *_ in got] == slots
        # the partial segments tile the k range in CTA order
        assert got[0][2] == 0 and got[-1][3] == nk
        assert all(a[3] == b[2] for a, b in zip(got, got[1:]))


@pytest.mark.parametrize("name", STREAM_TILES)
def test_streamk_workspace_bytes(name):
    t = sdt.tile_info(sdt.tile_id(name))
    for G in (1, 7, 152, 304):
        assert sdt.streamk_workspace_bytes(4096, 4096, 4096, name, G) == COUNTER_REGION + 2 * G * t["BM"] * t["BN"] * 4
    assert sdt.lib().sdt_streamk_workspace_bytes(4096, 4096, 4096, t["id"], 0) == 0       # G >= 1
    assert sdt.lib().sdt_streamk_workspace_bytes(0, 4096, 4096, t["id"], 152) == 0
    # at most 65536 output tiles (four counters each)
    big = 16384 * 4 if t["BM"] == 64 and t["BN"] == 64 else 1 << 20
    if not t["skinny"]:
        assert sdt.lib().sdt_streamk_workspace_bytes(big, big, 64, t["id"], 152) == 0


def test_streamk_tiles_and_default_ctas():
    for t in sdt.tiles():
        ok = t["name"] in STREAM_TILES
        assert (sdt.lib().sdt_streamk_workspace_bytes(512, 512, 512, t["id"], 152) > 0) == ok
        if ok:
            ctas = sdt.streamk_ctas(t["id"], sm_count=152)
            assert ctas % 152 == 0 and 152 <= ctas <= 152 * 4
        else:
            with pytest.raises(sdt.SdtError):
                sdt.streamk_ctas(t["id"], sm_count=152)


def test_workspace_queries_refuse_what_the_launches_refuse():
    # Dimensions above 2^30, or a grid of more than 2^30 - 1 output tiles, are refused by
    # the launches; the size queries return 0 for them instead of a product that wraps.
    L = sdt.lib()
    huge = 1 << 40
    for name in SPLIT_TILES + ["s128x16"]:
        tid = sdt.tile_id(name)
        assert L.sdt_splitk_ex_workspace_bytes(huge, huge, 4096, tid, 32) == 0
        assert L.sdt_splitk_ex_workspace_bytes(1 << 30, 1 << 30, 1 << 30, tid, 32) == 0   # too many tiles
        assert L.sdt_streamk_workspace_bytes(huge, huge, 4096, tid, 152) == 0
        assert L.sdt_streamk_workspace_bytes(64, 64, huge, tid, 152) == 0
    # the largest dimension the launches take still sizes exactly (one tile column)
    t = sdt.tile_info(sdt.tile_id("128x128"))
    M = 1 << 30
    want = COUNTER_REGION + 32 * M * t["BN"] * 4
    assert L.sdt_splitk_ex_workspace_bytes(M, 128, 1 << 30, t["id"], 32) == want
    assert L.sdt_splitk_workspace_bytes(M, 128, 1 << 30, t["id"], 32) == want
