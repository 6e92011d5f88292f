"""gemm_f16 on the GPU against the fp64 CPU oracle, through the C ABI.

Covers every tile of the ladder, stagger on and off, the square sweep, the
K-scan and the large squares, closed forms (identity, permutation), integer
inputs (bit-exact), empty and rejected shapes, and C poisoned with NaN before
each call so an unwritten tile cannot pass.
"""
import numpy as np
import pytest
import torch

import oracle
import shape_driven_tile_gb300 as sdt
from shape_driven_tile_gb300 import inputs
from _parity import assert_bit_exact_f16, assert_close, boundary_rows, nan_like, u16

pytestmark = pytest.mark.gpu


def run(A, B, dev, tile=None, stagger=-1):
    C = nan_like((A.shape[0], B.shape[1]), dev)
    if tile is None:
        sdt.gemm_f16(A, B, C)
    else:
        sdt.gemm_f16_with_tile(A, B, C, tile=tile, stagger=stagger)
    sdt.check_device_status()
    return C


def tile_ids():
    """Ladder tiles of power-of-two width (every shape below is a multiple of them); the
    skinny tiles are gemm_ex forms only, the 224-wide pair tile has its own shapes."""
    return [t["id"] for t in sdt.tiles() if not t["skinny"] and t["BN"] & (t["BN"] - 1) == 0]


def odd_tile_ids():
    return [t["id"] for t in sdt.tiles() if not t["skinny"] and t["BN"] & (t["BN"] - 1) != 0]


def tile_name(i):
    return sdt.tile_info(i)["name"]


# ---- configuration 1: 256^3, uniform and integer, every tile, stagger on/off ----------


@pytest.mark.parametrize("stagger", [0, 1])
@pytest.mark.parametrize("tile", tile_ids(), ids=tile_name)
def test_256_integer_bit_exact(cuda_device, tile, stagger):
    A = inputs.integers((256, 256), seed=inputs.seed_for(0, 0))
    B = inputs.integers((256, 256), seed=inputs.seed_for(0, 1))
    C = run(A.to(cuda_device), B.to(cuda_device), cuda_device, tile, stagger)
    assert_bit_exact_f16(C, oracle.gemm(u16(A), u16(B)), f"256^3 integer {tile_name(tile)}")


@pytest.mark.parametrize("tile", tile_ids(), ids=tile_name)
def test_256_uniform(cuda_device, tile):
    A = inputs.uniform((256, 256), seed=inputs.seed_for(0, 0))
    B = inputs.uniform((256, 256), seed=inputs.seed_for(0, 1))
    C = run(A.to(cuda_device), B.to(cuda_device), cuda_device, tile)
    assert_close(C.cpu().double().numpy(), oracle.gemm(u16(A), u16(B)), 256, tile_name(tile))


# ---- shapes that span several tiles, non-square, k-tile counts pow2 and not -----------

SHAPES = [(512, 768, 320), (768, 512, 1024), (1024, 256, 128), (256, 1024, 2112)]


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("tile", tile_ids(), ids=tile_name)
def test_multi_tile_shapes(cuda_device, tile, M, N, K):
    A = inputs.uniform((M, K), seed=11)
    B = inputs.uniform((K, N), seed=12)
    Ad, Bd = A.to(cuda_device), B.to(cuda_device)
    ref = oracle.gemm(u16(A), u16(B))
    for stagger in (0, 1):
        C = run(Ad, Bd, cuda_device, tile, stagger)
        assert_close(C.cpu().double().numpy(), ref, K, f"{M}x{N}x{K} {tile_name(tile)} stagger={stagger}")


@pytest.mark.parametrize("M,N,K", [(192, 320, 448), (64, 64, 128), (320, 64, 192)])
def test_shapes_only_small_tiles_divide(cuda_device, M, N, K):
    feas = sdt.feasible_tiles(M, N, K)
    assert feas
    A = inputs.integers((M, K), seed=13)
    B = inputs.integers((K, N), seed=14)
    ref = oracle.gemm(u16(A), u16(B))
    for t in feas:
        C = run(A.to(cuda_device), B.to(cuda_device), cuda_device, t)
        assert_bit_exact_f16(C, ref, f"{M}x{N}x{K} {tile_name(t)}")
    C = run(A.to(cuda_device), B.to(cuda_device), cuda_device)
    assert_bit_exact_f16(C, ref, f"{M}x{N}x{K} pick_tile")


# ---- closed forms -----------------------------------------------------------------------


@pytest.mark.parametrize("tile", tile_ids(), ids=tile_name)
def test_identity_and_permutation(cuda_device, tile):
    n = 512
    B = inputs.uniform((n, 768), seed=21)
    eye = torch.eye(n, dtype=torch.float16)
    C = run(eye.to(cuda_device), B.to(cuda_device), cuda_device, tile)
    assert torch.equal(C.cpu().view(torch.int16), B.view(torch.int16)), "I @ B != B"
    perm = torch.from_numpy(np.random.default_rng(5).permutation(n))
    P = torch.zeros((n, n), dtype=torch.float16)
    P[torch.arange(n), perm] = 1
    C = run(P.to(cuda_device), B.to(cuda_device), cuda_device, tile)
    assert torch.equal(C.cpu().view(torch.int16), B[perm].view(torch.int16)), "P @ B != B[perm]"
    A = inputs.uniform((768, n), seed=22)
    C = run(A.to(cuda_device), eye.to(cuda_device), cuda_device, tile)
    assert torch.equal(C.cpu().view(torch.int16), A.view(torch.int16)), "A @ I != A"


def test_rank1_closed_form(cuda_device):
    M, N, K = 512, 512, 1024
    u = torch.randint(-3, 4, (M, 1), generator=torch.Generator().manual_seed(3)).half() * 0.5
    v = torch.randint(-3, 4, (1, N), generator=torch.Generator().manual_seed(4)).half() * 0.25
    A = u.expand(M, K).contiguous()
    B = v.expand(K, N).contiguous()
    C = run(A.to(cuda_device), B.to(cuda_device), cuda_device)
    want = (K * u.double() * v.double()).numpy()
    assert np.array_equal(C.cpu().double().numpy(), want)


# ---- configuration 2: the square sweep with pick_tile -------------------------------------

SWEEP = [256, 512, 768, 1024, 1536, 2048, 2560, 3072, 3584, 4096]


@pytest.mark.parametrize("n", SWEEP)
def test_square_sweep_pick_tile(cuda_device, n):
    A = inputs.uniform((n, n), seed=inputs.seed_for(1, 0))
    B = inputs.uniform((n, n), seed=inputs.seed_for(1, 1))
    C = run(A.to(cuda_device), B.to(cuda_device), cuda_device).cpu().double().numpy()
    if n <= 1024:
        assert_close(C, oracle.gemm(u16(A), u16(B)), n, f"{n}^3")
    else:
        rows = boundary_rows(n, step=128, extra=8)
        rows = rows[:: max(1, len(rows) // 48)]
        assert_close(C[rows], oracle.gemm(u16(A), u16(B), rows=rows), n, f"{n}^3 rows")


@pytest.mark.parametrize("n", [1024, 2048])
def test_square_every_feasible_tile(cuda_device, n):
    A = inputs.uniform((n, n), seed=inputs.seed_for(1, 0))
    B = inputs.uniform((n, n), seed=inputs.seed_for(1, 1))
    Ad, Bd = A.to(cuda_device), B.to(cuda_device)
    rows = boundary_rows(n, step=64, extra=4)[:: 1 if n <= 1024 else 4]
    ref = oracle.gemm(u16(A), u16(B), rows=rows)
    for t in sdt.feasible_tiles(n, n, n):
        C = run(Ad, Bd, cuda_device, t).cpu().double().numpy()
        assert_close(C[rows], ref, n, f"{n}^3 {tile_name(t)}")


# ---- configuration 3: K-scan at M = N = 2048, fixed tile, stagger on and off ------------

KSCAN = [1920, 1984, 2048, 2112, 2176, 2304]


@pytest.mark.parametrize("K", KSCAN)
def test_kscan_stagger(cuda_device, K):
    M = N = 2048
    A = inputs.uniform((M, K), seed=inputs.seed_for(2, 0))
    B = inputs.uniform((K, N), seed=inputs.seed_for(2, 1))
    Ad, Bd = A.to(cuda_device), B.to(cuda_device)
    rows = boundary_rows(M, step=128, extra=8)[::3]
    ref = oracle.gemm(u16(A), u16(B), rows=rows)
    tile = sdt.tile_id("128x128")
    for stagger in (0, 1):
        C = run(Ad, Bd, cuda_device, tile, stagger).cpu().double().numpy()
        assert_close(C[rows], ref, K, f"K={K} stagger={stagger}")


@pytest.mark.parametrize("K", [2048, 1920])
def test_kscan_integer_stagger_bit_identical(cuda_device, K):
    M = N = 2048
    A = inputs.integers((M, K), seed=31)
    B = inputs.integers((K, N), seed=32)
    Ad, Bd = A.to(cuda_device), B.to(cuda_device)
    tile = sdt.tile_id("128x128")
    C0 = run(Ad, Bd, cuda_device, tile, 0)
    C1 = run(Ad, Bd, cuda_device, tile, 1)
    assert torch.equal(C0.view(torch.int16), C1.view(torch.int16))
    rows = boundary_rows(M, step=128, extra=8)[::4]
    assert_bit_exact_f16(C1.cpu()[rows], oracle.gemm(u16(A), u16(B), rows=rows), f"K={K}")


# ---- configuration 5: large squares (sampled rows) --------------------------------------


@pytest.mark.parametrize("n", [8192, 12288, 16384])
def test_large_square_sampled_rows(cuda_device, n):
    A = inputs.uniform((n, n), seed=inputs.seed_for(4, 0))
    B = inputs.uniform((n, n), seed=inputs.seed_for(4, 1))
    Ad, Bd = A.to(cuda_device), B.to(cuda_device)
    rng = np.random.default_rng(n)
    rows = np.unique(np.concatenate([[0, 127, 128, n // 2, n - 129, n - 1], rng.integers(0, n, 6)]))
    ref = oracle.gemm(u16(A), u16(B), rows=rows)
    C = run(Ad, Bd, cuda_device)
    assert_close(C[torch.from_numpy(rows).to(cuda_device)].cpu().double().numpy(), ref, n, f"{n}^3 pick")
    # the whole output is finite (no tile left unwritten)
    assert bool(torch.isfinite(C).all())
    del C
    C = run(Ad, Bd, cuda_device, sdt.tile_id("128x256"))
    assert_close(C[torch.from_numpy(rows).to(cuda_device)].cpu().double().numpy(), ref, n, f"{n}^3 128x256")


# ---- edge cases and the call contract ---------------------------------------------------------


def test_empty_and_zero_k(cuda_device):
    A = torch.empty((0, 256), dtype=torch.float16, device=cuda_device)
    B = torch.empty((256, 128), dtype=torch.float16, device=cuda_device)
    C = sdt.gemm_f16(A, B)
    assert C.shape == (0, 128)
    A = torch.empty((128, 0), dtype=torch.float16, device=cuda_device)
    B = torch.empty((0, 192), dtype=torch.float16, device=cuda_device)
    C = nan_like((128, 192), cuda_device)
    sdt.gemm_f16(A, B, C)
    torch.cuda.synchronize()
    assert bool((C == 0).all())


@pytest.mark.parametrize("M,N,K", [(100, 256, 256), (256, 200, 256), (256, 256, 100), (256, 256, 64)])
def test_ragged_shapes_rejected(cuda_device, M, N, K):
    A = torch.zeros((M, K), dtype=torch.float16, device=cuda_device)
    B = torch.zeros((K, N), dtype=torch.float16, device=cuda_device)
    with pytest.raises(sdt.SdtError) as e:
        sdt.gemm_f16(A, B)
    assert e.value.status == "SDT_ERR_SHAPE"


def test_infeasible_forced_tile(cuda_device):
    A = torch.zeros((192, 256), dtype=torch.float16, device=cuda_device)
    B = torch.zeros((256, 256), dtype=torch.float16, device=cuda_device)
    with pytest.raises(sdt.SdtError) as e:
        sdt.gemm_f16_with_tile(A, B, tile="128x128")
    assert e.value.status == "SDT_ERR_TILE"


def test_same_shape_different_operands(cuda_device):
    # The tensor-map cache is keyed by pointer and pitch: a second B of the same
    # shape must be read from its own memory.
    M = N = K = 512
    A = inputs.integers((M, K), seed=41).to(cuda_device)
    B1 = inputs.integers((K, N), seed=42)
    B2 = inputs.integers((K, N), seed=43)
    before = sdt.lib().sdt_debug_tensor_map_encodes()
    C1 = run(A, B1.to(cuda_device), cuda_device)
    C2 = run(A, B2.to(cuda_device), cuda_device)
    assert sdt.lib().sdt_debug_tensor_map_encodes() > before
    Ah = u16(A)
    assert_bit_exact_f16(C1, oracle.gemm(Ah, u16(B1)), "B1")
    assert_bit_exact_f16(C2, oracle.gemm(Ah, u16(B2)), "B2")


def test_graph_capture_replay(cuda_device):
    M, N, K = 1024, 512, 768
    A = inputs.uniform((M, K), seed=51).to(cuda_device)
    B = inputs.uniform((K, N), seed=52).to(cuda_device)
    C = torch.empty((M, N), dtype=torch.float16, device=cuda_device)
    eager = sdt.gemm_f16(A, B).clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        sdt.gemm_f16(A, B, C)  # first call outside capture (tensor maps, attributes)
        with torch.cuda.graph(g, stream=s):
            sdt.gemm_f16(A, B, C)
    C.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(C.view(torch.int16), eager.view(torch.int16))


def test_nondefault_stream(cuda_device):
    A = inputs.integers((512, 256), seed=61)
    B = inputs.integers((256, 384), seed=62)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        Ad, Bd = A.to(cuda_device), B.to(cuda_device)
        C = sdt.gemm_f16(Ad, Bd)
    s.synchronize()
    assert_bit_exact_f16(C, oracle.gemm(u16(A), u16(B)), "side stream")


@pytest.mark.parametrize("tile", tile_ids() + odd_tile_ids(), ids=tile_name)
def test_pipeline_phase_edges(cuda_device, tile):
    # k-tile counts around the ring depth: the first reuse of slot 0, the phase flip at
    # the ring's end, and one and two full turns of the ring, on one output tile
    info = sdt.tile_info(tile)
    S = info["stages"]
    M, N = info["BM"], info["BN"]
    for nk in sorted({2, S - 1, S, S + 1, 2 * S, 2 * S + 1} - {0, 1}):
        K = 64 * nk
        A = inputs.integers((M, K), seed=inputs.seed_for(90 + nk, 0))
        B = inputs.integers((K, N), seed=inputs.seed_for(90 + nk, 1))
        C = run(A.to(cuda_device), B.to(cuda_device), cuda_device, tile=tile)
        assert_bit_exact_f16(C, oracle.gemm(u16(A), u16(B)), f"{tile_name(tile)} nK={nk}")


# ---- the 224-wide two-CTA tile on shapes it divides -------------------------------------

@pytest.mark.parametrize("tile", odd_tile_ids(), ids=tile_name)
@pytest.mark.parametrize("M,N,K", [(256, 224, 256), (512, 672, 1024), (768, 448, 320), (256, 1344, 2112)])
def test_odd_width_integer_bit_exact(cuda_device, tile, M, N, K):
    A = inputs.integers((M, K), seed=inputs.seed_for(95, 0))
    B = inputs.integers((K, N), seed=inputs.seed_for(95, 1))
    ref = oracle.gemm(u16(A), u16(B))
    for stagger in (0, 1):
        C = run(A.to(cuda_device), B.to(cuda_device), cuda_device, tile, stagger)
        assert_bit_exact_f16(C, ref, f"{M}x{N}x{K} {tile_name(tile)} stagger={stagger}")


@pytest.mark.parametrize("tile", odd_tile_ids(), ids=tile_name)
def test_odd_width_uniform_and_picked(cuda_device, tile):
    M, N, K = 1024, 1792, 1536
    A = inputs.uniform((M, K), seed=inputs.seed_for(96, 0))
    B = inputs.uniform((K, N), seed=inputs.seed_for(96, 1))
    C = run(A.to(cuda_device), B.to(cuda_device), cuda_device, tile)
    rows = boundary_rows(M, step=64, extra=4)[::2]
    assert_close(C.cpu().double().numpy()[rows], oracle.gemm(u16(A), u16(B), rows=rows), K, tile_name(tile))
    assert tile in sdt.feasible_tiles(3584, 3584, 3584)


# ---- opt-in measured sweep (SDT_AUTOTUNE=1) ------------------------------------------


def test_autotune_times_the_feasible_tiles_and_remembers_one(cuda_device, monkeypatch):
    M, N, K = 512, 768, 1024
    A = inputs.integers((M, K), seed=inputs.seed_for(9, 0))
    B = inputs.integers((K, N), seed=inputs.seed_for(9, 1))
    want = oracle.gemm(u16(A), u16(B))
    Ad, Bd = A.to(cuda_device), B.to(cuda_device)
    sdt.clear_tune_table()
    try:
        monkeypatch.setenv("SDT_AUTOTUNE", "1")
        C = run(Ad, Bd, cuda_device)
        tid = sdt.tune_table_lookup(M, N, K)
        assert tid in sdt.feasible_tiles(M, N, K)
        assert_bit_exact_f16(C, want, f"autotuned {tile_name(tid)}")
        # the remembered tile serves the next call without the variable
        monkeypatch.delenv("SDT_AUTOTUNE")
        C2 = run(Ad, Bd, cuda_device)
        assert sdt.tune_table_lookup(M, N, K) == tid
        assert_bit_exact_f16(C2, want, "served from the table")
    finally:
        sdt.clear_tune_table()
