"""gemm_f16_splitk on the GPU against the fp64 oracle: every split-K tile, several
split counts (even, uneven, one k-tile per split), both reduction algorithms,
integer inputs bit-exact, a reused workspace, and the argument checks."""
import numpy as np
import pytest
import torch

import oracle
import shape_driven_tile_gb300 as sdt
from shape_driven_tile_gb300 import inputs
from _parity import assert_bit_exact_f16, assert_close, nan_like, u16

pytestmark = pytest.mark.gpu

SPLIT_TILES = ["64x64", "64x128", "128x64", "128x128", "128x256"]
ALGOS = [sdt.SPLITK_REDUCE_KERNEL, sdt.SPLITK_IN_KERNEL]


def run(A, B, ws, tile, splits, algo):
    C = nan_like((A.shape[0], B.shape[1]), A.device)
    sdt.gemm_f16_splitk(A, B, C, workspace=ws, tile=tile, splits=splits, algo=algo)
    sdt.check_device_status()
    return C


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("tile", SPLIT_TILES)
def test_integer_bit_exact_all_split_counts(cuda_device, tile, algo):
    M, N, K = 512, 512, 1280  # 20 k-tiles
    A = inputs.integers((M, K), seed=201)
    B = inputs.integers((K, N), seed=202)
    ref = oracle.gemm(u16(A), u16(B))
    Ad, Bd = A.to(cuda_device), B.to(cuda_device)
    for splits in (1, 2, 3, 7, 20):
        ws = sdt.splitk_workspace(M, N, K, tile, splits, device=cuda_device)
        C = run(Ad, Bd, ws, tile, splits, algo)
        assert_bit_exact_f16(C, ref, f"{tile} splits={splits} algo={algo}")


@pytest.mark.parametrize("algo", ALGOS)
def test_uniform_deep_k_picked(cuda_device, algo):
    M, N, K = 256, 512, 8192
    A = inputs.uniform((M, K), seed=211)
    B = inputs.uniform((K, N), seed=212)
    tid, sp = sdt.pick_splitk(M, N, K, sm_count=sdt.device_sm_count())
    assert sp > 1
    ws = sdt.splitk_workspace(M, N, K, tid, sp, device=cuda_device)
    C = run(A.to(cuda_device), B.to(cuda_device), ws, -1, 0, algo)
    assert_close(C.cpu().double().numpy(), oracle.gemm(u16(A), u16(B)), K, f"picked {sdt.tile_info(tid)['name']} x{sp}")


def test_workspace_reused_across_calls(cuda_device):
    # the in-kernel reduction resets its counters, so back-to-back calls on one
    # workspace (different operands) both come out right
    M, N, K = 256, 256, 2048
    tile, splits = "64x64", 8
    ws = sdt.splitk_workspace(M, N, K, tile, splits, device=cuda_device)
    for seed in (221, 223, 225):
        A = inputs.integers((M, K), seed=seed)
        B = inputs.integers((K, N), seed=seed + 1)
        C = run(A.to(cuda_device), B.to(cuda_device), ws, tile, splits, sdt.SPLITK_IN_KERNEL)
        assert_bit_exact_f16(C, oracle.gemm(u16(A), u16(B)), f"seed {seed}")


def test_splitk_matches_unsplit_bitwise_on_integers(cuda_device):
    M, N, K = 1024, 768, 4096
    A = inputs.integers((M, K), seed=231).to(cuda_device)
    B = inputs.integers((K, N), seed=232).to(cuda_device)
    C0 = sdt.gemm_f16_with_tile(A, B, tile="128x128")
    ws = sdt.splitk_workspace(M, N, K, "128x128", 4, device=cuda_device)
    C1 = run(A, B, ws, "128x128", 4, sdt.SPLITK_IN_KERNEL)
    assert torch.equal(C0.view(torch.int16), C1.view(torch.int16))


def test_splitk_errors(cuda_device):
    M, N, K = 256, 256, 1024
    A = torch.zeros((M, K), dtype=torch.float16, device=cuda_device)
    B = torch.zeros((K, N), dtype=torch.float16, device=cuda_device)
    ws = sdt.splitk_workspace(M, N, K, "64x64", 2, device=cuda_device)
    with pytest.raises(sdt.SdtError) as e:
        sdt.gemm_f16_splitk(A, B, workspace=ws, tile="64x64", splits=8)   # workspace sized for 2
    assert e.value.status == "SDT_ERR_ARG"
    with pytest.raises(sdt.SdtError) as e:
        sdt.gemm_f16_splitk(A, B, workspace=ws, tile="p128x256", splits=2)
    assert e.value.status == "SDT_ERR_TILE"
    with pytest.raises(sdt.SdtError) as e:
        sdt.gemm_f16_splitk(A, B, workspace=ws[16:], tile="64x64", splits=2)
    assert e.value.status == "SDT_ERR_ALIGN"
    with pytest.raises(sdt.SdtError) as e:
        sdt.gemm_f16_splitk(A, B, workspace=ws, tile="64x64", splits=99)
    assert e.value.status == "SDT_ERR_ARG"
