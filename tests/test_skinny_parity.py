"""Skinny tiles (s128x16, s128x32) on the GPU against the fp64 oracle: gemm_ex and
gemm_ex_splitk run them on C^T = op(B)^T . op(A)^T and write C back transposed --
few-row problems (M = 1 .. 40), both B layouts, fp16 and bf16, ragged N and K, both
split-K reductions, padded C."""
import pytest
import torch

import shape_driven_tile_gb300 as sdt
from _parity import assert_bit_exact_bf16, assert_bit_exact_f16, assert_close, assert_close_bf16
from test_gemm_ex_parity import DTYPES, operand, ref_of

pytestmark = pytest.mark.gpu
SKINNY = ["s128x16", "s128x32"]


def check(C, Av, Bv, dt, K, integer, what):
    ref = ref_of(Av, Bv, dt)
    if integer:
        (assert_bit_exact_bf16 if dt == torch.bfloat16 else assert_bit_exact_f16)(C, ref, what)
    else:
        got = C.float().cpu().double().numpy()
        (assert_close_bf16 if dt == torch.bfloat16 else assert_close)(got, ref, K, what)


@pytest.mark.parametrize("tile", SKINNY)
@pytest.mark.parametrize("dname", list(DTYPES))
@pytest.mark.parametrize("b_t", [False, True], ids=["NN", "TN"])
@pytest.mark.parametrize("M,N,K", [(1, 8, 64), (5, 200, 100), (16, 4096, 4096), (17, 136, 1000), (32, 256, 640),
                                   (40, 512, 2048)])
def test_integer_bit_exact(cuda_device, tile, dname, b_t, M, N, K):
    dt = DTYPES[dname]
    A, Av = operand(M, K, False, dt, 601, True, cuda_device)
    B, Bv = operand(K, N, b_t, dt, 602, True, cuda_device)
    C = torch.full((M, N), float("nan"), dtype=dt, device=cuda_device)
    sdt.gemm_ex(A, B, C, tile=tile)
    sdt.check_device_status()
    check(C, Av, Bv, dt, K, True, f"{tile} {dname} {'TN' if b_t else 'NN'} {M}x{N}x{K}")


@pytest.mark.parametrize("tile", SKINNY)
@pytest.mark.parametrize("dname", list(DTYPES))
def test_uniform_decode_rows(cuda_device, tile, dname):
    dt = DTYPES[dname]
    M, N, K = 16, 8192, 4096
    for b_t in (False, True):
        A, Av = operand(M, K, False, dt, 611, False, cuda_device)
        B, Bv = operand(K, N, b_t, dt, 612, False, cuda_device)
        C = sdt.gemm_ex(A, B, tile=tile)
        sdt.check_device_status()
        check(C, Av, Bv, dt, K, False, f"{tile} {dname} b_t={b_t}")


@pytest.mark.parametrize("tile", SKINNY)
@pytest.mark.parametrize("algo", [sdt.SPLITK_REDUCE_KERNEL, sdt.SPLITK_IN_KERNEL])
@pytest.mark.parametrize("M,N,K,splits", [(16, 4096, 4096, 4), (3, 264, 1000, 5), (33, 1024, 8192, 8)])
def test_splitk(cuda_device, tile, algo, M, N, K, splits):
    for dt in DTYPES.values():
        for b_t in (False, True):
            A, Av = operand(M, K, False, dt, 621, True, cuda_device)
            B, Bv = operand(K, N, b_t, dt, 622, True, cuda_device)
            nbytes = sdt.splitk_ex_workspace_bytes(M, N, K, tile, splits)
            ws = torch.zeros(nbytes + 256, dtype=torch.uint8, device=cuda_device)
            ws = ws[(-ws.data_ptr()) % 256:][:nbytes]
            C = torch.full((M, N), float("nan"), dtype=dt, device=cuda_device)
            for _ in range(2):
                sdt.gemm_ex_splitk(A, B, C, workspace=ws, tile=tile, splits=splits, algo=algo)
                sdt.check_device_status()
                check(C, Av, Bv, dt, K, True, f"{tile} split {splits} algo {algo} {M}x{N}x{K} b_t={b_t}")


def test_padded_c_untouched(cuda_device):
    M, N, K, pad = 20, 136, 512, 24
    A, Av = operand(M, K, False, torch.float16, 631, True, cuda_device)
    B, Bv = operand(K, N, True, torch.float16, 632, True, cuda_device)
    for tile in SKINNY:
        Cstore = torch.full((M + 1, N + pad), 7.0, dtype=torch.float16, device=cuda_device)
        C = Cstore[:M, :N]
        sdt.gemm_ex(A, B, C, tile=tile)
        sdt.check_device_status()
        assert_bit_exact_f16(C, ref_of(Av, Bv, torch.float16), f"padded C {tile}")
        assert bool((Cstore[:M, N:] == 7).all()) and bool((Cstore[M:] == 7).all())


def test_transposed_a_is_refused(cuda_device):
    A, _ = operand(16, 256, True, torch.float16, 641, True, cuda_device)   # A stored K x M
    B, _ = operand(256, 64, False, torch.float16, 642, True, cuda_device)
    with pytest.raises(sdt.SdtError) as e:
        sdt.gemm_ex(A, B, tile="s128x16")
    assert e.value.status == "SDT_ERR_TILE"
