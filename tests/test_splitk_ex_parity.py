"""gemm_ex_splitk on the GPU against the fp64 oracle: every operand layout, fp16 and
bf16, shapes no tile divides (including M = 16 decode rows), both reduction
algorithms, caller row strides."""
import numpy as np
import pytest
import torch

import shape_driven_tile_gb300 as sdt
from _parity import assert_bit_exact_bf16, assert_bit_exact_f16, assert_close, assert_close_bf16
from test_gemm_ex_parity import DTYPES, LAYOUTS, operand, ref_of

pytestmark = pytest.mark.gpu
ALGOS = {"reduce_kernel": sdt.SPLITK_REDUCE_KERNEL, "in_kernel": sdt.SPLITK_IN_KERNEL}


def workspace(M, N, K, tile, splits, dev):
    nbytes = sdt.splitk_ex_workspace_bytes(M, N, K, tile, splits)
    assert nbytes > 0
    ws = torch.zeros(nbytes + 256, dtype=torch.uint8, device=dev)
    off = (-ws.data_ptr()) % 256
    return ws[off:off + nbytes]


@pytest.mark.parametrize("algo", list(ALGOS))
@pytest.mark.parametrize("tile", ["64x64", "128x128", "128x256"])
@pytest.mark.parametrize("dname", list(DTYPES))
@pytest.mark.parametrize("lname", list(LAYOUTS))
def test_integer_bit_exact(cuda_device, lname, dname, tile, algo):
    # integer inputs: every partial and their sum in split order are exact
    ta, tb = LAYOUTS[lname]
    dt = DTYPES[dname]
    M, N, K = 200, 264, 1000  # ragged for every tile, K not a multiple of 64
    A, Av = operand(M, K, ta, dt, 501, True, cuda_device)
    B, Bv = operand(K, N, tb, dt, 502, True, cuda_device)
    C = torch.full((M, N), float("nan"), dtype=dt, device=cuda_device)
    ws = workspace(M, N, K, tile, 5, cuda_device)
    for _ in range(2):  # the in-kernel counters must come back to zero
        sdt.gemm_ex_splitk(A, B, C, workspace=ws, tile=tile, splits=5, algo=ALGOS[algo])
        sdt.check_device_status()
        (assert_bit_exact_bf16 if dt == torch.bfloat16 else assert_bit_exact_f16)(
            C, ref_of(Av, Bv, dt), f"{lname} {dname} {tile} {algo}")


@pytest.mark.parametrize("dname", list(DTYPES))
@pytest.mark.parametrize("M,N,K,splits", [(16, 4096, 4096, 8), (16, 16, 4096, 32), (16, 128, 8192, 16),
                                          (4096, 64, 4096, 4), (129, 136, 65, 2)])
def test_uniform_decode_and_skinny_shapes(cuda_device, M, N, K, splits, dname):
    dt = DTYPES[dname]
    for lname in ("NN", "TN"):
        ta, tb = LAYOUTS[lname]
        A, Av = operand(M, K, ta, dt, 511, False, cuda_device)
        B, Bv = operand(K, N, tb, dt, 512, False, cuda_device)
        for algo in ALGOS.values():
            C = torch.full((M, N), float("nan"), dtype=dt, device=cuda_device)
            ws = workspace(M, N, K, "64x64", splits, cuda_device)
            sdt.gemm_ex_splitk(A, B, C, workspace=ws, tile="64x64", splits=splits, algo=algo)
            sdt.check_device_status()
            got = C.float().cpu().double().numpy()
            (assert_close_bf16 if dt == torch.bfloat16 else assert_close)(got, ref_of(Av, Bv, dt), K,
                                                                         f"{M}x{N}x{K} {lname} s{splits} a{algo}")


def test_padded_c_and_picked(cuda_device):
    M, N, K, pad = 300, 136, 2000, 24
    A, Av = operand(M, K, False, torch.float16, 521, True, cuda_device)
    B, Bv = operand(K, N, True, torch.float16, 522, True, cuda_device)
    Cstore = torch.full((M + 1, N + pad), 7.0, dtype=torch.float16, device=cuda_device)
    C = Cstore[:M, :N]
    tid, sp = sdt.pick_splitk_any(M, N, K)
    ws = workspace(M, N, K, tid, sp, cuda_device)
    for algo in ALGOS.values():
        Cstore.fill_(7.0)
        sdt.gemm_ex_splitk(A, B, C, workspace=ws, tile=-1, splits=0, algo=algo)
        sdt.check_device_status()
        assert_bit_exact_f16(C, ref_of(Av, Bv, torch.float16), f"padded C algo {algo}")
        assert bool((Cstore[:M, N:] == 7).all()) and bool((Cstore[M:] == 7).all())


def test_matches_gemm_f16_splitk_bitwise(cuda_device):
    # on a shape the tile divides the general form is the same computation
    M = N = 512
    K = 4096
    A, _ = operand(M, K, False, torch.float16, 531, False, cuda_device)
    B, _ = operand(K, N, False, torch.float16, 532, False, cuda_device)
    A, B = A.contiguous(), B.contiguous()
    for algo in ALGOS.values():
        ws = workspace(M, N, K, "128x128", 4, cuda_device)
        C0 = sdt.gemm_f16_splitk(A, B, workspace=ws, tile="128x128", splits=4, algo=algo)
        C1 = sdt.gemm_ex_splitk(A, B, workspace=ws, tile="128x128", splits=4, algo=algo)
        torch.cuda.synchronize()
        assert torch.equal(C0.view(torch.int16), C1.view(torch.int16))


def test_errors(cuda_device):
    A = torch.zeros((16, 64), dtype=torch.float16, device=cuda_device)
    B = torch.zeros((64, 16), dtype=torch.float16, device=cuda_device)
    ws = workspace(16, 16, 64, "64x64", 1, cuda_device)
    with pytest.raises(sdt.SdtError) as e:
        sdt.gemm_ex_splitk(A, B, workspace=ws, tile="p128x256", splits=2)
    assert e.value.status == "SDT_ERR_TILE"
    with pytest.raises(sdt.SdtError) as e:
        sdt.gemm_ex_splitk(A, B, workspace=ws[:64], tile="64x64", splits=1)
    assert e.value.status == "SDT_ERR_ARG"


def test_one_workspace_serves_any_sequence_of_configurations(cuda_device):
    # zeroed once, then in-kernel reductions with different tiles and split counts in turn
    # (each configuration's partial planes must never land on another's counters)
    M, N, K = 256, 384, 2048
    A, Av = operand(M, K, False, torch.float16, 541, True, cuda_device)
    B, Bv = operand(K, N, False, torch.float16, 542, True, cuda_device)
    ref = ref_of(Av, Bv, torch.float16)
    cfgs = [("64x64", 2), ("128x128", 5), ("64x128", 3), ("64x64", 7), ("128x64", 2), ("128x256", 4)]
    need = max(sdt.splitk_ex_workspace_bytes(M, N, K, t, s) for t, s in cfgs)
    ws = torch.zeros(need + 256, dtype=torch.uint8, device=cuda_device)
    ws = ws[(-ws.data_ptr()) % 256:][:need]
    for rep in range(2):
        for tile, splits in cfgs:
            for algo in (sdt.SPLITK_IN_KERNEL, sdt.SPLITK_REDUCE_KERNEL):
                C = torch.full((M, N), float("nan"), dtype=torch.float16, device=cuda_device)
                sdt.gemm_ex_splitk(A, B, C, workspace=ws, tile=tile, splits=splits, algo=algo)
                sdt.check_device_status()
                assert_bit_exact_f16(C, ref, f"{tile} s{splits} a{algo} rep{rep}")
