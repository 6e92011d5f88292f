"""gemm_ex on the GPU against the fp64 oracle: transposed operands (NN, NT, TN,
TT), fp16 and bf16, shapes no tile divides, caller row strides, through every
kernel family (one-CTA tile, persistent, two-CTA pair) and the picker."""
import numpy as np
import pytest
import torch

import oracle
import shape_driven_tile_gb300 as sdt
from shape_driven_tile_gb300 import inputs
from _parity import (assert_bit_exact_bf16, assert_bit_exact_f16, assert_close, assert_close_bf16, u16)

pytestmark = pytest.mark.gpu

LAYOUTS = {"NN": (False, False), "NT": (False, True), "TN": (True, False), "TT": (True, True)}
DTYPES = {"f16": torch.float16, "bf16": torch.bfloat16}
TILES = ["64x64", "128x128", "p128x256", "2cta_256x256", "2cta_256x224", -1]


def operand(rows, cols, trans, dtype, seed, integer, dev, pad=0):
    """Logical [rows, cols] view; stored row-major (trans=False) or as its transpose,
    with `pad` extra elements per stored row (at least enough to make stored rows a
    multiple of 8 elements: the row stride of every operand is a multiple of 16 bytes)."""
    vals = (inputs.integers((rows, cols), seed=seed, dtype=torch.float32) if integer
            else inputs.uniform((rows, cols), seed=seed, dtype=torch.float32)).to(dtype)
    pad = max(pad, (-(rows if trans else cols)) % 8)
    if not trans:
        store = torch.zeros((rows, cols + pad), dtype=dtype)
        store[:, :cols] = vals
        return store.to(dev)[:, :cols], vals
    store = torch.zeros((cols, rows + pad), dtype=dtype)
    store[:, :rows] = vals.t()
    return store.to(dev)[:, :rows].t(), vals


def ref_of(Av, Bv, dtype):
    return oracle.gemm(u16(Av), u16(Bv), dtype="bf16" if dtype == torch.bfloat16 else "f16")


@pytest.mark.parametrize("tile", TILES, ids=str)
@pytest.mark.parametrize("dname", list(DTYPES))
@pytest.mark.parametrize("lname", list(LAYOUTS))
def test_layouts_dtypes_integer_bit_exact(cuda_device, lname, dname, tile):
    ta, tb = LAYOUTS[lname]
    dt = DTYPES[dname]
    M, N, K = 384, 320, 448  # ragged for the 128- and 256-wide tiles
    A, Av = operand(M, K, ta, dt, 401, True, cuda_device)
    B, Bv = operand(K, N, tb, dt, 402, True, cuda_device)
    C = sdt.gemm_ex(A, B, tile=tile)
    sdt.check_device_status()
    ref = ref_of(Av, Bv, dt)
    (assert_bit_exact_bf16 if dt == torch.bfloat16 else assert_bit_exact_f16)(C, ref, f"{lname} {dname} {tile}")


@pytest.mark.parametrize("dname", list(DTYPES))
@pytest.mark.parametrize("M,N,K", [(1, 8, 1), (7, 8, 9), (129, 136, 65), (300, 200, 100), (1000, 1000, 1000),
                                   (2049, 1032, 777), (64, 4096, 4096), (4096, 64, 4096)])
def test_ragged_uniform_picked(cuda_device, M, N, K, dname):
    dt = DTYPES[dname]
    for lname in ("NN", "TN"):
        ta, tb = LAYOUTS[lname]
        A, Av = operand(M, K, ta, dt, 411, False, cuda_device)
        B, Bv = operand(K, N, tb, dt, 412, False, cuda_device)
        C = sdt.gemm_ex(A, B)
        sdt.check_device_status()
        ref = ref_of(Av, Bv, dt)
        got = C.float().cpu().double().numpy()
        if dt == torch.bfloat16:
            assert_close_bf16(got, ref, K, f"{M}x{N}x{K} {lname}")
        else:
            assert_close(got, ref, K, f"{M}x{N}x{K} {lname}")


def test_padded_c_leaves_padding_untouched(cuda_device):
    M, N, K, pad = 300, 136, 200, 24
    A, Av = operand(M, K, False, torch.float16, 421, True, cuda_device)
    B, Bv = operand(K, N, False, torch.float16, 422, True, cuda_device)
    Cstore = torch.full((M + 1, N + pad), 7.0, dtype=torch.float16, device=cuda_device)
    C = Cstore[:M, :N]
    for tile in TILES:
        Cstore.fill_(7.0)
        sdt.gemm_ex(A, B, C, tile=tile)
        sdt.check_device_status()
        assert_bit_exact_f16(C, ref_of(Av, Bv, torch.float16), f"padded C {tile}")
        assert bool((Cstore[:M, N:] == 7).all()), f"{tile} wrote into the row padding"
        assert bool((Cstore[M:] == 7).all()), f"{tile} wrote past the last row"


def test_padded_and_tight_operands_agree(cuda_device):
    # A padded operand and a tight one of the same shape must get their own tensor maps
    # (the map cache is keyed by the row stride): results are identical.
    M, N, K = 512, 512, 1024
    Ap, Av = operand(M, K, False, torch.float16, 431, False, cuda_device, pad=64)
    Bp, Bv = operand(K, N, False, torch.float16, 432, False, cuda_device, pad=32)
    At, Bt = Ap.contiguous(), Bp.contiguous()
    before = sdt.lib().sdt_debug_tensor_map_encodes()
    C1 = sdt.gemm_ex(At, Bt, tile="128x128")
    C2 = sdt.gemm_ex(Ap, Bp, tile="128x128")
    assert sdt.lib().sdt_debug_tensor_map_encodes() >= before + 2
    assert torch.equal(C1.view(torch.int16), C2.view(torch.int16))
    assert_close(C2.cpu().double().numpy(), ref_of(Av, Bv, torch.float16), K, "padded")


def test_gemm_ex_matches_gemm_f16_bitwise(cuda_device):
    M = N = K = 2048
    A = inputs.uniform((M, K), seed=441).to(cuda_device)
    B = inputs.uniform((K, N), seed=442).to(cuda_device)
    for tile in ("128x128", "p128x256", "2cta_256x256"):
        C0 = sdt.gemm_f16_with_tile(A, B, tile=tile, stagger=0)
        import os
        old = os.environ.get("SDT_STAGGER")
        os.environ["SDT_STAGGER"] = "0"
        try:
            C1 = sdt.gemm_ex(A, B, tile=tile)
        finally:
            if old is None:
                del os.environ["SDT_STAGGER"]
            else:
                os.environ["SDT_STAGGER"] = old
        assert torch.equal(C0.view(torch.int16), C1.view(torch.int16)), tile


def test_large_tn_bf16_sampled_rows(cuda_device):
    M = N = K = 4096
    A, Av = operand(M, K, True, torch.bfloat16, 451, False, cuda_device)
    B, Bv = operand(K, N, False, torch.bfloat16, 452, False, cuda_device)
    C = sdt.gemm_ex(A, B)
    sdt.check_device_status()
    rows = np.array([0, 1, 255, 256, 2047, 4095])
    ref = oracle.gemm(u16(Av), u16(Bv), rows=rows, dtype="bf16")
    assert_close_bf16(C.float().cpu().double().numpy()[rows], ref, K, "4096 TN bf16")


def test_k_zero_and_errors(cuda_device):
    A = torch.empty((16, 0), dtype=torch.float16, device=cuda_device)
    B = torch.empty((0, 24), dtype=torch.float16, device=cuda_device)
    Cs = torch.full((16, 32), 5.0, dtype=torch.float16, device=cuda_device)
    sdt.gemm_ex(A, B, Cs[:, :24])
    torch.cuda.synchronize()
    assert bool((Cs[:, :24] == 0).all()) and bool((Cs[:, 24:] == 5).all())
    A = torch.zeros((16, 16), dtype=torch.float16, device=cuda_device)
    B = torch.zeros((16, 12), dtype=torch.float16, device=cuda_device)
    with pytest.raises(sdt.SdtError) as e:
        sdt.gemm_ex(A, B)                      # N % 8 != 0
    assert e.value.status == "SDT_ERR_SHAPE"
    with pytest.raises(TypeError):
        sdt.gemm_ex(A, B.to(torch.bfloat16))   # mixed types


@pytest.mark.parametrize("tile", ["p128x128", "p128x256", "2cta_256x128", "2cta_256x256", "2cta_256x224"])
@pytest.mark.parametrize("M,N,K", [(1, 8, 1), (3, 40, 70), (257, 264, 130), (130, 1000, 64)])
def test_tma_store_tiles_on_tiny_ragged_shapes(cuda_device, tile, M, N, K):
    # the persistent and two-CTA kernels store C through 32 x 32 TMA boxes: rows and
    # columns past C (most of the tile here) must be dropped, the rest exact
    for dname, dt in DTYPES.items():
        A, Av = operand(M, K, False, dt, 451, True, cuda_device)
        B, Bv = operand(K, N, True, dt, 452, True, cuda_device)
        Cstore = torch.full((M + 2, N + 16), 3.0, dtype=dt, device=cuda_device)
        C = Cstore[:M, :N]
        sdt.gemm_ex(A, B, C, tile=tile)
        sdt.check_device_status()
        (assert_bit_exact_bf16 if dt == torch.bfloat16 else assert_bit_exact_f16)(C, ref_of(Av, Bv, dt),
                                                                                   f"{tile} {M}x{N}x{K} {dname}")
        assert bool((Cstore[:M, N:] == 3).all()) and bool((Cstore[M:] == 3).all()), f"{tile} wrote outside C"
