"""The two-CTA tile's last round split in K (gemm_f16_ws / gemm_ex_ws) against the fp64
oracle: forced split counts 2..8 on every two-CTA tile, ragged shapes, all four layouts
in fp16 and bf16, the planned split at the sizes where it applies (4096^3: two k-ranges
per leftover tile; 2560^3: three), integer-valued inputs bit for bit, repeat calls bit
for bit, the workspace's counters back at zero after every call, and the argument
checks."""
import numpy as np
import pytest
import torch

import oracle
import shape_driven_tile_gb300 as sdt
from shape_driven_tile_gb300 import inputs
from _parity import (assert_bit_exact_bf16, assert_bit_exact_f16, assert_close, assert_close_bf16,
                     boundary_rows, u16)
from shape_driven_tile_gb300._lib import SdtError

pytestmark = pytest.mark.gpu

COUNTER_BYTES = 1 << 20
PAIR_TILES = ["2cta_256x256", "2cta_256x224", "2cta_256x128"]
LAYOUTS = {"NN": (False, False), "NT": (False, True), "TN": (True, False), "TT": (True, True)}
DTYPES = {"f16": torch.float16, "bf16": torch.bfloat16}


@pytest.fixture(scope="module")
def ws(cuda_device):
    return sdt.gemm_workspace(cuda_device)


def counters_zero(ws):
    torch.cuda.synchronize()
    return bool((ws[:COUNTER_BYTES].view(torch.int32) == 0).all())


def operand(rows, cols, trans, dtype, seed, integer, dev):
    """Logical [rows, cols] view, stored row-major or as its transpose (rows padded to 8 elements)."""
    vals = (inputs.integers((rows, cols), seed=seed, dtype=torch.float32) if integer
            else inputs.uniform((rows, cols), seed=seed, dtype=torch.float32)).to(dtype)
    if not trans:
        store = torch.zeros((rows, cols + (-cols) % 8), dtype=dtype)
        store[:, :cols] = vals
        return store.to(dev)[:, :cols], vals
    store = torch.zeros((cols, rows + (-rows) % 8), dtype=dtype)
    store[:, :rows] = vals.t()
    return store.to(dev)[:, :rows].t(), vals


def ref_of(Av, Bv, dtype):
    return oracle.gemm(u16(Av), u16(Bv), dtype="bf16" if dtype == torch.bfloat16 else "f16")


def plan(M, N, K, tile, tail_splits=-1):
    return sdt.pair_tail_plan(M, N, K, tile, sdt.device_sm_count(), sdt.lib().sdt_device_smem_optin(),
                              tail_splits=tail_splits)


@pytest.mark.parametrize("tile", PAIR_TILES)
@pytest.mark.parametrize("S", [2, 3, 5, 7])
def test_forced_splits_integer_bit_exact(cuda_device, ws, tile, S):
    # 2 x 2 tiles (2 x 4 for the 128-wide tile: fewer than the pairs, so every tile is in the
    # last round); K = 2112 is 33 k-tiles, which no split count above divides
    M, N, K = 512, 448 if tile == "2cta_256x224" else 512, 2112
    bn = sdt.tile_info(sdt.tile_id(tile))["BN"]
    tail_start, items, splits, long_k = plan(M, N, K, tile, S)
    assert (tail_start, splits) == (0, S) and items == (M // 256) * (N // bn) * S
    assert 33 // S <= long_k <= 33 - (S - 1)
    A, Av = operand(M, K, False, torch.float16, 701, True, cuda_device)
    B, Bv = operand(K, N, False, torch.float16, 702, True, cuda_device)
    C = torch.full((M, N), float("nan"), dtype=torch.float16, device=cuda_device)
    sdt.gemm_ex_ws(A, B, C, workspace=ws, tile=tile, tail_splits=S)
    sdt.check_device_status()
    assert counters_zero(ws)
    assert_bit_exact_f16(C, ref_of(Av, Bv, torch.float16), f"{tile} S={S}")
    plain = sdt.gemm_ex(A, B, tile=tile)
    assert torch.equal(C.view(torch.int16), plain.view(torch.int16))


@pytest.mark.parametrize("dname", list(DTYPES))
@pytest.mark.parametrize("lname", list(LAYOUTS))
def test_ragged_layouts_dtypes(cuda_device, ws, lname, dname):
    ta, tb = LAYOUTS[lname]
    dt = DTYPES[dname]
    M, N, K = 300, 520, 1000  # ragged in every dimension; K not a multiple of 64
    A, Av = operand(M, K, ta, dt, 711, False, cuda_device)
    B, Bv = operand(K, N, tb, dt, 712, False, cuda_device)
    ref = ref_of(Av, Bv, dt)
    for tile, S in (("2cta_256x256", 3), ("2cta_256x128", 2), ("2cta_256x224", 4)):
        C = sdt.gemm_ex_ws(A, B, workspace=ws, tile=tile, tail_splits=S)
        sdt.check_device_status()
        got = C.float().cpu().double().numpy()
        what = f"{lname} {dname} {tile} S={S}"
        (assert_close_bf16 if dt == torch.bfloat16 else assert_close)(got, ref, K, what)
    assert counters_zero(ws)
    # integer-valued operands: bit for bit
    A, Av = operand(M, K, ta, dt, 713, True, cuda_device)
    B, Bv = operand(K, N, tb, dt, 714, True, cuda_device)
    C = sdt.gemm_ex_ws(A, B, workspace=ws, tile="2cta_256x256", tail_splits=5)
    sdt.check_device_status()
    (assert_bit_exact_bf16 if dt == torch.bfloat16 else assert_bit_exact_f16)(C, ref_of(Av, Bv, dt), lname)


def test_padded_c_outside_untouched(cuda_device, ws):
    M, N, K, pad = 260, 264, 640, 24
    A, Av = operand(M, K, False, torch.float16, 721, True, cuda_device)
    B, Bv = operand(K, N, False, torch.float16, 722, True, cuda_device)
    store = torch.full((M + 1, N + pad), 7.0, dtype=torch.float16, device=cuda_device)
    C = store[:M, :N]
    sdt.gemm_ex_ws(A, B, C, workspace=ws, tile="2cta_256x256", tail_splits=4)
    sdt.check_device_status()
    assert_bit_exact_f16(C.contiguous(), ref_of(Av, Bv, torch.float16), "padded C")
    assert bool((store[:M, N:] == 7.0).all()) and bool((store[M:] == 7.0).all())


@pytest.mark.parametrize("n,splits", [(4096, -1), (2560, 3), (8192, -1)])
def test_planned_split_square(cuda_device, ws, n, splits):
    # 4096^3 and 8192^3 as planned (two k-ranges per leftover tile on a 152-SM GPU), 2560^3
    # with a forced count (the estimate keeps half-width items there)
    tile = sdt.pick_tile(n, n, n)
    assert sdt.tile_info(tile)["name"] == "2cta_256x256"
    if splits < 0 and sdt.device_sm_count() != 152:
        pytest.skip("the planned split count is that of a 152-SM GPU")
    assert plan(n, n, n, tile, splits)[2] == (splits if splits > 0 else 2)
    A = inputs.uniform((n, n), seed=inputs.seed_for(1, 0))
    B = inputs.uniform((n, n), seed=inputs.seed_for(1, 1))
    Ad, Bd = A.to(cuda_device), B.to(cuda_device)
    C = torch.full((n, n), float("nan"), dtype=torch.float16, device=cuda_device)
    sdt.gemm_ex_ws(Ad, Bd, C, workspace=ws, tile=tile, tail_splits=splits)
    sdt.check_device_status()
    assert counters_zero(ws)
    assert bool(torch.isfinite(C).all())
    # rows of the last round's tiles (the leftover tiles are the last in raster order) and
    # the tile-row boundaries
    rows = np.unique(np.concatenate([boundary_rows(n, step=256, extra=8)[::2], np.arange(n - 256, n, 37)]))
    ref = oracle.gemm(u16(A), u16(B), rows=rows)
    assert_close(C.cpu().double().numpy()[rows], ref, n, f"{n}^3 ws")
    # the same launch without a workspace agrees within the tolerance, and a second call
    # with the workspace is bit-identical to the first
    plain = sdt.gemm_f16(Ad, Bd).cpu().double().numpy()
    assert_close(plain[rows], ref, n, f"{n}^3 plain")
    C2 = sdt.gemm_ex_ws(Ad, Bd, workspace=ws, tile=tile, tail_splits=splits)
    assert torch.equal(C.view(torch.int16), C2.view(torch.int16))


def test_split_integer_4096_bit_exact(cuda_device, ws):
    n = 4096
    A = inputs.integers((n, n), seed=731)
    B = inputs.integers((n, n), seed=732)
    Ad, Bd = A.to(cuda_device), B.to(cuda_device)
    C = sdt.gemm_ex_ws(Ad, Bd, workspace=ws, tail_splits=2)
    plain = sdt.gemm_f16(Ad, Bd)
    sdt.check_device_status()
    assert torch.equal(C.view(torch.int16), plain.view(torch.int16))
    rows = np.concatenate([np.arange(0, 8), np.arange(n - 300, n, 13)])
    assert_bit_exact_f16(C.cpu()[rows], oracle.gemm(u16(A), u16(B), rows=rows), "4096^3 integer")


def test_dirty_partial_slots(cuda_device, ws):
    # every slot is written before it is read: garbage left in the partials changes nothing
    M, N, K = 512, 512, 1024
    A, Av = operand(M, K, False, torch.float16, 741, True, cuda_device)
    B, Bv = operand(K, N, False, torch.float16, 742, True, cuda_device)
    ws[COUNTER_BYTES:].view(torch.float16).fill_(float("nan"))
    C = sdt.gemm_ex_ws(A, B, workspace=ws, tile="2cta_256x256", tail_splits=6)
    sdt.check_device_status()
    assert_bit_exact_f16(C, ref_of(Av, Bv, torch.float16), "dirty slots")
    assert counters_zero(ws)


def test_graph_capture_replay(cuda_device, ws):
    n = 2560
    A = inputs.uniform((n, n), seed=751).to(cuda_device)
    B = inputs.uniform((n, n), seed=752).to(cuda_device)
    C = torch.empty((n, n), dtype=torch.float16, device=cuda_device)
    eager = sdt.gemm_f16_ws(A, B, workspace=ws).clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        sdt.gemm_f16_ws(A, B, C, workspace=ws)
        with torch.cuda.graph(g, stream=s):
            for _ in range(3):
                sdt.gemm_f16_ws(A, B, C, workspace=ws)
    C.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(C.view(torch.int16), eager.view(torch.int16))
    assert counters_zero(ws)


def test_no_workspace_is_gemm_f16(cuda_device):
    n = 4096
    A = inputs.uniform((n, n), seed=761).to(cuda_device)
    B = inputs.uniform((n, n), seed=762).to(cuda_device)
    a = sdt.gemm_f16_ws(A, B, workspace=None)
    b = sdt.gemm_f16(A, B)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    c = sdt.gemm_ex_ws(A, B, workspace=None, tail_splits=4)
    assert torch.equal(c.view(torch.int16), b.view(torch.int16))


def test_workspace_argument_checks(cuda_device, ws):
    A = torch.zeros((512, 512), dtype=torch.float16, device=cuda_device)
    B = torch.zeros((512, 512), dtype=torch.float16, device=cuda_device)
    need = sdt.gemm_workspace_bytes()
    assert need == sdt.gemm_workspace_bytes(sdt.device_sm_count())
    raw = torch.zeros(need + 512, dtype=torch.uint8, device=cuda_device)
    base = (-raw.data_ptr()) % 256
    with pytest.raises(SdtError) as e:  # not 256-byte aligned
        sdt.gemm_f16_ws(A, B, workspace=raw[base + 16:base + 16 + need])
    assert e.value.status == "SDT_ERR_ALIGN"
    with pytest.raises(SdtError) as e:  # too small
        sdt.gemm_f16_ws(A, B, workspace=raw[base:base + need - 256])
    assert e.value.status == "SDT_ERR_ARG"
    for bad in (1, -2, 9):
        with pytest.raises(SdtError) as e:
            sdt.gemm_ex_ws(A, B, workspace=ws, tile="2cta_256x256", tail_splits=bad)
        assert e.value.status == "SDT_ERR_ARG"
    # K == 0 and empty outputs through the workspace entry points
    C = torch.full((512, 512), 3.0, dtype=torch.float16, device=cuda_device)
    A0 = torch.empty((512, 0), dtype=torch.float16, device=cuda_device)
    B0 = torch.empty((0, 512), dtype=torch.float16, device=cuda_device)
    sdt.gemm_ex_ws(A0, B0, C, workspace=ws, tile="2cta_256x256", tail_splits=2)
    torch.cuda.synchronize()
    assert bool((C == 0).all())
    sdt.gemm_ex_ws(torch.empty((0, 512), dtype=torch.float16, device=cuda_device), B, workspace=ws)
    assert counters_zero(ws)
