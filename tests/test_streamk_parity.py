"""Stream-K (gemm_ex_splitk / gemm_f16_splitk with algo=SPLITK_STREAM) on the GPU
against the fp64 oracle: every tile with a stream-K form, operand layouts, fp16 and
bf16, ragged shapes, CTA counts from 1 to more than the unit count, decode rows,
run-to-run determinism, padded C, and one workspace shared with split-K calls."""
import pytest
import torch

import shape_driven_tile_gb300 as sdt
from _parity import assert_bit_exact_bf16, assert_bit_exact_f16, assert_close, assert_close_bf16
from test_gemm_ex_parity import DTYPES, LAYOUTS, operand, ref_of

pytestmark = pytest.mark.gpu
TILES = ["64x64", "64x128", "128x64", "128x128", "128x256", "s128x16", "s128x32"]


def workspace(nbytes, dev):
    ws = torch.zeros(nbytes + 256, dtype=torch.uint8, device=dev)
    return ws[(-ws.data_ptr()) % 256:][:nbytes]


ALGOS = [sdt.SPLITK_STREAM, sdt.SPLITK_STREAM_REDUCE]


def run(A, B, C, tile, ctas, ws=None, algo=sdt.SPLITK_STREAM):
    M, K = A.shape
    N = B.shape[1]
    if ws is None:
        ws = workspace(sdt.streamk_workspace_bytes(M, N, K, tile, ctas), A.device)
    sdt.gemm_ex_splitk(A, B, C, workspace=ws, tile=tile, splits=ctas or 0, algo=algo)
    sdt.check_device_status()
    return C


def check(C, Av, Bv, dt, K, integer, what):
    ref = ref_of(Av, Bv, dt)
    if integer:
        (assert_bit_exact_bf16 if dt == torch.bfloat16 else assert_bit_exact_f16)(C, ref, what)
    else:
        (assert_close_bf16 if dt == torch.bfloat16 else assert_close)(C.float().cpu().double().numpy(), ref, K, what)


@pytest.mark.parametrize("tile", TILES)
@pytest.mark.parametrize("dname", list(DTYPES))
@pytest.mark.parametrize("lname", list(LAYOUTS))
def test_layouts_integer_bit_exact(cuda_device, tile, dname, lname):
    ta, tb = LAYOUTS[lname]
    if ta and tile.startswith("s"):
        pytest.skip("skinny tiles take A stored M x K")
    dt = DTYPES[dname]
    M, N, K = 200, 264, 1000  # ragged for every tile; 16 k-tiles, the last one partial
    A, Av = operand(M, K, ta, dt, 701, True, cuda_device)
    B, Bv = operand(K, N, tb, dt, 702, True, cuda_device)
    for ctas in (None, 5):
        for algo in ALGOS:
            C = torch.full((M, N), float("nan"), dtype=dt, device=cuda_device)
            run(A, B, C, tile, ctas, algo=algo)
            check(C, Av, Bv, dt, K, True, f"{tile} {dname} {lname} ctas={ctas} algo={algo}")


@pytest.mark.parametrize("tile", TILES)
@pytest.mark.parametrize("ctas", [1, 2, 3, 7, 64, 151, 152, 1000, 100000])
def test_cta_counts(cuda_device, tile, ctas):
    # from one CTA doing everything to more CTAs than units (lowered to one unit each)
    M, N, K = 256, 384, 1024
    A, Av = operand(M, K, False, torch.float16, 711, True, cuda_device)
    B, Bv = operand(K, N, True, torch.float16, 712, True, cuda_device)
    for algo in ALGOS:
        C = torch.full((M, N), float("nan"), dtype=torch.float16, device=cuda_device)
        run(A, B, C, tile, ctas, algo=algo)
        check(C, Av, Bv, torch.float16, K, True, f"{tile} ctas={ctas} algo={algo}")


@pytest.mark.parametrize("tile", TILES)
@pytest.mark.parametrize("M,N,K", [(1, 8, 64), (16, 16, 4096), (16, 4096, 16384), (16, 8192, 4096), (3, 200, 65),
                                   (33, 1000, 3000), (1, 4096, 64), (5, 40, 17), (130, 136, 1), (64, 64, 63)])
def test_decode_and_tiny_shapes(cuda_device, tile, M, N, K):
    for dt in DTYPES.values():
        A, Av = operand(M, K, False, dt, 721, True, cuda_device)
        B, Bv = operand(K, N, True, dt, 722, True, cuda_device)
        for algo in ALGOS:
            C = torch.full((M, N), float("nan"), dtype=dt, device=cuda_device)
            run(A, B, C, tile, None, algo=algo)
            check(C, Av, Bv, dt, K, True, f"{tile} {M}x{N}x{K} {dt} algo={algo}")


@pytest.mark.parametrize("tile", ["128x256", "s128x16", "64x64"])
def test_uniform_within_tolerance_and_deterministic(cuda_device, tile):
    M, N, K = 48, 4096, 8192
    for dt in DTYPES.values():
        A, Av = operand(M, K, False, dt, 731, False, cuda_device)
        B, Bv = operand(K, N, True, dt, 732, False, cuda_device)
        ws = workspace(sdt.streamk_workspace_bytes(M, N, K, tile, None), cuda_device)
        C1 = run(A, B, torch.empty((M, N), dtype=dt, device=cuda_device), tile, None, ws)
        check(C1, Av, Bv, dt, K, False, f"{tile} {dt}")
        for _ in range(3):  # partials are summed in CTA order, whatever the order of arrival
            C2 = run(A, B, torch.empty((M, N), dtype=dt, device=cuda_device), tile, None, ws)
            assert torch.equal(C1.view(torch.int16), C2.view(torch.int16))
        # the second-kernel fix-up sums in the same order: the same bits
        C3 = run(A, B, torch.empty((M, N), dtype=dt, device=cuda_device), tile, None, ws, algo=sdt.SPLITK_STREAM_REDUCE)
        assert torch.equal(C1.view(torch.int16), C3.view(torch.int16))


def test_padded_c_untouched(cuda_device):
    M, N, K, pad = 130, 264, 777, 24
    A, Av = operand(M, K, False, torch.bfloat16, 741, True, cuda_device)
    B, Bv = operand(K, N, False, torch.bfloat16, 742, True, cuda_device)
    for tile in TILES:
        Cstore = torch.full((M + 1, N + pad), 7.0, dtype=torch.bfloat16, device=cuda_device)
        C = Cstore[:M, :N]
        run(A, B, C, tile, 37)
        assert_bit_exact_bf16(C, ref_of(Av, Bv, torch.bfloat16), f"padded C {tile}")
        assert bool((Cstore[:M, N:] == 7).all()) and bool((Cstore[M:] == 7).all())


def test_one_workspace_with_split_k(cuda_device):
    # stream-K and split-K calls in turn on one workspace zeroed once, with tile counts
    # well past what a 256-byte counter block would hold
    M, N, K = 1024, 1536, 1024
    A, Av = operand(M, K, False, torch.float16, 751, True, cuda_device)
    B, Bv = operand(K, N, False, torch.float16, 752, True, cuda_device)
    ref = ref_of(Av, Bv, torch.float16)
    cfgs = [("64x64", 152, sdt.SPLITK_STREAM), ("64x64", 3, sdt.SPLITK_IN_KERNEL), ("128x256", 4, sdt.SPLITK_REDUCE_KERNEL),
            ("128x128", 77, sdt.SPLITK_STREAM), ("64x64", 2, sdt.SPLITK_IN_KERNEL), ("128x256", 300, sdt.SPLITK_STREAM),
            ("64x128", 152, sdt.SPLITK_STREAM_REDUCE)]
    need = max(sdt.streamk_workspace_bytes(M, N, K, t, s) if a in ALGOS
               else sdt.splitk_ex_workspace_bytes(M, N, K, t, s) for t, s, a in cfgs)
    ws = workspace(need, cuda_device)
    for rep in range(2):
        for tile, s, algo in cfgs:
            C = torch.full((M, N), float("nan"), dtype=torch.float16, device=cuda_device)
            sdt.gemm_ex_splitk(A, B, C, workspace=ws, tile=tile, splits=s, algo=algo)
            sdt.check_device_status()
            assert_bit_exact_f16(C, ref, f"{tile} {s} algo {algo} rep {rep}")


def test_tight_entry_and_errors(cuda_device):
    M, N, K = 512, 512, 2048
    A, Av = operand(M, K, False, torch.float16, 761, True, cuda_device)
    B, Bv = operand(K, N, False, torch.float16, 762, True, cuda_device)
    ws = workspace(sdt.streamk_workspace_bytes(M, N, K, "128x128", None), cuda_device)
    C = sdt.gemm_f16_splitk(A, B, workspace=ws, tile="128x128", splits=0, algo=sdt.SPLITK_STREAM)
    sdt.check_device_status()
    assert_bit_exact_f16(C, ref_of(Av, Bv, torch.float16), "gemm_f16_splitk stream-K")
    with pytest.raises(sdt.SdtError) as e:  # persistent tile: no stream-K form
        sdt.gemm_ex_splitk(A, B, workspace=ws, tile="p128x256", splits=0, algo=sdt.SPLITK_STREAM)
    assert e.value.status == "SDT_ERR_TILE"
    small = ws[: sdt.streamk_workspace_bytes(M, N, K, "128x128", 8) - 256]
    with pytest.raises(sdt.SdtError) as e:  # workspace too small for 8 CTAs
        sdt.gemm_ex_splitk(A, B, workspace=small, tile="128x128", splits=8, algo=sdt.SPLITK_STREAM)
    assert e.value.status == "SDT_ERR_ARG"


def test_empty_and_refused_cases(cuda_device):
    # K = 0: the empty sum, C = 0; M = 0: nothing to do; skinny tiles refuse A stored K x M
    ws = workspace(sdt.streamk_workspace_bytes(64, 64, 64, "128x128", 4), cuda_device)
    A = torch.empty((40, 0), dtype=torch.float16, device=cuda_device)
    B = torch.empty((0, 24), dtype=torch.float16, device=cuda_device)
    C = torch.full((40, 24), 3.0, dtype=torch.float16, device=cuda_device)
    sdt.gemm_ex_splitk(A, B, C, workspace=ws, tile="128x128", splits=4, algo=sdt.SPLITK_STREAM)
    sdt.check_device_status()
    assert bool((C == 0).all())
    A0 = torch.empty((0, 64), dtype=torch.float16, device=cuda_device)
    B0 = torch.ones((64, 16), dtype=torch.float16, device=cuda_device)
    C0 = sdt.gemm_ex_splitk(A0, B0, workspace=ws, tile="128x128", splits=4, algo=sdt.SPLITK_STREAM)
    assert C0.shape == (0, 16)
    At, _ = operand(16, 256, True, torch.float16, 771, True, cuda_device)
    Bn, _ = operand(256, 64, False, torch.float16, 772, True, cuda_device)
    with pytest.raises(sdt.SdtError) as e:
        sdt.gemm_ex_splitk(At, Bn, workspace=ws, tile="s128x16", splits=4, algo=sdt.SPLITK_STREAM)
    assert e.value.status == "SDT_ERR_TILE"
