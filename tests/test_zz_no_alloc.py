"""The split-K entry point that allocates nothing (gemm_f16_splitk_noalloc).

It exists for callers that cannot allocate device memory where they multiply
(code that must not synchronise the device, plugin hosts with a fixed memory
budget and no allocator, allocator-free latency-critical loops): its workspace
is a fixed 16 MiB array the library keeps in device memory, the 1 MiB counter
region of the split-K workspace layout followed by 15 MiB of fp32 partials.

These tests call it through the C ABI.  Its kernels and summation order are
those of gemm_f16_splitk with the separate reduction kernel, so its output
must equal that entry point's bit for bit; it is also held to the oracle's
tolerance.  The checked calls start on an array left dirty (NaN partials of
a larger shape with another tile and split count), because nothing in the
array is cleared between calls.  The file is collected last so a
first-failure stop has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import shape_driven_tile_gb300 as sdt
from shape_driven_tile_gb300 import inputs
from _parity import assert_close, boundary_rows, u16

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 16 << 20


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _noalloc(A, B, C, tile, splits):
    L = sdt.lib()
    M, K = A.shape
    N = B.shape[1]
    rc = L.gemm_f16_splitk_noalloc(M, N, K, A.data_ptr(), B.data_ptr(), C.data_ptr(), tile, splits, _stream())
    assert rc == 0, L.sdt_last_error()
    sdt.check_device_status()
    return C


def _splitk(A, B, tile, splits, device):
    M, K = A.shape
    N = B.shape[1]
    ws = sdt.splitk_workspace(M, N, K, tile, splits, device=device)
    return sdt.gemm_f16_splitk(A, B, workspace=ws, tile=tile, splits=splits, algo=sdt.SPLITK_REDUCE_KERNEL)


def _dirty_scratch(device):
    """A call that fills 13 MiB of the array (counters + 12 MiB of partials) with NaN:
    1024x1024x2048, 128x128, 3 splits, A all NaN."""
    M = N = 1024
    K = 2048
    tid = sdt.tile_id("128x128")
    assert sdt.splitk_workspace_bytes(M, N, K, tid, 3) == (1 << 20) + 3 * M * N * 4
    A = torch.full((M, K), float("nan"), dtype=torch.float16, device=device)
    B = torch.ones((K, N), dtype=torch.float16, device=device)
    C = torch.empty((M, N), dtype=torch.float16, device=device)
    _noalloc(A, B, C, tid, 3)
    assert torch.isnan(C).all()


def _oracle_rows(A, B, rows=None):
    return oracle.gemm(u16(A), u16(B), rows=rows)


def test_noalloc_bit_identical_to_workspace_entry_point_two_calls(cuda_device):
    M, N, K = 512, 768, 4096
    tid, splits = sdt.tile_id("64x64"), 8
    assert sdt.splitk_workspace_bytes(M, N, K, tid, splits) <= SCRATCH_BYTES
    _dirty_scratch(cuda_device)
    for call in range(2):
        A_h = inputs.uniform((M, K), seed=301 + 2 * call)
        B_h = inputs.uniform((K, N), seed=302 + 2 * call)
        A, B = A_h.to(cuda_device), B_h.to(cuda_device)
        C = torch.full((M, N), float("nan"), dtype=torch.float16, device=cuda_device)
        _noalloc(A, B, C, tid, splits)
        ref = _splitk(A, B, tid, splits, cuda_device)
        assert torch.equal(C, ref), f"call {call}: differs from gemm_f16_splitk"
        assert_close(C.cpu().double().numpy(), _oracle_rows(A_h, B_h), K, f"call {call} vs oracle")


def test_noalloc_picks_tile_and_splits(cuda_device):
    L = sdt.lib()
    M, N, K = 256, 256, 8192
    A_h, B_h = inputs.uniform((M, K), seed=311), inputs.uniform((K, N), seed=312)
    A, B = A_h.to(cuda_device), B_h.to(cuda_device)
    tid, splits = sdt.pick_splitk(M, N, K, sm_count=sdt.device_sm_count(), smem_limit=L.sdt_device_smem_optin())
    assert sdt.splitk_workspace_bytes(M, N, K, tid, splits) <= SCRATCH_BYTES
    _dirty_scratch(cuda_device)
    C = torch.full((M, N), float("nan"), dtype=torch.float16, device=cuda_device)
    _noalloc(A, B, C, -1, 0)
    assert torch.equal(C, _splitk(A, B, tid, splits, cuda_device))
    assert_close(C.cpu().double().numpy(), _oracle_rows(A_h, B_h), K, "picked")


def test_noalloc_lowers_a_picked_split_count_to_fit(cuda_device):
    # a shape whose picked split count needs more than the array; the call runs the
    # same tile with the largest split count that fits
    L = sdt.lib()
    sm, smem = sdt.device_sm_count(), L.sdt_device_smem_optin()
    found = None
    for M, N, K in [(1024, 1536, 16384), (1536, 1024, 16384), (1024, 1024, 32768), (768, 1536, 16384)]:
        tid, splits = sdt.pick_splitk(M, N, K, sm_count=sm, smem_limit=smem)
        if sdt.splitk_workspace_bytes(M, N, K, tid, splits) > SCRATCH_BYTES and \
                sdt.splitk_workspace_bytes(M, N, K, tid, 1) <= SCRATCH_BYTES:
            found = (M, N, K, tid, splits)
            break
    assert found, "no candidate shape makes the pick exceed the scratch (the test lost its case)"
    M, N, K, tid, picked = found
    fit = max(s for s in range(1, picked) if sdt.splitk_workspace_bytes(M, N, K, tid, s) <= SCRATCH_BYTES)
    A_h, B_h = inputs.uniform((M, K), seed=321), inputs.uniform((K, N), seed=322)
    A, B = A_h.to(cuda_device), B_h.to(cuda_device)
    C = torch.full((M, N), float("nan"), dtype=torch.float16, device=cuda_device)
    _noalloc(A, B, C, -1, 0)
    assert torch.equal(C, _splitk(A, B, tid, fit, cuda_device)), f"{M}x{N}x{K}: not tile {tid} with {fit} splits"
    rows = boundary_rows(M, step=128, extra=4, seed=5)
    assert_close(C.cpu().double().numpy()[rows], _oracle_rows(A_h, B_h, rows), K, f"{M}x{N}x{K} lowered")


def test_noalloc_scratch_boundary(cuda_device):
    # 512x512 with 15 splits needs exactly 16 MiB (1 MiB counters + 15 MiB partials): runs;
    # 512x512 with 16 splits needs 17 MiB: refused before any launch
    L = sdt.lib()
    tid = sdt.tile_id("64x64")
    M = N = 512
    K = 15 * 64
    assert sdt.splitk_workspace_bytes(M, N, K, tid, 15) == SCRATCH_BYTES
    A_h, B_h = inputs.uniform((M, K), seed=331), inputs.uniform((K, N), seed=332)
    A, B = A_h.to(cuda_device), B_h.to(cuda_device)
    C = torch.full((M, N), float("nan"), dtype=torch.float16, device=cuda_device)
    _noalloc(A, B, C, tid, 15)
    assert torch.equal(C, _splitk(A, B, tid, 15, cuda_device))
    assert_close(C.cpu().double().numpy(), _oracle_rows(A_h, B_h), K, "exactly 16 MiB")
    K = 16 * 64
    assert sdt.splitk_workspace_bytes(M, N, K, tid, 16) == SCRATCH_BYTES + (1 << 20)
    A = torch.zeros((M, K), dtype=torch.float16, device=cuda_device)
    B = torch.zeros((K, N), dtype=torch.float16, device=cuda_device)
    C = torch.full((M, N), float("nan"), dtype=torch.float16, device=cuda_device)
    rc = L.gemm_f16_splitk_noalloc(M, N, K, A.data_ptr(), B.data_ptr(), C.data_ptr(), tid, 16, _stream())
    assert rc == -10
    assert b"scratch" in L.sdt_last_error()
    torch.cuda.synchronize()
    assert torch.isnan(C).all()  # nothing launched


def test_noalloc_rejects_shapes_beyond_the_scratch(cuda_device):
    L = sdt.lib()
    M, N, K = 2048, 2048, 4096          # 2 splits of 2048x2048 fp32 = 32 MiB of partials
    tid = sdt.tile_id("128x128")
    assert sdt.splitk_workspace_bytes(M, N, K, tid, 2) > SCRATCH_BYTES
    A = torch.zeros((M, K), dtype=torch.float16, device=cuda_device)
    B = torch.zeros((K, N), dtype=torch.float16, device=cuda_device)
    C = torch.zeros((M, N), dtype=torch.float16, device=cuda_device)
    rc = L.gemm_f16_splitk_noalloc(M, N, K, A.data_ptr(), B.data_ptr(), C.data_ptr(), tid, 2, _stream())
    assert rc == -10
    assert b"scratch" in L.sdt_last_error()
    # picked: even one split of 2048x2048 (16 MiB of partials) does not fit
    rc = L.gemm_f16_splitk_noalloc(M, N, K, A.data_ptr(), B.data_ptr(), C.data_ptr(), -1, 0, _stream())
    assert rc == -10
    assert b"scratch" in L.sdt_last_error()


def test_noalloc_empty_sum_with_a_picked_tile(cuda_device):
    # K == 0 is the empty sum: C = 0, also when the call is asked to pick tile and splits
    M, N = 256, 384
    for tile, splits in ((-1, 0), (sdt.tile_id("64x64"), 4)):
        C = torch.full((M, N), float("nan"), dtype=torch.float16, device=cuda_device)
        L = sdt.lib()
        rc = L.gemm_f16_splitk_noalloc(M, N, 0, None, None, C.data_ptr(), tile, splits,
                                       _stream())
        assert rc == 0, L.sdt_last_error()
        sdt.check_device_status()
        assert (C == 0).all().item()
        assert np.all(C.cpu().numpy() == 0)
