"""The split-K entry point that allocates nothing (gemm_f16_splitk_noalloc).

It exists for callers that cannot allocate device memory where they multiply
(code that must not synchronise the device, plugin hosts with a fixed memory
budget and no allocator, allocator-free latency-critical loops): its workspace
is a fixed array the library keeps in device memory.  These tests call it
through the C ABI and check its output against the workspace entry point
(gemm_f16_splitk) within the parity tolerance, on two calls in a row, and
that a shape needing more than the fixed scratch is refused.  The file is
collected last so a first-failure stop has already run every other test.
"""
import ctypes

import pytest
import torch

import shape_driven_tile_gb300 as sdt
from shape_driven_tile_gb300 import inputs
from _parity import assert_close

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 16 << 20


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def test_noalloc_matches_workspace_entry_point_two_calls(cuda_device):
    L = sdt.lib()
    M, N, K = 512, 768, 4096
    tid, splits = sdt.tile_id("64x64"), 8
    assert sdt.splitk_workspace_bytes(M, N, K, tid, splits) <= SCRATCH_BYTES
    ws = sdt.splitk_workspace(M, N, K, tid, splits, device=cuda_device)
    for call in range(2):
        A = inputs.uniform((M, K), seed=301 + 2 * call).to(cuda_device)
        B = inputs.uniform((K, N), seed=302 + 2 * call).to(cuda_device)
        ref = sdt.gemm_f16_splitk(A, B, workspace=ws, tile=tid, splits=splits, algo=sdt.SPLITK_REDUCE_KERNEL)
        C = torch.full((M, N), float("nan"), dtype=torch.float16, device=cuda_device)
        rc = L.gemm_f16_splitk_noalloc(M, N, K, A.data_ptr(), B.data_ptr(), C.data_ptr(), tid, splits, _stream())
        assert rc == 0, L.sdt_last_error()
        sdt.check_device_status()
        assert_close(C.cpu().double().numpy(), ref.cpu().double().numpy(), K, f"call {call}")


def test_noalloc_picks_tile_and_splits(cuda_device):
    L = sdt.lib()
    M, N, K = 256, 256, 8192
    A = inputs.uniform((M, K), seed=311).to(cuda_device)
    B = inputs.uniform((K, N), seed=312).to(cuda_device)
    tid, splits = sdt.pick_splitk(M, N, K, sm_count=sdt.device_sm_count(), smem_limit=L.sdt_device_smem_optin())
    ws = sdt.splitk_workspace(M, N, K, tid, splits, device=cuda_device)
    ref = sdt.gemm_f16_splitk(A, B, workspace=ws, tile=tid, splits=splits, algo=sdt.SPLITK_REDUCE_KERNEL)
    C = torch.full((M, N), float("nan"), dtype=torch.float16, device=cuda_device)
    rc = L.gemm_f16_splitk_noalloc(M, N, K, A.data_ptr(), B.data_ptr(), C.data_ptr(), -1, 0, _stream())
    assert rc == 0, L.sdt_last_error()
    sdt.check_device_status()
    assert_close(C.cpu().double().numpy(), ref.cpu().double().numpy(), K, "picked")


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
