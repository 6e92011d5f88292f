"""Argument checks of the Python binding: operands that are not CUDA tensors on the current
device are refused before anything reaches the library (a host pointer handed to a kernel
would fault the GPU)."""
import pytest
import torch

import shape_driven_tile_gb300 as sdt


def host(*shape, dtype=torch.float16):
    return torch.zeros(*shape, dtype=dtype)


@pytest.mark.parametrize("call", [
    lambda: sdt.gemm_f16(host(64, 64), host(64, 64)),
    lambda: sdt.gemm_f16_with_tile(host(64, 64), host(64, 64), tile="64x64"),
    lambda: sdt.gemm_ex(host(64, 64), host(64, 64)),
    lambda: sdt.gemm_ex(host(64, 64, dtype=torch.bfloat16), host(64, 64, dtype=torch.bfloat16)),
    lambda: sdt.gemv_m1(host(64, dtype=torch.bfloat16), host(8, 64, dtype=torch.bfloat16)),
    lambda: sdt.gemv_m1(host(64, dtype=torch.bfloat16), host(8, 64, dtype=torch.int8), host(8, 2)),
    lambda: sdt.gemm_f16_splitk(host(64, 64), host(64, 64), workspace=host(16, dtype=torch.uint8)),
    lambda: sdt.gemm_ex_splitk(host(64, 64), host(64, 64), workspace=host(16, dtype=torch.uint8)),
], ids=["gemm_f16", "with_tile", "gemm_ex", "gemm_ex_bf16", "gemv_bf16", "gemv_q8", "splitk", "ex_splitk"])
def test_host_operands_are_refused(call):
    with pytest.raises((TypeError, ValueError)):
        call()


def test_gemm_ex_refuses_non_tensors_and_bad_ranks():
    with pytest.raises(TypeError):
        sdt.gemm_ex([[1.0]], host(64, 64))
    with pytest.raises(TypeError):
        sdt.gemm_ex(host(64, 64), host(64, 64, dtype=torch.bfloat16))


@pytest.mark.gpu
def test_host_output_or_workspace_with_device_operands(cuda_device):
    A = torch.zeros(128, 128, dtype=torch.float16, device=cuda_device)
    B = torch.zeros(128, 128, dtype=torch.float16, device=cuda_device)
    with pytest.raises(ValueError, match="C must be a CUDA tensor"):
        sdt.gemm_ex(A, B, host(128, 128))
    with pytest.raises(ValueError, match="C must be a CUDA tensor"):
        sdt.gemm_f16(A, B, host(128, 128))
    ws = sdt.splitk_workspace(128, 128, 128, "64x64", 2, device=cuda_device)
    with pytest.raises(ValueError, match="C must be a CUDA tensor"):
        sdt.gemm_ex_splitk(A, B, host(128, 128), workspace=ws, tile="64x64", splits=2)
    with pytest.raises(TypeError, match="workspace"):
        sdt.gemm_ex_splitk(A, B, workspace=host(1 << 21, dtype=torch.uint8), tile="64x64", splits=2)
    wide = torch.zeros(2, ws.numel(), dtype=torch.uint8, device=cuda_device)
    with pytest.raises(ValueError, match="contiguous"):
        sdt.gemm_f16_splitk(A, B, workspace=wide.t(), tile="64x64", splits=2)
    x = torch.zeros(128, dtype=torch.bfloat16, device=cuda_device)
    W = torch.zeros(64, 128, dtype=torch.bfloat16, device=cuda_device)
    with pytest.raises(ValueError, match="y must be a CUDA tensor"):
        sdt.gemv_m1(x, W, y=torch.zeros(64))
