"""The library called from several host threads at once, each on its own CUDA stream:
different shapes, tiles, layouts and entry points interleave through the shared
tensor-map cache, status word and lazily configured kernels.  Every result must equal
the fp64 oracle bit for bit (integer inputs)."""
import threading

import pytest
import torch

import shape_driven_tile_gb300 as sdt
from _parity import assert_bit_exact_f16
from test_gemm_ex_parity import operand, ref_of

pytestmark = pytest.mark.gpu

JOBS = [  # (M, N, K, tile, b_t, entry)
    (256, 256, 512, "64x64", False, "gemm_ex"),
    (384, 320, 448, "2cta_256x256", True, "gemm_ex"),
    (512, 448, 1024, "2cta_256x224", False, "gemm_ex"),
    (16, 4096, 2048, "s128x16", True, "gemm_ex"),
    (1024, 1024, 1024, -1, False, "gemm_f16"),
    (200, 264, 1000, "128x128", True, "stream"),
    (256, 384, 2048, "64x128", False, "splitk"),
    (300, 136, 777, "p128x256", True, "gemm_ex"),
]


def test_threads_on_separate_streams(cuda_device):
    data = []
    for i, (M, N, K, tile, b_t, entry) in enumerate(JOBS):
        A, Av = operand(M, K, False, torch.float16, 800 + 2 * i, True, cuda_device)
        B, Bv = operand(K, N, b_t, torch.float16, 801 + 2 * i, True, cuda_device)
        ws = None
        if entry == "stream":
            n = sdt.streamk_workspace_bytes(M, N, K, tile, None)
        elif entry == "splitk":
            n = sdt.splitk_ex_workspace_bytes(M, N, K, tile, 4)
        else:
            n = 0
        if n:
            w = torch.zeros(n + 256, dtype=torch.uint8, device=cuda_device)
            ws = w[(-w.data_ptr()) % 256:][:n]
        data.append((A, B, ws, ref_of(Av, Bv, torch.float16)))
    torch.cuda.synchronize()
    errors = []

    def worker(t):
        try:
            stream = torch.cuda.Stream(device=cuda_device)
            outs = []
            with torch.cuda.stream(stream):
                for r in range(6):
                    j = (t + r) % len(JOBS)
                    M, N, K, tile, b_t, entry = JOBS[j]
                    A, B, ws, _ = data[j] if entry not in ("stream", "splitk") else (data[j][0], data[j][1], None, None)
                    if entry in ("stream", "splitk"):
                        # workspaces are per call site: this thread's own copy
                        n = data[j][2].numel()
                        w = torch.zeros(n + 256, dtype=torch.uint8, device=cuda_device)
                        ws = w[(-w.data_ptr()) % 256:][:n]
                    C = torch.full((M, N), float("nan"), dtype=torch.float16, device=cuda_device)
                    if entry == "gemm_ex":
                        sdt.gemm_ex(A, B, C, tile=tile, stream=stream)
                    elif entry == "gemm_f16":
                        sdt.gemm_f16(A, B, C, stream=stream)
                    elif entry == "stream":
                        sdt.gemm_ex_splitk(A, B, C, workspace=ws, tile=tile, splits=0, algo=sdt.SPLITK_STREAM,
                                           stream=stream)
                    else:
                        sdt.gemm_ex_splitk(A, B, C, workspace=ws, tile=tile, splits=4, algo=sdt.SPLITK_IN_KERNEL,
                                           stream=stream)
                    outs.append((j, C, ws))
            stream.synchronize()
            for j, C, _ in outs:
                assert_bit_exact_f16(C, data[j][3], f"thread {t} job {j}")
        except Exception as e:  # reported on the main thread
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(t,)) for t in range(4)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    sdt.check_device_status()
    if errors:
        raise errors[0]
