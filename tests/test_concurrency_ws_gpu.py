"""Workspace-taking entry points from several streams and host threads at once: each
stream with its own workspace (the k-split last round's counters and partials, split-K's)
gives the same bits as the same calls one after another, and every workspace's counters
are back at zero afterwards."""
import threading

import numpy as np
import pytest
import torch

import shape_driven_tile_gb300 as sdt
from shape_driven_tile_gb300 import inputs

pytestmark = pytest.mark.gpu


def problem(i, dev):
    rng = np.random.default_rng(500 + i)
    M = int(rng.integers(1, 1200))
    N = 8 * int(rng.integers(1, 150))
    K = 8 * int(rng.integers(1, 190))  # tight row-major operands: rows of a multiple of 16 bytes
    A = inputs.integers((M, K), seed=600 + 2 * i).to(dev)
    B = inputs.integers((K, N), seed=601 + 2 * i).to(dev)
    kind = ["ex", "ws", "splitk", "f16"][i % 4]
    return kind, A, B


def run(kind, A, B, ws, sk_ws, stream):
    M, K = A.shape
    N = B.shape[1]
    if kind == "ex":
        return sdt.gemm_ex(A, B, stream=stream)
    if kind == "ws":
        return sdt.gemm_ex_ws(A, B, workspace=ws, tile="2cta_256x256", tail_splits=2, stream=stream)
    if kind == "splitk":
        splits = min(2, -(-K // 64))
        need = sdt.splitk_ex_workspace_bytes(M, N, K, "64x64", splits)
        return sdt.gemm_ex_splitk(A, B, workspace=sk_ws[:need], tile="64x64", splits=splits,
                                  algo=sdt.SPLITK_IN_KERNEL, stream=stream)
    return sdt.gemm_ex(A, B, tile="p128x128", stream=stream)


def workspaces(dev):
    return sdt.gemm_workspace(dev), torch.zeros(64 << 20, dtype=torch.uint8, device=dev)


def test_two_streams_own_workspaces_match_sequential(cuda_device):
    probs = [problem(i, cuda_device) for i in range(24)]
    ws0, sk0 = workspaces(cuda_device)
    want = [run(k, A, B, ws0, sk0, None).clone() for k, A, B in probs]
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    wss = [workspaces(cuda_device) for _ in streams]
    for s in streams:
        s.wait_stream(torch.cuda.current_stream())
    got = []
    for i, (k, A, B) in enumerate(probs):
        s = streams[i % 2]
        ws, sk = wss[i % 2]
        with torch.cuda.stream(s):
            got.append(run(k, A, B, ws, sk, s))
    torch.cuda.synchronize()
    sdt.check_device_status()
    for i, (g, w) in enumerate(zip(got, want)):
        assert torch.equal(g.view(torch.int16), w.view(torch.int16)), f"problem {i} ({probs[i][0]})"
    for ws, sk in wss:
        assert bool((ws[: 1 << 20] == 0).all()) and bool((sk[: 1 << 20] == 0).all())


def test_host_threads_each_on_its_own_stream(cuda_device):
    probs = [problem(100 + i, cuda_device) for i in range(32)]
    ws0, sk0 = workspaces(cuda_device)
    want = [run(k, A, B, ws0, sk0, None).clone() for k, A, B in probs]
    torch.cuda.synchronize()
    got = [None] * len(probs)
    errors = []

    def worker(t):
        try:
            torch.cuda.set_device(cuda_device)
            s = torch.cuda.Stream()
            ws, sk = workspaces(cuda_device)
            torch.cuda.synchronize()
            with torch.cuda.stream(s):
                for i in range(t, len(probs), 4):
                    k, A, B = probs[i]
                    got[i] = run(k, A, B, ws, sk, s)
            s.synchronize()
        except Exception as e:  # reported on the main thread
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(t,)) for t in range(4)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    torch.cuda.synchronize()
    sdt.check_device_status()
    for i, (g, w) in enumerate(zip(got, want)):
        assert torch.equal(g.view(torch.int16), w.view(torch.int16)), f"problem {i} ({probs[i][0]})"
