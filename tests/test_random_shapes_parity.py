"""Seeded random problems through every GEMM entry point against the fp64 oracle: shapes
from 1 to ~700 in each dimension (N a multiple of 8), all four operand layouts, fp16 and
bf16, caller row strides with padding, every ladder tile (the skinny ones where their
layout rule allows), split-K with both reductions, Stream-K with both fix-ups, and the
two-CTA tiles' k-split last round.  Integer-valued operands, so each result must equal
the oracle's value rounded to the output type, bit for bit; C's padding must be left
untouched."""
import numpy as np
import pytest
import torch

import oracle
import shape_driven_tile_gb300 as sdt
from shape_driven_tile_gb300 import inputs
from _parity import assert_bit_exact_bf16, assert_bit_exact_f16, u16

pytestmark = pytest.mark.gpu

CASES = 160
SENTINEL = 3.0  # written into C's padding; a write outside C would change it


def operand(rows, cols, trans, dtype, seed, pad, dev):
    vals = inputs.integers((rows, cols), seed=seed, dtype=torch.float32).to(dtype)
    if not trans:
        store = torch.zeros((rows, cols + pad), dtype=dtype)
        store[:, :cols] = vals
        return store.to(dev)[:, :cols], vals
    store = torch.zeros((cols, rows + pad), dtype=dtype)
    store[:, :rows] = vals.t()
    return store.to(dev)[:, :rows].t(), vals


def draw(rng):
    M = int(rng.integers(1, 700))
    N = 8 * int(rng.integers(1, 88))
    K = int(rng.integers(1, 700))
    ta, tb = bool(rng.integers(0, 2)), bool(rng.integers(0, 2))
    dtype = torch.bfloat16 if rng.integers(0, 2) else torch.float16
    # row padding keeps every stored row a multiple of 8 elements (16 bytes)
    pads = [8 * int(rng.integers(0, 3)) for _ in range(3)]
    return M, N, K, ta, tb, dtype, pads


def run_case(i, rng, dev, ws, sk_ws):
    M, N, K, ta, tb, dtype, (pa, pb, pc) = draw(rng)
    pa += (-(M if ta else K)) % 8  # A stored [M][K] or, transposed, [K][M]
    pb += (-(K if tb else N)) % 8  # B stored [K][N] or, transposed, [N][K]
    A, Av = operand(M, K, ta, dtype, 9000 + 2 * i, pa, dev)
    B, Bv = operand(K, N, tb, dtype, 9001 + 2 * i, pb, dev)
    store = torch.full((M, N + pc), SENTINEL, dtype=dtype, device=dev)
    C = store[:, :N]
    names = [t["name"] for t in sdt.tiles() if not (t["skinny"] and ta)]
    entry = ["ex", "ex", "ws", "splitk", "streamk"][int(rng.integers(0, 5))]
    what = f"case {i}: {M}x{N}x{K} {'T' if ta else 'N'}{'T' if tb else 'N'} {dtype} {entry}"
    if entry == "ex":
        tile = names[int(rng.integers(0, len(names)))] if rng.integers(0, 4) else -1
        sdt.gemm_ex(A, B, C, tile=tile)
        what += f" tile {tile}"
    elif entry == "ws":
        tile = ["2cta_256x256", "2cta_256x224", "2cta_256x128"][int(rng.integers(0, 3))]
        splits = int(rng.choice([-1, 0, 2, 3, 5]))
        sdt.gemm_ex_ws(A, B, C, workspace=ws, tile=tile, tail_splits=splits)
        what += f" tile {tile} tail_splits {splits}"
    else:
        sk_tiles = [n for n in names if not n.startswith(("p", "2cta"))]
        tile = sk_tiles[int(rng.integers(0, len(sk_tiles)))]
        if entry == "splitk":
            algo = int(rng.choice([sdt.SPLITK_REDUCE_KERNEL, sdt.SPLITK_IN_KERNEL]))
            splits = int(rng.integers(1, max(2, min(8, -(-K // 64)) + 1)))
            need = sdt.splitk_ex_workspace_bytes(M, N, K, tile, splits)
        else:
            algo = int(rng.choice([sdt.SPLITK_STREAM, sdt.SPLITK_STREAM_REDUCE]))
            splits = int(rng.integers(1, 300))
            need = sdt.streamk_workspace_bytes(M, N, K, tile, splits)
        assert 0 < need <= sk_ws.numel(), (what, need)
        sdt.gemm_ex_splitk(A, B, C, workspace=sk_ws[:need], tile=tile, splits=splits, algo=algo)
        what += f" tile {tile} splits {splits} algo {algo}"
    sdt.check_device_status()
    ref = oracle.gemm(u16(Av), u16(Bv), dtype="bf16" if dtype == torch.bfloat16 else "f16")
    (assert_bit_exact_bf16 if dtype == torch.bfloat16 else assert_bit_exact_f16)(C.contiguous(), ref, what)
    assert bool((store[:, N:] == SENTINEL).all()), f"{what}: wrote outside C"


def test_random_problems_every_entry_point(cuda_device):
    ws = sdt.gemm_workspace(cuda_device)
    sk_ws = torch.zeros(128 << 20, dtype=torch.uint8, device=cuda_device)
    rng = np.random.default_rng(20261202)
    for i in range(CASES):
        run_case(i, rng, cuda_device, ws, sk_ws)
    torch.cuda.synchronize()
    assert bool((ws[: 1 << 20] == 0).all()) and bool((sk_ws[: 1 << 20] == 0).all()), "counters left non-zero"
