"""Shape-driven fp16 GEMM and M=1 decode GEMV for GB300 (sm_103a).

Thin binding over libsdt.so (C ABI in include/sdt.h): the functions below only
check and marshal arguments (tensor pointers, shapes, the current CUDA stream)
and call the C entry points of the same names.  Every step of the computation
runs in the library's CUDA kernels; there is no fallback path.
"""
from __future__ import annotations

import ctypes

import torch

from ._lib import SdtError, check, lib, sdt_tile_desc

__all__ = [
    "SdtError", "gemm_f16", "gemm_f16_with_tile", "gemv_m1", "gemv_m1_bf16", "gemv_m1_q8",
    "feasible_tiles", "pick_tile", "tile_estimate_us", "seed_tile", "tile_info", "tiles", "tile_id",
    "load_tune_table", "clear_tune_table", "tune_table_lookup", "check_device_status",
    "debug_timeout_probe", "device_sm_count", "lib", "gemm_f16_splitk", "splitk_workspace",
    "splitk_workspace_bytes", "pick_splitk", "pick_tile_any", "gemm_ex_splitk",
    "splitk_ex_workspace_bytes", "pick_splitk_any", "SPLITK_REDUCE_KERNEL", "SPLITK_IN_KERNEL", "gemm_ex",
    "SPLITK_STREAM", "SPLITK_STREAM_REDUCE", "streamk_ctas", "streamk_workspace_bytes",
    "gemm_f16_ws", "gemm_ex_ws", "gemm_workspace_bytes", "gemm_workspace", "pair_tail_plan",
]


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _one_device(**tensors):
    """Every operand must be a CUDA tensor on the current device: the library launches on
    the current device, so a host pointer or another GPU's memory would reach its kernels."""
    current = None
    for name, t in tensors.items():
        if not isinstance(t, torch.Tensor):
            raise TypeError(f"{name} must be a torch.Tensor")
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if current is None:
            current = torch.cuda.current_device()
        if t.device.index != current:
            raise ValueError(f"{name} is on {t.device}, but the current device is cuda:{current}")


def _workspace(workspace):
    if not isinstance(workspace, torch.Tensor) or not workspace.is_cuda:
        raise TypeError("workspace must be a CUDA tensor")
    if not workspace.is_contiguous():
        raise ValueError("workspace must be contiguous")
    return workspace.numel() * workspace.element_size()


def _need(t, name, dtype, ndim):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must be {ndim}-D")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous (tight row-major)")


def _gemm_args(A, B, C):
    _need(A, "A", torch.float16, 2)
    _need(B, "B", torch.float16, 2)
    M, K = A.shape
    K2, N = B.shape
    if K != K2:
        raise ValueError(f"inner dimensions differ: A is {tuple(A.shape)}, B is {tuple(B.shape)}")
    if C is None:
        C = torch.empty((M, N), dtype=torch.float16, device=A.device)
    else:
        _need(C, "C", torch.float16, 2)
        if tuple(C.shape) != (M, N):
            raise ValueError(f"C must be {(M, N)}, got {tuple(C.shape)}")
    _one_device(A=A, B=B, C=C)
    return M, N, K, C


def gemm_f16(A: torch.Tensor, B: torch.Tensor, C: torch.Tensor | None = None, *, stream=None):
    """C = A @ B (fp16 in, fp32 accumulate, fp16 out) with the tile chosen from the shape."""
    M, N, K, C = _gemm_args(A, B, C)
    check(lib().gemm_f16(M, N, K, A.data_ptr(), B.data_ptr(), C.data_ptr(), _stream(stream)))
    return C


def gemm_f16_with_tile(A, B, C=None, *, tile, stagger: int = -1, stream=None):
    """gemm_f16 with a forced ladder tile (id or name); stagger -1 auto, 0 off, 1 on."""
    M, N, K, C = _gemm_args(A, B, C)
    tid = tile_id(tile) if isinstance(tile, str) else int(tile)
    check(lib().gemm_f16_with_tile(M, N, K, A.data_ptr(), B.data_ptr(), C.data_ptr(),
                                   _stream(stream), tid, int(stagger)))
    return C


def _gemv_args(x, W, y, wdtype):
    _need(x, "x", torch.bfloat16, 1)
    _need(W, "W", wdtype, 2)
    N, K = W.shape
    if x.shape[0] != K:
        raise ValueError(f"x has length {x.shape[0]}, W is {tuple(W.shape)} (K-major [N, K])")
    if y is None:
        y = torch.empty(N, dtype=torch.float32, device=x.device)
    else:
        _need(y, "y", torch.float32, 1)
        if y.shape[0] != N:
            raise ValueError("y must have length N")
    _one_device(x=x, W=W, y=y)
    return K, N, y


def gemv_m1_bf16(x, W, y=None, *, stream=None):
    """y[n] = sum_k x[k] W[n, k]; x bf16 [K], W bf16 [N, K] (K-major), y fp32 [N]."""
    K, N, y = _gemv_args(x, W, y, torch.bfloat16)
    check(lib().gemv_m1_bf16(K, N, x.data_ptr(), W.data_ptr(), y.data_ptr(), _stream(stream)))
    return y


def gemv_m1_q8(x, q, scales, y=None, *, stream=None):
    """q8 decode: W[n, k] = q[n, k] * scales[n, k // 32]; q int8 [N, K], scales fp16 [N, K/32]."""
    K, N, y = _gemv_args(x, q, y, torch.int8)
    _need(scales, "scales", torch.float16, 2)
    if K % 32 or tuple(scales.shape) != (N, K // 32):
        raise ValueError(f"scales must be {(N, K // 32)} with K % 32 == 0")
    _one_device(x=x, scales=scales)
    check(lib().gemv_m1_q8(K, N, x.data_ptr(), q.data_ptr(), scales.data_ptr(), y.data_ptr(),
                           _stream(stream)))
    return y


def gemv_m1(x, W, scales=None, y=None, *, stream=None):
    """M=1 decode GEMV: bf16 weights when scales is None, else q8 (int8 + fp16 scale per 32)."""
    if scales is None:
        return gemv_m1_bf16(x, W, y, stream=stream)
    return gemv_m1_q8(x, W, scales, y, stream=stream)


DTYPE_CODES = {torch.float16: 0, torch.bfloat16: 1}
LAYOUT_A_T, LAYOUT_B_T = 1, 2


def _layout_of(T, name):
    """(stored transposed?, leading dimension) of a 2-D view: row-major or a transposed row-major view."""
    if T.dim() != 2:
        raise ValueError(f"{name} must be 2-D")
    r, c = T.shape
    s0, s1 = T.stride()
    up8 = lambda v: (max(v, 1) + 7) // 8 * 8  # a single stored row never steps: any legal stride works
    if s1 == 1 or c == 1:
        return False, (s0 if r > 1 else up8(max(s0, c)))
    if s0 == 1 or r == 1:
        return True, (s1 if c > 1 else up8(max(s1, r)))
    raise ValueError(f"{name} needs unit stride in one dimension (row-major or transposed row-major)")


def _ex_args(A, B, C):
    """(M, N, K, lda, ldb, ldc, layout, C) of gemm_ex-style views."""
    if not isinstance(A, torch.Tensor) or not isinstance(B, torch.Tensor):
        raise TypeError("A and B must be torch.Tensors")
    if A.dtype not in DTYPE_CODES or B.dtype != A.dtype:
        raise TypeError("A and B must both be float16 or both bfloat16")
    _one_device(A=A, B=B)
    if A.dim() != 2 or B.dim() != 2:
        raise ValueError("A and B must be 2-D")
    M, K = A.shape
    K2, N = B.shape
    if K != K2:
        raise ValueError(f"inner dimensions differ: {tuple(A.shape)} @ {tuple(B.shape)}")
    a_t, lda = _layout_of(A, "A")
    b_t, ldb = _layout_of(B, "B")
    if C is None:
        C = torch.empty((M, N), dtype=A.dtype, device=A.device)
    else:
        if not isinstance(C, torch.Tensor):
            raise TypeError("C must be a torch.Tensor")
        if C.dtype != A.dtype or C.dim() != 2 or tuple(C.shape) != (M, N) or (C.stride(1) != 1 and N > 1):
            raise ValueError(f"C must be a row-major {A.dtype} [{M}, {N}] view")
        _one_device(A=A, C=C)
    ldc = C.stride(0) if M > 1 else max(C.stride(0), N)
    layout = (LAYOUT_A_T if a_t else 0) | (LAYOUT_B_T if b_t else 0)
    return M, N, K, lda, ldb, ldc, layout, C


def gemm_ex(A, B, C=None, *, tile=-1, stream=None):
    """C = A @ B for fp16 or bf16 views of any shape: A [M, K] and B [K, N] may be row-major
    (padded rows allowed) or transposed views (e.g. X.t()); C [M, N] row-major, padding allowed."""
    M, N, K, lda, ldb, ldc, layout, C = _ex_args(A, B, C)
    tid = tile_id(tile) if isinstance(tile, str) else int(tile)
    check(lib().gemm_ex(M, N, K, A.data_ptr(), lda, B.data_ptr(), ldb, C.data_ptr(), ldc, DTYPE_CODES[A.dtype],
                        layout, tid, _stream(stream)))
    return C


def gemm_workspace_bytes(sm_count: int | None = None) -> int:
    """Bytes of workspace gemm_f16_ws / gemm_ex_ws take (current device when sm_count is None)."""
    if sm_count is None:
        return int(lib().sdt_gemm_workspace_bytes())
    return int(lib().sdt_gemm_workspace_bytes_for(int(sm_count)))


def gemm_workspace(device=None) -> torch.Tensor:
    """A zeroed, 256-byte aligned workspace for gemm_f16_ws / gemm_ex_ws (owned by the caller)."""
    nbytes = gemm_workspace_bytes()
    if nbytes == 0:
        raise SdtError(-9, "no CUDA device")
    ws = torch.empty(nbytes + 256, dtype=torch.uint8, device=device or "cuda")
    off = (-ws.data_ptr()) % 256
    ws = ws[off:off + nbytes]
    check(lib().sdt_splitk_workspace_init(ws.data_ptr(), nbytes, _stream(None)))
    return ws


def gemm_f16_ws(A, B, C=None, *, workspace, stream=None):
    """gemm_f16 with a workspace (gemm_workspace()) in which a two-CTA tile's partly empty
    last round may split its tiles in K; workspace None runs gemm_f16."""
    M, N, K, C = _gemm_args(A, B, C)
    if workspace is None:
        check(lib().gemm_f16_ws(M, N, K, A.data_ptr(), B.data_ptr(), C.data_ptr(), None, 0, _stream(stream)))
        return C
    nbytes = _workspace(workspace)
    _one_device(A=A, workspace=workspace)
    check(lib().gemm_f16_ws(M, N, K, A.data_ptr(), B.data_ptr(), C.data_ptr(), workspace.data_ptr(), nbytes,
                            _stream(stream)))
    return C


def gemm_ex_ws(A, B, C=None, *, workspace, tile=-1, tail_splits: int = -1, stream=None):
    """gemm_ex with a gemm_f16_ws workspace; tail_splits -1 plans the last round, 0 never
    splits it, 2..8 forces that many k-ranges per leftover tile."""
    M, N, K, lda, ldb, ldc, layout, C = _ex_args(A, B, C)
    tid = tile_id(tile) if isinstance(tile, str) else int(tile)
    wptr, nbytes = None, 0
    if workspace is not None:
        nbytes = _workspace(workspace)
        _one_device(A=A, workspace=workspace)
        wptr = workspace.data_ptr()
    check(lib().gemm_ex_ws(M, N, K, A.data_ptr(), lda, B.data_ptr(), ldb, C.data_ptr(), ldc, DTYPE_CODES[A.dtype],
                           layout, tid, int(tail_splits), wptr, nbytes, _stream(stream)))
    return C


def pair_tail_plan(M: int, N: int, K: int, tile, sm_count: int = 152, smem_limit: int = 232448, *,
                   workspace: bool = True, tail_splits: int = -1) -> tuple[int, int, int, int]:
    """(tail_start, num_items, splits, split0_ktiles) of a two-CTA tile's last round (see
    sdt.h); no GPU needed."""
    tid = tile_id(tile) if isinstance(tile, str) else int(tile)
    a, b, c, d = ctypes.c_int(), ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    check(lib().sdt_pair_tail_plan(M, N, K, tid, int(sm_count), int(smem_limit), 1 if workspace else 0,
                                   int(tail_splits), ctypes.byref(a), ctypes.byref(b), ctypes.byref(c),
                                   ctypes.byref(d)))
    return a.value, b.value, c.value, d.value


SPLITK_REDUCE_KERNEL = 0
SPLITK_IN_KERNEL = 1
SPLITK_STREAM = 2  # stream-K: `splits` is the CTA count (<= 0: one per SM slot); fix-up in the kernel
SPLITK_STREAM_REDUCE = 3  # stream-K with the fix-up in a second kernel


def splitk_workspace_bytes(M: int, N: int, K: int, tile, splits: int) -> int:
    tid = tile_id(tile) if isinstance(tile, str) else int(tile)
    return int(lib().sdt_splitk_workspace_bytes(M, N, K, tid, int(splits)))


def splitk_workspace(M: int, N: int, K: int, tile, splits: int, device=None) -> torch.Tensor:
    """A zeroed workspace tensor for gemm_f16_splitk (allocated by torch, owned by the caller)."""
    nbytes = splitk_workspace_bytes(M, N, K, tile, splits)
    if nbytes == 0:
        raise ValueError("invalid split-K combination")
    ws = torch.empty(nbytes + 256, dtype=torch.uint8, device=device or "cuda")
    off = (-ws.data_ptr()) % 256
    ws = ws[off:off + nbytes]
    check(lib().sdt_splitk_workspace_init(ws.data_ptr(), nbytes, _stream(None)))
    return ws


def gemm_f16_splitk(A, B, C=None, *, workspace, tile=-1, splits: int = 0,
                    algo: int = SPLITK_REDUCE_KERNEL, stream=None):
    """Split-K GEMM with a caller-owned workspace (see sdt.h); tile -1 picks tile and splits."""
    M, N, K, C = _gemm_args(A, B, C)
    tid = tile_id(tile) if isinstance(tile, str) else int(tile)
    nbytes = _workspace(workspace)
    _one_device(A=A, workspace=workspace)
    check(lib().gemm_f16_splitk(M, N, K, A.data_ptr(), B.data_ptr(), C.data_ptr(), workspace.data_ptr(), nbytes,
                                tid, int(splits), int(algo), _stream(stream)))
    return C


def splitk_ex_workspace_bytes(M: int, N: int, K: int, tile, splits: int) -> int:
    tid = tile_id(tile) if isinstance(tile, str) else int(tile)
    return int(lib().sdt_splitk_ex_workspace_bytes(M, N, K, tid, int(splits)))


def gemm_ex_splitk(A, B, C=None, *, workspace, tile=-1, splits: int = 0, algo: int = SPLITK_REDUCE_KERNEL,
                   stream=None):
    """Split-K / Stream-K form of gemm_ex (same views); `workspace` as for gemm_f16_splitk,
    sized by splitk_ex_workspace_bytes (algo 0 and 1: `splits` k-slices per output tile) or
    streamk_workspace_bytes (algo SPLITK_STREAM or SPLITK_STREAM_REDUCE: `splits` is the CTA
    count, 0 = one per SM slot)."""
    M, N, K, lda, ldb, ldc, layout, C = _ex_args(A, B, C)
    tid = tile_id(tile) if isinstance(tile, str) else int(tile)
    nbytes = _workspace(workspace)
    _one_device(A=A, workspace=workspace)
    check(lib().gemm_ex_splitk(M, N, K, A.data_ptr(), lda, B.data_ptr(), ldb, C.data_ptr(), ldc,
                               DTYPE_CODES[A.dtype], layout, workspace.data_ptr(), nbytes, tid, int(splits),
                               int(algo), _stream(stream)))
    return C


def streamk_ctas(tile, sm_count: int | None = None, smem_limit: int = 232448) -> int:
    """Default stream-K CTA count of a tile (SMs x CTAs per SM); current device when sm_count is None."""
    tid = tile_id(tile) if isinstance(tile, str) else int(tile)
    if sm_count is None:
        return check(lib().sdt_streamk_ctas(tid))
    return check(lib().sdt_streamk_ctas_for(tid, int(sm_count), int(smem_limit)))


def streamk_workspace_bytes(M: int, N: int, K: int, tile, ctas: int | None = None) -> int:
    """Workspace bytes of gemm_ex_splitk / gemm_f16_splitk with algo=SPLITK_STREAM and `ctas`
    CTAs (None: the tile's default count on the current device)."""
    tid = tile_id(tile) if isinstance(tile, str) else int(tile)
    if ctas is None or ctas <= 0:
        ctas = streamk_ctas(tid)
    return int(lib().sdt_streamk_workspace_bytes(M, N, K, tid, int(ctas)))


def pick_splitk_any(M: int, N: int, K: int, sm_count: int = 152, smem_limit: int = 232448):
    t, sp = ctypes.c_int(0), ctypes.c_int(0)
    check(lib().sdt_pick_splitk_any_for(M, N, K, int(sm_count), int(smem_limit), ctypes.byref(t),
                                        ctypes.byref(sp)))
    return t.value, sp.value


def pick_splitk(M: int, N: int, K: int, sm_count: int = 152, smem_limit: int = 232448):
    t, sp = ctypes.c_int(0), ctypes.c_int(0)
    check(lib().sdt_pick_splitk_for(M, N, K, int(sm_count), int(smem_limit), ctypes.byref(t), ctypes.byref(sp)))
    return t.value, sp.value


# ---- tiles ---------------------------------------------------------------------


def tile_info(tile_id: int) -> dict:
    """The ladder tile's description; "skinny" marks the tiles (named s<BM>x<BN>) that
    gemm_ex and gemm_ex_splitk run with swapped operands and gemm_f16 never uses."""
    d = sdt_tile_desc()
    check(lib().sdt_tile_info(int(tile_id), ctypes.byref(d)))
    info = {f: (getattr(d, f).decode() if f == "name" else getattr(d, f)) for f, _ in d._fields_}
    info["skinny"] = info["name"].startswith("s")
    return info


def tiles() -> list[dict]:
    return [tile_info(i) for i in range(lib().sdt_num_tiles())]


def tile_id(name: str) -> int:
    for t in tiles():
        if t["name"] == name:
            return t["id"]
    raise KeyError(name)


def feasible_tiles(M: int, N: int, K: int, smem_limit: int | None = None) -> list[int]:
    cap = 64
    ids = (ctypes.c_int * cap)()
    if smem_limit is None:
        n = check(lib().sdt_feasible_tiles(M, N, K, ids, cap))
    else:
        n = check(lib().sdt_feasible_tiles_for(M, N, K, int(smem_limit), ids, cap))
    return list(ids[: min(n, cap)])


def pick_tile(M: int, N: int, K: int, sm_count: int | None = None, smem_limit: int | None = None) -> int:
    if sm_count is None:
        return check(lib().sdt_pick_tile(M, N, K))
    return check(lib().sdt_pick_tile_for(M, N, K, int(sm_count),
                                         int(smem_limit) if smem_limit is not None else 232448))


def pick_tile_any(M: int, N: int, K: int, sm_count: int | None = None, smem_limit: int | None = None) -> int:
    """The tile gemm_ex picks for any shape (tiles may overhang ragged edges)."""
    if sm_count is None:
        sm_count, smem_limit = device_sm_count(), lib().sdt_device_smem_optin()
    return check(lib().sdt_pick_tile_any_for(M, N, K, int(sm_count),
                                             int(smem_limit) if smem_limit is not None else 232448))


def tile_estimate_us(tile, M: int, N: int, K: int, sm_count: int = 152) -> float:
    """pick_tile's run-time estimate (microseconds) of a ladder tile (id or name) on the shape."""
    tid = tile_id(tile) if isinstance(tile, str) else int(tile)
    v = lib().sdt_tile_estimate_us(tid, M, N, K, int(sm_count))
    if v < 0:
        check(int(v))
    return v


def seed_tile(M: int, N: int, units: int) -> int:
    return check(lib().sdt_seed_tile(M, N, units))


def load_tune_table(path: str) -> None:
    check(lib().sdt_load_tune_table(str(path).encode()))


def clear_tune_table() -> None:
    lib().sdt_clear_tune_table()


def tune_table_lookup(M: int, N: int, K: int) -> int:
    return lib().sdt_tune_table_lookup(M, N, K)


# ---- diagnostics ------------------------------------------------------------------


def check_device_status(stream=None) -> int:
    """Synchronise the stream; raise SdtError(SDT_ERR_TIMEOUT) if a kernel gave up a wait."""
    where = ctypes.c_int(0)
    rc = lib().sdt_check_device_status(_stream(stream), ctypes.byref(where))
    if rc < 0:
        err = SdtError(rc, (lib().sdt_last_error() or b"").decode())
        err.where = where.value
        raise err
    return 0


def debug_timeout_probe(limit_us: int, stream=None) -> None:
    check(lib().sdt_debug_timeout_probe(_stream(stream), int(limit_us)))


def device_sm_count() -> int:
    return check(lib().sdt_device_sm_count())
