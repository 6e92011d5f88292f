"""ctypes declarations of libsdt.so (the C ABI in include/sdt.h)."""
from __future__ import annotations

import ctypes
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libsdt.so")

_lock = threading.Lock()
_lib = None

i64 = ctypes.c_int64
vp = ctypes.c_void_p
cint = ctypes.c_int


class sdt_tile_desc(ctypes.Structure):
    _fields_ = [
        ("id", cint), ("BM", cint), ("BN", cint), ("BK", cint), ("cta_group", cint),
        ("stages", cint), ("threads", cint), ("smem_bytes", cint), ("tmem_cols", cint),
        ("name", ctypes.c_char * 24),
    ]


# name -> (restype, argtypes); every symbol include/sdt.h declares.
SIGNATURES = {
    "gemm_f16": (cint, [i64, i64, i64, vp, vp, vp, vp]),
    "gemv_m1": (cint, [i64, i64, vp, vp, vp, vp, vp]),
    "gemv_m1_bf16": (cint, [i64, i64, vp, vp, vp, vp]),
    "gemv_m1_q8": (cint, [i64, i64, vp, vp, vp, vp, vp]),
    "sdt_num_tiles": (cint, []),
    "sdt_tile_info": (cint, [cint, ctypes.POINTER(sdt_tile_desc)]),
    "sdt_tile_name": (ctypes.c_char_p, [cint]),
    "sdt_feasible_tiles_for": (cint, [i64, i64, i64, cint, ctypes.POINTER(cint), cint]),
    "sdt_feasible_tiles": (cint, [i64, i64, i64, ctypes.POINTER(cint), cint]),
    "sdt_pick_tile_for": (cint, [i64, i64, i64, cint, cint]),
    "sdt_pick_tile": (cint, [i64, i64, i64]),
    "sdt_seed_tile": (cint, [i64, i64, cint]),
    "gemm_f16_with_tile": (cint, [i64, i64, i64, vp, vp, vp, vp, cint, cint]),
    "sdt_load_tune_table": (cint, [ctypes.c_char_p]),
    "sdt_clear_tune_table": (None, []),
    "sdt_tune_table_size": (cint, []),
    "sdt_tune_table_lookup": (cint, [i64, i64, i64]),
    "sdt_last_error": (ctypes.c_char_p, []),
    "sdt_check_device_status": (cint, [vp, ctypes.POINTER(cint)]),
    "sdt_debug_timeout_probe": (cint, [vp, i64]),
    "sdt_debug_tensor_map_encodes": (i64, []),
    "sdt_device_sm_count": (cint, []),
    "sdt_device_smem_optin": (cint, []),
    "sdt_abi_version": (cint, []),
    "gemm_f16_splitk": (cint, [i64, i64, i64, vp, vp, vp, vp, ctypes.c_size_t, cint, cint, cint, vp]),
    "sdt_splitk_workspace_bytes": (ctypes.c_size_t, [i64, i64, i64, cint, cint]),
    "sdt_splitk_workspace_init": (cint, [vp, ctypes.c_size_t, vp]),
    "sdt_pick_splitk_for": (cint, [i64, i64, i64, cint, cint, ctypes.POINTER(cint), ctypes.POINTER(cint)]),
    "gemm_f16_splitk_noalloc": (cint, [i64, i64, i64, vp, vp, vp, cint, cint, vp]),
    "gemm_ex": (cint, [i64, i64, i64, vp, i64, vp, i64, vp, i64, cint, cint, cint, vp]),
    "sdt_pick_tile_any_for": (cint, [i64, i64, i64, cint, cint]),
    "sdt_tile_estimate_us": (ctypes.c_double, [cint, i64, i64, i64, cint]),
    "gemm_ex_splitk": (cint, [i64, i64, i64, vp, i64, vp, i64, vp, i64, cint, cint, vp, ctypes.c_size_t, cint, cint,
                              cint, vp]),
    "sdt_splitk_ex_workspace_bytes": (ctypes.c_size_t, [i64, i64, i64, cint, cint]),
    "sdt_pick_splitk_any_for": (cint, [i64, i64, i64, cint, cint, ctypes.POINTER(cint), ctypes.POINTER(cint)]),
    "sdt_streamk_workspace_bytes": (ctypes.c_size_t, [i64, i64, i64, cint, cint]),
    "sdt_streamk_ctas_for": (cint, [cint, cint, cint]),
    "sdt_streamk_ctas": (cint, [cint]),
    "gemm_f16_ws": (cint, [i64, i64, i64, vp, vp, vp, vp, ctypes.c_size_t, vp]),
    "gemm_ex_ws": (cint, [i64, i64, i64, vp, i64, vp, i64, vp, i64, cint, cint, cint, cint, vp, ctypes.c_size_t,
                          vp]),
    "sdt_gemm_workspace_bytes": (ctypes.c_size_t, []),
    "sdt_gemm_workspace_bytes_for": (ctypes.c_size_t, [cint]),
    "sdt_pair_tail_plan": (cint, [i64, i64, i64, cint, cint, cint, cint, cint, ctypes.POINTER(cint),
                                  ctypes.POINTER(cint), ctypes.POINTER(cint), ctypes.POINTER(cint)]),
}

STATUS = {
    0: "SDT_OK", -1: "SDT_ERR_NULL", -2: "SDT_ERR_ALIGN", -3: "SDT_ERR_SHAPE",
    -4: "SDT_ERR_UNSUPPORTED_DEVICE", -5: "SDT_ERR_LAUNCH", -6: "SDT_ERR_TIMEOUT",
    -7: "SDT_ERR_TILE", -8: "SDT_ERR_TABLE", -9: "SDT_ERR_CUDA", -10: "SDT_ERR_ARG",
}


class SdtError(RuntimeError):
    def __init__(self, code: int, message: str):
        self.code = code
        self.status = STATUS.get(code, str(code))
        super().__init__(f"{self.status}: {message}")


def lib():
    """The loaded library; raises (never falls back) when it is missing."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise ImportError(
                    f"{LIB_PATH} is missing: build it with "
                    "`python -c 'import __graft_entry__ as g; g.build()'`")
            h = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(h, name)
                fn.restype = res
                fn.argtypes = args
            _lib = h
    return _lib


def check(rc: int) -> int:
    if rc < 0:
        msg = lib().sdt_last_error()
        raise SdtError(rc, msg.decode() if msg else "")
    return rc
