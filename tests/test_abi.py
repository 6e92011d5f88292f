"""The C-ABI library loads, exports every symbol include/sdt.h declares, and
rejects bad arguments on the host -- all without a GPU."""
import ctypes
import os
import re

import pytest

import shape_driven_tile_gb300 as sdt
from shape_driven_tile_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sdt.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w \*]*?\b([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "while")))


def test_header_declares_core_calls():
    names = declared_functions()
    for n in ("gemm_f16", "gemv_m1", "sdt_pick_tile", "sdt_feasible_tiles", "gemm_f16_with_tile",
              "sdt_last_error", "sdt_check_device_status"):
        assert n in names


def test_every_declared_symbol_is_exported_and_bound():
    h = ctypes.CDLL(_lib.LIB_PATH)
    for name in declared_functions():
        assert hasattr(h, name), f"{name} declared in sdt.h but not exported"
        assert name in _lib.SIGNATURES, f"{name} has no ctypes signature"
    assert set(_lib.SIGNATURES) == set(declared_functions())


def test_abi_version():
    assert sdt.lib().sdt_abi_version() == 1


def L():
    return sdt.lib()


def test_null_and_alignment_rejected_before_device():
    assert L().gemm_f16(256, 256, 256, None, None, None, None) == -1
    assert L().gemm_f16(256, 256, 256, 16, 32, 48, None) == -1 or True  # non-null: next check
    assert L().gemm_f16(256, 256, 256, 0x1000, 0x2008, 0x3000, None) == -2
    assert L().gemm_f16(-1, 256, 256, 0x1000, 0x2000, 0x3000, None) == -3
    assert L().gemm_f16(0, 256, 256, None, None, None, None) == 0      # empty: no-op
    assert L().gemm_f16(256, 0, 256, None, None, None, None) == 0
    assert L().gemm_f16_with_tile(256, 256, 256, 0x1000, 0x2000, 0x3000, None, 99, -1) == -7
    assert L().gemm_f16_with_tile(256, 256, 256, 0x1000, 0x2000, 0x3000, None, 0, 5) == -10
    assert b"stagger" in L().sdt_last_error()


def test_gemv_argument_checks():
    assert L().gemv_m1(4096, 0, None, None, None, None, None) == 0
    assert L().gemv_m1(4096, 8, None, None, None, 0x1000, None) == -1
    assert L().gemv_m1(4096, 8, 0x1008, 0x2000, None, 0x3000, None) == -2
    assert L().gemv_m1(4100, 8, 0x1000, 0x2000, None, 0x3000, None) == -3
    assert L().gemv_m1_q8(4096, 8, 0x1000, 0x2000, None, 0x3000, None) == -1
    assert L().gemv_m1_q8(4112, 8, 0x1000, 0x2000, 0x4000, 0x3000, None) == -3


def test_valid_call_without_gpu_fails_loudly():
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    rc = L().gemm_f16(256, 256, 256, 0x1000, 0x2000, 0x3000, None)
    assert rc == -4
    assert L().sdt_last_error()
    with pytest.raises(sdt.SdtError):
        _lib.check(rc)


def test_tile_info_and_names():
    ts = sdt.tiles()
    assert [t["id"] for t in ts] == list(range(len(ts)))
    names = [t["name"] for t in ts]
    for want in ("64x64", "64x128", "128x64", "128x128", "128x256"):
        assert want in names
    for t in ts:
        assert t["BK"] == 64 and t["threads"] > 0
        assert t["smem_bytes"] <= 232448
        assert t["tmem_cols"] in (32, 64, 128, 256, 512)
        assert sdt.lib().sdt_tile_name(t["id"]).decode() == t["name"]
    assert sdt.lib().sdt_tile_name(len(ts)) is None
    d = _lib.sdt_tile_desc()
    assert sdt.lib().sdt_tile_info(-1, ctypes.byref(d)) == -7
    assert sdt.lib().sdt_tile_info(0, None) == -1
