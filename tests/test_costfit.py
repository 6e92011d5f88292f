"""The cost-model constants in the library are the fit of the frozen sweep (host only).

shape_driven_tile_gb300.costfit restates pick_tile's estimate over the library's tile
geometry and fits its constants to a measured sweep; refitting the frozen GB300 sweep must
give the ladder's printed constants, and the restated estimate must pick the library's tile.
"""
import os
import re

import pytest

import shape_driven_tile_gb300 as sdt
from shape_driven_tile_gb300 import costfit

pytest.importorskip("scipy")

PKG = os.path.dirname(sdt.__file__)
TABLE = os.path.join(PKG, "tables", "gb300_tile_sweep.jsonl")
HOST = os.path.join(PKG, "csrc", "gemm_host.cu")
ROW = re.compile(r'SDT_(TILE|PTILE|PAIR)\([^"]*"([^"]+)",\s*((?:[-\d.]+,\s*){4,5})(true|false)\)')


def ladder_source():
    """name -> ((fixed, kt, round, bw, share), candidate); the persistent and pair rows
    carry no share constant (one CTA or pair per SM by construction)."""
    rows = {}
    with open(HOST) as f:
        for kind, name, nums, cand in ROW.findall(f.read()):
            vals = [float(v) for v in nums.replace(" ", "").strip(",").split(",")]
            if kind != "TILE":
                vals.append(0.0)
            rows[name] = (tuple(vals), cand == "true")
    return rows


def test_source_rows_cover_the_ladder():
    rows = ladder_source()
    assert set(rows) == set(costfit.geometry())
    for name, (_, candidate) in rows.items():
        assert candidate == (name not in costfit.NOT_CANDIDATES), name


def test_refit_reproduces_the_ladder_constants():
    fitted = costfit.ladder_rows(costfit.fit(costfit.load(TABLE)))
    for name, (consts, _) in ladder_source().items():
        got = fitted[name]
        for field, want, have, unit in zip(costfit.FIELDS, consts, got, (1e-3, 1e-5, 1e-3, 1e-5, 1e-3)):
            assert abs(want - have) <= unit * 1.01, (name, field, want, have)


def test_restated_estimate_picks_the_library_tile():
    records = costfit.load(TABLE)
    consts = {n: list(c) for n, c in costfit.ladder_rows(costfit.fit(records)).items()}
    geo = costfit.geometry()
    for r in records:
        M, N, K = r["shape"]
        lib_pick = sdt.tile_info(sdt.pick_tile(M, N, K, sm_count=152, smem_limit=232448))["name"]
        assert costfit.pick(consts, r, geo=geo) == lib_pick, r["shape"]


def test_each_fit_term_is_needed_somewhere():
    # the fit is non-negative; a term that fits to zero on every tile would be dead weight
    consts = costfit.fit(costfit.load(TABLE))
    for i, field in enumerate(costfit.FIELDS):
        assert any(c[i] > 0 for c in consts.values()), field


def test_restated_estimate_equals_the_library_estimate():
    # the same numbers, not only the same picks: costfit's restatement with the printed
    # constants against sdt_tile_estimate_us, over the recorded shapes and a ragged grid
    consts = {n: list(c) for n, c in ladder_source_consts().items()}
    geo = costfit.geometry()
    shapes = [tuple(r["shape"]) for r in costfit.load(TABLE)]
    shapes += [(m, n, k) for m in (1, 100, 1000, 5000) for n in (8, 300, 4096) for k in (1, 70, 4096)]
    for M, N, K in shapes:
        for name in geo:
            want = costfit.estimate(consts, name, M, N, K, geo=geo)
            have = sdt.tile_estimate_us(name, M, N, K, sm_count=152)
            assert abs(have - want) <= 1e-9 * max(1.0, want), (name, M, N, K, have, want)
    with pytest.raises(sdt.SdtError):
        sdt.tile_estimate_us(99, 64, 64, 64)
    with pytest.raises(sdt.SdtError):
        sdt.tile_estimate_us("64x64", 0, 64, 64)


def ladder_source_consts():
    return {name: vals for name, (vals, _) in ladder_source().items()}
