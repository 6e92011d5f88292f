"""The benchmark's protocol legs on the GPU, shortened (few launches, short warm-ups):
each returns its rows with the fields the benchmark line reports, and the numbers
are plausible (positive times, fractions of the peak below about 1.2).  The full
legs run after the benchmark's timed region."""
import pytest
import torch

import bench
import shape_driven_tile_gb300 as sdt

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def square_operands(cuda_device):
    A = {n: torch.empty((n, n), dtype=torch.float16, device=cuda_device).uniform_(-1, 1) for n in bench.SWEEP}
    B = {n: torch.empty((n, n), dtype=torch.float16, device=cuda_device).uniform_(-1, 1) for n in bench.SWEEP}
    C = {n: torch.empty((n, n), dtype=torch.float16, device=cuda_device) for n in bench.SWEEP}
    tiles = {n: sdt.tile_info(sdt.pick_tile(n, n, n))["name"] for n in bench.SWEEP}
    return A, B, C, tiles


def test_gemm_protocol_leg(cuda_device, square_operands):
    A, B, C, tiles = square_operands
    out = bench.gemm_protocol_leg(sdt.lib(), A, B, C, tiles, bench.load_peaks(), torch.cuda.current_stream(),
                                  cuda_device, launches=4, reps=2, warm_s=0.05)
    assert [r["size"] for r in out["rows"]] == bench.SWEEP
    for r in out["rows"]:
        assert 0 < r["us_min"] <= r["us_max"] and r["eager_us"] > 0
        assert 0 < r["pct_peak_best"] < 120
    sdt.check_device_status()
    assert all(bool(torch.isfinite(C[n]).all()) for n in bench.SWEEP)


def test_pick_check_leg(cuda_device, square_operands):
    A, B, C, tiles = square_operands
    out = bench.pick_check_leg(sdt.lib(), A, B, C, tiles, bench.load_peaks(), torch.cuda.current_stream(),
                               cuda_device, passes=1, launches=1, warm_s=0.05)
    assert [r["shape"] for r in out["rows"]] == ([[n, n, n] for n in bench.SWEEP]
                                                 + [[2048, 2048, k] for k in bench.KSCAN if k != 2048])
    for r in out["rows"]:
        assert r["pick"] in r["us"] and r["best"] in r["us"] and r["slowdown"] >= 0
        assert set(r["us"]) == {sdt.tile_info(t)["name"] for t in sdt.feasible_tiles(*r["shape"])}
    assert out["worst_slowdown"] == max(r["slowdown"] for r in out["rows"])
    sdt.check_device_status()


def test_kscan_and_large_legs(cuda_device):
    out = bench.kscan_leg(sdt.lib(), bench.load_peaks(), torch.cuda.current_stream(), cuda_device, passes=1,
                          launches=1, graph_launches=2, warm_s=0.05)
    assert [r["K"] for r in out["rows"]] == bench.KSCAN
    for r in out["rows"]:
        assert r["stagger_applies"] == (r["K"] == 2048)
        assert all(v > 0 for d in (r["cold_tflops"], r["warm_tflops"]) for v in d.values())
    out = bench.large_leg(sdt.lib(), bench.load_peaks(), torch.cuda.current_stream(), cuda_device, sizes=[8192],
                          reps=1, warm_s=0.05)
    (r,) = out["rows"]
    assert r["size"] == 8192 and r["tile"] == sdt.tile_info(sdt.pick_tile(8192, 8192, 8192))["name"]
    assert 0 < r["pct_peak_best"] < 120
    sdt.check_device_status()


def test_event_pair_cost(cuda_device):
    cost = bench.event_pair_cost(torch.cuda.current_stream(), cuda_device, reps=8)
    assert set(cost) == {"min", "median"}
    assert 0 < cost["min"] <= cost["median"] < 1e4  # microseconds
