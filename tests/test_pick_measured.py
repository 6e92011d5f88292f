"""pick_tile against the measured sweep it was fitted to (host only, no GPU).

The FlyDSL RDNA GEMM pull request checks the tile pick_tile returns for each
measured shape; here the measurements themselves are frozen with the package
(every feasible ladder tile timed cold on GB300) and the pick is held to them:
within 5 % of the best tile on every recorded shape (the square sweep, the
K-scan, rectangular, skinny and deep-K shapes), and within 1 % on average.
"""
import json
import os

import pytest

import shape_driven_tile_gb300 as sdt

TABLE = os.path.join(os.path.dirname(sdt.__file__), "tables", "gb300_tile_sweep.jsonl")
SMS, SMEM = 152, 232448


def records():
    with open(TABLE) as f:
        return [json.loads(line) for line in f if line.startswith("{")]


def slowdown(rec):
    M, N, K = rec["shape"]
    name = sdt.tile_info(sdt.pick_tile(M, N, K, sm_count=SMS, smem_limit=SMEM))["name"]
    assert name in rec["us"], (rec["shape"], name)  # the pick was one of the timed (feasible) tiles
    return rec["us"][name] / min(rec["us"].values()) - 1.0


def is_config_shape(shape):
    M, N, K = shape
    return M == N == K or (M == N == 2048 and 1920 <= K <= 2304)


def test_table_covers_the_configurations():
    shapes = {tuple(r["shape"]) for r in records()}
    for n in (256, 512, 768, 1024, 1536, 2048, 2560, 3072, 3584, 4096):
        assert (n, n, n) in shapes
    for k in (1920, 1984, 2048, 2112, 2176, 2304):
        assert (2048, 2048, k) in shapes
    assert len(shapes) >= 40


def test_timed_tiles_are_the_feasible_ones():
    ladder = {t["id"]: t["name"] for t in sdt.tiles()}
    for r in records():
        M, N, K = r["shape"]
        feas = {ladder[i] for i in sdt.feasible_tiles(M, N, K, smem_limit=SMEM)}
        assert set(r["us"]) <= feas, r["shape"]


@pytest.mark.parametrize("rec", [r for r in records() if is_config_shape(r["shape"])],
                         ids=lambda r: "run%d-%dx%dx%d" % (r["run"], *r["shape"]))
def test_pick_within_5_percent_on_the_configurations(rec):
    assert slowdown(rec) <= 0.05


def test_pick_on_every_recorded_shape():
    s = [slowdown(r) for r in records()]
    assert max(s) <= 0.05
    assert sum(s) / len(s) <= 0.01
