"""Fit of pick_tile's cost-model constants to a measured tile sweep (host only, no GPU).

pick_tile estimates each feasible tile's run time on a shape from five constants per
tile (microseconds) and takes the smallest estimate; the estimate has the form of
``model_us`` in csrc/gemm_host.cu:

  one-CTA tiles, in waves of co-resident CTAs (waves = ceil(tiles / (SMs x CTAs per SM))):
      fixed + waves * (round + max(0, nK - stages) * kt) + tiles * nK / (SMs x CTAs per SM) * bw
      + share * (CTAs beyond the first on the busiest SM, summed over the waves)
  persistent tiles, one worker per SM or per SM pair (rounds = ceil(tiles / workers), minus
  half a round when the two-CTA 256x256 tail runs as half-width items):
      fixed + max(0, rounds * nK - stages) * kt + rounds * round + tiles * nK / workers * bw

This module restates that form over the library's own tile geometry (``sdt.tiles()``), fits
the constants of every tile to a sweep by non-negative least squares weighted by 1 / sqrt(time)
(between absolute and relative error: a fit weighted by 1 / time let the few-microsecond
shapes pull the wide tiles' constants off the long shapes, and picked 7.6 % off the best
on the current sweep, against 2.7 % here; each tile's rows are independent, so the fit is
one small problem per tile), and prints
them as the ladder's rows.  A tile feasible on too few swept shapes takes a scaled copy of
another tile's constants (``DERIVED``).  The sweep is the JSON-lines output of
``bench.py --mode sweep`` (one object per shape with ``"shape"`` and ``"us"``), e.g. the
frozen ``tables/gb300_tile_sweep.jsonl``:

    python -m shape_driven_tile_gb300.costfit shape_driven_tile_gb300/tables/gb300_tile_sweep.jsonl
"""
from __future__ import annotations

import json
import math
import sys

import numpy as np

SM_COUNT = 152            # GB300
SMEM_PER_SM = 233472      # bytes of shared memory per SM the occupancy is computed from
KB = 64                   # k-tile depth of every ladder tile
NOT_CANDIDATES = {"128x256", "2cta_256x128"}  # tiles that never won the sweep
# name: (source tile, k-tile scale, streaming-term scale).  The 256x224 pair: an N = 224
# MMA takes 0.96 of an N = 256 one (measured at 3584^3 and 7168^3); operand bytes 480 / 512.
DERIVED = {"2cta_256x224": ("2cta_256x256", 0.96, 480 / 512)}
FIELDS = ("fixed", "kt", "round", "bw", "share")


def load(path):
    """The sweep's records: dicts with "shape" [M, N, K] and "us" {tile name: time}."""
    out = []
    with open(path) as f:
        for line in f:
            line = line.strip()
            if line.startswith("{") and '"shape"' in line:
                r = json.loads(line)
                if "us" in r:
                    out.append(r)
    return out


def geometry():
    """name -> (BM, BN, persistent, pair, CTAs per SM, stages) of the ladder tiles pick_tile
    can choose from (the skinny tiles are gemm_ex forms only)."""
    import shape_driven_tile_gb300 as sdt

    g = {}
    for t in sdt.tiles():
        if t["skinny"]:
            continue
        pair = t["cta_group"] == 2
        persistent = pair or t["name"].startswith("p")
        occ = min(SMEM_PER_SM // (t["smem_bytes"] + 1024), 512 // t["tmem_cols"], 2048 // t["threads"])
        g[t["name"]] = (t["BM"], t["BN"], persistent, pair, max(1, occ), t["stages"])
    return g


def features(geo, M, N, K, sm_count=SM_COUNT):
    """The multipliers of (fixed, kt, round, bw, share) for one tile on one shape."""
    BM, BN, persistent, pair, occ, stages = geo
    tiles = math.ceil(M / BM) * math.ceil(N / BN)
    nK = math.ceil(K / KB)
    if persistent:
        workers = sm_count // 2 if pair else sm_count
        rounds = math.ceil(tiles / workers)
        if pair and BN == 256 and tiles >= workers:
            tail = tiles - (tiles // workers) * workers
            if 0 < tail and 2 * tail <= workers:
                rounds -= 0.5
        return np.array([1.0, max(0.0, rounds * nK - stages), rounds, tiles * nK / workers, 0.0])
    per_wave = sm_count * occ
    waves = math.ceil(tiles / per_wave)
    full, rest = divmod(tiles, per_wave)
    extra = full * (occ - 1) + (min(occ, math.ceil(rest / sm_count)) - 1 if rest else 0)
    return np.array([1.0, waves * max(0, nK - stages), waves, tiles * nK / per_wave, extra])


def fit(records, sm_count=SM_COUNT):
    """name -> array (fixed, kt, round, bw, share) fitted to the records."""
    from scipy.optimize import nnls

    geo = geometry()
    consts = {}
    for name, g in geo.items():
        rows, times = [], []
        for r in records:
            if name in r["us"]:
                rows.append(features(g, *r["shape"], sm_count))
                times.append(r["us"][name])
        if not rows:
            continue
        X, y = np.array(rows), np.array(times)
        w = 1.0 / np.sqrt(y)
        consts[name], _ = nnls(X * w[:, None], y * w)
    for name, (src, kt_scale, bw_scale) in DERIVED.items():
        if name in geo and src in consts:
            c = consts[src].copy()
            c[1] *= kt_scale
            c[3] *= bw_scale
            consts[name] = c
    return consts


def estimate(consts, name, M, N, K, sm_count=SM_COUNT, geo=None):
    geo = geo or geometry()
    return float(np.dot(consts[name], features(geo[name], M, N, K, sm_count)))


def pick(consts, record, sm_count=SM_COUNT, geo=None):
    """The candidate with the smallest estimate among the tiles the record timed."""
    geo = geo or geometry()
    M, N, K = record["shape"]
    cands = [t for t in record["us"] if t in consts and t not in NOT_CANDIDATES]
    return min(cands, key=lambda t: estimate(consts, t, M, N, K, sm_count, geo))


def ladder_rows(consts):
    """The constants as printed in the ladder (fixed, round and share to 3 decimals, kt and bw to 5)."""
    return {name: (round(c[0], 3), round(c[1], 5), round(c[2], 3), round(c[3], 5), round(c[4], 3))
            for name, c in consts.items()}


def main(argv):
    if len(argv) != 2:
        print(__doc__.strip().splitlines()[-1].strip())
        return 2
    records = load(argv[1])
    consts = fit(records)
    for name, (f, kt, rnd, bw, shr) in ladder_rows(consts).items():
        print(f"{name:14s} fixed {f:.3f}  kt {kt:.5f}  round {rnd:.3f}  bw {bw:.5f}  share {shr:.3f}")
    slow = [r["us"][pick(consts, r)] / min(r["us"].values()) - 1 for r in records]
    print(f"pick slowdown over {len(records)} records: average {100 * sum(slow) / len(slow):.2f} %, "
          f"worst {100 * max(slow):.2f} %")
    return 0


if __name__ == "__main__":
    sys.exit(main(sys.argv))
