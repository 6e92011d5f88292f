"""Monotone coordinate-descent tuning of one GEMM problem.

"Iteratively Tuning hipBLASLt TensileLite Kernels", sections "The Iteration:
Principle and Design" and "The Six Rounds": the search opens one group of
parameters at a time while every other parameter stays pinned at the running
best, puts the running best into every round's candidate list, and adopts a
round's winner only when it is strictly faster, so the latency after each round
can only stay or fall; the groups run in order of impact, with the tail
handling last.  The starting point is the library's own choice (the page's warm
start from the kernel already in hand; here pick_tile's tile).

Groups for this library's kernels:

  1. ``tile``     -- the ladder tile (any tile that fits on chip; gemm_ex lets
                     tiles overhang ragged edges) with its ring depth (the
                     page opens DepthU in this round; 0 = the tile's own depth,
                     deeper rings are clamped to what fits in shared memory)
  2. ``split-K``  -- split count and reduction algorithm with the tile pinned
                     (gemm_ex_splitk, a form of the one-CTA tiles only: when the
                     held tile is persistent or a CTA pair, the round opens the
                     split-capable tiles too; candidates the library rejects are
                     dropped before timing, as the page's legality filter drops
                     configurations that cannot be generated)
  3. ``mapping``  -- how CTAs land on the output: the raster band height (m-tiles
                     per band) and the k-loop start stagger
  4. ``tail``     -- the two-CTA 256x256 tile's tail as half-width items or not
  5. ``stream-K`` -- the page's terminal branch ("Stream-K"): the split count is
                     set aside and Stream-K opened instead, with one CTA per SM
                     slot or one per SM and the fix-up in the kernel or in a
                     second kernel, on the held tile (or, when it has no
                     stream-K form, on the tiles that have one); being a strict-
                     win round it keeps the split-K best when Stream-K loses,
                     which is the page's try-and-fallback

The descent itself (``descend``) is pure host logic over a ``measure`` callable;
``GemmProblem`` supplies candidates and GPU timings for a problem.
"""
from __future__ import annotations

import os
import random
from typing import Callable, Iterable

import torch

import shape_driven_tile_gb300 as sdt

SPLITS = (2, 3, 4, 6, 8, 12, 16)
DEPTHS = (0, 3, 4, 6, 8, 12)
RASTER = (1, 2, 4, 8, 16, 32)
# 0 / -1 leave the library's own default for that knob (raster band, stagger "auto", ring depth)
DEFAULTS = {"tile": -1, "stages": 0, "splits": 1, "algo": 0, "raster": 0, "stagger": -1, "tail": 1}


def _key(cfg: dict) -> tuple:
    return tuple(sorted(cfg.items()))


def descend(rounds, start: dict, measure: Callable[[dict], float | None], passes: int = 1, seed: int = 0):
    """Run the rounds from `start`.

    rounds  : sequence of (name, propose) where propose(held) yields candidate configs
    measure : config -> latency (any unit, lower is better) or None when the
              configuration is illegal for the problem
    passes  : each round times its candidates `passes` times, every pass in a fresh
              shuffled order, and keeps each candidate's best time -- so a slow drift
              of the device (clocks, temperature) does not favour whichever candidate
              is always timed first
    Returns (held, trajectory).  trajectory[0] is the start ("base"); entry r > 0
    records the round's name, the latency held after it, the configuration held,
    and how many candidates were enumerated and how many were legal.  The held
    latency is always a measurement of the held configuration: the incumbent is
    timed again in every round with the challengers (keeping its best time), and
    a challenger replaces it only when its time is strictly lower.  So the held
    latency never rises from one round to the next, whatever the ranges or the
    noise, and the worst a round can do is keep what it started from.
    """
    rng = random.Random(seed)
    held = dict(start)
    t_held = measure(held)
    if t_held is None:
        raise ValueError("the starting configuration is not legal for the problem")
    traj = [{"round": "base", "us": t_held, "cfg": dict(held), "enumerated": 1, "legal": 1}]
    for name, propose in rounds:
        cands, seen = [], set()
        for c in [dict(held)] + list(propose(dict(held))):  # union the incumbent
            k = _key(c)
            if k not in seen:
                seen.add(k)
                cands.append(dict(c))
        best_of = {}
        order = list(range(len(cands)))
        for _ in range(max(1, passes)):
            rng.shuffle(order)
            for i in order:
                k = _key(cands[i])
                if best_of.get(k, 0.0) is None:
                    continue  # illegal: not timed again
                t = measure(cands[i])
                best_of[k] = None if t is None else min(t, best_of.get(k) or t)
        results = [(best_of[_key(c)], c) for c in cands if best_of[_key(c)] is not None]
        if not results:
            traj.append({"round": name, "us": t_held, "cfg": dict(held), "enumerated": len(cands), "legal": 0})
            continue
        for t, c in results:
            if _key(c) == _key(held):
                t_held = min(t_held, t)
        best_t, best_c = min(results, key=lambda r: r[0])
        if best_t < t_held and _key(best_c) != _key(held):
            held, t_held = best_c, best_t
        traj.append({"round": name, "us": t_held, "cfg": dict(held), "enumerated": len(cands),
                     "legal": len(results)})
    return held, traj


class _Env:
    """Sets the library's per-call environment knobs for one launch and restores them
    (a knob at its "library default" value is removed from the environment)."""

    NAMES = {"raster": "SDT_RASTER_GROUP", "stagger": "SDT_STAGGER", "tail": "SDT_TAIL_SPLIT", "stages": "SDT_STAGES"}
    LIBRARY_DEFAULT = {"raster": 0, "stagger": -1, "stages": 0}

    def __init__(self, cfg: dict):
        self.vals = {self.NAMES[k]: (None if self.LIBRARY_DEFAULT.get(k) == cfg[k] else str(int(cfg[k])))
                     for k in self.NAMES}

    def __enter__(self):
        self.old = {k: os.environ.get(k) for k in self.vals}
        for k, v in self.vals.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v

    def __exit__(self, *exc):
        for k, v in self.old.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v


class L2Flush:
    """Leaves L2 holding clean lines of an unrelated buffer: a read of 4x the L2 size.

    A flush by writing (zeroing a large buffer) leaves L2 full of dirty lines, and
    the next kernel then pays for their write-back inside its timed region -- up to
    the whole L2 (~129 MB) of extra DRAM writes, which on a memory-bound launch of
    tens of microseconds inflates its time by a fifth or more.  A read pass evicts
    the previous launch's operands just the same and leaves nothing to write back.
    """

    def __init__(self, device, nbytes: int = 512 << 20):
        self.buf = torch.ones(nbytes // 4, dtype=torch.float32, device=device)

    def __call__(self):
        self.buf.sum()


class GemmProblem:
    """One problem C = op(A) . op(B) on the GPU and the candidates of each round.

    A is [M, K] row-major; B is the logical [K, N] operand as a view (row-major, or
    the transpose of a row-major [N, K] tensor); C is [M, N] row-major.  Latency of
    a configuration: mean device time of `reps` launches, each after an L2 flush
    (``L2Flush``; CUDA events on the current stream around the launch).
    """

    def __init__(self, A: torch.Tensor, B: torch.Tensor, C: torch.Tensor, reps: int = 10,
                 flush_bytes: int = 512 << 20):
        self.A, self.B, self.C, self.reps = A, B, C, reps
        self.M, self.K = A.shape
        self.N = B.shape[1]
        self.dtype = A.dtype
        self.flush = L2Flush(A.device, flush_bytes)
        self.ws = None
        self.ntiles = len(sdt.tiles())

    # -- launching ----------------------------------------------------------------------
    def _workspace(self, nbytes: int) -> torch.Tensor:
        """One workspace for every split candidate, zeroed when it is (re)allocated: the
        library keeps a zeroed workspace valid across tiles, split counts and algorithms."""
        if self.ws is None or self.ws.numel() < nbytes:
            ws = torch.empty(max(nbytes, 256) + 256, dtype=torch.uint8, device=self.A.device)
            off = (-ws.data_ptr()) % 256
            self.ws = ws[off:off + max(nbytes, 256)]
            sdt.lib().sdt_splitk_workspace_init(self.ws.data_ptr(), self.ws.numel(),
                                                torch.cuda.current_stream().cuda_stream)
        return self.ws

    def launcher(self, cfg: dict):
        """A no-argument callable that launches cfg, or None when cfg is illegal here."""
        streamk = cfg["algo"] in (sdt.SPLITK_STREAM, sdt.SPLITK_STREAM_REDUCE)
        if streamk or cfg["splits"] > 1:
            if streamk:
                if sdt.lib().sdt_streamk_workspace_bytes(self.M, self.N, self.K, cfg["tile"], 1) == 0:
                    return None  # no stream-K form
                nbytes = sdt.streamk_workspace_bytes(self.M, self.N, self.K, cfg["tile"], cfg["splits"] or None)
            else:
                nbytes = sdt.splitk_ex_workspace_bytes(self.M, self.N, self.K, cfg["tile"], cfg["splits"])
            if nbytes == 0:
                return None
            ws = self._workspace(nbytes)

            def run():
                with _Env(cfg):
                    sdt.gemm_ex_splitk(self.A, self.B, self.C, workspace=ws, tile=cfg["tile"],
                                       splits=cfg["splits"], algo=cfg["algo"])
            return run

        def run():
            with _Env(cfg):
                sdt.gemm_ex(self.A, self.B, self.C, tile=cfg["tile"])
        return run

    def measure(self, cfg: dict) -> float | None:
        run = self.launcher(cfg)
        if run is None:
            return None
        try:
            run()  # also rejects configurations the library refuses (tile/shape/split rules)
            torch.cuda.synchronize()
        except sdt.SdtError:
            return None
        stream = torch.cuda.current_stream()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(self.reps)]
        for e0, e1 in evs:
            self.flush()
            e0.record(stream)
            run()
            e1.record(stream)
        torch.cuda.synchronize()
        return 1e3 * sum(e0.elapsed_time(e1) for e0, e1 in evs) / self.reps

    # -- rounds -------------------------------------------------------------------------
    def start(self) -> dict:
        cfg = dict(DEFAULTS)
        cfg["tile"] = sdt.pick_tile_any(self.M, self.N, self.K)
        return cfg

    def rounds(self):
        def tiles(held):
            for t in range(self.ntiles):
                for d in DEPTHS:
                    yield dict(held, tile=t, stages=d, splits=1, algo=0)

        def split(held):
            # The page opens the split with the tile pinned.  Here split-K is a form of the
            # one-CTA tiles only, so when the held tile is persistent or a CTA pair the round
            # opens the split-capable tiles with it; the held configuration stays a
            # candidate either way.  Candidates without a split-K form for the shape are
            # dropped by measure()'s legality check.
            if held["splits"] > 1 or held["algo"] in (sdt.SPLITK_STREAM, sdt.SPLITK_STREAM_REDUCE):
                return
            own = sdt.splitk_ex_workspace_bytes(self.M, self.N, self.K, held["tile"], 2) > 0
            tiles = [held["tile"]] if own else range(self.ntiles)
            for t in tiles:
                for s in SPLITS:
                    for a in (sdt.SPLITK_REDUCE_KERNEL, sdt.SPLITK_IN_KERNEL):
                        yield dict(held, tile=t, splits=s, algo=a)

        def mapping(held):
            for r in RASTER:
                for st in (-1, 0, 1):
                    yield dict(held, raster=r, stagger=st)

        def tail(held):
            info = sdt.tile_info(held["tile"])
            if info["cta_group"] == 2 and info["BN"] == 256 and held["splits"] == 1:
                for t in (0, 1):
                    yield dict(held, tail=t)

        def stream(held):
            def has_form(t):
                return sdt.lib().sdt_streamk_workspace_bytes(self.M, self.N, self.K, t, 1) > 0

            tiles = [held["tile"]] if has_form(held["tile"]) else [t for t in range(self.ntiles) if has_form(t)]
            sms = sdt.device_sm_count()
            for t in tiles:
                for g in (0, sms):  # one CTA per SM slot (0), and one per SM
                    for a in (sdt.SPLITK_STREAM, sdt.SPLITK_STREAM_REDUCE):  # fix-up in the kernel or after it
                        yield dict(held, tile=t, splits=g, algo=a, tail=1)

        return [("tile", tiles), ("split-K", split), ("mapping", mapping), ("tail", tail), ("stream-K", stream)]

    def tune(self, passes: int = 2):
        return descend(self.rounds(), self.start(), self.measure, passes=passes)
