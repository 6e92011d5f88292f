"""Integer tile rules of the pages, written out plainly (oracle side).

TEST INFRASTRUCTURE ONLY (see the package docstring).

* ``seed_tile(M, N, units)`` -- the launcher rule of "Beating hipBLASLt on a
  Gaming GPU", section "The part that actually mattered": count the
  128x128-equivalent blocks the grid would produce, (M/128)*(N/128); at least
  one block per compute unit (96 on that card) takes 128x128, at least 64 of 96
  takes 64x128, anything less takes 64x64.  The page prints the thresholds for
  a 96-unit part only; for another unit count this function scales them as
  ``units`` and ``2*units/3`` (our reading; at 96 it is exactly the page's).

* ``grid(M, N, BM, BN)`` -- the CTA grid a tile cuts, printed as
  "N-blocks x M-blocks" in the "Tile . warps . grid" column of the "mojo-baro"
  table ("Square fp16 GEMM vs hipBLASLt"), and the workgroup counts of the
  FlyDSL pull request "Speed up the RDNA3 GEMM up to 1.85x by choosing the tile
  from the shape", section "Motivation" (4 at 256x256, 16 at 512x512 for a
  128x128 tile).

* ``feasible(M, N, K, tile, smem_limit, tmem_cols_limit)`` -- the three
  feasibility rules of that pull request's "Changes" section: a feasible tile
  (i) divides the shape, (ii) can fill the prefetch pipeline, (iii) fits in
  on-chip memory.  Readings for this hardware: (ii) is "at least two k-tiles"
  (one k-tile leaves nothing to overlap); (iii) is the tile's declared shared
  memory footprint within the device's per-block opt-in limit and its
  accumulator within the 512 tensor-memory columns of an SM; a two-CTA tile
  covers BM rows with a pair of CTAs, so it needs M divisible by its full BM.

* ``kloop_order(cta, n_k, stride)`` -- the per-workgroup k-loop start stagger
  of the same pull request (third commit and "Changes"): start each workgroup
  at a different k-tile and wrap with a mask; wired only when the k-tile count
  is a power of two.  Our reading of the start: (cta * stride) mod n_k.
"""
from __future__ import annotations


def blocks_128(M: int, N: int) -> int:
    return (M // 128) * (N // 128)


def seed_tile(M: int, N: int, units: int) -> str:
    b = blocks_128(M, N)
    if b >= units:
        return "128x128"
    if 3 * b >= 2 * units:
        return "64x128"
    return "64x64"


def grid(M: int, N: int, BM: int, BN: int) -> tuple[int, int]:
    """(blocks along N, blocks along M) for a tile that divides the shape."""
    return (N // BN, M // BM)


def feasible(M: int, N: int, K: int, tile: dict, smem_limit: int,
             tmem_cols_limit: int = 512) -> bool:
    BM, BN, BK = tile["BM"], tile["BN"], tile["BK"]
    if M <= 0 or N <= 0 or K <= 0:
        return False
    # (i) divides the shape
    if M % BM or N % BN or K % BK:
        return False
    # (ii) can fill the pipeline
    if K // BK < 2:
        return False
    # (iii) fits on chip
    if tile["smem_bytes"] > smem_limit:
        return False
    if tile["tmem_cols"] > tmem_cols_limit:
        return False
    return True


def is_pow2(n: int) -> bool:
    return n > 0 and (n & (n - 1)) == 0


def kloop_order(cta: int, n_k: int, stride: int = 1, enabled: bool = True) -> list[int]:
    if not enabled or not is_pow2(n_k):
        return list(range(n_k))
    start = (cta * stride) % n_k
    return [(start + i) % n_k for i in range(n_k)]
