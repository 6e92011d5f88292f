"""Comparison helpers shared by the GPU parity tests.

Tolerances (the stated bar for this path): on uniform [-1, 1] inputs
max|C - C_ref| <= 1e-3 * sqrt(K) and ||C - C_ref||_F / ||C_ref||_F <= 1e-3,
with C_ref the oracle's fp64 value; on integer-valued inputs the fp16 result
must equal the oracle's value rounded to fp16 (nearest even) bit for bit.
"""
import numpy as np
import torch

import oracle


def u16(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu().contiguous()
    return t.view(torch.int16).numpy().view(np.uint16)


def assert_close(got, ref, K, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output (unwritten tile?)"
    err = np.abs(got - ref)
    max_err = float(err.max()) if err.size else 0.0
    bound = 1e-3 * np.sqrt(max(K, 1))
    assert max_err <= bound, f"{what}: max abs error {max_err:.3e} > {bound:.3e}"
    nref = float(np.linalg.norm(ref))
    if nref > 0:
        rel = float(np.linalg.norm(got - ref)) / nref
        assert rel <= 1e-3, f"{what}: relative Frobenius error {rel:.3e} > 1e-3"
    return max_err


def assert_bit_exact_f16(got_f16: torch.Tensor, ref_f64: np.ndarray, what=""):
    want = oracle.f64_to_f16(ref_f64)
    got = u16(got_f16)
    bad = got != want
    assert not bad.any(), f"{what}: {int(bad.sum())} of {bad.size} fp16 results differ from the oracle"


def boundary_rows(M: int, step: int = 64, extra: int = 8, seed: int = 0) -> np.ndarray:
    """Rows at every tile-row boundary (first and last row of each 64-row band) plus random rows."""
    rows = set()
    for b in range(0, M, step):
        rows.add(b)
        rows.add(min(M - 1, b + step - 1))
    rng = np.random.default_rng(seed)
    rows.update(int(r) for r in rng.integers(0, M, extra))
    return np.array(sorted(rows), dtype=np.int64)


def nan_like(shape, device, dtype=torch.float16):
    return torch.full(shape, float("nan"), dtype=dtype, device=device)


def bf16_ulp(x) -> np.ndarray:
    """Spacing of the bfloat16 values at |x| (8 significant bits): 2^(e-7) for
    2^e <= |x| < 2^(e+1) in the normal range, the subnormal spacing 2^-133 below it."""
    a = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a >= 2.0 ** -126, np.exp2(e - 7), 2.0 ** -133)


def assert_close_bf16(got, ref, K, what=""):
    """bf16 output against want = the oracle's value rounded to bf16 (nearest even):
      * |got - want| <= 1 bf16 ulp + 1e-3*sqrt(K) per element: the fp32 sum may sit on
        the other side of a rounding boundary of want, by at most the stated
        accumulation bound (max error 1e-3*sqrt(K));
      * at most 2 % of the results (at least 8) off want: the tensor cores' fp32
        accumulation error is far below half a bf16 ulp almost everywhere (measured on
        GB300 for these kernels and for cuBLAS on the same inputs: 0.02-0.43 % off), so
        nearly every result is the correctly rounded value;
      * ||got - C_ref||_F <= ||want - C_ref||_F + 1e-3 ||C_ref||_F: beyond what rounding
        the exact product to bf16 costs, the stated relative Frobenius bound (1e-3)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    want = oracle.bf16_to_f64(oracle.f64_to_bf16(ref))
    diff = np.abs(got - want)
    bound = bf16_ulp(np.maximum(np.abs(got), np.abs(want))) + 1e-3 * np.sqrt(max(K, 1))
    excess = diff - bound
    assert excess.size == 0 or excess.max() <= 0, f"{what}: error exceeds 1 ulp + 1e-3*sqrt(K) by {excess.max():.3e}"
    off = int(np.count_nonzero(diff))
    assert off <= max(8, 0.02 * diff.size), f"{what}: {off} of {diff.size} results are not RN_bf16(C_ref)"
    nref = float(np.linalg.norm(ref))
    if nref > 0:
        extra = float(np.linalg.norm(got - ref)) - float(np.linalg.norm(want - ref))
        assert extra <= 1e-3 * nref, \
            f"{what}: Frobenius error beyond the rounding of C_ref is {extra / nref:.3e} of ||C_ref|| > 1e-3"


def assert_bit_exact_bf16(got_bf16, ref_f64, what=""):
    want = oracle.f64_to_bf16(ref_f64)
    got = u16(got_bf16)
    bad = got != want
    assert not bad.any(), f"{what}: {int(bad.sum())} of {bad.size} bf16 results differ from the oracle"


def q8_rounding_bound(x64, q, s64):
    """Bound on |y_gpu - y_ref| of the q8 kernel's arithmetic (the reading of the q8
    arithmetic in the design notes): each group g of 32 activations is scaled by
    2^(14 - E_g), E_g = the group's largest binary exponent (at least -111), and rounded
    to an integer, so an activation moves by at most 2^(E_g - 15); the group sums are
    exact in int32 and the fp32 work after them (int -> float, the scale product, the
    FMA and the sums across groups and threads) takes at most G + 2 roundings of 2^-24
    per term (bounded here with 2^-23).  Per output n:
        B_n = sum_g s[n,g] * sum_{k in g} |q[n,k]| * (2^(E_g - 15) * (1 + c) + c * |x_k|),
    c = (G + 2) * 2^-23, G = K / 32."""
    K = x64.size
    G = K // 32
    xg = np.abs(x64).reshape(G, 32)
    gmax = xg.max(axis=1)
    E = np.where(gmax > 0, np.floor(np.log2(np.where(gmax > 0, gmax, 1.0))), -111.0)
    E = np.maximum(E, -111.0)
    c = (G + 2) * 2.0 ** -23
    qa = np.abs(q.astype(np.float64)).reshape(q.shape[0], G, 32)
    act = np.exp2(E - 15)[None, :, None] * (1 + c) + c * xg[None, :, :]
    return (s64 * (qa * act).sum(axis=2)).sum(axis=1)
