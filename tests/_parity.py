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


def assert_close_bf16(got, ref, K, what=""):
    """bf16 output: the fp32 accumulation bound 1e-3*sqrt(K) plus half a bf16 ulp of the
    result (2^-8 relative), and a relative Frobenius error within 2^-8 (the bf16
    rounding of C alone is up to 2^-8 relative)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    bound = 1e-3 * np.sqrt(max(K, 1)) + 2.0 ** -8 * np.abs(ref)
    excess = np.abs(got - ref) - bound
    assert excess.max() <= 0, f"{what}: error exceeds bound by {excess.max():.3e}"
    nref = float(np.linalg.norm(ref))
    if nref > 0:
        rel = float(np.linalg.norm(got - ref)) / nref
        assert rel <= 2.0 ** -8, f"{what}: relative Frobenius error {rel:.3e} > 2^-8"


def assert_bit_exact_bf16(got_bf16, ref_f64, what=""):
    want = oracle.f64_to_bf16(ref_f64)
    got = u16(got_bf16)
    bad = got != want
    assert not bad.any(), f"{what}: {int(bad.sum())} of {bad.size} bf16 results differ from the oracle"
