"""CPU checks of the comparison helpers the GPU parity tests use (no GPU): the bf16
spacing against the format's definition (8 significant bits), and that the bf16
comparison passes the correctly rounded value and values one rounding step away,
and fails two steps, a dropped term and a wrong sign."""
import numpy as np
import pytest

import oracle
from _parity import assert_close, assert_close_bf16, bf16_ulp, q8_rounding_bound


def test_bf16_ulp_is_the_spacing_of_the_format():
    # next representable bf16 above x: bit pattern + 1 (positive normals)
    xs = np.array([1.0, 1.5, 2.0, 3.0, 0.75, 1e-3, 255.0, 256.0, 40000.0, 2.0 ** -126])
    pat = oracle.f64_to_bf16(xs)
    nxt = oracle.bf16_to_f64(pat + 1)
    assert np.array_equal(nxt - oracle.bf16_to_f64(pat), bf16_ulp(xs))
    assert bf16_ulp(np.array([1.0]))[0] == 2.0 ** -7
    assert bf16_ulp(np.array([-3.0]))[0] == 2.0 ** -6
    assert bf16_ulp(np.array([0.0]))[0] == 2.0 ** -133


def _case(seed=0, n=4096, K=64):
    rng = np.random.default_rng(seed)
    ref = rng.normal(0, np.sqrt(K) / 3, n)
    want = oracle.bf16_to_f64(oracle.f64_to_bf16(ref))
    return ref, want, K


def test_bf16_comparison_accepts_rounded_and_one_step_off():
    ref, want, K = _case()
    assert_close_bf16(want, ref, K)
    got = want.copy()
    got[:40] += bf16_ulp(got[:40])  # one rounding step (1 %): the fp32 sum on the other side
    assert_close_bf16(got, ref, K)
    small_ref, small_want = ref[:300], want[:300].copy()
    small_want[:8] -= bf16_ulp(small_want[:8])  # a small sample: eight one-step misses pass
    assert_close_bf16(small_want, small_ref, K)


def test_bf16_comparison_rejects_mistakes():
    ref, want, K = _case(1)
    bad = want.copy()
    bad[5] += 3 * bf16_ulp(bad[5]) + 1e-3 * np.sqrt(K)  # beyond 1 ulp + accumulation bound
    with pytest.raises(AssertionError):
        assert_close_bf16(bad, ref, K)
    many = want + bf16_ulp(want) * (np.arange(want.size) % 20 == 0)  # 5 % one step off
    with pytest.raises(AssertionError):
        assert_close_bf16(many, ref, K)
    with pytest.raises(AssertionError):
        assert_close_bf16(-want, ref, K)  # wrong sign
    rng = np.random.default_rng(2)
    term = rng.uniform(-1, 1, ref.size) * 0.5  # one product dropped from every sum
    with pytest.raises(AssertionError):
        assert_close_bf16(oracle.bf16_to_f64(oracle.f64_to_bf16(ref - term)), ref, K)


def test_fp16_comparison_bounds():
    ref, _, K = _case(3, K=1024)
    got = ref.copy()
    got[7] += 0.9e-3 * np.sqrt(K)  # one element near the max-error bound
    assert_close(got, ref, K)
    got[7] = ref[7] + 1.1e-3 * np.sqrt(K)
    with pytest.raises(AssertionError):
        assert_close(got, ref, K)
    with pytest.raises(AssertionError):  # every element off by 2e-3 relative: Frobenius
        assert_close(ref * (1 + 2e-3), ref, K)


def test_q8_rounding_bound_closed_form():
    # CPU check of the bound itself: integer activations within 2^7 of their group's
    # largest convert exactly, so only the fp32 term remains (tiny against |y|)
    K, N = 256, 4
    x = np.tile(np.arange(-16, 16, dtype=np.float64), K // 32)
    q = np.ones((N, K), dtype=np.int8)
    s = np.full((N, K // 32), 2.0 ** -7)
    b = q8_rounding_bound(x, q, s)
    # E_g = 4 for every group (largest |x| = 16): 2^(4-15) * 32 * 2^-7 per group, 8 groups
    assert np.allclose(b, 8 * 32 * 2.0 ** -7 * (2.0 ** -11 * (1 + 10 * 2.0 ** -23))
                       + 8 * 2.0 ** -7 * 10 * 2.0 ** -23 * np.abs(x[:32]).sum(), rtol=1e-12)


def _group_scaled(x, q, s, rnd):
    """y of the scheme the bound describes, in fp64: group scaling by 2^(14 - E_g), rnd
    to an integer, exact group sums."""
    N = q.shape[0]
    E = np.floor(np.log2(np.abs(x).reshape(-1, 32).max(axis=1)))
    scale = np.repeat(np.exp2(14 - E), 32)
    xr = rnd(x * scale) / scale
    return (s * (xr.reshape(-1, 32)[None] * q.reshape(N, -1, 32)).sum(axis=2)).sum(axis=1)


def _exact(x, q, s):
    N = q.shape[0]
    return (s * (x.reshape(-1, 32)[None] * q.reshape(N, -1, 32)).sum(axis=2)).sum(axis=1)


def test_q8_rounding_bound_covers_the_group_scaling():
    # random activations over 2^-24 .. 2^24: the scheme's error stays within the bound
    rng = np.random.default_rng(11)
    K, N = 1024, 64
    x = oracle.bf16_to_f64(oracle.f64_to_bf16(rng.uniform(-1, 1, K) * np.exp2(rng.integers(-24, 25, K))))
    q = rng.integers(-127, 128, (N, K)).astype(np.int8)
    s = oracle.f16_to_f64(oracle.f64_to_f16(rng.uniform(1e-3, 1e-2, (N, K // 32))))
    assert (np.abs(_group_scaled(x, q, s, np.rint) - _exact(x, q, s)) <= q8_rounding_bound(x, q, s)).all()
    # a group whose small activations all sit 7/8 of a quantum above an integer, same-sign
    # weights: rounding moves each by 1/8 quantum (inside), truncating by 7/8 (a plausible
    # mistake that the bound catches)
    x = np.concatenate([[1.0], (np.arange(1, 32) + 0.875) * 2.0 ** -14])
    q = np.full((1, 32), 127, dtype=np.int8)
    s = np.full((1, 1), 2.0 ** -7)
    b = q8_rounding_bound(x, q, s)
    assert (np.abs(_group_scaled(x, q, s, np.rint) - _exact(x, q, s)) <= b).all()
    assert (np.abs(_group_scaled(x, q, s, np.trunc) - _exact(x, q, s)) > b).all()
