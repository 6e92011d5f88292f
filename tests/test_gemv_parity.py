"""gemv_m1 (M=1 decode) on the GPU against the fp64 CPU oracle, through the C ABI."""
import os

import numpy as np
import pytest
import torch

import oracle
import shape_driven_tile_gb300 as sdt
from shape_driven_tile_gb300 import inputs
from _parity import assert_close, q8_rounding_bound, u16

pytestmark = pytest.mark.gpu

K_DEC, N_DEC = 4096, 12288
VARIANTS = ["ring", "stream", "stream1", "stream2", "1,4", "2,4", "4,4", "dp2", "dp4", "dp8"]


@pytest.fixture
def variant(request):
    old = os.environ.get("SDT_GEMV_VARIANT")
    os.environ["SDT_GEMV_VARIANT"] = request.param
    yield request.param
    if old is None:
        del os.environ["SDT_GEMV_VARIANT"]
    else:
        os.environ["SDT_GEMV_VARIANT"] = old


def bf16_case(K, N, seed):
    x = inputs.uniform((K,), seed=seed, dtype=torch.bfloat16)
    W = inputs.uniform((N, K), seed=seed + 1, dtype=torch.bfloat16)
    return x, W


@pytest.mark.parametrize("variant", VARIANTS, indirect=True)
def test_decode_bf16_full(cuda_device, variant):
    x, W = bf16_case(K_DEC, N_DEC, inputs.seed_for(3, 0))
    y = torch.full((N_DEC,), float("nan"), device=cuda_device)
    sdt.gemv_m1(x.to(cuda_device), W.to(cuda_device), y=y)
    sdt.check_device_status()
    assert_close(y.cpu().numpy(), oracle.gemv_bf16(u16(x), u16(W)), K_DEC, f"bf16 {variant}")


@pytest.mark.parametrize("variant", VARIANTS, indirect=True)
def test_decode_q8_full(cuda_device, variant):
    x = inputs.uniform((K_DEC,), seed=inputs.seed_for(3, 0), dtype=torch.bfloat16)
    q, s = inputs.q8_weights(N_DEC, K_DEC, seed=inputs.seed_for(3, 1))
    y = torch.full((N_DEC,), float("nan"), device=cuda_device)
    sdt.gemv_m1(x.to(cuda_device), q.to(cuda_device), s.to(cuda_device), y=y)
    sdt.check_device_status()
    ref = oracle.gemv_q8(u16(x), q.numpy(), u16(s))
    # the q8 weights carry a scale of ~5e-3: the absolute bound is met with room to spare
    assert_close(y.cpu().numpy(), ref, K_DEC, f"q8 {variant}")


def test_decode_bf16_integer_exact(cuda_device):
    x = inputs.integers((K_DEC,), seed=71, dtype=torch.bfloat16)
    W = inputs.integers((N_DEC, K_DEC), seed=72, dtype=torch.bfloat16)
    y = sdt.gemv_m1(x.to(cuda_device), W.to(cuda_device)).cpu().double().numpy()
    assert np.array_equal(y, oracle.gemv_bf16(u16(x), u16(W)))


def test_decode_q8_integer_exact(cuda_device):
    x = inputs.integers((K_DEC,), seed=73, dtype=torch.bfloat16)
    q, s = inputs.q8_weights_exact(N_DEC, K_DEC, seed=74)
    y = sdt.gemv_m1(x.to(cuda_device), q.to(cuda_device), s.to(cuda_device)).cpu().double().numpy()
    assert np.array_equal(y, oracle.gemv_q8(u16(x), q.numpy(), u16(s)))


@pytest.mark.parametrize("K,N", [(8, 5), (40, 17), (256, 1), (4096, 12291), (4104, 333), (12288, 4096)])
def test_ragged_bf16(cuda_device, K, N):
    x, W = bf16_case(K, N, 81)
    y = sdt.gemv_m1(x.to(cuda_device), W.to(cuda_device)).cpu().numpy()
    assert_close(y, oracle.gemv_bf16(u16(x), u16(W)), K, f"bf16 K={K} N={N}")


@pytest.mark.parametrize("K,N", [(32, 3), (96, 17), (4096, 12291), (4128, 65), (12288, 4096)])
def test_ragged_q8(cuda_device, K, N):
    x = inputs.uniform((K,), seed=91, dtype=torch.bfloat16)
    q, s = inputs.q8_weights(N, K, seed=92)
    y = sdt.gemv_m1(x.to(cuda_device), q.to(cuda_device), s.to(cuda_device)).cpu().numpy()
    assert_close(y, oracle.gemv_q8(u16(x), q.numpy(), u16(s)), K, f"q8 K={K} N={N}")


def test_zero_k_and_empty(cuda_device):
    x = torch.empty(0, dtype=torch.bfloat16, device=cuda_device)
    W = torch.empty((7, 0), dtype=torch.bfloat16, device=cuda_device)
    y = torch.full((7,), float("nan"), device=cuda_device)
    sdt.gemv_m1(x, W, y=y)
    torch.cuda.synchronize()
    assert bool((y == 0).all())
    W = torch.empty((0, 64), dtype=torch.bfloat16, device=cuda_device)
    assert sdt.gemv_m1(torch.zeros(64, dtype=torch.bfloat16, device=cuda_device), W).shape == (0,)


def test_rotating_buffers_each_correct(cuda_device):
    # The benchmark cycles through several weight buffers; each must give its own product.
    x = inputs.uniform((K_DEC,), seed=101, dtype=torch.bfloat16)
    xd = x.to(cuda_device)
    for i in range(3):
        W = inputs.uniform((2048, K_DEC), seed=102 + i, dtype=torch.bfloat16)
        y = sdt.gemv_m1(xd, W.to(cuda_device)).cpu().numpy()
        assert_close(y, oracle.gemv_bf16(u16(x), u16(W)), K_DEC, f"buffer {i}")


@pytest.mark.parametrize("variant", ["dp2", "dp4", "dp8"], indirect=True)
@pytest.mark.parametrize("K,N", [(32, 3), (4096, 12291), (4128, 65), (8192, 300), (12288, 4096), (16384, 77)])
def test_ragged_q8_integer_kernel(cuda_device, variant, K, N):
    # K = 32 (one group), a ragged group count, one and two groups per thread
    x = inputs.uniform((K,), seed=93, dtype=torch.bfloat16)
    q, s = inputs.q8_weights(N, K, seed=94)
    y = sdt.gemv_m1(x.to(cuda_device), q.to(cuda_device), s.to(cuda_device)).cpu().numpy()
    assert_close(y, oracle.gemv_q8(u16(x), q.numpy(), u16(s)), K, f"q8 {variant} K={K} N={N}")


def test_q8_integer_exact_large_k(cuda_device):
    # two groups per thread: still bit-exact on integer activations and power-of-two scales
    K, N = 12288, 1000
    x = inputs.integers((K,), seed=95, dtype=torch.bfloat16)
    q, s = inputs.q8_weights_exact(N, K, seed=96)
    y = sdt.gemv_m1(x.to(cuda_device), q.to(cuda_device), s.to(cuda_device)).cpu().double().numpy()
    assert np.array_equal(y, oracle.gemv_q8(u16(x), q.numpy(), u16(s)))


def test_q8_wide_dynamic_range(cuda_device):
    # activations spread over 2^-24 .. 2^24: each group is rescaled by its own power of two,
    # and an activation far below its group's largest is rounded to the group's quantum
    K, N = 4096, 2048
    g = torch.Generator().manual_seed(97)
    mag = torch.exp2(torch.randint(-24, 25, (K,), generator=g).to(torch.float32))
    x = ((torch.rand(K, generator=g) * 2 - 1) * mag).to(torch.bfloat16)
    q, s = inputs.q8_weights(N, K, seed=98)
    y = sdt.gemv_m1(x.to(cuda_device), q.to(cuda_device), s.to(cuda_device)).cpu().numpy()
    ref = oracle.gemv_q8(u16(x), q.numpy(), u16(s))
    bound = q8_rounding_bound(oracle.bf16_to_f64(u16(x)), q.numpy(), oracle.f16_to_f64(u16(s)))
    err = np.abs(y - ref)
    assert (err <= bound).all(), f"worst error / stated bound {np.max(err / bound):.3f}"
    assert np.linalg.norm(y - ref) <= 1e-3 * np.linalg.norm(ref)
    # the bound is tight enough to mean something: far inside the stated absolute bound (1e-3*sqrt(K))
    assert bound.max() <= 1e-3 * np.sqrt(K) * np.abs(ref).max()


def test_q8_weights_16_byte_aligned(cuda_device):
    # weights 16- but not 32-byte aligned take the fp32 register kernel; same result
    K, N = 4096, 513
    x = inputs.uniform((K,), seed=99, dtype=torch.bfloat16)
    q, s = inputs.q8_weights(N, K, seed=100)
    buf = torch.empty(N * K + 16, dtype=torch.int8, device=cuda_device)
    Wd = buf[16:].view(N, K)
    Wd.copy_(q.to(cuda_device))
    assert Wd.data_ptr() % 32 == 16
    y = sdt.gemv_m1(x.to(cuda_device), Wd, s.to(cuda_device)).cpu().numpy()
    assert_close(y, oracle.gemv_q8(u16(x), q.numpy(), u16(s)), K, "q8 16-byte aligned W")


@pytest.mark.parametrize("N", [12288, 1217])
def test_q8_scales_2_byte_aligned(cuda_device, N):
    # scales at an address that is 2- but not 4-byte aligned: the integer kernel loads each
    # scale's fp16 bits on their own and asks L2 for no scale rows (that needs 16 bytes);
    # integer inputs, so the result is exact.  N = 1217 leaves one CTA with two rows.
    K = 4096
    x = inputs.integers((K,), seed=103, dtype=torch.bfloat16)
    q, s = inputs.q8_weights_exact(N, K, seed=104)
    buf = torch.empty(N * (K // 32) + 1, dtype=torch.float16, device=cuda_device)
    sd = buf[1:].view(N, K // 32)
    sd.copy_(s.to(cuda_device))
    assert sd.data_ptr() % 4 == 2
    y = sdt.gemv_m1(x.to(cuda_device), q.to(cuda_device), sd).cpu().double().numpy()
    sdt.check_device_status()
    assert np.array_equal(y, oracle.gemv_q8(u16(x), q.numpy(), u16(s)))


def test_q8_nonfinite_activation_gives_nan(cuda_device):
    K, N = 4096, 64
    x = inputs.uniform((K,), seed=101, dtype=torch.bfloat16)
    x[1000] = float("inf")
    q, s = inputs.q8_weights(N, K, seed=102)
    y = sdt.gemv_m1(x.to(cuda_device), q.to(cuda_device), s.to(cuda_device)).cpu().numpy()
    assert not np.isfinite(y).any()


@pytest.mark.parametrize("variant", ["ring"], indirect=True)
@pytest.mark.parametrize("K,N", [(256, 1), (256, 5), (512, 151), (4096, 12291), (8192, 153), (16384, 300),
                                 (4352, 1000)])
def test_ragged_q8_ring_kernel(cuda_device, variant, K, N):
    # one row; fewer rows than SMs; one and two rows per CTA; a partial last stage; two and
    # four 32-byte slices per consumer thread (K 8192, 16384); K a multiple of 256 only
    x = inputs.uniform((K,), seed=121, dtype=torch.bfloat16)
    q, s = inputs.q8_weights(N, K, seed=122)
    y = sdt.gemv_m1(x.to(cuda_device), q.to(cuda_device), s.to(cuda_device)).cpu().numpy()
    sdt.check_device_status()
    assert_close(y, oracle.gemv_q8(u16(x), q.numpy(), u16(s)), K, f"q8 ring K={K} N={N}")


@pytest.mark.parametrize("variant", ["ring"], indirect=True)
@pytest.mark.parametrize("K,N", [(16, 3), (48, 1), (4096, 12291), (8192, 153), (16384, 77), (4112, 1000),
                                 (6144, 152)])
def test_ragged_bf16_ring_kernel(cuda_device, variant, K, N):
    x, W = bf16_case(K, N, 131)
    y = sdt.gemv_m1(x.to(cuda_device), W.to(cuda_device)).cpu().numpy()
    sdt.check_device_status()
    assert_close(y, oracle.gemv_bf16(u16(x), u16(W)), K, f"bf16 ring K={K} N={N}")


@pytest.mark.parametrize("variant", ["ring"], indirect=True)
def test_ring_integer_exact_and_repeatable(cuda_device, variant):
    # exact in fp32 whatever the order (integer activations, power-of-two scales), and
    # bit-identical from launch to launch (fixed summation order)
    x = inputs.integers((K_DEC,), seed=141, dtype=torch.bfloat16)
    q, s = inputs.q8_weights_exact(N_DEC, K_DEC, seed=142)
    xd, qd, sd = x.to(cuda_device), q.to(cuda_device), s.to(cuda_device)
    y1 = sdt.gemv_m1(xd, qd, sd)
    y2 = sdt.gemv_m1(xd, qd, sd)
    assert torch.equal(y1, y2)
    assert np.array_equal(y1.cpu().double().numpy(), oracle.gemv_q8(u16(x), q.numpy(), u16(s)))
    W = inputs.integers((N_DEC, K_DEC), seed=143, dtype=torch.bfloat16)
    yb = sdt.gemv_m1(xd, W.to(cuda_device)).cpu().double().numpy()
    assert np.array_equal(yb, oracle.gemv_bf16(u16(x), u16(W)))


@pytest.mark.parametrize("variant", ["ring"], indirect=True)
@pytest.mark.parametrize("ring_kb", ["36", "60", "100"])
def test_ring_depths(cuda_device, variant, ring_kb, monkeypatch):
    # rings of two stages up to the default depth (wraparound of the stage phases)
    monkeypatch.setenv("SDT_GEMV_RING_KB", ring_kb)
    x = inputs.uniform((K_DEC,), seed=151, dtype=torch.bfloat16)
    q, s = inputs.q8_weights(2048, K_DEC, seed=152)
    y = sdt.gemv_m1(x.to(cuda_device), q.to(cuda_device), s.to(cuda_device)).cpu().numpy()
    assert_close(y, oracle.gemv_q8(u16(x), q.numpy(), u16(s)), K_DEC, f"q8 ring {ring_kb} KB")
    W = inputs.uniform((2048, K_DEC), seed=153, dtype=torch.bfloat16)
    y = sdt.gemv_m1(x.to(cuda_device), W.to(cuda_device)).cpu().numpy()
    assert_close(y, oracle.gemv_bf16(u16(x), u16(W)), K_DEC, f"bf16 ring {ring_kb} KB")
    sdt.check_device_status()


@pytest.mark.parametrize("variant", ["dp2"], indirect=True)
@pytest.mark.parametrize("K,N", [(16, 3), (48, 17), (4096, 12291), (4112, 65), (8192, 300), (4104, 33)])
def test_ragged_bf16_row_range_kernel(cuda_device, variant, K, N):
    # one unit, a ragged unit count, one and two units per thread; K % 16 != 0 falls back
    x, W = bf16_case(K, N, 111)
    y = sdt.gemv_m1(x.to(cuda_device), W.to(cuda_device)).cpu().numpy()
    assert_close(y, oracle.gemv_bf16(u16(x), u16(W)), K, f"bf16 {variant} K={K} N={N}")


@pytest.mark.parametrize("variant", ["dp2"], indirect=True)
def test_bf16_row_range_integer_exact(cuda_device, variant):
    K, N = 8192, 1000
    x = inputs.integers((K,), seed=113, dtype=torch.bfloat16)
    W = inputs.integers((N, K), seed=114, dtype=torch.bfloat16)
    y = sdt.gemv_m1(x.to(cuda_device), W.to(cuda_device)).cpu().double().numpy()
    assert np.array_equal(y, oracle.gemv_bf16(u16(x), u16(W)))
