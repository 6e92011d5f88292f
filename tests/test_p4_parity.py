"""The GEMM problem matrix of "Iteratively Tuning hipBLASLt TensileLite Kernels"
("Experiment Setup": 24 shapes, fp16 / bf16, NN / TN) through gemm_ex with the
library's pick, and through configurations the coordinate-descent tuner adopts,
against the fp64 oracle on sampled rows of C."""
import numpy as np
import pytest
import torch

import oracle
import shape_driven_tile_gb300 as sdt
from shape_driven_tile_gb300 import inputs, tune
from _parity import assert_close, assert_close_bf16, u16

pytestmark = pytest.mark.gpu

SHAPES = {s[0]: s[1:] for s in inputs.P4_SHAPES}
SMALL = ["sn_16_dec", "sn_32_dec", "sn_128_dec", "sqS", "sn_16_pf", "sn_64_pf", "d4k_qkv_dec", "sqL"]
CASES = ([(n, "f16", "NN") for n in SHAPES] + [(n, "bf16", "TN") for n in SHAPES]
         + [(n, d, l) for n in SMALL for d, l in (("f16", "TN"), ("bf16", "NN"))])
DT = {"f16": torch.float16, "bf16": torch.bfloat16}


def sample_rows(M, seed):
    rng = np.random.default_rng(seed)
    rows = {0, M - 1, M // 2, min(M - 1, 63), min(M - 1, 64), min(M - 1, 127), min(M - 1, 128)}
    rows.update(int(r) for r in rng.integers(0, M, 5))
    return np.array(sorted(rows), dtype=np.int64)


def problem(name, dt, layout, dev):
    M, N, K = SHAPES[name]
    dtype = DT[dt]
    A_h, B_h = inputs.p4_operands(M, N, K, layout, seed=900 + 7 * len(name), dtype=dtype)
    A = A_h.to(dev)
    B = B_h.to(dev) if layout == "NN" else B_h.to(dev).t()
    B_logical = B_h if layout == "NN" else B_h.t().contiguous()
    return M, N, K, A, B, A_h, B_logical


def check(C, A_h, B_logical, K, dt, what, seed=0):
    rows = sample_rows(A_h.shape[0], seed)
    ref = oracle.gemm(u16(A_h), u16(B_logical), rows=rows, dtype=dt)
    got = C.cpu()[torch.from_numpy(rows)].double().numpy()
    (assert_close if dt == "f16" else assert_close_bf16)(got, ref, K, what)


@pytest.mark.parametrize("name,dt,layout", CASES, ids=[f"{n}-{d}-{l}" for n, d, l in CASES])
def test_p4_problem_pick(cuda_device, name, dt, layout):
    M, N, K, A, B, A_h, B_logical = problem(name, dt, layout, cuda_device)
    C = torch.full((M, N), float("nan"), dtype=DT[dt], device=cuda_device)
    sdt.gemm_ex(A, B, C)
    sdt.check_device_status()
    check(C, A_h, B_logical, K, dt, f"{name} {dt} {layout} pick")


@pytest.mark.parametrize("name,dt,layout", [("sqS", "f16", "NN"), ("sn_64_pf", "f16", "NN"),
                                            ("d4k_qkv_dec", "bf16", "TN"), ("thinK", "f16", "NN")])
def test_tuned_configuration_matches_oracle(cuda_device, name, dt, layout):
    # the descent's held latency never rises, and what it adopts computes the same product
    M, N, K, A, B, A_h, B_logical = problem(name, dt, layout, cuda_device)
    C = torch.empty((M, N), dtype=DT[dt], device=cuda_device)
    prob = tune.GemmProblem(A, B, C, reps=3)
    held, traj = prob.tune()
    us = [t["us"] for t in traj]
    assert all(b <= a for a, b in zip(us, us[1:])), us
    C.fill_(float("nan"))
    prob.launcher(held)()
    sdt.check_device_status()
    check(C, A_h, B_logical, K, dt, f"{name} {dt} {layout} tuned {held}")
