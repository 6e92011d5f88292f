"""Bounded waits: a kernel that waits on a barrier nothing arrives at gives up,
records its site in the status word and returns; the context stays usable."""
import pytest
import torch

import shape_driven_tile_gb300 as sdt
from shape_driven_tile_gb300 import inputs

pytestmark = pytest.mark.gpu


def test_timeout_probe_reports_and_clears(cuda_device):
    sdt.check_device_status()  # clean start
    sdt.debug_timeout_probe(20_000)  # 20 ms limit on a barrier nothing arrives at
    with pytest.raises(sdt.SdtError) as e:
        sdt.check_device_status()
    assert e.value.status == "SDT_ERR_TIMEOUT"
    assert e.value.where & 0xF == 5
    sdt.check_device_status()  # the word was cleared by the read
    # the context is still usable
    A = inputs.integers((256, 256), seed=1).to(cuda_device)
    C = sdt.gemm_f16(A, A)
    sdt.check_device_status()
    assert bool(torch.isfinite(C).all())


def test_probe_limit_validated(cuda_device):
    with pytest.raises(sdt.SdtError):
        sdt.debug_timeout_probe(0)
