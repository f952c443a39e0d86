"""Failure detection on the GPU without a fault: a bounded wait that runs out.

The self-test kernel waits on an mbarrier that nothing arrives at, through
the same bounded-wait code every pipelined kernel uses, with a 20 ms limit.
It must give up, set the SWAB_ERR_TIMEOUT bit of the device status word and
return; afterwards the context must still run kernels correctly.
"""
import numpy as np
import pytest
import torch

import oracle
import sliding_window_attention_band_gb300 as swab
from sliding_window_attention_band_gb300 import build as swab_build

pytestmark = pytest.mark.gpu

TIMEOUT_BIT = 1 << 5  # SWAB_ERR_TIMEOUT


def test_bounded_wait_reports_timeout_and_context_survives():
    swab_build.build()
    swab.load()
    swab.device_status(reset=True)
    swab.selftest_wait_timeout(20000)
    flags = swab.device_status(reset=True)
    assert flags & TIMEOUT_BIT
    assert swab.device_status(reset=True) == 0  # the reset cleared it
    # the context still works: a small band_qk matches the oracle
    d = swab.Desc(1, 1, 300, 64, 8, 8, 0, 0.0, torch.float16)
    A, B = swab.seeded_qkvo(1, 300, 64, torch.float16, seed=3, count=2)
    S = torch.empty(1, 300, d.D, dtype=torch.float16, device="cuda")
    swab.band_qk(d, 0.125, A.cuda(), B.cuda(), S)
    ref = oracle.band_qk(A.double().numpy(), B.double().numpy(), 8, 8, 0, 0.125, 0.0)
    got = S.double().cpu().numpy()
    assert np.max(np.abs(got - ref)) <= 2e-3 * np.max(np.abs(ref))
    assert swab.device_status(reset=True) == 0
