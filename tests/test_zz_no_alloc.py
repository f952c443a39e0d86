"""The allocation-free backward entry point (band_attention_bwd_noalloc).

Some callers cannot allocate device memory (they run under an allocator they
do not control, or are handed only input and output pointers), so the library
offers a backward that keeps its per-row scratch in a module-scope device
array instead of a caller workspace.  This file checks, through the C ABI,
that two consecutive calls give the same gradients as the regular entry point
with a workspace, within the tolerance the other parity tests use.  It is
named to be collected last.
"""
import numpy as np
import pytest
import torch

import sliding_window_attention_band_gb300 as swab
from sliding_window_attention_band_gb300 import build as swab_build

pytestmark = pytest.mark.gpu

ABS_TOL = 1e-2
UNIT_ROUNDOFF = {torch.float16: 2.0 ** -11, torch.bfloat16: 2.0 ** -8}


def run_both(d, seed):
    Q, K, V, dO = (x.cuda() for x in swab.seeded_qkvo(d.BH, d.n, 64, d.dtype, seed=seed))
    O = torch.empty_like(Q)
    lse = torch.empty(d.BH, d.n, dtype=torch.float32, device="cuda")
    swab.band_attention(d, 0.125, Q, K, V, O, lse)
    ref = [torch.empty_like(Q) for _ in range(3)]
    ws = torch.empty(swab.band_attention_bwd_workspace(d) // 4, dtype=torch.float32,
                     device="cuda")
    swab.band_attention_bwd(d, 0.125, Q, K, V, O, dO, lse, *ref, ws)
    got = [torch.full_like(Q, float("nan")) for _ in range(3)]
    swab.band_attention_bwd_noalloc(d, 0.125, Q, K, V, O, dO, lse, *got)
    torch.cuda.synchronize()
    return [x.double().cpu().numpy() for x in ref], [x.double().cpu().numpy() for x in got]


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_noalloc_backward_matches_workspace_backward_twice(dtype):
    swab_build.build()
    swab.load()
    shapes = [swab.Desc(1, 3, 1000, 64, 64, 64, 0, 0.0, dtype),   # first call on the device
              swab.Desc(1, 2, 777, 64, 100, 37, 2, 0.0, dtype)]   # second call, other shape
    for k, d in enumerate(shapes):
        ref, got = run_both(d, seed=60 + k)
        for r, g in zip(ref, got):
            assert np.all(np.abs(g - r) <= ABS_TOL + UNIT_ROUNDOFF[dtype] * np.abs(r))
    assert swab.device_status(reset=True) == 0


def test_noalloc_rejects_oversized_problem():
    swab_build.build()
    swab.load()
    d = swab.Desc(1, 2, swab._binding.NOALLOC_MAX_ROWS // 2 + 1, 64, 4, 4, 0, 0.0, torch.float16)
    z = torch.zeros(1, dtype=torch.float16, device="cuda")
    import ctypes
    P = ctypes.c_void_p
    rc = swab.load().band_attention_bwd_noalloc(ctypes.byref(d.c), 0.125, *[P(z.data_ptr())] * 9,
                                                None)
    assert rc == 2  # SWAB_ERR_UNSUPPORTED, checked before any launch
