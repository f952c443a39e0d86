"""The allocation-free backward entry point (band_attention_bwd_noalloc).

Some callers cannot allocate device memory (they run under an allocator they
do not control, or are handed only input and output pointers), so the library
offers a backward that keeps its per-row scratch in a module-scope device
array instead of a caller workspace.  This file checks, through the C ABI,
that two consecutive calls (the first one on the device, then one of another
shape) give the same gradients as the regular entry point with a workspace and
as the fp64 oracle, within the tolerances the other parity tests use, and that
a repeated call on the same inputs gives bitwise the same gradients.  It is
named to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import sliding_window_attention_band_gb300 as swab
from sliding_window_attention_band_gb300 import build as swab_build

pytestmark = pytest.mark.gpu

ABS_TOL = 1e-2
F32_TOL = 1e-5


def abs_bound(ref, dtype):
    """The chained-output bound of the parity tests: plain 1e-2 for fp16, plus
    one output rounding (2^-8 |ref|) for bf16."""
    return ABS_TOL + (2.0 ** -8 * np.abs(ref) if dtype == torch.bfloat16 else 0.0)


def f64(t):
    return t.double().cpu().numpy()


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
    again = [torch.full_like(Q, float("nan")) for _ in range(3)]
    swab.band_attention_bwd_noalloc(d, 0.125, Q, K, V, O, dO, lse, *again)
    torch.cuda.synchronize()
    orc = oracle.attention_bwd(*(f64(x) for x in (Q, K, V, dO)), d.w, d.w_upper, d.dilation, 0.125)
    return [f64(x) for x in ref], [f64(x) for x in got], [f64(x) for x in again], orc


def normwise(got, ref):
    den = np.max(np.abs(ref))
    return float(np.max(np.abs(got - ref)) / (den if den > 0 else 1.0))


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16, torch.float32])
def test_noalloc_backward_matches_workspace_backward_and_oracle_twice(dtype):
    swab_build.build()
    swab.load()
    shapes = [swab.Desc(1, 3, 1000, 64, 64, 64, 0, 0.0, dtype),   # first call on the device
              swab.Desc(1, 2, 777, 64, 100, 37, 2, 0.0, dtype)]   # second call, other shape
    for k, d in enumerate(shapes):
        ref, got, again, orc = run_both(d, seed=60 + k)
        for name, r, g, a, o in zip(("dQ", "dK", "dV"), ref, got, again, orc):
            # the same call on the same inputs repeats bitwise (one writer per row)
            np.testing.assert_array_equal(a, g, err_msg=name)
            if dtype == torch.float32:
                assert normwise(g, o) <= F32_TOL, name
                assert normwise(g, r) <= F32_TOL, name
            else:
                assert np.all(np.abs(g - o) <= abs_bound(o, dtype)), name
                # both entry points are within the bound of the oracle, so of
                # each other within twice it
                assert np.all(np.abs(g - r) <= 2 * abs_bound(o, dtype)), name
    assert swab.device_status(reset=True) == 0


def test_noalloc_rejects_oversized_problem():
    swab_build.build()
    swab.load()
    d = swab.Desc(1, 2, swab._binding.NOALLOC_MAX_ROWS // 2 + 1, 64, 4, 4, 0, 0.0, torch.float16)
    z = torch.zeros(1, dtype=torch.float16, device="cuda")
    P = ctypes.c_void_p
    rc = swab.load().band_attention_bwd_noalloc(ctypes.byref(d.c), 0.125, *[P(z.data_ptr())] * 9,
                                                None)
    assert rc == 2  # SWAB_ERR_UNSUPPORTED, checked before any launch
