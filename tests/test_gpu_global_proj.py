"""Global queries with their own projections (ONNX Runtime issue "[WIP]
Improve LongformerAttention performance", item (3), compact global_q):
global_attention / global_attention_bwd against the fp64 oracle, and the
composition with the band path (local rows through the band calls with
global_idx, global rows replaced by the global queries' outputs; in the
backward dO's global rows zeroed for the band path) against the oracle's
composition, which is pinned to dense torch autograd.  Tolerances as in
test_gpu_parity.py."""
import numpy as np
import pytest
import torch

import oracle
import sliding_window_attention_band_gb300 as swab
from sliding_window_attention_band_gb300.inputs import WORKLOADS, seeded_qkvo

from test_gpu_globals import gpu_chain_globals
from test_gpu_parity import F32_TOL, f64, normwise, within_abs

pytestmark = [pytest.mark.gpu, pytest.mark.usefixtures("device_status_guard")]

CASES = [  # BH, n, G, dtype
    (2, 1000, 16, torch.float16),
    (3, 777, 5, torch.bfloat16),
    (1, 4096, 16, torch.float16),
    (2, 333, 17, torch.float32),   # two query chunks, the second of one query
    (1, 100, 1, torch.bfloat16),   # fewer keys than one forward chunk
    (1, 515, 40, torch.float16),
]


def ids(c):
    return f"BH{c[0]}-n{c[1]}-G{c[2]}-{str(c[3]).split('.')[-1]}"


def inputs(BH, n, G, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    mk = lambda *s: torch.randn(*s, generator=g).to(dtype)   # noqa: E731
    return mk(BH, G, 64), mk(BH, n, 64), mk(BH, n, 64), mk(BH, G, 64)


def run_global(d, scale, Qg, Kg, Vg, dOg):
    Qg, Kg, Vg, dOg = (x.cuda() for x in (Qg, Kg, Vg, dOg))
    ws = torch.empty(swab.global_attention_workspace(d) // 4 + 4, dtype=torch.float32,
                     device="cuda")
    Og = torch.empty_like(Qg)
    lseg = torch.empty(d.BH, d.G, dtype=torch.float32, device="cuda")
    swab.global_attention(d, scale, Qg, Kg, Vg, Og, lseg, ws)
    dQg, dKg, dVg = torch.empty_like(Qg), torch.empty_like(Kg), torch.empty_like(Vg)
    swab.global_attention_bwd(d, scale, Qg, Kg, Vg, Og, dOg, lseg, dQg, dKg, dVg, ws)
    torch.cuda.synchronize()
    return Og, lseg, dQg, dKg, dVg


def check(got, ref, dtype, name):
    if dtype == torch.float32:
        assert normwise(f64(got), ref) <= F32_TOL, name
    else:
        assert within_abs(f64(got), ref, dtype), name


@pytest.mark.parametrize("case", CASES, ids=ids)
def test_global_attention_unit(case):
    BH, n, G, dtype = case
    gidx = tuple(range(0, n, max(1, n // G)))[:G]
    d = swab.Desc(1, BH, n, 64, 8, 8, 0, 0.0, dtype, gidx)
    Qg, Kg, Vg, dOg = inputs(BH, n, G, dtype, seed=n + G)
    Og, lseg, dQg, dKg, dVg = run_global(d, 0.125, Qg, Kg, Vg, dOg)
    rO, rl = oracle.global_attention_fwd(f64(Qg), f64(Kg), f64(Vg), 0.125)
    rq, rk, rv = oracle.global_attention_bwd(f64(Qg), f64(Kg), f64(Vg), f64(dOg), 0.125)
    check(Og.cpu(), rO, dtype, "Og")
    np.testing.assert_allclose(f64(lseg), rl, rtol=1e-5, atol=1e-4)
    for name, got, ref in (("dQg", dQg, rq), ("dKg", dKg, rk), ("dVg", dVg, rv)):
        check(got.cpu(), ref, dtype, name)


def test_global_attention_bwd_repeatable():
    """dQg sums per-tile partials in a fixed order: two runs agree bitwise."""
    d = swab.Desc(1, 2, 2048, 64, 8, 8, 0, 0.0, torch.float16, tuple(range(16)))
    args = inputs(2, 2048, 16, torch.float16, seed=5)
    a = run_global(d, 0.125, *args)
    b = run_global(d, 0.125, *args)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def composed(d, scale, Q, K, V, dO, Qg, Kg, Vg):
    """The band path with global_idx for the local rows; global rows from the
    global queries' own projections."""
    gidx = list(d.global_idx)
    dO_local = dO.clone()
    dO_local[:, gidx] = 0
    out = gpu_chain_globals(d, Q.cuda(), K.cuda(), V.cuda(), dO_local.cuda(), scale)
    Og, lseg, dQg, dKg, dVg = run_global(d, scale, Qg, Kg, Vg, dO[:, gidx].contiguous())
    out["O"][:, gidx] = Og
    return out, dict(Og=Og, dQg=dQg, dKg=dKg, dVg=dVg)


def check_composed(d, scale, Q, K, V, dO, Qg, Kg, Vg, slices):
    band, glob = composed(d, scale, Q, K, V, dO, Qg, Kg, Vg)
    gidx = list(d.global_idx)
    sl = list(slices)
    q, k, v, go = (f64(x[sl]) for x in (Q, K, V, dO))
    rO, _ = oracle.attention_fwd(q, k, v, d.w, d.w_upper, d.dilation, scale, gidx)
    rOg, _ = oracle.global_attention_fwd(f64(Qg[sl]), f64(Kg[sl]), f64(Vg[sl]), scale)
    rO[:, gidx] = rOg
    go_local = go.copy()
    go_local[:, gidx] = 0.0
    rq, rk, rv = oracle.attention_bwd(q, k, v, go_local, d.w, d.w_upper, d.dilation, scale, gidx)
    rgq, rgk, rgv = oracle.global_attention_bwd(f64(Qg[sl]), f64(Kg[sl]), f64(Vg[sl]),
                                                go[:, gidx], scale)
    for name, got, ref in (("O", band["O"], rO), ("dQ", band["dQ"], rq), ("dK", band["dK"], rk),
                           ("dV", band["dV"], rv), ("dQg", glob["dQg"], rgq),
                           ("dKg", glob["dKg"], rgk), ("dVg", glob["dVg"], rgv)):
        check(got[sl].cpu(), ref, d.dtype, name)


def test_separate_projections_small():
    BH, n, w, gidx = 3, 1100, 64, tuple(range(16))
    d = swab.Desc(1, BH, n, 64, w, w, 0, 0.0, torch.bfloat16, gidx)
    Q, K, V, dO = seeded_qkvo(BH, n, 64, torch.bfloat16, seed=61)
    Qg, Kg, Vg, _ = inputs(BH, n, len(gidx), torch.bfloat16, seed=62)
    check_composed(d, 0.125, Q, K, V, dO, Qg, Kg, Vg, range(BH))


def test_separate_projections_training_workload_sampled():
    """b = 12, h = 12, n = 4096, w = 256, 16 global tokens (positions 0..15),
    bf16, with separate global projections (slices 0 and 77 compared)."""
    wl = WORKLOADS[4]
    d = swab.Desc.from_workload(wl)
    g = torch.Generator().manual_seed(4004)
    mk = lambda *s: torch.randn(*s, generator=g).to(wl.dtype)   # noqa: E731
    Q, K, V, dO = (mk(wl.BH, wl.n, 64) for _ in range(4))
    Qg, Kg, Vg = mk(wl.BH, d.G, 64), mk(wl.BH, wl.n, 64), mk(wl.BH, wl.n, 64)
    check_composed(d, wl.scale, Q, K, V, dO, Qg, Kg, Vg, (0, 77))
