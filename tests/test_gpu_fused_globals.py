"""The fused forward with global tokens (ONNX Runtime issue "[WIP] Improve
LongformerAttention performance", item (1)): band_attention gives the same O
and lse as the attention with global tokens on explicit key sets (the fp64
oracle) -- local rows over their band keys outside G plus G, global rows over
every key.  Tolerances as in test_gpu_parity.py."""
import numpy as np
import pytest
import torch

import oracle
import sliding_window_attention_band_gb300 as swab
from sliding_window_attention_band_gb300.inputs import WORKLOADS, seeded_qkvo, workload_inputs

from test_gpu_parity import f64, within_abs

pytestmark = [pytest.mark.gpu, pytest.mark.usefixtures("device_status_guard")]

CASES = [  # BH, n, w, w_upper, dilation, dtype, global idx
    (2, 1000, 64, 64, 0, torch.float16, (0, 1, 7, 500, 999)),
    (3, 777, 100, 37, 2, torch.bfloat16, (3, 20, 21, 400)),
    (1, 640, 0, 127, 1, torch.float16, tuple(range(16))),
    (2, 515, 3, 3, 3, torch.float16, (64,)),
    (1, 1100, 300, 300, 0, torch.bfloat16, tuple(range(0, 1100, 37))),
]


def ids(c):
    return f"BH{c[0]}-n{c[1]}-w{c[2]}-wu{c[3]}-d{c[4]}-{str(c[5]).split('.')[-1]}-G{len(c[6])}"


def run(d, Q, K, V, scale):
    O = torch.empty(d.BH, d.n, 64, dtype=d.dtype, device="cuda")
    lse = torch.empty(d.BH, d.n, dtype=torch.float32, device="cuda")
    swab.band_attention(d, scale, Q.cuda(), K.cuda(), V.cuda(), O, lse)
    torch.cuda.synchronize()
    return O, lse


def check(d, Q, K, V, scale, slices):
    O, lse = run(d, Q, K, V, scale)
    sl = list(slices)
    rO, rl = oracle.attention_fwd(f64(Q[sl]), f64(K[sl]), f64(V[sl]), d.w, d.w_upper, d.dilation,
                                  scale, list(d.global_idx))
    assert within_abs(f64(O[sl].cpu()), rO, d.dtype)
    np.testing.assert_allclose(f64(lse[sl].cpu()), rl, rtol=1e-4, atol=2e-3)


@pytest.mark.parametrize("case", CASES, ids=ids)
def test_fused_forward_globals(case):
    BH, n, w, wu, dil, dtype, gidx = case
    d = swab.Desc(1, BH, n, 64, w, wu, dil, 0.0, dtype, gidx)
    Q, K, V, _ = seeded_qkvo(BH, n, 64, dtype, seed=n + 71)
    check(d, Q, K, V, 0.125, range(BH))


# enough (16-query chunk, slice) pairs to fill the GPU, so the dense global
# rows run on the tensor-core kernel: ragged key tails (777 = 6 x 128 + 9,
# 129 = 128 + 1), a single key chunk (n = 50), a partial last query chunk
# (G = 21) and four query chunks (G = 63); three slices checked
TC_ROWS_CASES = [
    (80, 777, 100, 37, 2, torch.bfloat16, (0, 3, 20, 21, 400) + tuple(range(500, 776, 18))),
    (96, 129, 0, 0, 0, torch.float16, (0, 128)),
    (100, 50, 10, 10, 0, torch.float16, (3, 49)),
    (24, 1000, 64, 64, 0, torch.float16, tuple(range(0, 1000, 16))[:64]),
]


@pytest.mark.parametrize("case", TC_ROWS_CASES, ids=ids)
def test_fused_forward_globals_tensor_core_rows(case):
    BH, n, w, wu, dil, dtype, gidx = case
    assert 2 * ((len(gidx) + 15) // 16) * BH >= torch.cuda.get_device_properties(0).multi_processor_count
    d = swab.Desc(1, BH, n, 64, w, wu, dil, 0.0, dtype, gidx)
    Q, K, V, _ = seeded_qkvo(BH, n, 64, dtype, seed=n + 5)
    check(d, Q, K, V, 0.125, (0, BH // 2 + 1, BH - 1))


def test_fused_forward_globals_matches_materialised():
    """The fused forward and the materialised chain agree with global tokens."""
    BH, n, gidx = 2, 900, (0, 5, 450, 899)
    d = swab.Desc(1, BH, n, 64, 128, 128, 0, 0.0, torch.float16, gidx)
    Q, K, V, _ = (x.cuda() for x in seeded_qkvo(BH, n, 64, torch.float16, seed=3))
    O, lse = run(d, Q, K, V, 0.125)
    S = torch.empty(BH, n, d.D, dtype=torch.float16, device="cuda")
    Sg = (torch.empty(BH, n, d.G, dtype=torch.float16, device="cuda"),
          torch.empty(BH, d.G, n, dtype=torch.float16, device="cuda"))
    Pg = tuple(torch.empty_like(x) for x in Sg)
    P = torch.empty_like(S)
    O2 = torch.empty_like(O)
    lse2 = torch.empty_like(lse)
    swab.band_qk(d, 0.125, Q, K, S, Sg)
    swab.band_softmax(d, S, P, lse2, Sg=Sg, Pg=Pg)
    swab.band_pv(d, 1.0, P, V, O2, Pg=Pg)
    torch.cuda.synchronize()
    assert float((O.float() - O2.float()).abs().max()) <= 1e-2
    assert float((lse - lse2).abs().max()) <= 2e-3


def test_fused_forward_globals_training_workload_sampled():
    """b = 12, h = 12, n = 4096, w = 256, 16 global tokens, bf16 (slices 0, 77, 143)."""
    wl = WORKLOADS[4]
    Q, K, V = workload_inputs(wl, count=3)
    check(swab.Desc.from_workload(wl), Q, K, V, wl.scale, (0, 77, 143))


# ---------------------------------------------------------------------------
# the fused backward with global tokens: band_attention_bwd gives the dQ, dK,
# dV of the attention with global tokens on explicit key sets (the fp64
# oracle's scatter) -- the band with global keys and queries left out, the
# global columns and the global rows
# ---------------------------------------------------------------------------
def run_bwd(d, Q, K, V, dO, scale):
    q, k, v, go = (x.cuda() for x in (Q, K, V, dO))
    O = torch.empty_like(q)
    lse = torch.empty(d.BH, d.n, dtype=torch.float32, device="cuda")
    swab.band_attention(d, scale, q, k, v, O, lse)
    dQ, dK, dV = (torch.full_like(q, float("nan")) for _ in range(3))
    ws = torch.empty(swab.band_attention_bwd_workspace(d) // 4, dtype=torch.float32, device="cuda")
    ws.fill_(float("nan"))  # contents on entry must not matter
    swab.band_attention_bwd(d, scale, q, k, v, O, go, lse, dQ, dK, dV, ws)
    torch.cuda.synchronize()
    return dQ, dK, dV


def check_bwd(d, Q, K, V, dO, scale, slices):
    dQ, dK, dV = run_bwd(d, Q, K, V, dO, scale)
    for b in slices:
        sl = slice(b, b + 1)
        refs = oracle.attention_bwd(f64(Q[sl]), f64(K[sl]), f64(V[sl]), f64(dO[sl]), d.w, d.w_upper,
                                    d.dilation, scale, list(d.global_idx))
        for name, got, ref in (("dQ", dQ, refs[0]), ("dK", dK, refs[1]), ("dV", dV, refs[2])):
            assert within_abs(f64(got[sl].cpu()), ref, d.dtype), (name, b)


@pytest.mark.parametrize("case", CASES, ids=ids)
def test_fused_backward_globals(case):
    BH, n, w, wu, dil, dtype, gidx = case
    d = swab.Desc(1, BH, n, 64, w, wu, dil, 0.0, dtype, gidx)
    Q, K, V, dO = seeded_qkvo(BH, n, 64, dtype, seed=n + 91)
    check_bwd(d, Q, K, V, dO, 0.125, range(BH))


def test_fused_backward_globals_more_than_128():
    """G = 150 global tokens: the global columns take two tiles of gathered
    keys per slice (the second one ragged); with dilation."""
    BH, n, gidx = 2, 900, tuple(range(0, 900, 6))
    assert len(gidx) == 150
    d = swab.Desc(1, BH, n, 64, 40, 40, 1, 0.0, torch.float16, gidx)
    Q, K, V, dO = seeded_qkvo(BH, n, 64, torch.float16, seed=17)
    check_bwd(d, Q, K, V, dO, 0.125, range(BH))


def test_fused_globals_largest_count():
    """G = 256 global tokens (the largest count), dilated: the forward's
    global columns and rows off the tensor-core paths' limits, the backward's
    global columns as two tiles of gathered keys."""
    BH, n, gidx = 2, 700, tuple(range(0, 512, 2))
    assert len(gidx) == swab._binding.MAX_GLOBAL
    d = swab.Desc(1, BH, n, 64, 24, 40, 1, 0.0, torch.bfloat16, gidx)
    Q, K, V, dO = seeded_qkvo(BH, n, 64, torch.bfloat16, seed=19)
    check(d, Q, K, V, 0.125, range(BH))
    check_bwd(d, Q, K, V, dO, 0.125, range(BH))


def test_fused_backward_globals_training_workload_sampled():
    """b = 12, h = 12, n = 4096, w = 256, 16 global tokens, bf16 (slices 0, 77, 143)."""
    wl = WORKLOADS[4]
    Q, K, V, dO = workload_inputs(wl)
    check_bwd(swab.Desc.from_workload(wl), Q, K, V, dO, wl.scale, (0, 77, 143))
