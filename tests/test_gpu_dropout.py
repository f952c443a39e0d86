"""Dropout of the attention probabilities in the fused forward and backward
(nvFuser issue "HuggingFace BertForMaskedLM - Log Softmax Fusion with Autocast
has bad perf", fusion 1: probabilities dropped with probability p, the kept
ones scaled by 1/(1-p)), the keep decisions drawn from Philox4x64-10, against
the fp64 oracle that draws them the same way.

The keep decision of (slice, query, key) depends on the slice number, so the
oracle always sees every slice of the batch; only the comparison is sampled.
"""
import numpy as np
import pytest
import torch

import oracle
import sliding_window_attention_band_gb300 as swab
from sliding_window_attention_band_gb300.inputs import WORKLOADS, seeded_qkvo, workload_inputs

from test_gpu_key_bias import make_bias, per_slice
from test_gpu_parity import F32_TOL, empty_dense, f64, normwise, within_abs

pytestmark = [pytest.mark.gpu, pytest.mark.usefixtures("device_status_guard")]

CASES = [  # b, h, n, w, w_upper, dilation, dtype, with key bias
    (2, 2, 700, 64, 64, 0, torch.float16, False),
    (1, 3, 777, 100, 37, 2, torch.bfloat16, False),
    (2, 1, 1100, 300, 0, 0, torch.float16, True),
    (1, 2, 515, 3, 3, 3, torch.float16, True),
    (1, 2, 640, 45, 70, 1, torch.bfloat16, True),
    (2, 2, 333, 7, 30, 2, torch.float32, False),
    (1, 2, 300, 40, 9, 0, torch.float32, True),
]


def ids(c):
    return (f"b{c[0]}h{c[1]}-n{c[2]}-w{c[3]}-wu{c[4]}-d{c[5]}-{str(c[6]).split('.')[-1]}"
            f"{'-bias' if c[7] else ''}")


def run_pair(d, Q, K, V, dO, scale):
    q, k, v, go = (x.cuda() for x in (Q, K, V, dO))
    O = empty_dense(d)
    lse = torch.empty((d.BH, d.n), dtype=torch.float32, device="cuda")
    swab.band_attention(d, scale, q, k, v, O, lse)
    dQ, dK, dV = (empty_dense(d) for _ in range(3))
    ws = torch.empty(swab.band_attention_bwd_workspace(d) // 4, dtype=torch.float32, device="cuda")
    ws.fill_(float("nan"))
    swab.band_attention_bwd(d, scale, q, k, v, O, go, lse, dQ, dK, dV, ws)
    torch.cuda.synchronize()
    return O, lse, dQ, dK, dV


def check_dropout(b, h, n, w, wu, dil, dtype, Q, K, V, dO, bias, p, seed, slices):
    d = swab.Desc(b, h, n, 64, w, wu, dil, 0.0, dtype,
                  key_bias=bias.cuda() if bias is not None else None, dropout_p=p,
                  dropout_seed=seed)
    scale = 0.125
    O, lse, dQ, dK, dV = run_pair(d, Q, K, V, dO, scale)
    args = dict(key_bias=per_slice(bias, h) if bias is not None else None, drop_t=d.drop_t,
                seed=seed)
    refO, reflse = oracle.attention_fwd(f64(Q), f64(K), f64(V), w, wu, dil, scale, **args)
    refs = oracle.attention_bwd(f64(Q), f64(K), f64(V), f64(dO), w, wu, dil, scale, **args)
    sl = list(slices)
    np.testing.assert_allclose(lse[sl].cpu().double().numpy(), reflse[sl], rtol=1e-4, atol=2e-3)
    for name, got, ref in (("O", O, refO), ("dQ", dQ, refs[0]), ("dK", dK, refs[1]),
                           ("dV", dV, refs[2])):
        g_ = f64(got[sl].cpu())
        if dtype == torch.float32:
            assert normwise(g_, ref[sl]) <= F32_TOL, name
        else:
            assert within_abs(g_, ref[sl], dtype), name


@pytest.mark.parametrize("case", CASES, ids=ids)
def test_fused_dropout(case):
    b, h, n, w, wu, dil, dtype, with_bias = case
    Q, K, V, dO = seeded_qkvo(b * h, n, 64, dtype, seed=n + 11)
    bias = make_bias(b, n, seed=n + 12) if with_bias else None
    check_dropout(b, h, n, w, wu, dil, dtype, Q, K, V, dO, bias, 0.1, 987654321 + n,
                  range(b * h))


def test_dropout_high_p():
    """p = 0.9 (threshold byte 230): most probabilities dropped."""
    Q, K, V, dO = seeded_qkvo(2, 520, 64, torch.float16, seed=77)
    check_dropout(1, 2, 520, 64, 64, 0, torch.float16, Q, K, V, dO, None, 0.9, 2**63 + 5,
                  range(2))


def test_dropout_zero_is_no_dropout():
    """p = 0 gives bitwise the results of a descriptor without dropout."""
    Q, K, V, dO = seeded_qkvo(2, 600, 64, torch.float16, seed=3)
    outs = []
    for kw in ({}, {"dropout_p": 0.0, "dropout_seed": 5}):
        d = swab.Desc(1, 2, 600, 64, 64, 64, 0, 0.0, torch.float16, **kw)
        outs.append([t.cpu() for t in run_pair(d, Q, K, V, dO, 0.125)[:2]])
    for a, b_ in zip(*outs):
        assert torch.equal(a, b_)


def test_dropout_seed_changes_mask():
    """Two seeds give different outputs and the same lse (lse is pre-dropout)."""
    Q, K, V, dO = seeded_qkvo(2, 600, 64, torch.float16, seed=4)
    res = []
    for seed in (1, 2):
        d = swab.Desc(1, 2, 600, 64, 64, 64, 0, 0.0, torch.float16, dropout_p=0.2,
                      dropout_seed=seed)
        res.append([t.cpu() for t in run_pair(d, Q, K, V, dO, 0.125)[:2]])
    assert not torch.equal(res[0][0], res[1][0])
    assert torch.equal(res[0][1], res[1][1])


def test_dropout_workload():
    """The n=4096, w=256 fp16 workload with p = 0.1 (slices 0 and 7 compared)."""
    wl = WORKLOADS[2]
    Q, K, V, dO = workload_inputs(wl)
    check_dropout(wl.b, wl.h, wl.n, wl.w, wl.w_upper, wl.dilation, wl.dtype, Q, K, V, dO, None,
                  0.1, 42, (0, 7))


@pytest.mark.parametrize("case", [c for c in CASES if c[6] != torch.float32], ids=ids)
def test_dropout_keep_bit_cache(case):
    """With the keep-bit cache the forward stores the bits it draws and the
    backward reads them instead of drawing them: O, lse, dK, dV are bitwise
    those of the run without the cache (whose parity test_fused_dropout
    checks), dQ within the rounding of its run-to-run accumulation order."""
    b, h, n, w, wu, dil, dtype, with_bias = case
    Q, K, V, dO = seeded_qkvo(b * h, n, 64, dtype, seed=n + 21)
    bias = make_bias(b, n, seed=n + 22).cuda() if with_bias else None
    kw = dict(key_bias=bias, dropout_p=0.15, dropout_seed=4242 + n)
    plain = swab.Desc(b, h, n, 64, w, wu, dil, 0.0, dtype, **kw)
    mask = torch.full((swab.band_attention_dropout_mask_bytes(plain) // 4,), -1, dtype=torch.int32,
                      device="cuda")   # every bit set: the forward must write what is read
    cached = swab.Desc(b, h, n, 64, w, wu, dil, 0.0, dtype, dropout_mask=mask, **kw)
    r0 = run_pair(plain, Q, K, V, dO, 0.125)
    r1 = run_pair(cached, Q, K, V, dO, 0.125)
    for name, x0, x1 in zip(("O", "lse", "dQ", "dK", "dV"), r0, r1):
        if name == "dQ":
            torch.testing.assert_close(x1.float(), x0.float(), rtol=1e-2, atol=1e-3)
        else:
            assert torch.equal(x0, x1), name
