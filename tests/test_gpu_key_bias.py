"""Key-padding bias on the GPU: (1 - mask) * -10000 per key added to the scaled
scores before the softmax (nvFuser issue "HuggingFace BertForMaskedLM - Log
Softmax Fusion with Autocast has bad perf", fusion 1), in band_softmax and the
fused forward and backward, against the fp64 oracle -- also together with
global tokens (ONNX Runtime issue "[WIP] Improve LongformerAttention
performance", item (1)), where it applies to every key a row attends to."""
import numpy as np
import pytest
import torch

import oracle
import sliding_window_attention_band_gb300 as swab
from sliding_window_attention_band_gb300.inputs import WORKLOADS, seeded_qkvo, workload_inputs

from test_gpu_parity import F32_TOL, empty_dense, f64, normwise, within_abs

pytestmark = [pytest.mark.gpu, pytest.mark.usefixtures("device_status_guard")]

CASES = [  # b, h, n, w, w_upper, dilation, dtype
    (2, 2, 700, 64, 64, 0, torch.float16),
    (1, 3, 777, 100, 37, 2, torch.bfloat16),
    (2, 1, 1100, 300, 0, 0, torch.float16),
    (1, 2, 515, 3, 3, 3, torch.float16),
    (2, 2, 333, 7, 30, 2, torch.float32),
]


def ids(c):
    return f"b{c[0]}h{c[1]}-n{c[2]}-w{c[3]}-wu{c[4]}-d{c[5]}-{str(c[6]).split('.')[-1]}"


def make_bias(b, n, seed):
    """(1 - mask) * -10000 for a seeded 0/1 key mask (a quarter of the keys
    masked) plus a small seeded per-key term; [b, n] fp32."""
    g = torch.Generator().manual_seed(seed)
    keep = torch.rand(b, n, generator=g) > 0.25
    return torch.where(keep, 0.0, -10000.0) + 0.3 * torch.randn(b, n, generator=g)


def per_slice(bias, h):
    """[b, n] -> [b*h, n] (the bias is shared by the heads of a batch)."""
    return bias.repeat_interleave(h, dim=0).double().numpy()


@pytest.mark.parametrize("case", CASES, ids=ids)
def test_band_softmax_key_bias(case):
    b, h, n, w, wu, dil, dtype = case
    bias = make_bias(b, n, seed=n)
    d = swab.Desc(b, h, n, 64, w, wu, dil, 0.0, dtype, key_bias=bias.cuda())
    S = (torch.randn(b * h, n, d.D, generator=torch.Generator().manual_seed(n + 1)) * 2).to(dtype)
    P = torch.empty_like(S, device="cuda")
    lse = torch.empty(b * h, n, dtype=torch.float32, device="cuda")
    swab.band_softmax(d, S.cuda(), P, lse)
    torch.cuda.synchronize()
    refP, reflse = oracle.band_softmax(f64(S), w, wu, dil, key_bias=per_slice(bias, h))
    s = dil + 1
    i = np.arange(n)[:, None]
    t = np.arange(d.D)[None, :]
    j = i + (t - w) * s
    valid = (j >= 0) & (j < n)
    got = f64(P.cpu())
    if dtype == torch.float32:
        assert normwise(got[:, valid], refP[:, valid]) <= F32_TOL
    else:
        assert within_abs(got[:, valid], refP[:, valid], dtype)
    np.testing.assert_allclose(lse.cpu().double().numpy(), reflse, rtol=1e-4, atol=2e-3)


def check_fused_bias(b, h, n, w, wu, dil, dtype, Q, K, V, dO, bias, slices, gidx=None):
    d = swab.Desc(b, h, n, 64, w, wu, dil, 0.0, dtype, global_idx=gidx, key_bias=bias.cuda())
    gi = list(gidx) if gidx else None
    q, k, v, go = (x.cuda() for x in (Q, K, V, dO))
    scale = 0.125
    O = empty_dense(d)
    lse = torch.empty((d.BH, n), dtype=torch.float32, device="cuda")
    swab.band_attention(d, scale, q, k, v, O, lse)
    dQ, dK, dV = (empty_dense(d) for _ in range(3))
    ws = torch.empty(swab.band_attention_bwd_workspace(d) // 4, dtype=torch.float32, device="cuda")
    ws.fill_(float("nan"))
    swab.band_attention_bwd(d, scale, q, k, v, O, go, lse, dQ, dK, dV, ws)
    torch.cuda.synchronize()
    kb = per_slice(bias, h)
    for sl_i in slices:
        sl = slice(sl_i, sl_i + 1)
        refO, reflse = oracle.attention_fwd(f64(Q[sl]), f64(K[sl]), f64(V[sl]), w, wu, dil, scale,
                                            global_idx=gi, key_bias=kb[sl])
        refs = oracle.attention_bwd(f64(Q[sl]), f64(K[sl]), f64(V[sl]), f64(dO[sl]), w, wu, dil,
                                    scale, global_idx=gi, key_bias=kb[sl])
        np.testing.assert_allclose(lse[sl].cpu().double().numpy(), reflse, rtol=1e-4, atol=2e-3)
        for name, got, ref in (("O", O, refO), ("dQ", dQ, refs[0]), ("dK", dK, refs[1]),
                               ("dV", dV, refs[2])):
            g_ = f64(got[sl].cpu())
            if dtype == torch.float32:
                assert normwise(g_, ref) <= F32_TOL, name
            else:
                assert within_abs(g_, ref, dtype), name


@pytest.mark.parametrize("case", CASES, ids=ids)
def test_fused_key_bias(case):
    b, h, n, w, wu, dil, dtype = case
    Q, K, V, dO = seeded_qkvo(b * h, n, 64, dtype, seed=n + 7)
    check_fused_bias(b, h, n, w, wu, dil, dtype, Q, K, V, dO, make_bias(b, n, seed=n + 8),
                     range(b * h))


def test_fused_key_bias_workload():
    """The n=4096, w=256 fp16 workload with a quarter of the keys masked."""
    wl = WORKLOADS[2]
    Q, K, V, dO = workload_inputs(wl)
    check_fused_bias(wl.b, wl.h, wl.n, wl.w, wl.w_upper, wl.dilation, wl.dtype, Q, K, V, dO,
                     make_bias(wl.b, wl.n, seed=4096), (0, 7))


GLOBAL_CASES = [  # b, h, n, w, w_upper, dilation, dtype, global idx
    # few global tokens: global columns on the tensor cores, rows on FFMA
    (2, 2, 700, 64, 64, 0, torch.float16, (0, 1, 350, 699)),
    # more than 64: global columns on FFMA; dilated
    (1, 3, 777, 100, 37, 2, torch.bfloat16, tuple(range(0, 777, 9))),
    # enough (16-query chunk, slice) pairs for the tensor-core global rows
    (12, 2, 600, 32, 32, 0, torch.float16, tuple(range(0, 600, 9))[:64]),
]


def gids(c):
    return ids(c[:7]) + f"-G{len(c[7])}"


@pytest.mark.parametrize("case", GLOBAL_CASES, ids=gids)
def test_fused_key_bias_with_globals(case):
    b, h, n, w, wu, dil, dtype, gidx = case
    Q, K, V, dO = seeded_qkvo(b * h, n, 64, dtype, seed=n + 9)
    slices = range(b * h) if b * h <= 6 else (0, b * h // 2, b * h - 1)
    check_fused_bias(b, h, n, w, wu, dil, dtype, Q, K, V, dO, make_bias(b, n, seed=n + 10), slices, gidx)


def test_fused_key_bias_with_globals_training_workload_sampled():
    """b = 12, h = 12, n = 4096, w = 256, 16 global tokens, bf16, with a quarter
    of the keys masked (a padded batch): slices 0, 77, 143."""
    wl = WORKLOADS[4]
    Q, K, V, dO = workload_inputs(wl)
    check_fused_bias(wl.b, wl.h, wl.n, wl.w, wl.w_upper, wl.dilation, wl.dtype, Q, K, V, dO,
                     make_bias(wl.b, wl.n, seed=4097), (0, 77, 143), wl.global_idx)
