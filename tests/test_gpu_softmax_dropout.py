"""Dropout in the materialised path: band_softmax_dropout writes the
probabilities P and the dropped, rescaled Pd (nvFuser issue "HuggingFace
BertForMaskedLM - Log Softmax Fusion with Autocast has bad perf", fusion 1,
outputs both), band_softmax_bwd takes P and the gradient of Pd.  Against the
fp64 oracle, which draws the same Philox4x64-10 keep bytes.  The keep
pattern is compared exactly (a wrong bit on a small probability would hide
inside an absolute tolerance)."""
import numpy as np
import pytest
import torch

import oracle
import sliding_window_attention_band_gb300 as swab
from sliding_window_attention_band_gb300.inputs import (WORKLOADS, seeded_band, seeded_qkvo,
                                                        workload_inputs)

from test_gpu_key_bias import make_bias, per_slice
from test_gpu_parity import (ABS_TOL, F32_TOL, UNIT_CASES, empty_band, empty_dense, f64,
                             normwise, poison_invalid, score_tol, unit_ids, valid_mask,
                             within_abs)

pytestmark = [pytest.mark.gpu, pytest.mark.usefixtures("device_status_guard")]

P_DROP = 0.1
SEED = 0x5EED1234ABCD


def ddesc(BH, n, w, wu, dil, dtype, bias=None, p=P_DROP):
    return swab.Desc(1, BH, n, 64, w, wu, dil, 0.0, dtype, dropout_p=p, dropout_seed=SEED,
                     key_bias=bias.cuda() if bias is not None else None)


@pytest.mark.parametrize("with_bias", [False, True], ids=["", "bias"])
@pytest.mark.parametrize("case", UNIT_CASES, ids=unit_ids)
def test_band_softmax_dropout_unit(case, with_bias):
    BH, n, w, wu, dil, dtype = case
    bias = make_bias(1, n, seed=n + 3) if with_bias else None
    d = ddesc(BH, n, w, wu, dil, dtype, bias)
    S = (seeded_band(BH, n, d.D, torch.float32, seed=21) * 3).to(dtype)
    P, Pd = empty_band(d), empty_band(d)
    lse = torch.empty((BH, n), dtype=torch.float32, device="cuda")
    swab.band_softmax_dropout(d, poison_invalid(S, n, w, wu, dil).cuda(), Pd, P=P, lse=lse)
    kb = per_slice(bias, BH) if with_bias else None
    refP, reflse, refPd = oracle.band_softmax(f64(S), w, wu, dil, key_bias=kb, drop_t=d.drop_t,
                                              seed=SEED)
    gP, gPd = f64(P), f64(Pd)
    m = valid_mask(n, w, wu, dil)
    assert np.all(gP[:, ~m] == 0.0) and np.all(gPd[:, ~m] == 0.0)
    dscale = 256.0 / (256.0 - d.drop_t)
    tol = 1e-6 if dtype == torch.float32 else ABS_TOL
    assert np.max(np.abs(gP - refP)) <= tol
    assert np.max(np.abs(gPd - refPd)) <= tol * dscale
    assert np.max(np.abs(f64(lse) - reflse)) <= 1e-4 * max(1.0, np.max(np.abs(reflse)))
    # exact keep pattern wherever the probability is representable
    live = m[None] & (gP != 0.0)
    assert np.array_equal((gPd != 0.0)[live], (refPd != 0.0)[live])
    kept = (refPd != 0.0)[m[None] & (refP > 0.0)]   # masked keys have P = 0 exactly
    e = 1 - d.drop_t / 256
    assert abs(kept.mean() - e) < 5 * np.sqrt(e * (1 - e) / kept.size)


def test_band_softmax_dropout_zero_p_and_no_P():
    """p = 0 keeps everything: Pd equals band_softmax's P up to rounding (rows
    with dropout stream, the register path takes the max first); P may be
    omitted."""
    BH, n, w, wu, dil, dtype = 2, 600, 64, 64, 1, torch.float16
    d0 = swab.Desc(1, BH, n, 64, w, wu, dil, 0.0, dtype)
    d = ddesc(BH, n, w, wu, dil, dtype, p=0.0)
    S = (seeded_band(BH, n, d.D, torch.float32, seed=22) * 3).to(dtype).cuda()
    P, Pd = empty_band(d0), empty_band(d)
    swab.band_softmax(d0, S, P)
    swab.band_softmax_dropout(d, S, Pd)
    torch.cuda.synchronize()
    a, b_ = P.float().cpu(), Pd.float().cpu()
    assert torch.allclose(a, b_, rtol=2.0 ** -10, atol=1e-7)
    assert bool(((a > 1e-4) <= (b_ > 0)).all())


@pytest.mark.parametrize("case", UNIT_CASES, ids=unit_ids)
def test_band_softmax_bwd_dropout_unit(case):
    BH, n, w, wu, dil, dtype = case
    d = ddesc(BH, n, w, wu, dil, dtype)
    P = seeded_band(BH, n, d.D, dtype, seed=23)
    dP = seeded_band(BH, n, d.D, dtype, seed=24)
    dS = empty_band(d)
    swab.band_softmax_bwd(d, poison_invalid(P, n, w, wu, dil).cuda(),
                          poison_invalid(dP, n, w, wu, dil).cuda(), dS)
    ref = oracle.band_softmax_bwd(f64(P), f64(dP), w, wu, dil, drop_t=d.drop_t, seed=SEED)
    got = f64(dS)
    m = valid_mask(n, w, wu, dil)
    assert np.all(got[:, ~m] == 0.0)
    assert normwise(got, ref, m) <= score_tol(dtype)


def gpu_chain_dropout(d, Q, K, V, dO, scale):
    S, P, Pd, dPd, dS = (empty_band(d) for _ in range(5))
    lse = torch.empty((d.BH, d.n), dtype=torch.float32, device="cuda")
    O, dQ, dK, dV = (empty_dense(d) for _ in range(4))
    swab.band_qk(d, scale, Q, K, S)
    swab.band_softmax_dropout(d, S, Pd, P=P, lse=lse)
    swab.band_pv(d, 1.0, Pd, V, O)
    swab.band_qk(d, 1.0, dO, V, dPd)
    swab.band_softmax_bwd(d, P, dPd, dS)
    swab.band_pv(d, scale, dS, K, dQ)
    swab.band_qk_bwd_t(d, scale, dS, Q, dK)
    swab.band_pv_bwd_t(d, 1.0, Pd, dO, dV)
    torch.cuda.synchronize()
    return dict(O=O, lse=lse, dQ=dQ, dK=dK, dV=dV)


def check_chain_dropout(b, h, n, w, wu, dil, dtype, Q, K, V, dO, scale, slices, bias=None):
    d = swab.Desc(b, h, n, 64, w, wu, dil, 0.0, dtype, dropout_p=P_DROP, dropout_seed=SEED,
                  key_bias=bias.cuda() if bias is not None else None)
    out = gpu_chain_dropout(d, *(x.cuda() for x in (Q, K, V, dO)), scale)
    # the keep decisions depend on the slice number: the oracle sees every slice
    args = dict(drop_t=d.drop_t, seed=SEED, key_bias=per_slice(bias, h) if bias is not None else None)
    refO, reflse = oracle.attention_fwd(f64(Q), f64(K), f64(V), w, wu, dil, scale, **args)
    refs = oracle.attention_bwd(f64(Q), f64(K), f64(V), f64(dO), w, wu, dil, scale, **args)
    sl = list(slices)
    np.testing.assert_allclose(f64(out["lse"])[sl], reflse[sl], rtol=1e-4, atol=2e-2)
    for name, ref in (("O", refO), ("dQ", refs[0]), ("dK", refs[1]), ("dV", refs[2])):
        got = f64(out[name])[sl]
        if dtype == torch.float32:
            assert normwise(got, ref[sl]) <= F32_TOL, name
        else:
            assert within_abs(got, ref[sl], dtype), name


@pytest.mark.parametrize("case", [(1, 2, 700, 64, 64, 0, torch.float16, False),
                                  (1, 3, 777, 100, 37, 2, torch.bfloat16, True),
                                  (2, 1, 333, 7, 30, 2, torch.float32, False)],
                         ids=["fp16", "bf16-dil-bias", "fp32-dil"])
def test_chain_dropout_unit(case):
    b, h, n, w, wu, dil, dtype, with_bias = case
    Q, K, V, dO = seeded_qkvo(b * h, n, 64, dtype, seed=n + 31)
    bias = make_bias(b, n, seed=n + 32) if with_bias else None
    check_chain_dropout(b, h, n, w, wu, dil, dtype, Q, K, V, dO, 0.125, range(b * h), bias)


def test_chain_dropout_workload():
    """The materialised chain with p = 0.1 on the n=4096, w=256 fp16 workload
    (slices 0 and 7 compared)."""
    wl = WORKLOADS[2]
    Q, K, V, dO = workload_inputs(wl)
    check_chain_dropout(wl.b, wl.h, wl.n, wl.w, wl.w_upper, wl.dilation, wl.dtype, Q, K, V, dO,
                        wl.scale, (0, 7))


def test_chain_dropout_matches_fused():
    """The materialised chain and the fused pair draw the same keep decisions:
    their outputs agree to the rounding of the band tensors."""
    b, h, n, w, wu = 1, 2, 1000, 128, 128
    Q, K, V, dO = (x.cuda() for x in seeded_qkvo(b * h, n, 64, torch.float16, seed=41))
    d = swab.Desc(b, h, n, 64, w, wu, 0, 0.0, torch.float16, dropout_p=0.25, dropout_seed=99)
    ch = gpu_chain_dropout(d, Q, K, V, dO, 0.125)
    O = empty_dense(d)
    lse = torch.empty((d.BH, n), dtype=torch.float32, device="cuda")
    swab.band_attention(d, 0.125, Q, K, V, O, lse)
    torch.cuda.synchronize()
    assert np.max(np.abs(f64(O) - f64(ch["O"]))) <= 2e-2
