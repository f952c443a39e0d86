"""band_softmax / band_softmax_bwd on long band rows, where a CTA of eight
warps holds one row (rows of more than four 16-byte pieces a lane for one
warp, up to 32 values a thread), and one row length past that (the two-pass
streaming kernel).  Against the fp64 oracle with the unit tests' tolerances:
plain, with the key bias, with dropout (keep pattern exact), dilation,
ragged sequence ends, fp16 / bf16 / fp32 ("Developing a faster schedule for
Longformer's kernel", post 3: windows up to 8192; the long causal workload's
4097 diagonals)."""
import numpy as np
import pytest
import torch

import oracle
import sliding_window_attention_band_gb300 as swab
from sliding_window_attention_band_gb300.inputs import seeded_band

from test_gpu_key_bias import make_bias, per_slice
from test_gpu_parity import (ABS_TOL, empty_band, f64, normwise, poison_invalid, score_tol,
                             valid_mask)

pytestmark = [pytest.mark.gpu, pytest.mark.usefixtures("device_status_guard")]

SEED = 0x5EED1234ABCD

CASES = [  # BH, n, w, w_upper, dilation, dtype
    (1, 2000, 768, 768, 0, torch.float16),     # 193 pieces: one a thread
    (1, 4500, 4096, 0, 0, torch.bfloat16),     # the causal band, 514 pieces
    (2, 900, 256, 256, 0, torch.float32),      # fp32 rows of 129-130 pieces
    (1, 1500, 512, 512, 0, torch.float32),     # fp32, two pieces a thread
    (1, 1900, 600, 300, 2, torch.float16),     # dilation, lopsided band
    (1, 1200, 4000, 4000, 0, torch.float16),   # 8001 slots: 1001 pieces, four a thread
    (1, 700, 4200, 4200, 0, torch.float16),    # 8401 slots: past the CTA, streamed
]


def ids(c):
    return f"BH{c[0]}-n{c[1]}-w{c[2]}-wu{c[3]}-d{c[4]}-{str(c[5]).split('.')[-1]}"


def desc(BH, n, w, wu, dil, dtype, bias=None, p=0.0):
    return swab.Desc(1, BH, n, 64, w, wu, dil, 0.0, dtype, dropout_p=p, dropout_seed=SEED,
                     key_bias=bias.cuda() if bias is not None else None)


@pytest.mark.parametrize("with_bias", [False, True], ids=["", "bias"])
@pytest.mark.parametrize("case", CASES, ids=ids)
def test_band_softmax_long_rows(case, with_bias):
    BH, n, w, wu, dil, dtype = case
    bias = make_bias(1, n, seed=n + 5) if with_bias else None
    d = desc(BH, n, w, wu, dil, dtype, bias)
    S = (seeded_band(BH, n, d.D, torch.float32, seed=31) * 3).to(dtype)
    P = empty_band(d)
    lse = torch.empty((BH, n), dtype=torch.float32, device="cuda")
    swab.band_softmax(d, poison_invalid(S, n, w, wu, dil).cuda(), P, lse)
    kb = per_slice(bias, BH) if with_bias else None
    refP, reflse = oracle.band_softmax(f64(S), w, wu, dil, key_bias=kb)
    got = f64(P)
    tol = 1e-6 if dtype == torch.float32 else ABS_TOL
    assert np.max(np.abs(got - refP)) <= tol
    assert np.max(np.abs(f64(lse) - reflse)) <= 1e-4 * max(1.0, np.max(np.abs(reflse)))
    assert np.all(got[:, ~valid_mask(n, w, wu, dil)] == 0.0)


@pytest.mark.parametrize("case", CASES, ids=ids)
def test_band_softmax_bwd_long_rows(case):
    BH, n, w, wu, dil, dtype = case
    d = desc(BH, n, w, wu, dil, dtype)
    P = seeded_band(BH, n, d.D, dtype, seed=32)
    dP = seeded_band(BH, n, d.D, dtype, seed=33)
    dS = empty_band(d)
    swab.band_softmax_bwd(d, poison_invalid(P, n, w, wu, dil).cuda(),
                          poison_invalid(dP, n, w, wu, dil).cuda(), dS)
    ref = oracle.band_softmax_bwd(f64(P), f64(dP), w, wu, dil)
    got = f64(dS)
    m = valid_mask(n, w, wu, dil)
    assert np.all(got[:, ~m] == 0.0)
    assert normwise(got, ref, m) <= score_tol(dtype)


@pytest.mark.parametrize("case", CASES[:5], ids=ids)
def test_band_softmax_dropout_long_rows(case):
    """Forward with dropout (P and the dropped Pd, keep pattern exact) and the
    backward through it."""
    BH, n, w, wu, dil, dtype = case
    d = desc(BH, n, w, wu, dil, dtype, p=0.1)
    S = (seeded_band(BH, n, d.D, torch.float32, seed=34) * 3).to(dtype)
    P, Pd = empty_band(d), empty_band(d)
    lse = torch.empty((BH, n), dtype=torch.float32, device="cuda")
    swab.band_softmax_dropout(d, poison_invalid(S, n, w, wu, dil).cuda(), Pd, P=P, lse=lse)
    refP, reflse, refPd = oracle.band_softmax(f64(S), w, wu, dil, drop_t=d.drop_t, seed=SEED)
    gP, gPd = f64(P), f64(Pd)
    dscale = 256.0 / (256.0 - d.drop_t)
    tol = 1e-6 if dtype == torch.float32 else ABS_TOL
    assert np.max(np.abs(gP - refP)) <= tol
    assert np.max(np.abs(gPd - refPd)) <= tol * dscale
    m = valid_mask(n, w, wu, dil)
    live = m[None] & (gP != 0.0)
    assert np.array_equal((gPd != 0.0)[live], (refPd != 0.0)[live])
    dPd = seeded_band(BH, n, d.D, dtype, seed=35)
    dS = empty_band(d)
    swab.band_softmax_bwd(d, P, poison_invalid(dPd, n, w, wu, dil).cuda(), dS)
    ref = oracle.band_softmax_bwd(gP, f64(dPd), w, wu, dil, drop_t=d.drop_t, seed=SEED)
    assert normwise(f64(dS), ref, m) <= score_tol(dtype)
