"""GPU parity: every kernel of the library against the fp64 CPU oracle.

Both sides get the same dtype-rounded inputs (upcast to fp64 for the oracle,
exactly).  Tolerances:
  * fp16 banded scores: normwise  max|gpu - ref| / max|ref|  <= 2e-3 over
    valid slots (one RNE rounding of the fp32 accumulator costs at most
    2^-11 = 4.9e-4 relative); padding slots bit-exact;
  * bf16 banded scores: 2e-3 is below the format's own resolution -- one
    correctly rounded bf16 store is off by up to 2^-8 = 3.9e-3 relative -- so
    the bound is that unit roundoff plus 1e-4 of fp32-accumulation slack;
  * dense outputs of the unit kernels fed random (non-probability) bands:
    the same per-dtype bounds;
  * attention chains (O, P, dQ, dK, dV): max abs 1e-2.  fp16 is held to that
    plain bound; bf16 adds one rounding of the output itself (2^-8 x |ref|),
    since a correctly rounded bf16 value above 2.56 is already off by up to
    1e-2;
  * fp32 inputs: normwise relative 1e-5 (FFMA path, no TF32);
  * band indexing probes: bit-exact.
Invalid slots of every band INPUT are filled with NaN: the kernels must
ignore them.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import sliding_window_attention_band_gb300 as swab
from sliding_window_attention_band_gb300 import build as swab_build
from sliding_window_attention_band_gb300.inputs import (WORKLOADS, seeded_band, seeded_qkvo,
                                                        workload_inputs)

pytestmark = pytest.mark.gpu

SCORE_TOL = 2e-3
ABS_TOL = 1e-2
F32_TOL = 1e-5


@pytest.fixture(scope="module", autouse=True)
def _lib():
    swab_build.build()
    swab.load()
    swab.device_status(reset=True)
    yield
    assert swab.device_status(reset=True) == 0, "a kernel raised the device status word"


UNIT_ROUNDOFF = {torch.float16: 2.0 ** -11, torch.bfloat16: 2.0 ** -8, torch.float32: 2.0 ** -24}


def abs_bound(ref, dtype):
    """Element-wise bound on |got - ref| for a chained output: the plain 1e-2
    for fp16 (one fp16 rounding stays below 1e-2 up to |ref| = 20); for bf16
    1e-2 plus one rounding of the output, 2^-8 |ref|, because one correctly
    rounded bf16 store above |ref| = 2.56 already exceeds 1e-2."""
    if dtype == torch.bfloat16:
        return ABS_TOL + UNIT_ROUNDOFF[dtype] * np.abs(ref)
    return ABS_TOL


def within_abs(got, ref, dtype):
    """|got - ref| <= abs_bound(ref, dtype) everywhere."""
    return bool(np.all(np.abs(got - ref) <= abs_bound(ref, dtype)))


def f64(t):
    return t.detach().float().cpu().double().numpy()


def valid_mask(n, w, wu, dil):
    """[n, D] bool: slot t of row i holds a key inside the sequence."""
    s = dil + 1
    i = np.arange(n)[:, None]
    t = np.arange(w + wu + 1)[None, :]
    j = i + (t - w) * s
    return (j >= 0) & (j < n)


def poison_invalid(band, n, w, wu, dil):
    m = torch.from_numpy(~valid_mask(n, w, wu, dil))
    out = band.clone()
    out[:, m] = float("nan")
    return out


def normwise(got, ref, mask=None):
    if mask is not None:
        got, ref = got[..., mask], ref[..., mask]
    den = np.max(np.abs(ref))
    return float(np.max(np.abs(got - ref)) / (den if den > 0 else 1.0))


def dev(*ts):
    return [t.cuda() for t in ts]


def empty_band(d, dtype=None):
    return torch.empty((d.BH, d.n, d.D), dtype=dtype or d.dtype, device="cuda")


def empty_dense(d):
    return torch.empty((d.BH, d.n, d.head_dim), dtype=d.dtype, device="cuda")


# ---------------------------------------------------------------------------
# unit parity, small ragged cases spanning several tiles
# ---------------------------------------------------------------------------
UNIT_CASES = [  # BH, n, w, w_upper, dilation, dtype
    (2, 1000, 64, 64, 0, torch.float16),
    (3, 777, 100, 37, 2, torch.bfloat16),
    (1, 300, 256, 256, 0, torch.float16),
    (2, 640, 0, 127, 1, torch.float16),
    (1, 1100, 300, 0, 0, torch.bfloat16),
    (2, 515, 3, 3, 3, torch.float16),
    (1, 129, 1, 2, 0, torch.bfloat16),
    (2, 200, 20, 20, 0, torch.float32),
    (1, 333, 7, 30, 2, torch.float32),
    (2, 900, 9, 9, 2, torch.float16),     # dilated, s*D - 1 a multiple of 8: one gather shift
    # degenerate and extreme geometries
    (2, 1, 0, 0, 0, torch.float16),       # n = 1, D = 1: one key per row
    (3, 257, 0, 0, 0, torch.bfloat16),    # D = 1: the diagonal alone
    (1, 20, 2, 3, 15, torch.float16),     # the largest dilation (s = 16)
    (2, 10, 4, 4, 15, torch.bfloat16),    # n < s: six residues empty, one row per residue
    (1, 100, 256, 256, 0, torch.float16), # a window wider than the sequence
    (2, 50, 0, 0, 1, torch.float32),      # fp32, D = 1, dilated
]


def unit_ids(c):
    return f"BH{c[0]}-n{c[1]}-w{c[2]}-wu{c[3]}-d{c[4]}-{str(c[5]).split('.')[-1]}"


def mkdesc(BH, n, w, wu, d, dtype, padding=0.0, hd=64):
    return swab.Desc(1, BH, n, hd, w, wu, d, padding, dtype)


BF16_SCORE_TOL = 2.0 ** -8 + 1e-4


def score_tol(dtype):
    return {torch.float32: F32_TOL, torch.float16: SCORE_TOL, torch.bfloat16: BF16_SCORE_TOL}[dtype]


@pytest.mark.parametrize("case", UNIT_CASES, ids=unit_ids)
def test_band_qk_unit(case):
    BH, n, w, wu, dil, dtype = case
    d = mkdesc(BH, n, w, wu, dil, dtype, padding=-3.25)
    A, B = seeded_qkvo(BH, n, 64, dtype, seed=11, count=2)
    S = empty_band(d)
    swab.band_qk(d, 0.125, *dev(A, B), S)
    ref = oracle.band_qk(f64(A), f64(B), w, wu, dil, alpha=0.125, padding=-3.25)
    got = f64(S)
    m = valid_mask(n, w, wu, dil)
    assert np.all(got[:, ~m] == -3.25), "padding slots must hold the padding value exactly"
    assert normwise(got, ref, m) <= score_tol(dtype)


@pytest.mark.parametrize("case", UNIT_CASES, ids=unit_ids)
def test_band_softmax_unit(case):
    BH, n, w, wu, dil, dtype = case
    d = mkdesc(BH, n, w, wu, dil, dtype)
    S = (seeded_band(BH, n, d.D, torch.float32, seed=12) * 3).to(dtype)
    P = empty_band(d)
    lse = torch.empty((BH, n), dtype=torch.float32, device="cuda")
    swab.band_softmax(d, poison_invalid(S, n, w, wu, dil).cuda(), P, lse)
    refP, reflse = oracle.band_softmax(f64(S), w, wu, dil)
    got = f64(P)
    tol = 1e-6 if dtype == torch.float32 else ABS_TOL
    assert np.max(np.abs(got - refP)) <= tol
    assert np.max(np.abs(f64(lse) - reflse)) <= 1e-4 * max(1.0, np.max(np.abs(reflse)))
    assert np.all(got[:, ~valid_mask(n, w, wu, dil)] == 0.0)


@pytest.mark.parametrize("case", UNIT_CASES, ids=unit_ids)
def test_band_pv_unit(case):
    BH, n, w, wu, dil, dtype = case
    d = mkdesc(BH, n, w, wu, dil, dtype)
    P = seeded_band(BH, n, d.D, dtype, seed=13)
    (V,) = seeded_qkvo(BH, n, 64, dtype, seed=14, count=1)
    O = empty_dense(d)
    swab.band_pv(d, 0.75, poison_invalid(P, n, w, wu, dil).cuda(), V.cuda(), O)
    ref = oracle.band_pv(f64(P), f64(V), w, wu, dil, alpha=0.75)
    assert normwise(f64(O), ref) <= score_tol(dtype)


@pytest.mark.parametrize("case", UNIT_CASES, ids=unit_ids)
@pytest.mark.parametrize("name", ["band_qk_bwd_t", "band_pv_bwd_t"])
def test_band_t_unit(case, name):
    BH, n, w, wu, dil, dtype = case
    d = mkdesc(BH, n, w, wu, dil, dtype)
    Bd = seeded_band(BH, n, d.D, dtype, seed=15)
    (Y,) = seeded_qkvo(BH, n, 64, dtype, seed=16, count=1)
    X = empty_dense(d)
    getattr(swab, name)(d, 0.5, poison_invalid(Bd, n, w, wu, dil).cuda(), Y.cuda(), X)
    ref = oracle.band_t(f64(Bd), f64(Y), w, wu, dil, alpha=0.5)
    assert normwise(f64(X), ref) <= score_tol(dtype)


@pytest.mark.parametrize("case", UNIT_CASES, ids=unit_ids)
def test_band_softmax_bwd_unit(case):
    BH, n, w, wu, dil, dtype = case
    d = mkdesc(BH, n, w, wu, dil, dtype)
    P = seeded_band(BH, n, d.D, dtype, seed=17)
    dP = seeded_band(BH, n, d.D, dtype, seed=18)
    dS = empty_band(d)
    swab.band_softmax_bwd(d, poison_invalid(P, n, w, wu, dil).cuda(),
                          poison_invalid(dP, n, w, wu, dil).cuda(), dS)
    ref = oracle.band_softmax_bwd(f64(P), f64(dP), w, wu, dil)
    got = f64(dS)
    m = valid_mask(n, w, wu, dil)
    assert np.all(got[:, ~m] == 0.0)
    assert normwise(got, ref, m) <= score_tol(dtype)


# ---------------------------------------------------------------------------
# bit-exact band indexing probes
# ---------------------------------------------------------------------------
PROBE_CASES = [  # BH, n, w, w_upper, dilation, dtype
    (2, 1000, 64, 64, 0, torch.float16),
    (1, 4100, 256, 256, 3, torch.bfloat16),
    (1, 2049, 500, 0, 1, torch.float16),
    (1, 1500, 5, 5, 2, torch.bfloat16),   # dilated, s*D - 1 a multiple of 8
    (1, 10, 4, 4, 15, torch.float16),     # n < s: empty residues, the largest dilation
    (2, 1, 0, 0, 0, torch.bfloat16),      # n = 1
]


def digit(j, k):
    return (j >> (5 * k)) & 31  # base-32 digits: exact in fp16 and bf16


@pytest.mark.parametrize("case", PROBE_CASES, ids=unit_ids)
def test_index_probe_band_qk(case):
    BH, n, w, wu, dil, dtype = case
    d = mkdesc(BH, n, w, wu, dil, dtype, padding=-1.0)
    j = torch.arange(n)
    for k in range(3):
        Q = torch.zeros(BH, n, 64)
        Q[:, :, k] = 1.0
        K = torch.zeros(BH, n, 64)
        K[:, :, k] = digit(j, k).float()
        Q, K = Q.to(dtype), K.to(dtype)
        S = empty_band(d)
        swab.band_qk(d, 1.0, *dev(Q, K), S)
        ref = oracle.band_qk(f64(Q), f64(K), w, wu, dil, alpha=1.0, padding=-1.0)
        np.testing.assert_array_equal(f64(S), ref)


def one_hot_band(BH, n, w, wu, dil, dtype, seed):
    """One valid slot per row set to 1, other valid slots 0, invalid slots NaN."""
    D = w + wu + 1
    m = valid_mask(n, w, wu, dil)
    rng = np.random.default_rng(seed)
    band = np.zeros((BH, n, D), dtype=np.float32)
    for i in range(n):
        ts = np.nonzero(m[i])[0]
        for b in range(BH):
            band[b, i, rng.choice(ts)] = 1.0
    band[:, ~m] = np.nan
    return torch.from_numpy(band).to(dtype)


@pytest.mark.parametrize("case", PROBE_CASES, ids=unit_ids)
def test_index_probe_band_pv_and_t(case):
    BH, n, w, wu, dil, dtype = case
    d = mkdesc(BH, n, w, wu, dil, dtype)
    band = one_hot_band(BH, n, w, wu, dil, dtype, seed=19)
    Y = torch.zeros(BH, n, 64)
    for k in range(3):
        Y[:, :, k] = digit(torch.arange(n), k).float()
    Y = Y.to(dtype)
    clean = torch.nan_to_num(band.float(), nan=0.0)
    O = empty_dense(d)
    swab.band_pv(d, 1.0, band.cuda(), Y.cuda(), O)
    np.testing.assert_array_equal(f64(O), oracle.band_pv(f64(clean), f64(Y), w, wu, dil))
    if dtype == torch.float16:  # column sums of digits stay exact in fp16
        X = empty_dense(d)
        swab.band_pv_bwd_t(d, 1.0, band.cuda(), Y.cuda(), X)
        np.testing.assert_array_equal(f64(X), oracle.band_t(f64(clean), f64(Y), w, wu, dil))


# ---------------------------------------------------------------------------
# the full chain (forward + backward) on the named workloads
# ---------------------------------------------------------------------------
def gpu_chain(d, Q, K, V, dO, scale):
    S, P, dP, dS = (empty_band(d) for _ in range(4))
    lse = torch.empty((d.BH, d.n), dtype=torch.float32, device="cuda")
    O, dQ, dK, dV = (empty_dense(d) for _ in range(4))
    swab.band_qk(d, scale, Q, K, S)
    swab.band_softmax(d, S, P, lse)
    swab.band_pv(d, 1.0, P, V, O)
    swab.band_qk(d, 1.0, dO, V, dP)
    swab.band_softmax_bwd(d, P, dP, dS)
    swab.band_pv(d, scale, dS, K, dQ)
    swab.band_qk_bwd_t(d, scale, dS, Q, dK)
    swab.band_pv_bwd_t(d, 1.0, P, dO, dV)
    torch.cuda.synchronize()
    return dict(S=S, P=P, lse=lse, O=O, dQ=dQ, dK=dK, dV=dV)


def check_chain(wl, slices, backward=True):
    Q, K, V, dO = workload_inputs(wl)
    d = swab.Desc.from_workload(wl)
    out = gpu_chain(d, *dev(Q, K, V, dO), wl.scale)
    w, wu, dil = wl.w, wl.w_upper, wl.dilation
    m = valid_mask(wl.n, w, wu, dil)
    f32 = wl.dtype == torch.float32
    for b in slices:
        sl = slice(b, b + 1)
        q, k, v, go = (f64(x[sl]) for x in (Q, K, V, dO))
        refS = oracle.band_qk(q, k, w, wu, dil, alpha=wl.scale, padding=wl.padding)
        gotS = f64(out["S"][sl])
        assert np.all(gotS[:, ~m] == wl.padding)
        assert normwise(gotS, refS, m) <= score_tol(wl.dtype)
        refO, reflse = oracle.attention_fwd(q, k, v, w, wu, dil, wl.scale)
        refP, _ = oracle.band_softmax(refS, w, wu, dil)
        if f32:
            assert normwise(f64(out["P"][sl]), refP) <= F32_TOL
            assert normwise(f64(out["O"][sl]), refO) <= F32_TOL
        else:
            assert within_abs(f64(out["P"][sl]), refP, wl.dtype)
            assert within_abs(f64(out["O"][sl]), refO, wl.dtype)
        assert np.max(np.abs(f64(out["lse"][sl]) - reflse)) <= (1e-5 if f32 else 2e-2)
        if backward:
            rq, rk, rv = oracle.attention_bwd(q, k, v, go, w, wu, dil, wl.scale)
            for name, ref in (("dQ", rq), ("dK", rk), ("dV", rv)):
                got = f64(out[name][sl])
                if f32:
                    assert normwise(got, ref) <= F32_TOL, name
                else:
                    assert within_abs(got, ref, wl.dtype), name


def test_chain_config1_fp32_full():
    check_chain(WORKLOADS[1], slices=range(WORKLOADS[1].BH))


@pytest.mark.parametrize("cfg", [2, 3])
def test_chain_config_fp16_sampled(cfg):
    check_chain(WORKLOADS[cfg], slices=(0, 7))


def test_chain_config5_materialised_sampled():
    """The long causal workload through the eight materialised calls, forward
    and backward, on one sampled slice."""
    check_chain(WORKLOADS[5], slices=(5,), backward=True)


# ---------------------------------------------------------------------------
# fused forward: scores kept on chip
# ---------------------------------------------------------------------------
def check_fused(d, Q, K, V, scale, slices, f32):
    O = empty_dense(d)
    lse = torch.empty((d.BH, d.n), dtype=torch.float32, device="cuda")
    swab.band_attention(d, scale, *dev(Q, K, V), O, lse)
    torch.cuda.synchronize()
    for b in slices:
        sl = slice(b, b + 1)
        refO, reflse = oracle.attention_fwd(f64(Q[sl]), f64(K[sl]), f64(V[sl]), d.w, d.w_upper,
                                            d.dilation, scale)
        gotO, gotl = f64(O[sl]), f64(lse[sl])
        if f32:
            assert normwise(gotO, refO) <= F32_TOL
            assert np.max(np.abs(gotl - reflse)) <= 1e-5
        else:
            assert within_abs(gotO, refO, d.dtype)
            assert np.max(np.abs(gotl - reflse)) <= 2e-2


@pytest.mark.parametrize("case", UNIT_CASES, ids=unit_ids)
def test_band_attention_unit(case):
    BH, n, w, wu, dil, dtype = case
    d = mkdesc(BH, n, w, wu, dil, dtype)
    Q, K, V = seeded_qkvo(BH, n, 64, dtype, seed=21, count=3)
    check_fused(d, Q, K, V, 0.125, range(BH), dtype == torch.float32)


@pytest.mark.parametrize("cfg,slices", [(1, (0, 1)), (2, (0, 11)), (3, (4,)), (5, (2,))])
def test_band_attention_config(cfg, slices):
    wl = WORKLOADS[cfg]
    Q, K, V, _ = workload_inputs(wl)
    check_fused(swab.Desc.from_workload(wl), Q, K, V, wl.scale, slices,
                wl.dtype == torch.float32)


# ---------------------------------------------------------------------------
# fused backward: band probabilities recomputed on chip from lse
# ---------------------------------------------------------------------------
def check_fused_bwd(d, Q, K, V, dO, scale, slices, f32):
    q, k, v, go = dev(Q, K, V, dO)
    O = empty_dense(d)
    lse = torch.empty((d.BH, d.n), dtype=torch.float32, device="cuda")
    swab.band_attention(d, scale, q, k, v, O, lse)
    dQ, dK, dV = (empty_dense(d) for _ in range(3))
    ws = torch.empty(swab.band_attention_bwd_workspace(d) // 4, dtype=torch.float32, device="cuda")
    ws.fill_(float("nan"))  # contents on entry must not matter
    swab.band_attention_bwd(d, scale, q, k, v, O, go, lse, dQ, dK, dV, ws)
    torch.cuda.synchronize()
    for b in slices:
        sl = slice(b, b + 1)
        refs = oracle.attention_bwd(f64(Q[sl]), f64(K[sl]), f64(V[sl]), f64(dO[sl]), d.w,
                                    d.w_upper, d.dilation, scale)
        for name, got, ref in (("dQ", dQ, refs[0]), ("dK", dK, refs[1]), ("dV", dV, refs[2])):
            g_ = f64(got[sl])
            if f32:
                assert normwise(g_, ref) <= F32_TOL, name
            else:
                assert within_abs(g_, ref, d.dtype), name


@pytest.mark.parametrize("case", UNIT_CASES, ids=unit_ids)
def test_band_attention_bwd_unit(case):
    BH, n, w, wu, dil, dtype = case
    d = mkdesc(BH, n, w, wu, dil, dtype)
    Q, K, V, dO = seeded_qkvo(BH, n, 64, dtype, seed=23)
    check_fused_bwd(d, Q, K, V, dO, 0.125, range(BH), dtype == torch.float32)


@pytest.mark.parametrize("cfg,slices", [(1, (0, 1)), (2, (0, 11)), (3, (6,)), (5, (3,))])
def test_band_attention_bwd_config(cfg, slices):
    wl = WORKLOADS[cfg]
    Q, K, V, dO = workload_inputs(wl)
    check_fused_bwd(swab.Desc.from_workload(wl), Q, K, V, dO, wl.scale, slices,
                    wl.dtype == torch.float32)


# ---------------------------------------------------------------------------
# rows with a single key: the softmax weight is exactly 1, so the attention
# returns V exactly and passes dO straight to dV (closed forms, bitwise)
# ---------------------------------------------------------------------------
SINGLE_KEY_CASES = [  # BH, n, w, w_upper, dilation: every row's band holds only its own key
    (2, 1, 0, 0, 0),      # n = 1
    (3, 300, 0, 0, 0),    # D = 1
    (2, 12, 3, 5, 15),    # n <= s: one row per residue
]


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16, torch.float32],
                         ids=lambda t: str(t).split(".")[-1])
@pytest.mark.parametrize("case", SINGLE_KEY_CASES, ids=lambda c: "BH{}-n{}-w{}-wu{}-d{}".format(*c))
def test_single_key_rows_return_v(case, dtype):
    BH, n, w, wu, dil = case
    d = mkdesc(BH, n, w, wu, dil, dtype)
    Q, K, V, dO = dev(*seeded_qkvo(BH, n, 64, dtype, seed=29))
    # fused forward and backward
    O = empty_dense(d)
    lse = torch.empty((BH, n), dtype=torch.float32, device="cuda")
    swab.band_attention(d, 0.125, Q, K, V, O, lse)
    dQ, dK, dV = (empty_dense(d) for _ in range(3))
    ws = torch.empty(swab.band_attention_bwd_workspace(d) // 4, dtype=torch.float32, device="cuda")
    swab.band_attention_bwd(d, 0.125, Q, K, V, O, dO, lse, dQ, dK, dV, ws)
    # the materialised forward
    S, P = empty_band(d), empty_band(d)
    Om = empty_dense(d)
    swab.band_qk(d, 0.125, Q, K, S)
    swab.band_softmax(d, S, P)
    swab.band_pv(d, 1.0, P, V, Om)
    torch.cuda.synchronize()
    assert torch.equal(O, V) and torch.equal(Om, V)
    assert torch.equal(dV, dO)
    m = torch.from_numpy(valid_mask(n, w, wu, dil))   # the diagonal slot alone
    assert torch.all(P.cpu()[:, m] == 1) and torch.all(P.cpu()[:, ~m] == 0)
    # lse is the row's own scaled score; dS = P (dP - delta) = 0 up to the
    # rounding of two dot products of the same vectors
    qk = (Q.double() * K.double()).sum(-1) * 0.125
    assert torch.allclose(lse.double(), qk, rtol=1e-5, atol=2e-3 if dtype != torch.float32 else 1e-5)
    for g in (dQ, dK):
        assert float(g.double().abs().max()) <= 2e-3
