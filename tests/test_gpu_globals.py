"""GPU parity with global tokens (one global index shared by the batch).

Every input a kernel must ignore is poisoned with NaN: invalid band slots,
band slots whose key is global, the band and cols rows of global queries.
Tolerances as in test_gpu_parity.py.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import sliding_window_attention_band_gb300 as swab
from sliding_window_attention_band_gb300 import build as swab_build
from sliding_window_attention_band_gb300.inputs import (WORKLOADS, seeded_band, seeded_qkvo,
                                                        seeded_uniform, workload_inputs)

from test_gpu_parity import (ABS_TOL, dev, empty_band, empty_dense, f64, normwise, score_tol,
                             valid_mask, within_abs)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    swab_build.build()
    swab.load()
    swab.device_status(reset=True)
    yield
    assert swab.device_status(reset=True) == 0


CASES = [  # BH, n, w, w_upper, dilation, dtype, global idx
    (2, 1000, 64, 64, 0, torch.float16, (0, 1, 7, 500, 999)),
    (3, 777, 100, 37, 2, torch.bfloat16, (3, 20, 21, 400)),
    (1, 640, 0, 127, 1, torch.float16, tuple(range(16))),
    (2, 300, 20, 20, 0, torch.float32, (0, 150, 299)),
    (1, 129, 1, 2, 0, torch.bfloat16, (64,)),
    # more than 64 global tokens: the band products' global term on FFMA
    (1, 700, 30, 30, 0, torch.float16, tuple(range(0, 700, 9))),
    # the largest number of global tokens (256), dilated
    (1, 600, 16, 16, 1, torch.bfloat16, tuple(range(0, 512, 2))),
]


def ids(c):
    return f"BH{c[0]}-n{c[1]}-w{c[2]}-wu{c[3]}-d{c[4]}-{str(c[5]).split('.')[-1]}-G{len(c[6])}"


def mk(BH, n, w, wu, dil, dtype, gidx):
    return swab.Desc(1, BH, n, 64, w, wu, dil, 0.0, dtype, gidx)


def ignorable_band(n, w, wu, dil, gidx):
    """[n, D] True where a consumer must ignore the band slot."""
    s = dil + 1
    i = np.arange(n)[:, None]
    t = np.arange(w + wu + 1)[None, :]
    j = i + (t - w) * s
    bad = (j < 0) | (j >= n)
    g = np.zeros(n, dtype=bool)
    g[list(gidx)] = True
    jj = np.clip(j, 0, n - 1)
    bad |= g[jj] & ~((j < 0) | (j >= n))
    bad |= g[:, None]
    return bad


def poison(band, cols, n, w, wu, dil, gidx):
    band = band.clone()
    band[:, torch.from_numpy(ignorable_band(n, w, wu, dil, gidx))] = float("nan")
    cols = cols.clone()
    cols[:, list(gidx), :] = float("nan")
    return band, cols


def glob_pair(BH, n, G, dtype, seed, uniform=False):
    if uniform:
        return (seeded_uniform((BH, n, G), dtype, seed), seeded_uniform((BH, G, n), dtype, seed + 1))
    return (seeded_band(BH, n, G, dtype, seed), seeded_band(BH, G, n, dtype, seed + 1))


def empty_glob(d):
    return (torch.empty(d.BH, d.n, d.G, dtype=d.dtype, device="cuda"),
            torch.empty(d.BH, d.G, d.n, dtype=d.dtype, device="cuda"))


@pytest.mark.parametrize("case", CASES, ids=ids)
def test_band_qk_globals(case):
    BH, n, w, wu, dil, dtype, gidx = case
    d = mk(*case)
    A, B = seeded_qkvo(BH, n, 64, dtype, seed=31, count=2)
    S = empty_band(d)
    Sg = empty_glob(d)
    swab.band_qk(d, 0.125, *dev(A, B), S, Sg)
    refS, refc, refr = oracle.band_qk(f64(A), f64(B), w, wu, dil, 0.125, 0.0, gidx)
    tol = score_tol(dtype)
    assert normwise(f64(Sg[0]), refc) <= tol
    assert normwise(f64(Sg[1]), refr) <= tol
    assert normwise(f64(S), refS, valid_mask(n, w, wu, dil)) <= tol


@pytest.mark.parametrize("case", CASES, ids=ids)
def test_band_softmax_globals(case):
    BH, n, w, wu, dil, dtype, gidx = case
    d = mk(*case)
    S = (seeded_band(BH, n, d.D, torch.float32, seed=32) * 3).to(dtype)
    Sc, Sr = glob_pair(BH, n, d.G, dtype, seed=33)
    Sp, Scp = poison(S, Sc, n, w, wu, dil, gidx)
    P = empty_band(d)
    Pg = empty_glob(d)
    lse = torch.empty(BH, n, dtype=torch.float32, device="cuda")
    swab.band_softmax(d, Sp.cuda(), P, lse, Sg=(Scp.cuda(), Sr.cuda()), Pg=Pg)
    refP, reflse, refPc, refPr = oracle.band_softmax(f64(S), w, wu, dil, gidx, f64(Sc), f64(Sr))
    tol = 1e-6 if dtype == torch.float32 else ABS_TOL
    assert np.max(np.abs(f64(P) - refP)) <= tol
    assert np.max(np.abs(f64(Pg[0]) - refPc)) <= tol
    assert np.max(np.abs(f64(Pg[1]) - refPr)) <= tol
    assert np.max(np.abs(f64(lse) - reflse)) <= 1e-4 * max(1.0, np.max(np.abs(reflse)))


@pytest.mark.parametrize("case", CASES, ids=ids)
def test_band_softmax_globals_key_bias(case):
    """With a key-padding bias (a quarter of the keys masked by -10000, plus a
    small per-key term): added to the band slots, the global columns (key
    G[g]) and the dense global rows."""
    BH, n, w, wu, dil, dtype, gidx = case
    gen = torch.Generator().manual_seed(n + 34)
    kb = torch.where(torch.rand(1, n, generator=gen) > 0.25, 0.0, -10000.0) + 0.3 * torch.randn(1, n, generator=gen)
    d = swab.Desc(1, BH, n, 64, w, wu, dil, 0.0, dtype, gidx, key_bias=kb.cuda())
    S = (seeded_band(BH, n, d.D, torch.float32, seed=35) * 3).to(dtype)
    Sc, Sr = glob_pair(BH, n, d.G, dtype, seed=36)
    Sp, Scp = poison(S, Sc, n, w, wu, dil, gidx)
    P = empty_band(d)
    Pg = empty_glob(d)
    lse = torch.empty(BH, n, dtype=torch.float32, device="cuda")
    swab.band_softmax(d, Sp.cuda(), P, lse, Sg=(Scp.cuda(), Sr.cuda()), Pg=Pg)
    refP, reflse, refPc, refPr = oracle.band_softmax(f64(S), w, wu, dil, gidx, f64(Sc), f64(Sr),
                                                     key_bias=kb.repeat(BH, 1).double().numpy())
    tol = 1e-6 if dtype == torch.float32 else ABS_TOL
    assert np.max(np.abs(f64(P) - refP)) <= tol
    assert np.max(np.abs(f64(Pg[0]) - refPc)) <= tol
    assert np.max(np.abs(f64(Pg[1]) - refPr)) <= tol
    assert np.max(np.abs(f64(lse) - reflse)) <= 1e-4 * max(1.0, np.max(np.abs(reflse)))


@pytest.mark.parametrize("case", CASES, ids=ids)
def test_band_pv_globals(case):
    BH, n, w, wu, dil, dtype, gidx = case
    d = mk(*case)
    P = seeded_band(BH, n, d.D, dtype, seed=34)
    Pc, Pr = glob_pair(BH, n, d.G, dtype, seed=35)
    (V,) = seeded_qkvo(BH, n, 64, dtype, seed=36, count=1)
    Pp, Pcp = poison(P, Pc, n, w, wu, dil, gidx)
    O = empty_dense(d)
    swab.band_pv(d, 0.75, Pp.cuda(), V.cuda(), O, Pg=(Pcp.cuda(), Pr.cuda()))
    ref = oracle.band_pv(f64(P), f64(V), w, wu, dil, 0.75, gidx, f64(Pc), f64(Pr))
    assert normwise(f64(O), ref) <= score_tol(dtype)


@pytest.mark.parametrize("case", CASES, ids=ids)
@pytest.mark.parametrize("name", ["band_qk_bwd_t", "band_pv_bwd_t"])
def test_band_t_globals(case, name):
    BH, n, w, wu, dil, dtype, gidx = case
    d = mk(*case)
    Bd = seeded_band(BH, n, d.D, dtype, seed=37)
    Bc, Br = glob_pair(BH, n, d.G, dtype, seed=38)
    (Y,) = seeded_qkvo(BH, n, 64, dtype, seed=39, count=1)
    Bp, Bcp = poison(Bd, Bc, n, w, wu, dil, gidx)
    X = empty_dense(d)
    getattr(swab, name)(d, 0.5, Bp.cuda(), Y.cuda(), X, (Bcp.cuda(), Br.cuda()))
    ref = oracle.band_t(f64(Bd), f64(Y), w, wu, dil, 0.5, gidx, f64(Bc), f64(Br))
    assert normwise(f64(X), ref) <= score_tol(dtype)


@pytest.mark.parametrize("case", CASES, ids=ids)
def test_band_softmax_bwd_globals(case):
    BH, n, w, wu, dil, dtype, gidx = case
    d = mk(*case)
    P = seeded_band(BH, n, d.D, dtype, seed=40)
    dP = seeded_band(BH, n, d.D, dtype, seed=41)
    Pc, Pr = glob_pair(BH, n, d.G, dtype, seed=42)
    dPc, dPr = glob_pair(BH, n, d.G, dtype, seed=44)
    Pp, Pcp = poison(P, Pc, n, w, wu, dil, gidx)
    dPp, dPcp = poison(dP, dPc, n, w, wu, dil, gidx)
    dS = empty_band(d)
    dSg = empty_glob(d)
    swab.band_softmax_bwd(d, Pp.cuda(), dPp.cuda(), dS, Pg=(Pcp.cuda(), Pr.cuda()),
                          dPg=(dPcp.cuda(), dPr.cuda()), dSg=dSg)
    rS, rSc, rSr = oracle.band_softmax_bwd(f64(P), f64(dP), w, wu, dil, gidx, f64(Pc), f64(dPc),
                                           f64(Pr), f64(dPr))
    tol = score_tol(dtype)
    assert normwise(f64(dS), rS) <= tol
    assert normwise(f64(dSg[0]), rSc) <= tol
    assert normwise(f64(dSg[1]), rSr) <= tol


# ---------------------------------------------------------------------------
# chains: forward + backward with globals against the definition
# ---------------------------------------------------------------------------
def gpu_chain_globals(d, Q, K, V, dO, scale):
    S, P, dP, dS = (empty_band(d) for _ in range(4))
    Sg, Pg, dPg, dSg = (empty_glob(d) for _ in range(4))
    lse = torch.empty((d.BH, d.n), dtype=torch.float32, device="cuda")
    O, dQ, dK, dV = (empty_dense(d) for _ in range(4))
    swab.band_qk(d, scale, Q, K, S, Sg)
    swab.band_softmax(d, S, P, lse, Sg=Sg, Pg=Pg)
    swab.band_pv(d, 1.0, P, V, O, Pg=Pg)
    swab.band_qk(d, 1.0, dO, V, dP, dPg)
    swab.band_softmax_bwd(d, P, dP, dS, Pg=Pg, dPg=dPg, dSg=dSg)
    swab.band_pv(d, scale, dS, K, dQ, Pg=dSg)
    swab.band_qk_bwd_t(d, scale, dS, Q, dK, dSg)
    swab.band_pv_bwd_t(d, 1.0, P, dO, dV, Pg)
    torch.cuda.synchronize()
    return dict(O=O, lse=lse, dQ=dQ, dK=dK, dV=dV)


def storage_bounds(d, q, k, v, go, scale):
    """Element-wise error bounds of the materialised bf16 chain with global
    tokens, derived from the roundings of its stored band and global tensors.

    Every stored value (S, P, dP, dS and the outputs) is one round-to-nearest
    of an fp32 result, so it carries a relative error of at most u = 2^-8.  To
    first order:
      |dP_ij err| (the softmax of rounded scores, then rounded)
          <= u P_ij (1 + |S_ij| + sum_k P_ik |S_ik|)                =: E_P
      |O_i err|   <= sum_j E_P,ij |v_j| + u |O_i|
      |dP err|    <= u |dP|                                          =: E_dP
      |delta err| <= sum_j (E_P |dP| + P E_dP)_ij                    =: E_delta
      |dS err|    <= E_P |dP - delta| + P (E_dP + E_delta) + u |dS|  =: E_dS
      |dQ err| <= scale sum_j E_dS,ij |k_j| + u |dQ|,  dK likewise with |q|,
      |dV err| <= sum_i E_P,ij |dO_i| + u |dV|.
    The first-order terms are doubled (second-order terms and the fp32 sums),
    and the plain 1e-2 of the other chains is added.  Row sums run over a
    row's band slots and global columns (local rows) or its dense row (global
    rows); the oracle's P is 0 on every slot attention does not use."""
    u = 2.0 ** -8
    w, wu, dil, gi = d.w, d.w_upper, d.dilation, d.global_idx
    S, Sc, Sr = oracle.band_qk(q, k, w, wu, dil, scale, 0.0, gi)
    P, _, Pc, Pr = oracle.band_softmax(S, w, wu, dil, gi, Sc, Sr)
    dP, dPc, dPr = oracle.band_qk(go, v, w, wu, dil, 1.0, 0.0, gi)
    dS, dSc, dSr = oracle.band_softmax_bwd(P, dP, w, wu, dil, gi, Pc, dPc, Pr, dPr)
    O = oracle.band_pv(P, v, w, wu, dil, 1.0, gi, Pc, Pr)

    def rowsum(b, c, r):  # per local row over band + cols; per global row over its dense row
        return b.sum(-1) + c.sum(-1), r.sum(-1)

    ls, gs = rowsum(P * np.abs(S), Pc * np.abs(Sc), Pr * np.abs(Sr))
    EP = u * P * (1 + np.abs(S) + ls[..., None])
    EPc = u * Pc * (1 + np.abs(Sc) + ls[..., None])
    EPr = u * Pr * (1 + np.abs(Sr) + gs[..., None])
    ld, gd = rowsum(P * dP, Pc * dPc, Pr * dPr)           # delta
    le, ge = rowsum(EP * np.abs(dP) + P * u * np.abs(dP), EPc * np.abs(dPc) + Pc * u * np.abs(dPc),
                    EPr * np.abs(dPr) + Pr * u * np.abs(dPr))   # its error
    EdS = EP * np.abs(dP - ld[..., None]) + P * (u * np.abs(dP) + le[..., None]) + u * np.abs(dS)
    EdSc = EPc * np.abs(dPc - ld[..., None]) + Pc * (u * np.abs(dPc) + le[..., None]) + u * np.abs(dSc)
    EdSr = EPr * np.abs(dPr - gd[..., None]) + Pr * (u * np.abs(dPr) + ge[..., None]) + u * np.abs(dSr)
    rq, rk, rv = oracle.attention_bwd(q, k, v, go, w, wu, dil, scale, gi)
    aq, ak, av, ago = (np.abs(x) for x in (q, k, v, go))
    first = {
        "O": oracle.band_pv(EP, av, w, wu, dil, 1.0, gi, EPc, EPr),
        "dQ": oracle.band_pv(EdS, ak, w, wu, dil, scale, gi, EdSc, EdSr),
        "dK": oracle.band_t(EdS, aq, w, wu, dil, scale, gi, EdSc, EdSr),
        "dV": oracle.band_t(EP, ago, w, wu, dil, 1.0, gi, EPc, EPr),
    }
    refs = {"O": O, "dQ": rq, "dK": rk, "dV": rv}
    return {nm: ABS_TOL + u * np.abs(refs[nm]) + 2.0 * first[nm] for nm in refs}


def check_chain_globals(d, Q, K, V, dO, scale, slices, derived_bf16_bound=False):
    out = gpu_chain_globals(d, *dev(Q, K, V, dO), scale)
    f32 = d.dtype == torch.float32
    for b in slices:
        sl = slice(b, b + 1)
        q, k, v, go = (f64(x[sl]) for x in (Q, K, V, dO))
        rO, rl = oracle.attention_fwd(q, k, v, d.w, d.w_upper, d.dilation, scale, d.global_idx)
        rq, rk, rv = oracle.attention_bwd(q, k, v, go, d.w, d.w_upper, d.dilation, scale,
                                          d.global_idx)
        bounds = storage_bounds(d, q, k, v, go, scale) if derived_bf16_bound else None
        for name, ref in (("O", rO), ("dQ", rq), ("dK", rk), ("dV", rv)):
            got = f64(out[name][sl])
            if f32:
                assert normwise(got, ref) <= 1e-5, name
            elif bounds is not None:
                assert np.all(np.abs(got - ref) <= bounds[name]), name
            else:
                assert within_abs(got, ref, d.dtype), name
        assert np.max(np.abs(f64(out["lse"][sl]) - rl)) <= (1e-5 if f32 else 2e-2)


@pytest.mark.parametrize("case", CASES, ids=ids)
def test_chain_globals_small(case):
    BH, n, w, wu, dil, dtype, gidx = case
    # A window of a handful of keys, with S, P, dP and dS each stored once in
    # bf16 (2^-8 relative each), puts the outputs beyond the plain 1e-2 + one
    # output rounding; that case is held to the bound derived from those
    # roundings (storage_bounds), in bf16.
    tiny_bf16 = dtype == torch.bfloat16 and w + wu + 1 < 32
    d = mk(BH, n, w, wu, dil, dtype, gidx)
    Q, K, V, dO = seeded_qkvo(BH, n, 64, dtype, seed=45)
    check_chain_globals(d, Q, K, V, dO, 0.125, range(BH), derived_bf16_bound=tiny_bf16)


def test_chain_config4_bf16_globals_sampled():
    wl = WORKLOADS[4]
    Q, K, V, dO = workload_inputs(wl)
    check_chain_globals(swab.Desc.from_workload(wl), Q, K, V, dO, wl.scale, slices=(0, 77, 143))
