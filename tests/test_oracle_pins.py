"""Pins for the fp64 CPU oracle (no GPU).

The oracle is checked against things other than itself:
  * torch fp64 dense attention with a mask built from the OFFSET condition
    (j - i = k*(dilation+1), k in [-w, w_upper]) -- a different formulation
    from the oracle's slot loop -- and torch autograd for the gradients;
  * closed forms: the valid slot range, full-window = dense softmax attention,
    one-sided window = causal attention (torch.tril mask);
  * invariants: softmax rows sum to 1, dilation = interleave of undilated
    bands on x[r::s], adjoint identities of the three banded products;
  * central finite differences of the forward;
  * a hand-worked tiny example (tests/golden/band_qk_tiny.txt);
  * planted mistakes: textual mutants of band_oracle.c must fail these pins.
"""
from __future__ import annotations

import ctypes
import os
import shutil
import subprocess
import tempfile

import numpy as np
import pytest
import torch

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
RNG_SEED = 4242


def rng(seed=RNG_SEED):
    return np.random.default_rng(seed)


def dense_mask(n, w, wu, dil, gidx=()):
    """Allowed (query, key) pairs from the offset condition, built with torch."""
    s = dil + 1
    i = torch.arange(n).view(-1, 1)
    j = torch.arange(n).view(1, -1)
    off = j - i
    m = (off >= -w * s) & (off <= wu * s) & (torch.remainder(off, s) == 0)
    if len(gidx):
        g = torch.zeros(n, dtype=torch.bool)
        g[list(gidx)] = True
        m = (m & ~g.view(1, -1)) | g.view(1, -1) | g.view(-1, 1)
    return m


def torch_attention(Q, K, V, mask, scale):
    """Dense masked softmax attention in fp64 (library routines only)."""
    s = scale * Q @ K.transpose(-1, -2)
    s = s.masked_fill(~mask, float("-inf"))
    return torch.softmax(s, -1) @ V, torch.logsumexp(s, -1)


def closed_form_range(i, n, w, wu, s):
    """First/last valid slot of row i: t_lo = max(0, w - floor(i/s)),
    t_hi = min(D-1, w + floor((n-1-i)/s))."""
    D = w + wu + 1
    return max(0, w - i // s), min(D - 1, w + (n - 1 - i) // s)


def randn(*shape, seed=0):
    return rng(seed).standard_normal(shape)


# --------------------------------------------------------------------------
# hand-worked example
# --------------------------------------------------------------------------
def load_golden():
    cases, cur = [], None
    with open(os.path.join(HERE, "golden", "band_qk_tiny.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if line.startswith("case"):
                _, w, wu, d = line.split()
                cur = (int(w), int(wu), int(d), [])
                cases.append(cur)
            else:
                cur[3].append([float(x) for x in line.split()])
    return cases


GOLD_Q = np.array([[1, 0], [0, 1], [1, 1], [2, 0], [0, 2]], dtype=np.float64)[None]
GOLD_K = np.array([[1, 2], [3, 4], [5, 6], [7, 8], [9, 10]], dtype=np.float64)[None]


def pin_golden():
    for w, wu, d, rows in load_golden():
        S = oracle.band_qk(GOLD_Q, GOLD_K, w, wu, d, alpha=1.0, padding=-7.0)
        np.testing.assert_array_equal(S[0], np.array(rows))


def test_golden_tiny():
    pin_golden()


# --------------------------------------------------------------------------
# band scores against the dense product
# --------------------------------------------------------------------------
SCORE_CASES = [  # n, w, w_upper, dilation
    (37, 5, 3, 0), (37, 4, 4, 2), (50, 3, 0, 1), (8, 20, 20, 0), (1, 2, 2, 0),
    (29, 0, 0, 0), (33, 0, 6, 3), (64, 16, 16, 0),
]


def pin_scores(n, w, wu, d, alpha=0.37, padding=-3.5):
    A, B = randn(2, n, 5, seed=1), randn(2, n, 5, seed=2)
    S = oracle.band_qk(A, B, w, wu, d, alpha=alpha, padding=padding)
    dense = alpha * torch.from_numpy(A) @ torch.from_numpy(B).transpose(-1, -2)
    mask = dense_mask(n, w, wu, d)
    s = d + 1
    for i in range(n):
        keys = torch.nonzero(mask[i]).flatten()
        lo, hi = closed_form_range(i, n, w, wu, s)
        assert len(keys) == hi - lo + 1
        np.testing.assert_allclose(S[:, i, lo:hi + 1], dense[:, i, keys].numpy(), rtol=1e-12,
                                   atol=1e-12)
        assert np.all(S[:, i, :lo] == padding) and np.all(S[:, i, hi + 1:] == padding)


@pytest.mark.parametrize("n,w,wu,d", SCORE_CASES)
def test_band_scores_vs_dense(n, w, wu, d):
    pin_scores(n, w, wu, d)


# --------------------------------------------------------------------------
# attention forward: definition and the per-kernel chain against torch
# --------------------------------------------------------------------------
ATTN_CASES = [  # n, hd, w, w_upper, dilation, global idx
    (24, 8, 30, 30, 0, ()),         # full window: dense attention
    (24, 8, 27, 0, 0, ()),          # one-sided window >= n: causal attention
    (41, 6, 4, 2, 0, ()),
    (41, 6, 3, 3, 1, ()),
    (45, 4, 2, 5, 3, ()),
    (40, 6, 3, 3, 0, (0, 1, 7, 39)),
    (43, 5, 2, 4, 2, (3, 20)),
    (12, 4, 2, 2, 0, tuple(range(12))),  # every token global: dense attention
]


def chain_fwd(Q, K, V, w, wu, d, scale, gidx):
    if gidx:
        S, Sg, Sr = oracle.band_qk(Q, K, w, wu, d, alpha=scale, padding=11.0, global_idx=gidx)
        P, lse, Pg, Pr = oracle.band_softmax(S, w, wu, d, gidx, Sg, Sr)
        O = oracle.band_pv(P, V, w, wu, d, 1.0, gidx, Pg, Pr)
    else:
        S = oracle.band_qk(Q, K, w, wu, d, alpha=scale, padding=11.0)
        P, lse = oracle.band_softmax(S, w, wu, d)
        O = oracle.band_pv(P, V, w, wu, d, 1.0)
    return O, lse


def pin_attention(n, hd, w, wu, d, gidx):
    Q, K, V = (randn(3, n, hd, seed=s) for s in (3, 4, 5))
    scale = 1.0 / np.sqrt(hd)
    mask = dense_mask(n, w, wu, d, gidx)
    O_t, lse_t = torch_attention(*(torch.from_numpy(x) for x in (Q, K, V)), mask, scale)
    O, lse = oracle.attention_fwd(Q, K, V, w, wu, d, scale, gidx)
    np.testing.assert_allclose(O, O_t.numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(lse, lse_t.numpy(), rtol=1e-12, atol=1e-12)
    O2, lse2 = chain_fwd(Q, K, V, w, wu, d, scale, gidx)
    np.testing.assert_allclose(O2, O_t.numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(lse2, lse_t.numpy(), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("n,hd,w,wu,d,gidx", ATTN_CASES)
def test_attention_vs_torch(n, hd, w, wu, d, gidx):
    pin_attention(n, hd, w, wu, d, gidx)


def test_causal_is_tril():
    """One-sided window covering the sequence = causal attention (torch.tril)."""
    n, hd = 19, 4
    Q, K, V = (randn(1, n, hd, seed=s) for s in (6, 7, 8))
    mask = torch.tril(torch.ones(n, n, dtype=torch.bool))
    O_t, _ = torch_attention(*(torch.from_numpy(x) for x in (Q, K, V)), mask, 0.5)
    O, _ = oracle.attention_fwd(Q, K, V, n + 3, 0, 0, 0.5)
    np.testing.assert_allclose(O, O_t.numpy(), rtol=1e-12, atol=1e-12)


def test_full_window_is_sdpa():
    """Full window = torch's scaled_dot_product_attention (no mask)."""
    n, hd = 21, 8
    Q, K, V = (randn(2, n, hd, seed=s) for s in (9, 10, 11))
    ref = torch.nn.functional.scaled_dot_product_attention(
        *(torch.from_numpy(x) for x in (Q, K, V)))
    O, _ = oracle.attention_fwd(Q, K, V, n, n, 0)
    np.testing.assert_allclose(O, ref.numpy(), rtol=1e-11, atol=1e-12)


# --------------------------------------------------------------------------
# softmax invariants
# --------------------------------------------------------------------------
def pin_softmax_rows(n=45, w=4, wu=6, d=1, gidx=(2, 9)):
    S = randn(2, n, w + wu + 1, seed=12) * 3
    Sg = randn(2, n, len(gidx), seed=13)
    Sr = randn(2, len(gidx), n, seed=14)
    P, lse, Pg, Pr = oracle.band_softmax(S, w, wu, d, gidx, Sg, Sr)
    s = d + 1
    g = set(gidx)
    for i in range(n):
        lo, hi = closed_form_range(i, n, w, wu, s)
        if i in g:
            assert np.all(P[:, i] == 0) and np.all(Pg[:, i] == 0)
            continue
        tot = P[:, i].sum(-1) + Pg[:, i].sum(-1)
        np.testing.assert_allclose(tot, 1.0, rtol=0, atol=1e-12)
        assert np.all(P[:, i, :lo] == 0) and np.all(P[:, i, hi + 1:] == 0)
        for t in range(lo, hi + 1):
            if i + (t - w) * s in g:
                assert np.all(P[:, i, t] == 0)
    np.testing.assert_allclose(Pr.sum(-1), 1.0, rtol=0, atol=1e-12)
    # no globals: rows sum to one over the closed-form range alone
    P0, _ = oracle.band_softmax(S, w, wu, d)
    np.testing.assert_allclose(P0.sum(-1), 1.0, rtol=0, atol=1e-12)


def test_softmax_rows_sum_to_one():
    pin_softmax_rows()


# --------------------------------------------------------------------------
# dilation = interleave of undilated bands on x[r::s]
# --------------------------------------------------------------------------
@pytest.mark.parametrize("d", [1, 3])
def test_dilation_interleave(d):
    n, hd, w, wu = 41, 5, 3, 2
    s = d + 1
    Q, K, V = (randn(2, n, hd, seed=s_) for s_ in (15, 16, 17))
    O, lse = oracle.attention_fwd(Q, K, V, w, wu, d, 0.4)
    S = oracle.band_qk(Q, K, w, wu, d, alpha=0.4, padding=-1.0)
    for r in range(s):
        sub = slice(r, None, s)
        O_r, lse_r = oracle.attention_fwd(Q[:, sub], K[:, sub], V[:, sub], w, wu, 0, 0.4)
        np.testing.assert_allclose(O[:, sub], O_r, rtol=1e-13, atol=1e-13)
        np.testing.assert_allclose(lse[:, sub], lse_r, rtol=1e-13, atol=1e-13)
        S_r = oracle.band_qk(Q[:, sub], K[:, sub], w, wu, 0, alpha=0.4, padding=-1.0)
        np.testing.assert_array_equal(S[:, sub], S_r)


# --------------------------------------------------------------------------
# adjoint identities of the three banded products
# --------------------------------------------------------------------------
def pin_adjoint(n=38, hd=6, w=5, wu=2, d=1, gidx=()):
    A, B = randn(2, n, hd, seed=18), randn(2, n, hd, seed=19)
    D = w + wu + 1
    X = randn(2, n, D, seed=20)
    # slots a consumer ignores carry no weight in <S, X>
    s = d + 1
    g = set(gidx)
    for i in range(n):
        for t in range(D):
            j = i + (t - w) * s
            if j < 0 or j >= n or j in g or i in g:
                X[:, i, t] = 0.0
    if gidx:
        G = len(gidx)
        Xg, Xr = randn(2, n, G, seed=21), randn(2, G, n, seed=22)
        Xg[:, list(gidx)] = 0.0
        S, Sg, Sr = oracle.band_qk(A, B, w, wu, d, 1.0, 0.0, gidx)
        lhs = (S * X).sum() + (Sg * Xg).sum() + (Sr * Xr).sum()
        mid = (A * oracle.band_pv(X, B, w, wu, d, 1.0, gidx, Xg, Xr)).sum()
        rhs = (B * oracle.band_t(X, A, w, wu, d, 1.0, gidx, Xg, Xr)).sum()
    else:
        S = oracle.band_qk(A, B, w, wu, d, 1.0, 0.0)
        lhs = (S * X).sum()
        mid = (A * oracle.band_pv(X, B, w, wu, d, 1.0)).sum()
        rhs = (B * oracle.band_t(X, A, w, wu, d, 1.0)).sum()
    assert abs(lhs - mid) <= 1e-12 * abs(lhs) + 1e-12
    assert abs(lhs - rhs) <= 1e-12 * abs(lhs) + 1e-12


@pytest.mark.parametrize("gidx", [(), (0, 5, 17)])
def test_adjoint_identities(gidx):
    pin_adjoint(gidx=gidx)


# --------------------------------------------------------------------------
# gradients
# --------------------------------------------------------------------------
GRAD_CASES = [  # n, hd, w, w_upper, dilation, gidx
    (33, 6, 4, 4, 0, ()),
    (37, 5, 3, 1, 2, ()),
    (30, 4, 3, 3, 0, (0, 4, 29)),
    (16, 4, 20, 0, 0, ()),
]


def torch_grads(Q, K, V, dO, mask, scale):
    t = [torch.from_numpy(x).clone().requires_grad_(True) for x in (Q, K, V)]
    O, _ = torch_attention(*t, mask, scale)
    O.backward(torch.from_numpy(dO))
    return [x.grad.numpy() for x in t]


def chain_bwd(Q, K, V, dO, w, wu, d, scale, gidx):
    """The backward as the five banded calls a GPU user makes."""
    if gidx:
        S, Sg, Sr = oracle.band_qk(Q, K, w, wu, d, scale, 0.0, gidx)
        P, _, Pg, Pr = oracle.band_softmax(S, w, wu, d, gidx, Sg, Sr)
        dP, dPg, dPr = oracle.band_qk(dO, V, w, wu, d, 1.0, 0.0, gidx)
        dS, dSg, dSr = oracle.band_softmax_bwd(P, dP, w, wu, d, gidx, Pg, dPg, Pr, dPr)
        dQ = oracle.band_pv(dS, K, w, wu, d, scale, gidx, dSg, dSr)
        dK = oracle.band_t(dS, Q, w, wu, d, scale, gidx, dSg, dSr)
        dV = oracle.band_t(P, dO, w, wu, d, 1.0, gidx, Pg, Pr)
    else:
        S = oracle.band_qk(Q, K, w, wu, d, scale, 0.0)
        P, _ = oracle.band_softmax(S, w, wu, d)
        dP = oracle.band_qk(dO, V, w, wu, d, 1.0, 0.0)
        dS = oracle.band_softmax_bwd(P, dP, w, wu, d)
        dQ = oracle.band_pv(dS, K, w, wu, d, scale)
        dK = oracle.band_t(dS, Q, w, wu, d, scale)
        dV = oracle.band_t(P, dO, w, wu, d, 1.0)
    return dQ, dK, dV


def pin_grads(n, hd, w, wu, d, gidx):
    Q, K, V, dO = (randn(2, n, hd, seed=s) for s in (23, 24, 25, 26))
    scale = 0.45
    ref = torch_grads(Q, K, V, dO, dense_mask(n, w, wu, d, gidx), scale)
    for got in (oracle.attention_bwd(Q, K, V, dO, w, wu, d, scale, gidx),
                chain_bwd(Q, K, V, dO, w, wu, d, scale, gidx)):
        for g, r in zip(got, ref):
            np.testing.assert_allclose(g, r, rtol=1e-10, atol=1e-11)


@pytest.mark.parametrize("n,hd,w,wu,d,gidx", GRAD_CASES)
def test_grads_vs_autograd(n, hd, w, wu, d, gidx):
    pin_grads(n, hd, w, wu, d, gidx)


def test_grads_finite_difference():
    n, hd, w, wu, d, gidx = 12, 3, 2, 1, 1, (5,)
    Q, K, V, dO = (randn(1, n, hd, seed=s) for s in (27, 28, 29, 30))
    scale, h = 0.7, 1e-6
    grads = oracle.attention_bwd(Q, K, V, dO, w, wu, d, scale, gidx)

    def loss(Q_, K_, V_):
        return float((oracle.attention_fwd(Q_, K_, V_, w, wu, d, scale, gidx)[0] * dO).sum())

    for which, g in enumerate(grads):
        for idx in [(0, 0, 0), (0, 5, 1), (0, 7, 2), (0, 11, 0), (0, 3, 1)]:
            args = [Q.copy(), K.copy(), V.copy()]
            args[which][idx] += h
            up = loss(*args)
            args[which][idx] -= 2 * h
            dn = loss(*args)
            fd = (up - dn) / (2 * h)
            assert abs(fd - g[idx]) <= 1e-6 * max(1.0, abs(fd)), (which, idx, fd, g[idx])


def test_bad_global_index_rejected():
    A = randn(1, 10, 2)
    for bad in ((3, 3), (5, 2), (10,), (-1,)):
        with pytest.raises(ValueError):
            oracle.band_qk(A, A, 1, 1, 0, global_idx=bad)


# --------------------------------------------------------------------------
# planted mistakes: every mutant of the oracle must fail at least one pin
# --------------------------------------------------------------------------
# ---------------------------------------------------------------------------
# key-padding bias: nvFuser issue "HuggingFace BertForMaskedLM - Log Softmax
# Fusion with Autocast has bad perf", fusion 1 adds (1 - mask) * -10000 per key
# to the scaled scores before the softmax
# ---------------------------------------------------------------------------
BIAS_CASES = [  # n, hd, w, w_upper, dilation
    (41, 6, 4, 2, 0),
    (45, 4, 2, 5, 3),
    (24, 8, 30, 30, 0),
]


def key_bias(BH, n, seed):
    """(1 - mask) * -10000 for a random 0/1 key mask, plus small per-key terms."""
    rng = np.random.default_rng(seed)
    keep = rng.random((BH, n)) > 0.25
    return np.where(keep, 0.0, -10000.0) + 0.3 * rng.standard_normal((BH, n))


def torch_attention_bias(Q, K, V, mask, scale, kb):
    s = scale * Q @ K.transpose(-1, -2) + kb[:, None, :]
    s = s.masked_fill(~mask, float("-inf"))
    return torch.softmax(s, -1) @ V, torch.logsumexp(s, -1)


def pin_bias(n, hd, w, wu, d, gidx=()):
    Q, K, V, dO = (randn(3, n, hd, seed=s) for s in (61, 62, 63, 64))
    kb = key_bias(3, n, seed=65)
    scale = 1.0 / np.sqrt(hd)
    mask = dense_mask(n, w, wu, d, gidx)
    tQ, tK, tV, tb = (torch.from_numpy(x) for x in (Q, K, V, kb))
    O_t, lse_t = torch_attention_bias(tQ, tK, tV, mask, scale, tb)
    gi = list(gidx) or None
    O, lse = oracle.attention_fwd(Q, K, V, w, wu, d, scale, global_idx=gi, key_bias=kb)
    np.testing.assert_allclose(O, O_t.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(lse, lse_t.numpy(), rtol=1e-12, atol=1e-9)
    if gidx:
        # gradients against autograd of the dense reference
        t = [x.clone().requires_grad_(True) for x in (tQ, tK, tV)]
        O_a, _ = torch_attention_bias(*t, mask, scale, tb)
        O_a.backward(torch.from_numpy(dO))
        got = oracle.attention_bwd(Q, K, V, dO, w, wu, d, scale, global_idx=gi, key_bias=kb)
        for g, r in zip(got, t):
            np.testing.assert_allclose(g, r.grad.numpy(), rtol=1e-9, atol=1e-11)
        # the materialised forward with global tokens: the bias in band_softmax
        # reaches the band slots, the global columns and the global rows
        S, Sg, Sr = oracle.band_qk(Q, K, w, wu, d, alpha=scale, padding=11.0, global_idx=gi)
        P, lse2, Pg, Pr = oracle.band_softmax(S, w, wu, d, global_idx=gi, Sg=Sg, Sr=Sr, key_bias=kb)
        O2 = oracle.band_pv(P, V, w, wu, d, 1.0, global_idx=gi, Pg=Pg, Pr=Pr)
        np.testing.assert_allclose(O2, O_t.numpy(), rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(lse2, lse_t.numpy(), rtol=1e-12, atol=1e-9)
        return
    # the materialised chain with the bias in band_softmax
    S = oracle.band_qk(Q, K, w, wu, d, alpha=scale, padding=11.0)
    P, lse2 = oracle.band_softmax(S, w, wu, d, key_bias=kb)
    O2 = oracle.band_pv(P, V, w, wu, d, 1.0)
    np.testing.assert_allclose(O2, O_t.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(lse2, lse_t.numpy(), rtol=1e-12, atol=1e-9)
    # gradients against autograd of the dense reference
    t = [x.clone().requires_grad_(True) for x in (tQ, tK, tV)]
    O_a, _ = torch_attention_bias(*t, mask, scale, tb)
    O_a.backward(torch.from_numpy(dO))
    got = oracle.attention_bwd(Q, K, V, dO, w, wu, d, scale, key_bias=kb)
    for g, r in zip(got, t):
        np.testing.assert_allclose(g, r.grad.numpy(), rtol=1e-9, atol=1e-11)


@pytest.mark.parametrize("n,hd,w,wu,d", BIAS_CASES)
def test_key_bias_vs_torch(n, hd, w, wu, d):
    pin_bias(n, hd, w, wu, d)


# The key-padding bias with global tokens: the bias is added to the scaled
# score of every key a row attends to, whatever its key set -- the band keys
# and the global columns of a local row, every key of a global row (the
# additive mask of the nvFuser fusion applied to the attention of ONNX
# Runtime's item (1)).
BIAS_GLOBAL_CASES = [  # n, hd, w, w_upper, dilation, global idx
    (41, 6, 4, 2, 0, (0, 7, 40)),
    (45, 4, 2, 5, 3, (3, 4, 22)),
    (24, 8, 30, 30, 0, (11,)),
]


@pytest.mark.parametrize("n,hd,w,wu,d,gidx", BIAS_GLOBAL_CASES)
def test_key_bias_with_globals_vs_torch(n, hd, w, wu, d, gidx):
    pin_bias(n, hd, w, wu, d, gidx)


def test_key_bias_constant_is_a_shift():
    """A bias equal for every key leaves P and O unchanged and shifts lse by it."""
    n, hd, w, wu, d = 33, 5, 3, 4, 1
    Q, K, V = (randn(2, n, hd, seed=s) for s in (66, 67, 68))
    O0, lse0 = oracle.attention_fwd(Q, K, V, w, wu, d, 0.4)
    O1, lse1 = oracle.attention_fwd(Q, K, V, w, wu, d, 0.4, key_bias=np.full((2, n), 2.5))
    np.testing.assert_allclose(O1, O0, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse1, lse0 + 2.5, rtol=1e-13, atol=1e-12)


def test_key_bias_huge_negative_removes_keys():
    """A bias of -1e6 on a key removes it from every row's key set."""
    n, hd, w, wu, d = 30, 4, 5, 5, 0
    Q, K, V = (randn(1, n, hd, seed=s) for s in (69, 70, 71))
    gone = [3, 4, 17]
    kb = np.zeros((1, n))
    kb[0, gone] = -1e6
    mask = dense_mask(n, w, wu, d)
    mask[:, gone] = False
    mask[gone, :] = mask[gone, :] | torch.eye(n, dtype=torch.bool)[gone]  # keep rows non-empty
    O, _ = oracle.attention_fwd(Q, K, V, w, wu, d, 0.5, key_bias=kb)
    rows = [i for i in range(n) if i not in gone]
    O_t, _ = torch_attention(*(torch.from_numpy(x) for x in (Q, K, V)), mask, 0.5)
    np.testing.assert_allclose(O[:, rows], O_t.numpy()[:, rows], rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------------------
# dropout of the probabilities (nvFuser issue, fusion 1: p with 1/(1-p)
# scaling) from the counter-based generator Philox4x64-10 (Salmon et al.,
# SC'11), pinned to numpy's implementation of the same generator
# ---------------------------------------------------------------------------
def numpy_philox_block(counter, key):
    """The Philox4x64-10 block at `counter` from numpy (which advances the
    counter before producing a block)."""
    c = np.array(counter, dtype=np.uint64)
    c[0] -= np.uint64(1)  # the tests use counter[0] >= 1
    bg = np.random.Philox(key=np.array(key, dtype=np.uint64), counter=c)
    return bg.random_raw(4).astype(np.uint64)


@pytest.mark.parametrize("counter,key", [((1, 0, 0, 0), (0, 0)), ((5, 7, 3, 0), (2024, 0)),
                                         ((1 << 40, 99, 12, 0), (0xDEADBEEF12345678, 0))])
def test_philox_matches_numpy(counter, key):
    np.testing.assert_array_equal(oracle.philox4x64(counter, key), numpy_philox_block(counter, key))


def test_dropout_factor_definition():
    """Element (bh, i, j): byte (b mod 32) of the block at (b // 32, i, bh, 0),
    b = j // s, little-endian bytes of the four words; kept iff byte >= t."""
    rng = np.random.default_rng(5)
    for _ in range(40):
        seed, t = int(rng.integers(1, 1 << 62)), int(rng.integers(1, 256))
        bh, i, s = int(rng.integers(0, 50)), int(rng.integers(0, 5000)), int(rng.integers(1, 4))
        j = int(rng.integers(32 * s, 5000))
        b = j // s
        blk = numpy_philox_block((b // 32, i, bh, 0), (seed, 0))
        k = b % 32
        byte = (int(blk[k // 8]) >> (8 * (k % 8))) & 0xFF
        want = 256.0 / (256.0 - t) if byte >= t else 0.0
        assert oracle.dropout_factor(seed, t, bh, i, j, s) == want


def test_dropout_keep_fraction():
    t, seed, kept, tot = 26, 77, 0, 0
    for i in range(64):
        for j in range(0, 2048, 3):
            kept += oracle.dropout_factor(seed, t, 1, i, j, 1) > 0
            tot += 1
    frac = kept / tot
    expect = 1 - t / 256
    assert abs(frac - expect) < 5 * np.sqrt(expect * (1 - expect) / tot)


def dense_drop_factors(BH, n, s, seed, t):
    F = np.ones((BH, n, n))
    for bh in range(BH):
        for i in range(n):
            for j in range(n):
                F[bh, i, j] = oracle.dropout_factor(seed, t, bh, i, j, s)
    return F


DROP_CASES = [  # n, hd, w, w_upper, dilation, threshold
    (37, 5, 4, 3, 0, 26),
    (41, 4, 3, 5, 2, 77),
]


@pytest.mark.parametrize("n,hd,w,wu,d,t", DROP_CASES)
def test_dropout_attention_vs_torch(n, hd, w, wu, d, t):
    Q, K, V, dO = (randn(2, n, hd, seed=sd) for sd in (81, 82, 83, 84))
    scale, seed = 0.4, 1234567
    F = torch.from_numpy(dense_drop_factors(2, n, d + 1, seed, t))
    mask = dense_mask(n, w, wu, d)
    t_in = [torch.from_numpy(x).clone().requires_grad_(True) for x in (Q, K, V)]
    sc = scale * t_in[0] @ t_in[1].transpose(-1, -2)
    sc = sc.masked_fill(~mask, float("-inf"))
    O_t = (torch.softmax(sc, -1) * F) @ t_in[2]
    O_t.backward(torch.from_numpy(dO))
    O, lse = oracle.attention_fwd(Q, K, V, w, wu, d, scale, drop_t=t, seed=seed)
    np.testing.assert_allclose(O, O_t.detach().numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(lse, torch.logsumexp(sc, -1).detach().numpy(), rtol=1e-12,
                               atol=1e-12)
    got = oracle.attention_bwd(Q, K, V, dO, w, wu, d, scale, drop_t=t, seed=seed)
    for g, r in zip(got, t_in):
        np.testing.assert_allclose(g, r.grad.numpy(), rtol=1e-9, atol=1e-11)
    # the materialised chain: band_softmax writes P and the dropped Pd, P.V
    # uses Pd, and band_softmax_bwd takes P with the gradient of Pd
    S = oracle.band_qk(Q, K, w, wu, d, alpha=scale, padding=-3.0)
    P, lse2, Pd = oracle.band_softmax(S, w, wu, d, drop_t=t, seed=seed)
    np.testing.assert_allclose(oracle.band_pv(Pd, V, w, wu, d), O_t.detach().numpy(),
                               rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(lse2, lse, rtol=1e-13, atol=1e-13)
    dPd = oracle.band_qk(dO, V, w, wu, d)
    dS = oracle.band_softmax_bwd(P, dPd, w, wu, d, drop_t=t, seed=seed)
    chain = (oracle.band_pv(dS, K, w, wu, d, alpha=scale), oracle.band_t(dS, Q, w, wu, d, scale),
             oracle.band_t(Pd, dO, w, wu, d))
    for g, r in zip(chain, t_in):
        np.testing.assert_allclose(g, r.grad.numpy(), rtol=1e-9, atol=1e-11)
    # threshold 0 is no dropout
    O0, _ = oracle.attention_fwd(Q, K, V, w, wu, d, scale, drop_t=0, seed=seed)
    O1, _ = oracle.attention_fwd(Q, K, V, w, wu, d, scale)
    np.testing.assert_array_equal(O0, O1)


def pin_dropout():
    test_dropout_attention_vs_torch(*DROP_CASES[0])


# ---------------------------------------------------------------------------
# AddBiasTranspose (ONNX Runtime issue, item (2)) against numpy broadcasting and
# an axis permutation
# ---------------------------------------------------------------------------
ABT_CASES = [(1, 7, 3, 2, 4), (2, 5, 1, 3, 8), (3, 4, 2, 1, 2)]  # b, n, M, h, hd


@pytest.mark.parametrize("b,n,M,h,hd", ABT_CASES)
def test_add_bias_transpose_vs_numpy(b, n, M, h, hd):
    rng = np.random.default_rng(b * 100 + n)
    X = rng.standard_normal((b, n, M, h, hd))
    bias = rng.standard_normal((M, h, hd))
    want = np.transpose(X + bias[None, None], (2, 0, 3, 1, 4))
    np.testing.assert_array_equal(oracle.add_bias_transpose(X, bias), want)
    np.testing.assert_array_equal(oracle.add_bias_transpose(X), np.transpose(X, (2, 0, 3, 1, 4)))


def test_add_bias_transpose_is_a_permutation():
    """Without a bias every input value lands in exactly one place: distinct
    integers come out as the same multiset, each at its own index."""
    b, n, M, h, hd = 2, 3, 3, 2, 4
    X = np.arange(b * n * M * h * hd, dtype=np.float64).reshape(b, n, M, h, hd)
    Y = oracle.add_bias_transpose(X)
    np.testing.assert_array_equal(np.sort(Y.ravel()), X.ravel())
    for (m, bb, hh, i, c) in [(0, 0, 0, 0, 0), (2, 1, 1, 2, 3), (1, 0, 1, 2, 0)]:
        assert Y[m, bb, hh, i, c] == (((bb * n + i) * M + m) * h + hh) * hd + c


def pin_add_bias_transpose():
    for c in ABT_CASES:
        test_add_bias_transpose_vs_numpy(*c)
    test_add_bias_transpose_is_a_permutation()


# ---------------------------------------------------------------------------
# global queries with their own projections (ONNX Runtime issue, item (3) and
# the compact global_q): dense attention of G compact queries over every key
# ---------------------------------------------------------------------------
GA_CASES = [(2, 3, 17, 5), (1, 1, 9, 4), (3, 4, 23, 8)]  # BH, G, n, hd


@pytest.mark.parametrize("BH,G,n,hd", GA_CASES)
def test_global_attention_vs_torch(BH, G, n, hd):
    rng = np.random.default_rng(BH * 97 + n)
    Qg, dOg = rng.standard_normal((BH, G, hd)), rng.standard_normal((BH, G, hd))
    Kg, Vg = rng.standard_normal((BH, n, hd)), rng.standard_normal((BH, n, hd))
    scale = 0.3
    t = [torch.from_numpy(x).clone().requires_grad_(True) for x in (Qg, Kg, Vg)]
    sc = scale * t[0] @ t[1].transpose(-1, -2)
    O_t = torch.softmax(sc, -1) @ t[2]
    O_t.backward(torch.from_numpy(dOg))
    Og, lseg = oracle.global_attention_fwd(Qg, Kg, Vg, scale)
    np.testing.assert_allclose(Og, O_t.detach().numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(lseg, torch.logsumexp(sc, -1).detach().numpy(), rtol=1e-12,
                               atol=1e-12)
    got = oracle.global_attention_bwd(Qg, Kg, Vg, dOg, scale)
    for g, r in zip(got, t):
        np.testing.assert_allclose(g, r.grad.numpy(), rtol=1e-9, atol=1e-11)


def test_global_attention_equals_shared_projection_rows():
    """With Qg = Q[G], Kg = K, Vg = V the global queries' outputs are the global
    rows of the attention with global tokens (key sets on explicit lists)."""
    BH, n, hd, w, wu = 2, 40, 6, 3, 2
    gidx = [0, 7, 31]
    Q, K, V = (randn(BH, n, hd, seed=s) for s in (91, 92, 93))
    O, lse = oracle.attention_fwd(Q, K, V, w, wu, 0, 0.4, global_idx=gidx)
    Og, lseg = oracle.global_attention_fwd(Q[:, gidx], K, V, 0.4)
    np.testing.assert_allclose(Og, O[:, gidx], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lseg, lse[:, gidx], rtol=1e-13, atol=1e-13)


def test_separate_global_projections_composition():
    """Longformer-style attention with separate global projections: local rows
    attend to their band keys outside G plus G (projections Q, K, V); global
    rows attend to every key through Qg (compact), Kg, Vg.  The composition --
    the band path with global_idx for the local rows, global_attention for the
    global rows, and in the backward dO's global rows zeroed for the band path
    and handed to global_attention_bwd -- equals dense torch attention under
    autograd."""
    BH, n, hd, w, wu, d = 2, 36, 5, 3, 4, 1
    gidx = [1, 12, 30]
    Q, K, V, dO = (randn(BH, n, hd, seed=s) for s in (101, 102, 103, 104))
    Qg = randn(BH, len(gidx), hd, seed=105)
    Kg, Vg = randn(BH, n, hd, seed=106), randn(BH, n, hd, seed=107)
    scale = 0.45
    t = [torch.from_numpy(x).clone().requires_grad_(True) for x in (Q, K, V, Qg, Kg, Vg)]
    mask = dense_mask(n, w, wu, d, gidx)
    local, _ = torch_attention(t[0], t[1], t[2], mask, scale)
    glob = torch.softmax(scale * t[3] @ t[4].transpose(-1, -2), -1) @ t[5]
    is_g = torch.zeros(n, dtype=torch.bool)
    is_g[gidx] = True
    out = local.clone()
    out[:, gidx] = glob
    out.backward(torch.from_numpy(dO))
    O, _ = oracle.attention_fwd(Q, K, V, w, wu, d, scale, global_idx=gidx)
    Og, _ = oracle.global_attention_fwd(Qg, Kg, Vg, scale)
    O[:, gidx] = Og
    np.testing.assert_allclose(O, out.detach().numpy(), rtol=1e-10, atol=1e-12)
    dO_local = dO.copy()
    dO_local[:, gidx] = 0.0
    grads = (oracle.attention_bwd(Q, K, V, dO_local, w, wu, d, scale, global_idx=gidx) +
             oracle.global_attention_bwd(Qg, Kg, Vg, dO[:, gidx], scale))
    for g, r in zip(grads, t):
        np.testing.assert_allclose(g, r.grad.numpy(), rtol=1e-9, atol=1e-11)


def pin_global_attention():
    for c in GA_CASES:
        test_global_attention_vs_torch(*c)
    test_global_attention_equals_shared_projection_rows()
    test_separate_global_projections_composition()


MUTANTS = {
    "key_offset": ("(long long)(t - w) * s;", "(long long)(t - w + 1) * s;"),
    "stride": ("const int D = w + wu + 1, s = dil + 1;",
               "const int D = w + wu + 1, s = dil + 1 + (dil > 0);"),
    "softmax_no_divide": ("? exp(srow[t] - m) / z : 0.0;", "? exp(srow[t] - m) : 0.0;"),
    "pv_alpha_dropped": ("for (int c = 0; c < hd; ++c) o[c] *= alpha;", ""),
    "t_operand": ("x[(size_t)j * hd + c] += alpha * b[t] * yi;",
                  "x[(size_t)j * hd + c] += alpha * b[t] * y[(size_t)j * hd + c];"),
    "softmax_bwd_sign": ("dP[r * D + t] - delta)", "dP[r * D + t] + delta)"),
    "softmax_bwd_dropout_delta": (
        """delta += P[r * D + t] * drop_factor(seed, drop_t, bh, i, i + (t - w) * s, s) *
                             dP[r * D + t];""", "delta += P[r * D + t] * dP[r * D + t];"),
    "softmax_dropped_unscaled": ("? drop_factor(seed, drop_t, bh, i, i + (t - w) * s, s) * prow[t]",
                                 "? (drop_factor(seed, drop_t, bh, i, i + (t - w) * s, s) > 0) *"
                                 " prow[t]"),
    "bwd_dk_scale": ("+= scale * sbuf[(size_t)bh * nnz + u] * qi;",
                     "+= sbuf[(size_t)bh * nnz + u] * qi;"),
    "global_cols_dropped_from_sum": (
        "for (int q = 0; q < G; ++q) z += exp(XG(q) - m);", ""),
    "global_key_not_excluded": ("if (gmask && gmask[j]) return 0;", ""),
    "global_cols_key_bias_ignored": ("(kbias ? kbias[(size_t)bh * n + gidx[q]] : 0.0)", "0.0"),
    "global_rows_key_bias_ignored": ("(kbias ? kbias[(size_t)bh * n + (j)] : 0.0)", "0.0"),
    "key_bias_ignored": ("(kbias ? kbias[(size_t)bh * n + ks.key[b0 + u]] : 0.0)", "0.0"),
    "softmax_key_bias_ignored": ("((kbias && j >= 0 && j < n) ? kbias[(size_t)bh * n + j] : 0.0)",
                                 "0.0"),
    "dropout_factor_dropped": ("""                    const double p = exp(x[u] - m) / z *
                                     drop_factor(seed, drop_t, bh, i, ks.key[b0 + u], s_);""",
                               """                    const double p = exp(x[u] - m) / z;"""),
    "abt_m_h_swapped": ("const size_t src = ((((size_t)bb * n + i) * M + m) * h + hh) * hd + c;",
                        "const size_t src = ((((size_t)bb * n + i) * h + hh) * M + m) * hd + c;"),
    "abt_bias_index": ("bias[((size_t)m * h + hh) * hd + c]", "bias[((size_t)hh * M + m) * hd + c]"),
    "global_attention_delta": ("const double delta = dot(dO, o, hd);", "const double delta = 0.0;"),
    "global_attention_dk_scale": ("dK[(size_t)j * hd + c] += scale * ds * q[c];",
                                  "dK[(size_t)j * hd + c] += ds * q[c];"),
    "dropout_byte_order": ("(out[k / 8] >> (8 * (k % 8)))", "(out[k % 4] >> (8 * (k / 4)))"),
    "qk_transposed": ("srow[t] = alpha * dot(a, B + ((size_t)bh * n + j) * hd, hd);",
                      "srow[t] = alpha * dot(B + ((size_t)bh * n + i) * hd,"
                      " A + ((size_t)bh * n + j) * hd, hd);"),
}


def run_all_pins():
    pin_golden()
    for c in SCORE_CASES:
        pin_scores(*c)
    for c in ATTN_CASES:
        pin_attention(*c)
    pin_softmax_rows()
    pin_adjoint()
    pin_adjoint(gidx=(0, 5, 17))
    for c in GRAD_CASES:
        pin_grads(*c)
    for c in BIAS_CASES:
        pin_bias(*c)
    for c in BIAS_GLOBAL_CASES:
        pin_bias(*c)
    pin_dropout()
    test_dropout_factor_definition()
    pin_add_bias_transpose()
    pin_global_attention()


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_fails_pins(name):
    old, new = MUTANTS[name]
    with open(os.path.join(os.path.dirname(oracle.__file__), "band_oracle.c")) as f:
        src = f.read()
    assert old in src, f"mutation anchor for {name} not found"
    with tempfile.TemporaryDirectory() as tmp:
        c = os.path.join(tmp, "mutant.c")
        so = os.path.join(tmp, "mutant.so")
        with open(c, "w") as f:
            f.write(src.replace(old, new))
        subprocess.check_call(["gcc", "-O1", "-std=c99", "-fopenmp", "-fPIC", "-shared", "-o",
                               so, c, "-lm"])
        saved = oracle._load()  # the real library, typed; the mutant borrows its signatures
        try:
            mut = ctypes.CDLL(so)
            for fname in ("orc_num_threads", "orc_band_qk", "orc_band_softmax", "orc_band_pv",
                          "orc_band_t", "orc_band_softmax_bwd", "orc_attention_fwd",
                          "orc_attention_bwd", "orc_philox4x64", "orc_dropout_factor",
                          "orc_add_bias_transpose", "orc_global_attention_fwd",
                          "orc_global_attention_bwd"):
                src_f, dst_f = getattr(oracle._lib, fname), getattr(mut, fname)
                dst_f.argtypes, dst_f.restype = src_f.argtypes, src_f.restype
            oracle._lib = mut
            with pytest.raises(AssertionError):
                run_all_pins()
        finally:
            oracle._lib = saved


def test_real_oracle_passes_all_pins():
    run_all_pins()
