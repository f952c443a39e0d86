"""fp64 CPU oracle for sliding-window (banded) attention.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  It shares no code with the CUDA library (``band_oracle.c`` is plain C
compiled with gcc) and the library never calls it.

Every function takes and returns float64 numpy arrays in the layouts below and
follows the definitions written at the top of ``band_oracle.c``:

* dense tensors ``[BH, n, hd]``; band tensors ``[BH, n, D]`` with
  ``D = w + w_upper + 1`` and slot ``t`` holding key ``i + (t - w) * (dilation+1)``;
* global pieces: ``cols`` ``[BH, n, G]`` (row i at key G[g]) and ``rows``
  ``[BH, G, n]`` (dense row of query G[g]); ``lse`` ``[BH, n]``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "band_oracle.c")
_LIBDIR = os.path.join(_HERE, "_lib")
_LIB = os.path.join(_LIBDIR, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile band_oracle.c into oracle/_lib/liboracle.so with gcc + OpenMP."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    os.makedirs(_LIBDIR, exist_ok=True)
    tmp = _LIB + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-std=c99", "-fopenmp", "-fPIC", "-shared",
                           "-o", tmp, _SRC, "-lm"])
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        d = ctypes.c_double
        i = ctypes.c_int
        p = ctypes.c_void_p
        _lib.orc_num_threads.restype = i
        _lib.orc_band_qk.argtypes = [i, i, i, i, i, i, d, d, p, p, p, i, p, p, p]
        u64 = ctypes.c_uint64
        _lib.orc_band_softmax.argtypes = [i, i, i, i, i, p, p, p, i, p, p, p, p, p, p, u64, i, p]
        _lib.orc_band_pv.argtypes = [i, i, i, i, i, i, d, p, p, p, i, p, p, p]
        _lib.orc_band_t.argtypes = [i, i, i, i, i, i, d, p, p, p, i, p, p, p]
        _lib.orc_band_softmax_bwd.argtypes = [i, i, i, i, i, p, p, p, i, p, p, p, p, p, p, p, u64,
                                              i]
        _lib.orc_attention_fwd.argtypes = [i, i, i, i, i, i, d, p, p, p, p, p, i, p, p, u64, i]
        _lib.orc_attention_bwd.argtypes = [i, i, i, i, i, i, d, p, p, p, p, p, p, p, i, p, p,
                                           u64, i]
        _lib.orc_philox4x64.argtypes = [p, p, p]
        _lib.orc_philox4x64.restype = i
        _lib.orc_dropout_factor.argtypes = [u64, i, i, i, i, i, ctypes.POINTER(ctypes.c_double)]
        _lib.orc_dropout_factor.restype = i
        _lib.orc_add_bias_transpose.argtypes = [i, i, i, i, i, p, p, p]
        _lib.orc_global_attention_fwd.argtypes = [i, i, i, i, d, p, p, p, p, p]
        _lib.orc_global_attention_bwd.argtypes = [i, i, i, i, d, p, p, p, p, p, p, p]
        for f in ("orc_add_bias_transpose", "orc_global_attention_fwd", "orc_global_attention_bwd", "orc_band_qk", "orc_band_softmax", "orc_band_pv",
                  "orc_band_t",
                  "orc_band_softmax_bwd", "orc_attention_fwd", "orc_attention_bwd"):
            getattr(_lib, f).restype = i
    return _lib


def num_threads() -> int:
    """Threads the oracle's OpenMP loops use (the host's cores unless limited)."""
    return int(_load().orc_num_threads())


def _f64(x):
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _gidx(global_idx):
    if global_idx is None or len(global_idx) == 0:
        return 0, None
    g = np.ascontiguousarray(np.asarray(global_idx, dtype=np.int32))
    return int(g.size), g


def _check(rc, name):
    if rc != 0:
        raise ValueError(f"{name}: bad arguments (code {rc})")


def band_qk(A, B, w, w_upper, dilation=0, alpha=1.0, padding=0.0, global_idx=None):
    """S = alpha * A.B^T on the band (+ global cols / rows).  Returns S or (S, Sg, Sr)."""
    A, B = _f64(A), _f64(B)
    BH, n, hd = A.shape
    D = w + w_upper + 1
    G, g = _gidx(global_idx)
    S = np.empty((BH, n, D))
    Sg = np.empty((BH, n, G)) if G else None
    Sr = np.empty((BH, G, n)) if G else None
    _check(_load().orc_band_qk(BH, n, hd, w, w_upper, dilation, alpha, padding, _ptr(A),
                               _ptr(B), _ptr(S), G, _ptr(g), _ptr(Sg), _ptr(Sr)), "band_qk")
    return (S, Sg, Sr) if G else S


def _kbias(key_bias, BH, n):
    """Key bias given per slice [BH, n] (callers expand a [b, n] bias over the heads)."""
    if key_bias is None:
        return None
    kb = _f64(key_bias)
    if kb.shape != (BH, n):
        raise ValueError(f"key_bias must be [BH, n] = {(BH, n)}, got {kb.shape}")
    return kb


def band_softmax(S, w, w_upper, dilation=0, global_idx=None, Sg=None, Sr=None, key_bias=None,
                 drop_t=0, seed=0):
    """Masked row softmax (key_bias[bh, j] added to the score of key j).  Returns
    (P, lse) or (P, lse, Pg, Pr) with globals; with dropout (threshold byte
    drop_t > 0) (P, lse, Pd), Pd the dropped and rescaled probabilities."""
    S = _f64(S)
    BH, n, D = S.shape
    kb = _kbias(key_bias, BH, n)
    G, g = _gidx(global_idx)
    P = np.empty_like(S)
    Pd = np.empty_like(S) if drop_t else None
    lse = np.empty((BH, n))
    Pg = np.empty((BH, n, G)) if G else None
    Pr = np.empty((BH, G, n)) if G else None
    Sg = _f64(Sg) if G else None
    Sr = _f64(Sr) if G else None
    _check(_load().orc_band_softmax(BH, n, w, w_upper, dilation, _ptr(S), _ptr(P), _ptr(lse),
                                    G, _ptr(g), _ptr(Sg), _ptr(Sr), _ptr(Pg), _ptr(Pr), _ptr(kb),
                                    seed, drop_t, _ptr(Pd)),
           "band_softmax")
    if drop_t:
        return P, lse, Pd
    return (P, lse, Pg, Pr) if G else (P, lse)


def band_pv(P, V, w, w_upper, dilation=0, alpha=1.0, global_idx=None, Pg=None, Pr=None):
    """O = alpha * band(P).V (+ global terms)."""
    P, V = _f64(P), _f64(V)
    BH, n, hd = V.shape
    G, g = _gidx(global_idx)
    O = np.empty((BH, n, hd))
    Pg = _f64(Pg) if G else None
    Pr = _f64(Pr) if G else None
    _check(_load().orc_band_pv(BH, n, hd, w, w_upper, dilation, alpha, _ptr(P), _ptr(V),
                               _ptr(O), G, _ptr(g), _ptr(Pg), _ptr(Pr)), "band_pv")
    return O


def band_t(Bd, Y, w, w_upper, dilation=0, alpha=1.0, global_idx=None, Bg=None, Br=None):
    """X = alpha * band(Bd)^T.Y by scatter (+ global terms)."""
    Bd, Y = _f64(Bd), _f64(Y)
    BH, n, hd = Y.shape
    G, g = _gidx(global_idx)
    X = np.empty((BH, n, hd))
    Bg = _f64(Bg) if G else None
    Br = _f64(Br) if G else None
    _check(_load().orc_band_t(BH, n, hd, w, w_upper, dilation, alpha, _ptr(Bd), _ptr(Y),
                              _ptr(X), G, _ptr(g), _ptr(Bg), _ptr(Br)), "band_t")
    return X


def band_softmax_bwd(P, dP, w, w_upper, dilation=0, global_idx=None, Pg=None, dPg=None,
                     Pr=None, dPr=None, drop_t=0, seed=0):
    """dS = P * (f dP - rowsum(P * f dP)), f the dropout keep-and-scale factor
    (1 without dropout; dP is then the gradient of the dropped probabilities).
    Returns dS or (dS, dSg, dSr)."""
    P, dP = _f64(P), _f64(dP)
    BH, n, D = P.shape
    G, g = _gidx(global_idx)
    dS = np.empty_like(P)
    if G:
        Pg, dPg, Pr, dPr = _f64(Pg), _f64(dPg), _f64(Pr), _f64(dPr)
        dSg = np.empty((BH, n, G))
        dSr = np.empty((BH, G, n))
    else:
        dSg = dSr = None
    _check(_load().orc_band_softmax_bwd(BH, n, w, w_upper, dilation, _ptr(P), _ptr(dP),
                                        _ptr(dS), G, _ptr(g), _ptr(Pg), _ptr(dPg), _ptr(dSg),
                                        _ptr(Pr), _ptr(dPr), _ptr(dSr), seed, drop_t),
           "band_softmax_bwd")
    return (dS, dSg, dSr) if G else dS


def philox4x64(counter, key):
    """Philox4x64-10 block of a 4-word counter and 2-word key (uint64)."""
    c = np.ascontiguousarray(counter, dtype=np.uint64)
    k = np.ascontiguousarray(key, dtype=np.uint64)
    out = np.empty(4, dtype=np.uint64)
    _check(_load().orc_philox4x64(_ptr(c), _ptr(k), _ptr(out)), "philox4x64")
    return out


def dropout_factor(seed, drop_t, bh, i, j, s):
    """Keep-and-scale factor of element (bh, i, j): 0 or 256 / (256 - drop_t)."""
    out = ctypes.c_double()
    _check(_load().orc_dropout_factor(seed, drop_t, bh, i, j, s, ctypes.byref(out)),
           "dropout_factor")
    return out.value


def attention_fwd(Q, K, V, w, w_upper, dilation=0, scale=None, global_idx=None, key_bias=None,
                  drop_t=0, seed=0):
    """Attention on explicit key sets (key_bias[bh, j] added to the scaled score of
    key j; dropout of the probabilities with threshold byte drop_t).  Returns
    (O, lse)."""
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    BH, n, hd = Q.shape
    kb = _kbias(key_bias, BH, n)
    scale = 1.0 / np.sqrt(hd) if scale is None else scale
    G, g = _gidx(global_idx)
    O = np.empty((BH, n, hd))
    lse = np.empty((BH, n))
    _check(_load().orc_attention_fwd(BH, n, hd, w, w_upper, dilation, scale, _ptr(Q),
                                     _ptr(K), _ptr(V), _ptr(O), _ptr(lse), G, _ptr(g), _ptr(kb),
                                     seed, drop_t), "attention_fwd")
    return O, lse


def attention_bwd(Q, K, V, dO, w, w_upper, dilation=0, scale=None, global_idx=None,
                  key_bias=None, drop_t=0, seed=0):
    """Gradients of attention_fwd's O.  Returns (dQ, dK, dV)."""
    Q, K, V, dO = _f64(Q), _f64(K), _f64(V), _f64(dO)
    BH, n, hd = Q.shape
    kb = _kbias(key_bias, BH, n)
    scale = 1.0 / np.sqrt(hd) if scale is None else scale
    G, g = _gidx(global_idx)
    dQ, dK, dV = (np.empty((BH, n, hd)) for _ in range(3))
    _check(_load().orc_attention_bwd(BH, n, hd, w, w_upper, dilation, scale, _ptr(Q),
                                     _ptr(K), _ptr(V), _ptr(dO), _ptr(dQ), _ptr(dK),
                                     _ptr(dV), G, _ptr(g), _ptr(kb), seed, drop_t),
           "attention_bwd")
    return dQ, dK, dV


def add_bias_transpose(X, bias=None):
    """X [b, n, M, h, hd] (+ bias [M, h, hd]) -> Y [M, b, h, n, hd]."""
    X = _f64(X)
    b, n, M, h, hd = X.shape
    bias = _f64(bias) if bias is not None else None
    if bias is not None and bias.shape != (M, h, hd):
        raise ValueError(f"bias must be [M, h, hd] = {(M, h, hd)}")
    Y = np.empty((M, b, h, n, hd))
    _check(_load().orc_add_bias_transpose(b, n, M, h, hd, _ptr(X), _ptr(bias), _ptr(Y)),
           "add_bias_transpose")
    return Y


def global_attention_fwd(Qg, Kg, Vg, scale):
    """Compact global queries Qg [BH, G, hd] over every key of Kg, Vg [BH, n, hd].
    Returns (Og [BH, G, hd], lseg [BH, G])."""
    Qg, Kg, Vg = _f64(Qg), _f64(Kg), _f64(Vg)
    BH, G, hd = Qg.shape
    n = Kg.shape[1]
    Og = np.empty((BH, G, hd))
    lseg = np.empty((BH, G))
    _check(_load().orc_global_attention_fwd(BH, G, n, hd, scale, _ptr(Qg), _ptr(Kg), _ptr(Vg),
                                            _ptr(Og), _ptr(lseg)), "global_attention_fwd")
    return Og, lseg


def global_attention_bwd(Qg, Kg, Vg, dOg, scale):
    """Gradients of global_attention_fwd's Og.  Returns (dQg, dKg, dVg)."""
    Qg, Kg, Vg, dOg = _f64(Qg), _f64(Kg), _f64(Vg), _f64(dOg)
    BH, G, hd = Qg.shape
    n = Kg.shape[1]
    dQg = np.empty((BH, G, hd))
    dKg, dVg = np.empty((BH, n, hd)), np.empty((BH, n, hd))
    _check(_load().orc_global_attention_bwd(BH, G, n, hd, scale, _ptr(Qg), _ptr(Kg), _ptr(Vg),
                                            _ptr(dOg), _ptr(dQg), _ptr(dKg), _ptr(dVg)),
           "global_attention_bwd")
    return dQg, dKg, dVg
