"""C-ABI boundary tests that need no GPU.

* the library builds, loads on a machine without a driver, and exports every
  function include/swab.h declares -- the regular build and the
  bounds-checked one (which says so; the regular one says it is not);
* invalid arguments come back as the documented status before any CUDA call
  (the pointers below are fake, never dereferenced: validation rejects the
  call first).
"""
from __future__ import annotations

import ctypes
import os
import re

import pytest
import torch

from sliding_window_attention_band_gb300 import _binding as B
from sliding_window_attention_band_gb300 import build as swab_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "swab.h")

OK, INVALID, UNSUPPORTED, MISALIGNED, CUDA = 0, 1, 2, 3, 4
FAKE = 0x10000  # 16-byte aligned, never dereferenced


@pytest.fixture(scope="module")
def lib():
    swab_build.build()
    return B.load()


def declared_functions():
    with open(HEADER) as f:
        text = f.read()
    return re.findall(r"SWAB_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)


def test_header_lists_every_binding():
    names = declared_functions()
    assert sorted(names) == sorted(B.API_FUNCTIONS)


def test_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_bounds_checked_build_exports_and_identifies_itself(lib):
    swab_build.build_all()
    checked = ctypes.CDLL(swab_build.LIB_BOUNDS)   # loading needs no driver
    for name in declared_functions():
        assert hasattr(checked, name), name
    checked.swab_bounds_checked.restype = ctypes.c_int32
    lib.swab_bounds_checked.restype = ctypes.c_int32
    assert checked.swab_bounds_checked() == 1
    assert lib.swab_bounds_checked() == 0
    # the report validates its argument before any CUDA call
    assert checked.swab_bounds_report(None, 0) == INVALID
    assert lib.swab_bounds_report(None, 0) == INVALID


def test_version_and_status_strings(lib):
    assert B.version() == "0.1.0"
    for code, name in enumerate(B.STATUS_NAMES):
        assert B.status_string(code) == name
    assert B.status_string(99) == "SWAB_UNKNOWN_STATUS"


def desc(**kw):
    base = dict(b=1, h=2, n=256, head_dim=64, w=16, w_upper=16, dilation=0, padding=0.0,
                dtype=torch.float16, global_idx=None)
    base.update(kw)
    return B.Desc(**base)


def call(lib, name, d, *ptrs, alpha=0.125):
    P = ctypes.c_void_p
    if name == "band_qk":
        return lib.band_qk(ctypes.byref(d.c), alpha, P(ptrs[0]), P(ptrs[1]), P(ptrs[2]), None,
                           None)
    if name == "band_softmax":
        return lib.band_softmax(ctypes.byref(d.c), P(ptrs[0]), None, P(ptrs[1]), None,
                                P(ptrs[2]) if len(ptrs) > 2 else None, None)
    if name in ("band_pv", "band_qk_bwd_t", "band_pv_bwd_t"):
        return getattr(lib, name)(ctypes.byref(d.c), alpha, P(ptrs[0]), None, P(ptrs[1]),
                                  P(ptrs[2]), None)
    if name == "band_softmax_bwd":
        return lib.band_softmax_bwd(ctypes.byref(d.c), P(ptrs[0]), None, P(ptrs[1]), None,
                                    P(ptrs[2]), None, None)
    if name == "band_attention":
        return lib.band_attention(ctypes.byref(d.c), alpha, P(ptrs[0]), P(ptrs[1]),
                                  P(ptrs[2]), P(ptrs[3]), None, None)
    raise KeyError(name)


ALL3 = ["band_qk", "band_softmax", "band_pv", "band_qk_bwd_t", "band_pv_bwd_t",
        "band_softmax_bwd"]


@pytest.mark.parametrize("name", ALL3 + ["band_attention"])
def test_null_descriptor(lib, name):
    P = ctypes.c_void_p
    fn = getattr(lib, name)
    if name == "band_attention":
        rc = fn(None, 1.0, P(FAKE), P(FAKE), P(FAKE), P(FAKE), None, None)
    elif name == "band_qk":
        rc = fn(None, 1.0, P(FAKE), P(FAKE), P(FAKE), None, None)
    elif name == "band_softmax":
        rc = fn(None, P(FAKE), None, P(FAKE), None, None, None)
    elif name == "band_softmax_bwd":
        rc = fn(None, P(FAKE), None, P(FAKE), None, P(FAKE), None, None)
    else:
        rc = fn(None, 1.0, P(FAKE), None, P(FAKE), P(FAKE), None)
    assert rc == INVALID


@pytest.mark.parametrize("name", ALL3)
@pytest.mark.parametrize("bad,expected", [
    (dict(n=0), INVALID), (dict(b=0), INVALID), (dict(w=-1), INVALID),
    (dict(w_upper=-2), INVALID), (dict(dilation=-1), INVALID), (dict(dilation=16), UNSUPPORTED),
    (dict(head_dim=128), UNSUPPORTED), (dict(head_dim=0), INVALID),
    (dict(global_idx=[3, 3]), INVALID), (dict(global_idx=[5, 2]), INVALID),
    (dict(global_idx=[256]), INVALID), (dict(global_idx=[-1]), INVALID),
    (dict(b=300, h=300), UNSUPPORTED),
])
def test_bad_descriptor(lib, name, bad, expected):
    assert call(lib, name, desc(**bad), FAKE, FAKE, FAKE) == expected


def test_bad_dtype(lib):
    d = desc()
    d.c.dtype = 7
    assert call(lib, "band_qk", d, FAKE, FAKE, FAKE) == INVALID


def test_too_many_globals(lib):
    d = desc(n=1000, global_idx=list(range(257)))
    assert call(lib, "band_qk", d, FAKE, FAKE, FAKE) == INVALID


def test_f32_head_dim_limit(lib):
    assert call(lib, "band_qk", desc(dtype=torch.float32, head_dim=129), FAKE, FAKE, FAKE) == \
        UNSUPPORTED


@pytest.mark.parametrize("name", ALL3)
def test_null_and_misaligned_pointers(lib, name):
    d = desc()
    assert call(lib, name, d, 0, FAKE, FAKE) == INVALID
    assert call(lib, name, d, FAKE, 0, FAKE) == INVALID
    assert call(lib, name, d, FAKE + 2, FAKE, FAKE) == MISALIGNED
    assert call(lib, name, d, FAKE, FAKE + 8, FAKE) == MISALIGNED
    assert call(lib, name, d, FAKE, FAKE, FAKE + 4) == MISALIGNED
    if name != "band_softmax":  # its third pointer (lse) is optional
        assert call(lib, name, d, FAKE, FAKE, 0) == INVALID


def test_lse_misaligned(lib):
    assert call(lib, "band_softmax", desc(), FAKE, FAKE, FAKE + 4) == MISALIGNED


def test_device_status_null(lib):
    assert lib.swab_device_status(None, 0) == INVALID


@pytest.mark.skipif(torch.cuda.is_available(), reason="only meaningful without a GPU")
@pytest.mark.parametrize("dtype", [torch.float16, torch.float32])
def test_valid_call_without_gpu_reports_cuda_error(lib, dtype):
    """Valid arguments on a machine with no GPU: the launch fails cleanly."""
    assert call(lib, "band_qk", desc(dtype=dtype), FAKE, FAKE, FAKE) == CUDA
    assert call(lib, "band_softmax", desc(dtype=dtype), FAKE, FAKE) == CUDA


def test_binding_shape_checks():
    d = desc()
    with pytest.raises(ValueError):
        B.band_qk(d, 1.0, torch.zeros(3), torch.zeros(3), torch.zeros(3))
    with pytest.raises(ValueError):
        B.Desc(1, 1, 8, 64, 1, 1, dtype=torch.int32)


def test_binding_raises_swab_error(lib):
    d = desc(n=0)
    with pytest.raises(B.SwabError) as ei:
        B._call("band_qk", ctypes.byref(d.c), 1.0, ctypes.c_void_p(FAKE),
                ctypes.c_void_p(FAKE), ctypes.c_void_p(FAKE), None, None)
    assert ei.value.status_name == "SWAB_ERR_INVALID_ARG"


def test_globals_need_companions(lib):
    """With global tokens every band tensor needs its (cols, rows) companion."""
    d = desc(n=512, global_idx=[0, 5, 9])
    P = ctypes.c_void_p
    assert lib.band_qk(ctypes.byref(d.c), 1.0, P(FAKE), P(FAKE), P(FAKE), None, None) == INVALID
    half = B._Glob(FAKE, None)
    assert lib.band_qk(ctypes.byref(d.c), 1.0, P(FAKE), P(FAKE), P(FAKE), ctypes.byref(half),
                       None) == INVALID
    mis = B._Glob(FAKE, FAKE + 2)
    assert lib.band_pv(ctypes.byref(d.c), 1.0, P(FAKE), ctypes.byref(mis), P(FAKE), P(FAKE),
                       None) == MISALIGNED
    ok = B._Glob(FAKE, FAKE)
    assert lib.band_softmax(ctypes.byref(d.c), P(FAKE), ctypes.byref(ok), P(FAKE), None, None,
                            None) == INVALID


def test_globals_need_head_dim_64(lib):
    d = desc(dtype=torch.float32, head_dim=32, global_idx=[1])
    ok = B._Glob(FAKE, FAKE)
    P = ctypes.c_void_p
    assert lib.band_qk(ctypes.byref(d.c), 1.0, P(FAKE), P(FAKE), P(FAKE), ctypes.byref(ok),
                       None) == UNSUPPORTED


def test_fused_forward_global_rules(lib):
    """With global tokens the fused forward needs lse (the global columns are
    merged by log-sum-exp), f16 / bf16 and the contiguous layout."""
    P = ctypes.c_void_p
    d = desc(global_idx=[1])
    assert lib.band_attention(ctypes.byref(d.c), 1.0, P(FAKE), P(FAKE), P(FAKE), P(FAKE), None,
                              None) == INVALID
    d32 = desc(global_idx=[1], dtype=torch.float32)
    assert lib.band_attention(ctypes.byref(d32.c), 1.0, P(FAKE), P(FAKE), P(FAKE), P(FAKE),
                              P(FAKE), None) == UNSUPPORTED
    ds = desc(global_idx=[1], qkv_row_stride=384)
    assert lib.band_attention(ctypes.byref(ds.c), 1.0, P(FAKE), P(FAKE), P(FAKE), P(FAKE),
                              P(FAKE), None) == UNSUPPORTED
    big = desc(n=200000, global_idx=[1])
    assert lib.band_attention(ctypes.byref(big.c), 1.0, P(FAKE), P(FAKE), P(FAKE), P(FAKE),
                              P(FAKE), None) == UNSUPPORTED
    # the fused backward takes global tokens in f16 / bf16 with the contiguous
    # layout and a key bitmap that fits in shared memory; the rest is refused
    # before anything is launched
    for bad in (d32, ds, desc(n=120000, global_idx=[1])):
        assert lib.band_attention_bwd(ctypes.byref(bad.c), 1.0, *(P(FAKE) for _ in range(10)),
                                      None) == UNSUPPORTED
    # the allocation-free backward takes no global tokens
    assert lib.band_attention_bwd_noalloc(ctypes.byref(d.c), 1.0, *(P(FAKE) for _ in range(9)),
                                          None) == UNSUPPORTED
    # with global tokens the workspace grows by the gathered rows, the global
    # keys' tiles and the global rows' dK, dV terms
    plain = desc()
    assert lib.band_attention_bwd_workspace(ctypes.byref(d.c)) > \
        lib.band_attention_bwd_workspace(ctypes.byref(plain.c))


def test_binding_checks_companion_shapes():
    d = desc(global_idx=[0, 3])
    bad = (torch.zeros(2, 256, 3, dtype=torch.float16), torch.zeros(2, 2, 256, dtype=torch.float16))
    with pytest.raises(ValueError):
        B._glob(bad, d, "Sg")


def test_key_bias_validation(lib):
    """The key-padding bias must be 4-byte aligned; the separate global
    projections and the allocation-free backward do not take it."""
    d = desc()
    d.c.key_bias = FAKE + 2
    assert call(lib, "band_softmax", d, FAKE, FAKE) == MISALIGNED
    P = ctypes.c_void_p
    dg = desc(n=512, global_idx=[0, 5])
    dg.c.key_bias = FAKE
    assert lib.global_attention(ctypes.byref(dg.c), 0.125, *(P(FAKE) for _ in range(6)), None) == UNSUPPORTED
    d.c.key_bias = FAKE
    assert lib.band_attention_bwd_noalloc(ctypes.byref(d.c), 0.125, *(P(FAKE) for _ in range(9)),
                                          None) == UNSUPPORTED


def test_binding_key_bias_shape():
    with pytest.raises(ValueError):
        B.Desc(2, 3, 64, 64, 4, 4, key_bias=torch.zeros(3, 64))
    with pytest.raises(ValueError):
        B.Desc(2, 3, 64, 64, 4, 4, key_bias=torch.zeros(2, 64, dtype=torch.float16))


def test_dropout_validation(lib):
    """dropout_p must lie in [0, 1); band_softmax, global tokens and the
    allocation-free backward do not take dropout."""
    P = ctypes.c_void_p
    for bad in (-0.1, 1.0, float("nan")):
        d = desc()
        d.c.dropout_p = bad
        assert call(lib, "band_attention", d, FAKE, FAKE, FAKE, FAKE) == INVALID
    d = desc(dropout_p=0.1)
    assert call(lib, "band_softmax", d, FAKE, FAKE) == UNSUPPORTED
    assert lib.band_attention_bwd_noalloc(ctypes.byref(d.c), 0.125, *(P(FAKE) for _ in range(9)),
                                          None) == UNSUPPORTED
    dg = desc(n=512, global_idx=[0, 5], dropout_p=0.1)
    assert call(lib, "band_qk", dg, FAKE, FAKE, FAKE) == UNSUPPORTED
    assert desc(dropout_p=0.1).drop_t == 26 and desc(dropout_p=0.999).drop_t == 255


def test_softmax_dropout_validation(lib):
    """band_softmax_dropout: S and Pd required and aligned, P and lse optional
    but aligned, no global tokens, bands of at most 65536 slots."""
    P = ctypes.c_void_p
    f = lib.band_softmax_dropout
    d = desc(dropout_p=0.1)
    assert f(None, P(FAKE), P(FAKE), P(FAKE), None, None) == INVALID
    assert f(ctypes.byref(d.c), None, None, P(FAKE), None, None) == INVALID
    assert f(ctypes.byref(d.c), P(FAKE), None, None, None, None) == INVALID
    assert f(ctypes.byref(d.c), P(FAKE), None, P(FAKE + 2), None, None) == MISALIGNED
    assert f(ctypes.byref(d.c), P(FAKE), P(FAKE + 8), P(FAKE), None, None) == MISALIGNED
    assert f(ctypes.byref(d.c), P(FAKE), None, P(FAKE), P(FAKE + 4), None) == MISALIGNED
    dg = desc(n=512, global_idx=[0, 5])
    assert f(ctypes.byref(dg.c), P(FAKE), None, P(FAKE), None, None) == UNSUPPORTED
    big = desc(n=256, w=40000, w_upper=30000, dropout_p=0.1)
    assert f(ctypes.byref(big.c), P(FAKE), None, P(FAKE), None, None) == UNSUPPORTED
    assert call(lib, "band_softmax_bwd", big, FAKE, FAKE, FAKE) == UNSUPPORTED
    # without dropout the long band is fine for band_softmax_bwd's validation
    big0 = desc(n=256, w=40000, w_upper=30000)
    if not torch.cuda.is_available():
        assert call(lib, "band_softmax_bwd", big0, FAKE, FAKE, FAKE) == CUDA


def test_strided_layout_validation(lib):
    """Row strides: >= h * head_dim, 16-byte multiples; the materialised band
    products and the allocation-free backward take the contiguous layout only."""
    P = ctypes.c_void_p
    for kw, want in ((dict(qkv_row_stride=-8), INVALID), (dict(qkv_row_stride=64), INVALID),
                     (dict(out_row_stride=100), INVALID), (dict(qkv_row_stride=132), MISALIGNED),
                     (dict(out_row_stride=136, dtype=torch.float32), OK)):
        d = desc(**kw)   # h = 2, head_dim = 64: h * head_dim = 128
        rc = call(lib, "band_attention", d, FAKE, FAKE, FAKE, FAKE)
        if want == OK:
            assert rc in (OK, CUDA)   # valid; without a GPU the launch fails cleanly
        else:
            assert rc == want, kw
    d = desc(qkv_row_stride=384)
    for name in ("band_qk", "band_pv", "band_qk_bwd_t", "band_pv_bwd_t"):
        assert call(lib, name, d, FAKE, FAKE, FAKE) == UNSUPPORTED, name
    d = desc(out_row_stride=256)
    assert lib.band_attention_bwd_noalloc(ctypes.byref(d.c), 0.125, *(P(FAKE) for _ in range(9)),
                                          None) == UNSUPPORTED


def test_add_bias_transpose_validation(lib):
    P = ctypes.c_void_p
    f = lib.add_bias_transpose
    d = desc()
    assert f(None, 3, P(FAKE), None, P(FAKE * 16), None) == INVALID
    assert f(ctypes.byref(d.c), 0, P(FAKE), None, P(FAKE * 16), None) == INVALID
    assert f(ctypes.byref(d.c), 3, None, None, P(FAKE * 16), None) == INVALID
    assert f(ctypes.byref(d.c), 3, P(FAKE + 8), None, P(FAKE * 16), None) == MISALIGNED
    assert f(ctypes.byref(d.c), 3, P(FAKE), P(FAKE + 2), P(FAKE * 16), None) == MISALIGNED
    assert f(ctypes.byref(d.c), 3, P(FAKE), None, P(FAKE + 4096), None) == INVALID  # overlap
    odd = desc(head_dim=12)   # 24 bytes per head row: not whole 16-byte chunks
    assert f(ctypes.byref(odd.c), 3, P(FAKE), None, P(FAKE * 16), None) == UNSUPPORTED


def test_binding_strided_views():
    d = desc(b=2, h=3, n=40, qkv_row_stride=3 * 3 * 64)
    qkv = torch.zeros(2, 40, 3, 3, 64, dtype=torch.float16)
    ptr = B._dense_ptr(d, "Q", qkv[:, :, 0], d.qkv_row_stride)
    assert ptr.value == qkv.data_ptr()
    with pytest.raises(ValueError):
        B._dense_ptr(d, "Q", qkv[:, :, 0].contiguous(), d.qkv_row_stride)
    with pytest.raises(ValueError):
        B.add_bias_transpose(d, torch.zeros(2, 40, 3, 2, 64, dtype=torch.float16), None,
                             torch.zeros(3, 2, 3, 40, 64, dtype=torch.float16))


def test_global_attention_validation(lib):
    P = ctypes.c_void_p
    f, fb = lib.global_attention, lib.global_attention_bwd
    d = desc(n=512, global_idx=[0, 3, 9])
    assert lib.global_attention_workspace(ctypes.byref(d.c)) > 0
    assert lib.global_attention_workspace(ctypes.byref(desc().c)) == 0   # no global tokens
    assert f(ctypes.byref(desc().c), 0.1, *(P(FAKE) for _ in range(4)), None, P(FAKE), None) == \
        INVALID
    assert f(ctypes.byref(d.c), 0.1, P(FAKE), P(FAKE), P(FAKE), P(FAKE), None, None, None) == \
        INVALID   # no workspace
    assert f(ctypes.byref(d.c), 0.1, P(FAKE), P(FAKE), P(FAKE), P(FAKE), P(FAKE + 4), P(FAKE),
             None) == MISALIGNED
    d32 = desc(n=512, global_idx=[0, 3], dtype=torch.float32, head_dim=32)
    assert f(ctypes.byref(d32.c), 0.1, *(P(FAKE) for _ in range(4)), None, P(FAKE), None) == \
        UNSUPPORTED
    ds = desc(n=512, global_idx=[0, 3], qkv_row_stride=384)
    assert f(ctypes.byref(ds.c), 0.1, *(P(FAKE) for _ in range(4)), None, P(FAKE), None) == \
        UNSUPPORTED
    assert fb(ctypes.byref(d.c), 0.1, *(P(FAKE) for _ in range(5)), None,
              *(P(FAKE) for _ in range(4)), None) == INVALID   # lseg required


def test_dropout_mask_size_and_validation(lib):
    """The fused dropout's keep-bit cache: b*h*n rows of ceil(D / 32) + 1 words,
    4-byte aligned when dropout is on, ignored without dropout."""
    d = desc(dropout_p=0.1)
    words = (d.D + 31) // 32 + 1
    assert lib.band_attention_dropout_mask_bytes(ctypes.byref(d.c)) == d.BH * d.n * words * 4
    assert lib.band_attention_dropout_mask_bytes(None) == 0
    assert B.band_attention_dropout_mask_bytes(desc(w=100, w_upper=27)) == 2 * 256 * 5 * 4
    d.c.dropout_mask = FAKE + 2
    assert call(lib, "band_attention", d, FAKE, FAKE, FAKE, FAKE) == MISALIGNED
    d.c.dropout_mask = FAKE
    assert call(lib, "band_attention", d, FAKE, FAKE, FAKE, FAKE) in (OK, CUDA)
    d0 = desc()
    d0.c.dropout_mask = FAKE + 2   # no dropout: the cache is not used
    assert call(lib, "band_attention", d0, FAKE, FAKE, FAKE, FAKE) in (OK, CUDA)
