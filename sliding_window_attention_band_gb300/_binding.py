"""ctypes binding of libswab.so (include/swab.h).

Argument marshalling only: every computation runs in the library's CUDA
kernels.  PyTorch supplies device memory and the current stream.  If the
library has not been built, every call raises ``SwabError`` -- there is no
fallback implementation.  With SWAB_BOUNDS_CHECK=1 in the environment at the
first call, the bounds-checked build (libswab_bounds.so) is loaded instead.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

SWAB_OK = 0
STATUS_NAMES = ["SWAB_OK", "SWAB_ERR_INVALID_ARG", "SWAB_ERR_UNSUPPORTED",
                "SWAB_ERR_MISALIGNED", "SWAB_ERR_CUDA", "SWAB_ERR_TIMEOUT", "SWAB_ERR_BOUNDS"]
MAX_GLOBAL = 256
MAX_DILATION = 15

_DTYPES = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}

# every symbol the header declares
API_FUNCTIONS = ("add_bias_transpose", "global_attention", "global_attention_bwd",
                 "global_attention_workspace", "band_qk", "band_softmax", "band_softmax_dropout", "band_pv", "band_qk_bwd_t", "band_pv_bwd_t",
                 "band_softmax_bwd", "band_attention", "band_attention_bwd",
                 "band_attention_bwd_workspace", "band_attention_bwd_noalloc",
                 "band_attention_dropout_mask_bytes",
                 "swab_status_string", "swab_device_status",
                 "swab_selftest_wait_timeout", "swab_bounds_checked", "swab_bounds_report",
                 "swab_selftest_bounds", "swab_version")


class SwabError(RuntimeError):
    def __init__(self, fn: str, status: int):
        name = STATUS_NAMES[status] if 0 <= status < len(STATUS_NAMES) else str(status)
        super().__init__(f"{fn} failed: {name}")
        self.status = status
        self.status_name = name


class _Desc(ctypes.Structure):
    _fields_ = [("b", ctypes.c_int32), ("h", ctypes.c_int32), ("n", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("w", ctypes.c_int32),
                ("w_upper", ctypes.c_int32), ("dilation", ctypes.c_int32),
                ("padding", ctypes.c_float), ("dtype", ctypes.c_int32),
                ("n_global", ctypes.c_int32), ("global_idx", ctypes.POINTER(ctypes.c_int32)),
                ("key_bias", ctypes.c_void_p), ("dropout_p", ctypes.c_float),
                ("dropout_seed", ctypes.c_uint64), ("qkv_row_stride", ctypes.c_int64),
                ("out_row_stride", ctypes.c_int64), ("dropout_mask", ctypes.c_void_p)]


class _Glob(ctypes.Structure):
    _fields_ = [("cols", ctypes.c_void_p), ("rows", ctypes.c_void_p)]


class Desc:
    """Problem description (swab_desc).  Keeps the host global index alive."""

    def __init__(self, b, h, n, head_dim, w, w_upper, dilation=0, padding=0.0,
                 dtype=torch.float16, global_idx=None, key_bias=None, dropout_p=0.0,
                 dropout_seed=0, qkv_row_stride=0, out_row_stride=0, dropout_mask=None):
        if dtype not in _DTYPES:
            raise ValueError(f"unsupported dtype {dtype}")
        self.b, self.h, self.n, self.head_dim = int(b), int(h), int(n), int(head_dim)
        self.w, self.w_upper, self.dilation = int(w), int(w_upper), int(dilation)
        self.padding = float(padding)
        self.dtype = dtype
        gi = list(global_idx) if global_idx is not None else []
        self.global_idx = tuple(int(x) for x in gi)
        self._gi = (ctypes.c_int32 * max(1, len(gi)))(*gi) if gi else None
        # key-padding bias: a [b, n] fp32 CUDA tensor (kept alive here), or None
        if key_bias is not None:
            if (key_bias.dtype != torch.float32 or tuple(key_bias.shape) != (self.b, self.n)
                    or not key_bias.is_contiguous()):
                raise ValueError(f"key_bias must be a contiguous float32 [b, n] = "
                                 f"{(self.b, self.n)} tensor")
        self.key_bias = key_bias
        self.dropout_p, self.dropout_seed = float(dropout_p), int(dropout_seed)
        # strided dense layout of the fused calls: rows of [b, n, stride]
        self.qkv_row_stride, self.out_row_stride = int(qkv_row_stride), int(out_row_stride)
        # keep-bit cache of the fused dropout: a CUDA tensor of at least
        # band_attention_dropout_mask_bytes bytes (kept alive here), or None
        self.dropout_mask = dropout_mask
        self.c = _Desc(self.b, self.h, self.n, self.head_dim, self.w, self.w_upper,
                       self.dilation, self.padding, _DTYPES[dtype], len(gi),
                       ctypes.cast(self._gi, ctypes.POINTER(ctypes.c_int32)) if gi else None,
                       key_bias.data_ptr() if key_bias is not None else None, self.dropout_p,
                       self.dropout_seed, self.qkv_row_stride, self.out_row_stride,
                       dropout_mask.data_ptr() if dropout_mask is not None else None)

    @property
    def drop_t(self):
        """Dropout threshold byte: round(256 * dropout_p), at most 255."""
        return min(255, int(round(256.0 * self.dropout_p)))

    @property
    def BH(self):
        return self.b * self.h

    @property
    def D(self):
        return self.w + self.w_upper + 1

    @property
    def G(self):
        return len(self.global_idx)

    @classmethod
    def from_workload(cls, wl):
        return cls(wl.b, wl.h, wl.n, wl.head_dim, wl.w, wl.w_upper, wl.dilation, wl.padding,
                   wl.dtype, wl.global_idx)


_lib = None
_lock = threading.Lock()


def library_path() -> str:
    """The library ``load()`` takes: the bounds-checked build when the
    environment sets SWAB_BOUNDS_CHECK=1, else the regular one."""
    return _build.LIB_BOUNDS if os.environ.get("SWAB_BOUNDS_CHECK") == "1" else _build.LIB


def load():
    """Load libswab.so (built by ``build.build()``); raises if it is missing."""
    global _lib
    with _lock:
        if _lib is None:
            path = library_path()
            if not os.path.exists(path):
                raise SwabError("load (libswab.so not built; run "
                                "sliding_window_attention_band_gb300.build.build())", 4)
            lib = ctypes.CDLL(path)
            P = ctypes.c_void_p
            D = ctypes.POINTER(_Desc)
            Gp = ctypes.POINTER(_Glob)
            f, i32 = ctypes.c_float, ctypes.c_int32
            sigs = {
                "band_qk": [D, f, P, P, P, Gp, P],
                "band_softmax": [D, P, Gp, P, Gp, P, P],
                "band_softmax_dropout": [D, P, P, P, P, P],
                "add_bias_transpose": [D, i32, P, P, P, P],
                "global_attention": [D, f, P, P, P, P, P, P, P],
                "global_attention_bwd": [D, f, P, P, P, P, P, P, P, P, P, P, P],
                "band_pv": [D, f, P, Gp, P, P, P],
                "band_qk_bwd_t": [D, f, P, Gp, P, P, P],
                "band_pv_bwd_t": [D, f, P, Gp, P, P, P],
                "band_softmax_bwd": [D, P, Gp, P, Gp, P, Gp, P],
                "band_attention": [D, f, P, P, P, P, P, P],
                "band_attention_bwd": [D, f, P, P, P, P, P, P, P, P, P, P, P],
                "band_attention_bwd_noalloc": [D, f, P, P, P, P, P, P, P, P, P, P],
                "swab_device_status": [ctypes.POINTER(i32), i32],
                "swab_selftest_wait_timeout": [ctypes.c_uint32, P],
                "swab_bounds_report": [ctypes.POINTER(ctypes.c_uint64), i32],
                "swab_selftest_bounds": [P],
            }
            for name, args in sigs.items():
                fn = getattr(lib, name)
                fn.argtypes = args
                fn.restype = ctypes.c_int
            lib.global_attention_workspace.argtypes = [D]
            lib.global_attention_workspace.restype = ctypes.c_size_t
            lib.band_attention_bwd_workspace.argtypes = [D]
            lib.band_attention_bwd_workspace.restype = ctypes.c_size_t
            lib.band_attention_dropout_mask_bytes.argtypes = [D]
            lib.band_attention_dropout_mask_bytes.restype = ctypes.c_size_t
            lib.swab_status_string.restype = ctypes.c_char_p
            lib.swab_status_string.argtypes = [ctypes.c_int]
            lib.swab_version.restype = ctypes.c_char_p
            lib.swab_bounds_checked.argtypes = []
            lib.swab_bounds_checked.restype = ctypes.c_int32
            _lib = lib
    return _lib


def version() -> str:
    return load().swab_version().decode()


def status_string(code: int) -> str:
    return load().swab_status_string(code).decode()


# ---------------------------------------------------------------------------
# marshalling helpers
# ---------------------------------------------------------------------------
def _ptr(t):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream, like):
    if stream is None:
        if like is not None and like.is_cuda:
            return ctypes.c_void_p(torch.cuda.current_stream(like.device).cuda_stream)
        return None
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _glob(g, desc=None, name="glob"):
    """(cols [BH, n, G], rows [BH, G, n]) -> swab_glob*, or None."""
    if g is None:
        return None
    cols, rows = g
    if desc is not None:
        _check_shape(f"{name}.cols", cols, (desc.BH, desc.n, desc.G), desc.dtype)
        _check_shape(f"{name}.rows", rows, (desc.BH, desc.G, desc.n), desc.dtype)
    for t in (cols, rows):
        if t is not None and not t.is_contiguous():
            raise ValueError("tensors must be contiguous")
    return ctypes.byref(_Glob(cols.data_ptr() if cols is not None else None,
                              rows.data_ptr() if rows is not None else None))


def _check_shape(name, t, shape, dtype):
    if t is None:
        return
    if t.numel() != _numel(shape):
        raise ValueError(f"{name}: expected {shape} elements, got shape {tuple(t.shape)}")
    if t.dtype != dtype:
        raise ValueError(f"{name}: expected dtype {dtype}, got {t.dtype}")


def _numel(shape):
    k = 1
    for s in shape:
        k *= s
    return k


def _call(name, *args):
    rc = getattr(load(), name)(*args)
    if rc != SWAB_OK:
        raise SwabError(name, rc)


def _dense(d):
    return (d.BH, d.n, d.head_dim)


def _band(d):
    return (d.BH, d.n, d.D)


# ---------------------------------------------------------------------------
# the entry points (same names as the C ABI)
# ---------------------------------------------------------------------------
def band_qk(desc: Desc, alpha, A, B, S, Sg=None, stream=None):
    """S = alpha * A.B^T on the band (padding outside the sequence)."""
    for n_, t, sh in (("A", A, _dense(desc)), ("B", B, _dense(desc)), ("S", S, _band(desc))):
        _check_shape(n_, t, sh, desc.dtype)
    _call("band_qk", ctypes.byref(desc.c), float(alpha), _ptr(A), _ptr(B), _ptr(S),
          _glob(Sg, desc, "Sg"),
          _stream(stream, S))


def band_softmax(desc: Desc, S, P, lse=None, Sg=None, Pg=None, stream=None):
    """P = masked row softmax of S; lse (fp32, optional) = log-sum-exp per row."""
    _check_shape("S", S, _band(desc), desc.dtype)
    _check_shape("P", P, _band(desc), desc.dtype)
    _check_shape("lse", lse, (desc.BH, desc.n), torch.float32)
    _call("band_softmax", ctypes.byref(desc.c), _ptr(S), _glob(Sg, desc, "Sg"), _ptr(P),
          _glob(Pg, desc, "Pg"),
          _ptr(lse), _stream(stream, P))


def band_softmax_dropout(desc: Desc, S, Pd, P=None, lse=None, stream=None):
    """Pd = dropout of the masked row softmax of S (the descriptor's dropout);
    P (optional) = the probabilities before dropout; lse (optional)."""
    _check_shape("S", S, _band(desc), desc.dtype)
    _check_shape("Pd", Pd, _band(desc), desc.dtype)
    _check_shape("P", P, _band(desc), desc.dtype)
    _check_shape("lse", lse, (desc.BH, desc.n), torch.float32)
    _call("band_softmax_dropout", ctypes.byref(desc.c), _ptr(S), _ptr(P), _ptr(Pd), _ptr(lse),
          _stream(stream, Pd))


def band_pv(desc: Desc, alpha, P, V, O, Pg=None, stream=None):
    """O = alpha * band(P).V."""
    _check_shape("P", P, _band(desc), desc.dtype)
    _check_shape("V", V, _dense(desc), desc.dtype)
    _check_shape("O", O, _dense(desc), desc.dtype)
    _call("band_pv", ctypes.byref(desc.c), float(alpha), _ptr(P), _glob(Pg, desc, "Pg"),
          _ptr(V), _ptr(O),
          _stream(stream, O))


def band_qk_bwd_t(desc: Desc, alpha, dS, Q, dK, dSg=None, stream=None):
    """dK = alpha * band(dS)^T.Q."""
    _check_shape("dS", dS, _band(desc), desc.dtype)
    _check_shape("Q", Q, _dense(desc), desc.dtype)
    _check_shape("dK", dK, _dense(desc), desc.dtype)
    _call("band_qk_bwd_t", ctypes.byref(desc.c), float(alpha), _ptr(dS),
          _glob(dSg, desc, "dSg"), _ptr(Q),
          _ptr(dK), _stream(stream, dK))


def band_pv_bwd_t(desc: Desc, alpha, P, dO, dV, Pg=None, stream=None):
    """dV = alpha * band(P)^T.dO."""
    _check_shape("P", P, _band(desc), desc.dtype)
    _check_shape("dO", dO, _dense(desc), desc.dtype)
    _check_shape("dV", dV, _dense(desc), desc.dtype)
    _call("band_pv_bwd_t", ctypes.byref(desc.c), float(alpha), _ptr(P),
          _glob(Pg, desc, "Pg"), _ptr(dO),
          _ptr(dV), _stream(stream, dV))


def band_softmax_bwd(desc: Desc, P, dP, dS, Pg=None, dPg=None, dSg=None, stream=None):
    """dS = P * (dP - rowsum(P * dP)) on the used slots."""
    for n_, t in (("P", P), ("dP", dP), ("dS", dS)):
        _check_shape(n_, t, _band(desc), desc.dtype)
    _call("band_softmax_bwd", ctypes.byref(desc.c), _ptr(P), _glob(Pg, desc, "Pg"), _ptr(dP),
          _glob(dPg, desc, "dPg"), _ptr(dS), _glob(dSg, desc, "dSg"), _stream(stream, dS))


def _dense_ptr(desc: Desc, name, t, stride):
    """Pointer to a dense tensor of a fused call: contiguous [b*h, n, hd] (or
    any contiguous shape of that size) when stride == 0, else a [b, n, h, hd]
    view whose rows are `stride` elements apart (e.g. a slice of the merged
    projection output [b, n, 3, h, hd])."""
    if stride == 0:
        _check_shape(name, t, _dense(desc), desc.dtype)
        return _ptr(t)
    want_shape = (desc.b, desc.n, desc.h, desc.head_dim)
    want_strides = (desc.n * stride, stride, desc.head_dim, 1)
    if t.dtype != desc.dtype or tuple(t.shape) != want_shape or tuple(t.stride()) != want_strides:
        raise ValueError(f"{name}: expected a {want_shape} view with strides {want_strides}, got "
                         f"{tuple(t.shape)} / {tuple(t.stride())} {t.dtype}")
    return ctypes.c_void_p(t.data_ptr())


def band_attention(desc: Desc, scale, Q, K, V, O, lse=None, stream=None):
    """Fused forward: O (and lse) of band_qk -> band_softmax -> band_pv, scores on chip."""
    ps, os_ = desc.qkv_row_stride, desc.out_row_stride
    args = [_dense_ptr(desc, "Q", Q, ps), _dense_ptr(desc, "K", K, ps),
            _dense_ptr(desc, "V", V, ps), _dense_ptr(desc, "O", O, os_)]
    _check_shape("lse", lse, (desc.BH, desc.n), torch.float32)
    _call("band_attention", ctypes.byref(desc.c), float(scale), *args, _ptr(lse),
          _stream(stream, O))


def band_attention_bwd_workspace(desc: Desc) -> int:
    """Bytes of device workspace band_attention_bwd needs."""
    return int(load().band_attention_bwd_workspace(ctypes.byref(desc.c)))


def band_attention_dropout_mask_bytes(desc: Desc) -> int:
    """Bytes of the fused dropout's keep-bit cache (Desc(dropout_mask=...))."""
    return int(load().band_attention_dropout_mask_bytes(ctypes.byref(desc.c)))


def band_attention_bwd(desc: Desc, scale, Q, K, V, O, dO, lse, dQ, dK, dV, workspace,
                       stream=None):
    """Fused backward: dQ, dK, dV from Q, K, V, O, dO and the forward's lse."""
    ps, os_ = desc.qkv_row_stride, desc.out_row_stride
    args = [_dense_ptr(desc, n_, t, st) for n_, t, st in
            (("Q", Q, ps), ("K", K, ps), ("V", V, ps), ("O", O, os_), ("dO", dO, os_))]
    outs = [_dense_ptr(desc, n_, t, ps) for n_, t in (("dQ", dQ), ("dK", dK), ("dV", dV))]
    _check_shape("lse", lse, (desc.BH, desc.n), torch.float32)
    if workspace.numel() * workspace.element_size() < band_attention_bwd_workspace(desc):
        raise ValueError("workspace too small")
    _call("band_attention_bwd", ctypes.byref(desc.c), float(scale), *args, _ptr(lse), *outs,
          _ptr(workspace), _stream(stream, dQ))


def global_attention_workspace(desc: Desc) -> int:
    """Bytes of device workspace global_attention / global_attention_bwd need."""
    return int(load().global_attention_workspace(ctypes.byref(desc.c)))


def _global_shapes(desc: Desc):
    return (desc.BH, desc.G, desc.head_dim), (desc.BH, desc.n, desc.head_dim)


def global_attention(desc: Desc, scale, Qg, Kg, Vg, Og, lseg, workspace, stream=None):
    """Global queries Qg [b*h, G, 64] over every key of their own projections
    Kg, Vg [b*h, n, 64]: Og [b*h, G, 64], lseg [b*h, G] (may be None)."""
    gs, ns = _global_shapes(desc)
    for n_, t, sh in (("Qg", Qg, gs), ("Kg", Kg, ns), ("Vg", Vg, ns), ("Og", Og, gs)):
        _check_shape(n_, t, sh, desc.dtype)
    _check_shape("lseg", lseg, (desc.BH, desc.G), torch.float32)
    if workspace.numel() * workspace.element_size() < global_attention_workspace(desc):
        raise ValueError("workspace too small")
    _call("global_attention", ctypes.byref(desc.c), float(scale), _ptr(Qg), _ptr(Kg), _ptr(Vg),
          _ptr(Og), _ptr(lseg), _ptr(workspace), _stream(stream, Og))


def global_attention_bwd(desc: Desc, scale, Qg, Kg, Vg, Og, dOg, lseg, dQg, dKg, dVg, workspace,
                         stream=None):
    """Gradients of global_attention: dQg [b*h, G, 64], dKg, dVg [b*h, n, 64]."""
    gs, ns = _global_shapes(desc)
    for n_, t, sh in (("Qg", Qg, gs), ("Kg", Kg, ns), ("Vg", Vg, ns), ("Og", Og, gs),
                      ("dOg", dOg, gs), ("dQg", dQg, gs), ("dKg", dKg, ns), ("dVg", dVg, ns)):
        _check_shape(n_, t, sh, desc.dtype)
    _check_shape("lseg", lseg, (desc.BH, desc.G), torch.float32)
    if workspace.numel() * workspace.element_size() < global_attention_workspace(desc):
        raise ValueError("workspace too small")
    _call("global_attention_bwd", ctypes.byref(desc.c), float(scale), _ptr(Qg), _ptr(Kg), _ptr(Vg),
          _ptr(Og), _ptr(dOg), _ptr(lseg), _ptr(dQg), _ptr(dKg), _ptr(dVg), _ptr(workspace),
          _stream(stream, dQg))


def add_bias_transpose(desc: Desc, X, bias, Y, stream=None):
    """Y[m] = transpose of X[:, :, m] + bias[m]: X rows of [b, n, M, h, hd] (the
    merged projection output), bias [M, h, hd] or None, Y [M, b, h, n, hd]."""
    if X.dim() != 5 or X.shape[0] != desc.b or X.shape[1] != desc.n or X.shape[3] != desc.h \
            or X.shape[4] != desc.head_dim:
        raise ValueError(f"X: expected [b, n, M, h, hd], got {tuple(X.shape)}")
    M = int(X.shape[2])
    _check_shape("X", X, tuple(X.shape), desc.dtype)
    _check_shape("bias", bias, (M, desc.h, desc.head_dim), desc.dtype)
    _check_shape("Y", Y, (M, desc.b, desc.h, desc.n, desc.head_dim), desc.dtype)
    _call("add_bias_transpose", ctypes.byref(desc.c), M, _ptr(X), _ptr(bias), _ptr(Y),
          _stream(stream, Y))


def selftest_wait_timeout(limit_us: int = 20000, stream=None):
    """Launch the bounded-wait self-test (a wait that must give up after limit_us)."""
    s = _stream(stream, None)
    if s is None and torch.cuda.is_available():
        s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    _call("swab_selftest_wait_timeout", int(limit_us), s)


NOALLOC_MAX_ROWS = 1 << 22


def band_attention_bwd_noalloc(desc: Desc, scale, Q, K, V, O, dO, lse, dQ, dK, dV, stream=None):
    """band_attention_bwd without a workspace argument, for callers that cannot
    allocate device memory: the library keeps the per-row scratch in a
    module-scope device array (b*h*n <= NOALLOC_MAX_ROWS).  Calls that overlap
    on the GPU share that array and race; the first call on a device resolves
    the array's address and should come before any stream capture."""
    for n_, t in (("Q", Q), ("K", K), ("V", V), ("O", O), ("dO", dO), ("dQ", dQ), ("dK", dK),
                  ("dV", dV)):
        _check_shape(n_, t, _dense(desc), desc.dtype)
    _check_shape("lse", lse, (desc.BH, desc.n), torch.float32)
    _call("band_attention_bwd_noalloc", ctypes.byref(desc.c), float(scale), _ptr(Q), _ptr(K),
          _ptr(V), _ptr(O), _ptr(dO), _ptr(lse), _ptr(dQ), _ptr(dK), _ptr(dV),
          _stream(stream, dQ))


def bounds_checked() -> bool:
    """True when the loaded library is the bounds-checked build."""
    return bool(load().swab_bounds_checked())


def bounds_report(reset: bool = True):
    """The first out-of-bounds access the checked build recorded since the
    last reset: (site, address, bytes), site = (file id << 16 | line) + 1, or
    None when there was none."""
    out = (ctypes.c_uint64 * 3)()
    _call("swab_bounds_report", out, 1 if reset else 0)
    return None if out[0] == 0 else (int(out[0]), int(out[1]), int(out[2]))


def selftest_bounds(stream=None):
    """Run the bounds checks' self-test (checked build); raises SwabError if
    the checks misbehave or the build has none (SWAB_ERR_UNSUPPORTED)."""
    s = _stream(stream, None)
    if s is None and torch.cuda.is_available():
        s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    _call("swab_selftest_bounds", s)


def device_status(reset: bool = True) -> int:
    """The library's device status word (bit k = status k raised by a kernel)."""
    flags = ctypes.c_int32(0)
    _call("swab_device_status", ctypes.byref(flags), 1 if reset else 0)
    return int(flags.value)
