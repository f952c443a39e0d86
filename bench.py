#!/usr/bin/env python3
"""Benchmark: banded attention forward + backward on one GB300 (sm_103a).

One step = one forward + backward pass of sliding-window attention over the
Longformer-base workload (b=1, h=12, n=4096, head_dim=64, w=w_upper=256,
fp16, dilation 0), every kernel launched through the C ABI.  Two variants,
both timed in every run (--step picks the headline):

  fused (default): band_attention(Q,K,V)->O,lse, then
      band_attention_bwd(Q,K,V,O,dO,lse)->dQ,dK,dV (scores never in HBM);
  materialised: band_qk(Q,K)->S, band_softmax(S)->P,lse, band_pv(P,V)->O,
      band_qk(dO,V)->dP, band_softmax_bwd(P,dP)->dS, band_pv(dS,K)->dQ,
      band_qk_bwd_t(dS,Q)->dK, band_pv_bwd_t(P,dO)->dV.

`value` is TFLOP/s on algorithmic flops (6 banded contractions x 2*head_dim
per valid (query, key) pair) over device time with inputs resident in HBM.
L2 is flushed (a 256 MB write, then read back) before every step, outside the
timed events.
`e2e` is the same metric with pinned-host inputs copied in and the outputs
(O, dQ, dK, dV) copied back inside the timed region, every step, through the
public API called eagerly; the copies of neighbouring steps run on two copy
streams while a step computes (see time_e2e).

--impl reference times the fp64 CPU oracle (the only reference this subject
has) on a bounded sample of the same workload.
Multi-GPU (torchrun): every rank runs its own replica of the workload (the
(b,h) slices are independent; there is no exchange), scaling "weak".
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from sliding_window_attention_band_gb300.inputs import WORKLOADS, workload_inputs  # noqa: E402

METRIC = "banded attention fwd+bwd ms & TFLOP/s at n=4096,w=256,d=0/3; % of roofline"
MAIN_CFG = 2
ALSO_CFG = 3
N_CONTRACTIONS = 6
FLUSH_BYTES = 256 << 20


# ---------------------------------------------------------------------------
# accounting (algorithmic work of one step)
# ---------------------------------------------------------------------------
def valid_pairs(wl) -> int:
    s = wl.dilation + 1
    i = np.arange(wl.n, dtype=np.int64)
    t_lo = np.maximum(0, wl.w - i // s)
    t_hi = np.minimum(wl.D - 1, wl.w + (wl.n - 1 - i) // s)
    return int((t_hi - t_lo + 1).sum()) * wl.BH


def valid_pairs_globals(wl) -> int:
    """(query, key) pairs with global tokens: a local row's band keys outside G
    plus the G global keys; a global row's n keys."""
    s = wl.dilation + 1
    i = np.arange(wl.n, dtype=np.int64)
    t_lo = np.maximum(0, wl.w - i // s)
    t_hi = np.minimum(wl.D - 1, wl.w + (wl.n - 1 - i) // s)
    per_row = t_hi - t_lo + 1
    gl = np.array(wl.global_idx, dtype=np.int64)
    for p_ in gl:   # rows whose band holds global key p_
        k = np.arange(-wl.w, wl.w_upper + 1, dtype=np.int64)
        rows = p_ - k * s
        rows = rows[(rows >= 0) & (rows < wl.n)]
        per_row[rows] -= 1
    per_row += len(gl)
    per_row[gl] = wl.n
    return int(per_row.sum()) * wl.BH


def step_flops(wl) -> float:
    return float(N_CONTRACTIONS * 2 * wl.head_dim * valid_pairs(wl))


def kernel_bytes(wl) -> dict:
    """Algorithmic bytes of one call: every input read once, every output written once."""
    e = torch.finfo(wl.dtype).bits // 8
    dense = wl.BH * wl.n * wl.head_dim * e
    band = wl.BH * wl.n * wl.D * e
    rowf = wl.BH * wl.n * 4
    return {
        "band_qk": 2 * dense + band,
        "band_softmax": 2 * band + rowf,
        "band_pv": band + 2 * dense,
        "band_softmax_bwd": 3 * band,
        "band_t": band + 2 * dense,
        "band_attention": 4 * dense + rowf,
        # Q, K, V, O, dO, lse in; dQ, dK, dV out; the per-row delta out and back in
        "band_attention_bwd": 8 * dense + 3 * rowf,
    }


def kernel_flops(wl) -> dict:
    """Algorithmic flops of one call (2*head_dim per valid pair per contraction)."""
    c = 2.0 * wl.head_dim * valid_pairs(wl)
    return {"band_qk": c, "band_softmax": 0.0, "band_pv": c, "band_softmax_bwd": 0.0,
            "band_t": c, "band_attention": 2 * c, "band_attention_bwd": 4 * c}


# ---------------------------------------------------------------------------
# the step
# ---------------------------------------------------------------------------
class Step:
    """Buffers and launches of one forward + backward step, materialised band
    tensors: every banded product and softmax is its own call."""

    NAMES = ["band_qk", "band_softmax", "band_pv", "band_qk", "band_softmax_bwd", "band_pv",
             "band_t", "band_t"]
    LAUNCHES = 8
    DESCRIPTION = ("materialised fwd+bwd: band_qk, band_softmax, band_pv, band_qk(dO,V), "
                   "band_softmax_bwd, band_pv(dS,K), band_qk_bwd_t, band_pv_bwd_t")

    def __init__(self, wl, device):
        import sliding_window_attention_band_gb300 as swab

        self.swab = swab
        self.wl = wl
        self.d = swab.Desc.from_workload(wl)
        Q, K, V, dO = workload_inputs(wl)
        self.host = [x.pin_memory() for x in (Q, K, V, dO)]
        self.Q, self.K, self.V, self.dO = (x.to(device) for x in (Q, K, V, dO))
        band = (wl.BH, wl.n, wl.D)
        dense = (wl.BH, wl.n, wl.head_dim)
        mk = lambda shape: torch.empty(shape, dtype=wl.dtype, device=device)  # noqa: E731
        self.S, self.P, self.dP, self.dS = (mk(band) for _ in range(4))
        self.O, self.dQ, self.dK, self.dV = (mk(dense) for _ in range(4))
        self.lse = torch.empty((wl.BH, wl.n), dtype=torch.float32, device=device)
        self.out_host = [torch.empty(dense, dtype=wl.dtype).pin_memory() for _ in range(4)]

    def launches(self):
        s, d, sc = self.swab, self.d, self.wl.scale
        return [
            lambda: s.band_qk(d, sc, self.Q, self.K, self.S),
            lambda: s.band_softmax(d, self.S, self.P, self.lse),
            lambda: s.band_pv(d, 1.0, self.P, self.V, self.O),
            lambda: s.band_qk(d, 1.0, self.dO, self.V, self.dP),
            lambda: s.band_softmax_bwd(d, self.P, self.dP, self.dS),
            lambda: s.band_pv(d, sc, self.dS, self.K, self.dQ),
            lambda: s.band_qk_bwd_t(d, sc, self.dS, self.Q, self.dK),
            lambda: s.band_pv_bwd_t(d, 1.0, self.P, self.dO, self.dV),
        ]

    def capture(self):
        """Capture each API call once into its own CUDA graph; run() then replays
        them: the same kernels, with no host work between the launches."""
        self.graphs = []
        for fn in self.launches():
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, capture_error_mode="thread_local"):
                fn()
            self.graphs.append(g)
        torch.cuda.synchronize()

    def run(self, events=None, eager=False):
        graphs = getattr(self, "graphs", None)
        fns = self.launches() if eager or not graphs else [g.replay for g in graphs]
        for k, fn in enumerate(fns):
            if events is not None:
                events[k].record()
            fn()
        if events is not None:
            events[-1].record()

    def h2d(self):
        for dst, src in zip((self.Q, self.K, self.V, self.dO), self.host):
            dst.copy_(src, non_blocking=True)

    def d2h(self):
        for dst, src in zip(self.out_host, (self.O, self.dQ, self.dK, self.dV)):
            dst.copy_(src, non_blocking=True)

    @property
    def h2d_bytes(self):
        return sum(x.numel() * x.element_size() for x in self.host)

    @property
    def d2h_bytes(self):
        return sum(x.numel() * x.element_size() for x in self.out_host)


class GlobStep(Step):
    """The materialised eight-call step with global tokens: every band tensor
    has its two dense companions (cols [b, h, n, G], rows [b, h, G, n])."""

    DESCRIPTION = ("materialised fwd+bwd with global tokens: band_qk, band_softmax, band_pv, "
                   "band_qk(dO,V), band_softmax_bwd, band_pv(dS,K), band_qk_bwd_t, band_pv_bwd_t, "
                   "each with its cols / rows companions")

    def __init__(self, wl, device):
        super().__init__(wl, device)
        G = len(wl.global_idx)
        mk = lambda: (torch.empty(wl.BH, wl.n, G, dtype=wl.dtype, device=device),  # noqa: E731
                      torch.empty(wl.BH, G, wl.n, dtype=wl.dtype, device=device))
        self.Sg, self.Pg, self.dPg, self.dSg = mk(), mk(), mk(), mk()

    def launches(self):
        s, d, sc = self.swab, self.d, self.wl.scale
        return [
            lambda: s.band_qk(d, sc, self.Q, self.K, self.S, self.Sg),
            lambda: s.band_softmax(d, self.S, self.P, self.lse, Sg=self.Sg, Pg=self.Pg),
            lambda: s.band_pv(d, 1.0, self.P, self.V, self.O, Pg=self.Pg),
            lambda: s.band_qk(d, 1.0, self.dO, self.V, self.dP, self.dPg),
            lambda: s.band_softmax_bwd(d, self.P, self.dP, self.dS, Pg=self.Pg, dPg=self.dPg, dSg=self.dSg),
            lambda: s.band_pv(d, sc, self.dS, self.K, self.dQ, Pg=self.dSg),
            lambda: s.band_qk_bwd_t(d, sc, self.dS, self.Q, self.dK, self.dSg),
            lambda: s.band_pv_bwd_t(d, 1.0, self.P, self.dO, self.dV, self.Pg),
        ]


class FusedStep(Step):
    """Forward + backward with the scores kept on chip: band_attention (O, lse),
    then band_attention_bwd (dQ, dK, dV: its row-sum kernel, the one-pass
    dK/dV/dQ kernel and the dQ rounding kernel)."""

    NAMES = ["band_attention", "band_attention_bwd"]
    LAUNCHES = 4
    DESCRIPTION = ("fused fwd+bwd: band_attention (O, lse), band_attention_bwd "
                   "(row sums, one-pass dK/dV/dQ kernel, dQ rounding)")

    def __init__(self, wl, device):
        super().__init__(wl, device)
        nbytes = self.swab.band_attention_bwd_workspace(self.d)
        self.ws = torch.empty(nbytes // 4, dtype=torch.float32, device=device)

    def launches(self):
        s, d, sc = self.swab, self.d, self.wl.scale
        return [
            lambda: s.band_attention(d, sc, self.Q, self.K, self.V, self.O, self.lse),
            lambda: s.band_attention_bwd(d, sc, self.Q, self.K, self.V, self.O, self.dO, self.lse,
                                         self.dQ, self.dK, self.dV, self.ws),
        ]


class FusedVariantStep(FusedStep):
    """The fused step with one of the optional features of the fused calls:
    dropout of the probabilities (p = 0.1; also with the keep-bit cache, the
    forward storing the keep bits for the backward), a key-padding bias (a
    quarter of the keys masked with -10000), or the strided layout (Q, K, V read from a
    merged [b, n, 3, h, 64] projection buffer, dQ, dK, dV written into one)."""

    def __init__(self, wl, device, feature):
        import sliding_window_attention_band_gb300 as swab

        super().__init__(wl, device)
        self.feature = feature
        self.DESCRIPTION = f"fused fwd+bwd with {feature}"
        kw = {}
        if feature == "dropout p=0.1":
            kw = dict(dropout_p=0.1, dropout_seed=1234)
        elif feature == "dropout p=0.1 keep-bit cache":
            # the forward stores its keep bits, the backward reads them
            d0 = swab.Desc(wl.b, wl.h, wl.n, wl.head_dim, wl.w, wl.w_upper, wl.dilation,
                           wl.padding, wl.dtype, dropout_p=0.1, dropout_seed=1234)
            self.mask = torch.empty(swab.band_attention_dropout_mask_bytes(d0) // 4,
                                    dtype=torch.int32, device=device)
            kw = dict(dropout_p=0.1, dropout_seed=1234, dropout_mask=self.mask)
        elif feature == "key bias":
            g = torch.Generator().manual_seed(77)
            keep = torch.rand(wl.b, wl.n, generator=g) > 0.25
            self.kbias = torch.where(keep, 0.0, -10000.0).to(device)
            kw = dict(key_bias=self.kbias)
        elif feature == "strided qkv":
            b, h, n, hd = wl.b, wl.h, wl.n, wl.head_dim
            self.qkv = torch.empty(b, n, 3, h, hd, dtype=wl.dtype, device=device)
            for m, x in enumerate((self.Q, self.K, self.V)):
                self.qkv[:, :, m] = x.view(b, h, n, hd).permute(0, 2, 1, 3)
            self.dqkv = torch.empty_like(self.qkv)
            self.Os = torch.empty(b, n, h, hd, dtype=wl.dtype, device=device)
            self.dOs = self.dO.view(b, h, n, hd).permute(0, 2, 1, 3).contiguous()
            kw = dict(qkv_row_stride=3 * h * hd, out_row_stride=h * hd)
        else:
            raise ValueError(feature)
        self.d = swab.Desc(wl.b, wl.h, wl.n, wl.head_dim, wl.w, wl.w_upper, wl.dilation,
                           wl.padding, wl.dtype, **kw)

    def launches(self):
        if self.feature != "strided qkv":
            return super().launches()
        s, d, sc = self.swab, self.d, self.wl.scale
        Q, K, V = (self.qkv[:, :, m] for m in range(3))
        dQ, dK, dV = (self.dqkv[:, :, m] for m in range(3))
        return [
            lambda: s.band_attention(d, sc, Q, K, V, self.Os, self.lse),
            lambda: s.band_attention_bwd(d, sc, Q, K, V, self.Os, self.dOs, self.lse, dQ, dK, dV,
                                         self.ws),
        ]


def time_graph(fn, steps, warmup, flush):
    """Mean device time (ms) of one call captured into a CUDA graph, L2 flushed
    before every timed replay."""
    for _ in range(warmup):
        flush_l2(flush)
        fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, capture_error_mode="thread_local"):
        fn()
    torch.cuda.synchronize()
    ts = []
    for _ in range(steps):
        flush_l2(flush)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        g.replay()
        b.record()
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b))
    return statistics.mean(ts)


def prologue_and_globals(device, steps, flush, peaks):
    """add_bias_transpose on the merged Q, K, V projection of the Longformer-base
    shape, and the global queries with their own projections on the training
    shape (b = 12, h = 12, n = 4096, 16 global tokens, bf16)."""
    import sliding_window_attention_band_gb300 as swab

    out = {}
    wl = WORKLOADS[MAIN_CFG]
    g = torch.Generator().manual_seed(5)
    X = torch.randn(wl.b, wl.n, 3, wl.h, wl.head_dim, generator=g).to(wl.dtype).to(device)
    bias = torch.randn(3, wl.h, wl.head_dim, generator=g).to(wl.dtype).to(device)
    Y = torch.empty(3, wl.b, wl.h, wl.n, wl.head_dim, dtype=wl.dtype, device=device)
    d = swab.Desc(wl.b, wl.h, wl.n, wl.head_dim, wl.w, wl.w_upper, dtype=wl.dtype)
    ms = time_graph(lambda: swab.add_bias_transpose(d, X, bias, Y), steps, 3, flush)
    nbytes = 2 * X.numel() * X.element_size() + bias.numel() * bias.element_size()
    out[f"add_bias_transpose:{wl.name}"] = {
        "ms": round(ms, 4), "gbs": round(nbytes / (ms * 1e-3) / 1e9, 1), "bound": "hbm",
        "roofline_frac": round(nbytes / (peaks["hbm_gbs"] * 1e9) / (ms * 1e-3), 4),
        "bytes": nbytes}
    w4 = WORKLOADS[4]
    # the fused forward with global tokens on the training shape
    Q4, K4, V4 = (x.to(device) for x in workload_inputs(w4, count=3))
    O4 = torch.empty_like(Q4)
    lse4 = torch.empty(w4.BH, w4.n, dtype=torch.float32, device=device)
    d4 = swab.Desc.from_workload(w4)
    ms4 = time_graph(lambda: swab.band_attention(d4, w4.scale, Q4, K4, V4, O4, lse4), steps, 3, flush)
    fl4 = 2 * 2.0 * w4.head_dim * valid_pairs_globals(w4)
    out[f"band_attention+globals:{w4.name}"] = {
        "ms": round(ms4, 4), "tflops": round(fl4 / (ms4 * 1e-3) / 1e12, 2),
        "roofline_frac": round(fl4 / (peaks["bf16_tflops"] * 1e12) / (ms4 * 1e-3), 4), "bound": "tensor",
        "note": "band part (global keys masked) + global columns merged + global rows"}
    # the fused training step with global tokens: forward, then the backward
    # (band pass with global keys and queries left out, global columns, global
    # rows), on the same shape
    dO4 = workload_inputs(w4)[3].to(device)
    dQ4, dK4, dV4 = (torch.empty_like(Q4) for _ in range(3))
    ws4 = torch.empty(swab.band_attention_bwd_workspace(d4) // 4 + 4, dtype=torch.float32, device=device)
    msb = time_graph(lambda: swab.band_attention_bwd(d4, w4.scale, Q4, K4, V4, O4, dO4, lse4, dQ4, dK4, dV4, ws4),
                     steps, 3, flush)
    fl4b = 2 * fl4
    out[f"fused+globals:{w4.name}"] = {
        "ms_per_step": round(ms4 + msb, 4), "fwd_ms": round(ms4, 4), "bwd_ms": round(msb, 4),
        "tflops": round((fl4 + fl4b) / ((ms4 + msb) * 1e-3) / 1e12, 2),
        "roofline_frac": round((fl4 + fl4b) / (peaks["bf16_tflops"] * 1e12) / ((ms4 + msb) * 1e-3), 4),
        "bound": "tensor",
        "note": "band_attention then band_attention_bwd with 16 global tokens, bf16; flops = 6 contractions x "
                "2 x head_dim over the attended (query, key) pairs"}
    # the same step on a padded batch: a key-padding bias (a quarter of the keys
    # masked) together with the global tokens
    kb4 = torch.where(torch.rand(w4.b, w4.n, generator=g) > 0.25, 0.0, -10000.0).to(device)
    d4b = swab.Desc(w4.b, w4.h, w4.n, w4.head_dim, w4.w, w4.w_upper, w4.dilation, w4.padding, w4.dtype,
                    w4.global_idx, key_bias=kb4)
    msf = time_graph(lambda: swab.band_attention(d4b, w4.scale, Q4, K4, V4, O4, lse4), steps, 3, flush)
    msbk = time_graph(lambda: swab.band_attention_bwd(d4b, w4.scale, Q4, K4, V4, O4, dO4, lse4, dQ4, dK4, dV4, ws4),
                      steps, 3, flush)
    out[f"fused+globals+key_bias:{w4.name}"] = {
        "ms_per_step": round(msf + msbk, 4), "fwd_ms": round(msf, 4), "bwd_ms": round(msbk, 4),
        "tflops": round((fl4 + fl4b) / ((msf + msbk) * 1e-3) / 1e12, 2),
        "roofline_frac": round((fl4 + fl4b) / (peaks["bf16_tflops"] * 1e12) / ((msf + msbk) * 1e-3), 4),
        "bound": "tensor",
        "note": "the step above with a key-padding bias (a quarter of the keys masked); flops counted as above"}
    del Q4, K4, V4, O4, dO4, dQ4, dK4, dV4, ws4, kb4
    dg = swab.Desc.from_workload(w4)
    G, BH, n = dg.G, w4.BH, w4.n
    mk = lambda *sh: torch.randn(*sh, generator=g).to(w4.dtype).to(device)  # noqa: E731
    Qg, dOg, Kg, Vg = mk(BH, G, 64), mk(BH, G, 64), mk(BH, n, 64), mk(BH, n, 64)
    Og, dQg, dKg, dVg = (torch.empty_like(x) for x in (Qg, Qg, Kg, Vg))
    lseg = torch.empty(BH, G, dtype=torch.float32, device=device)
    ws = torch.empty(swab.global_attention_workspace(dg) // 4 + 4, dtype=torch.float32,
                     device=device)
    fwd = time_graph(lambda: swab.global_attention(dg, w4.scale, Qg, Kg, Vg, Og, lseg, ws),
                     steps, 3, flush)
    bwd = time_graph(lambda: swab.global_attention_bwd(dg, w4.scale, Qg, Kg, Vg, Og, dOg, lseg,
                                                       dQg, dKg, dVg, ws), steps, 3, flush)
    es = Kg.element_size()
    fb = 2 * BH * n * 64 * es                      # Kg, Vg read
    bb = 2 * fb                                    # Kg, Vg read, dKg, dVg written
    out[f"global_attention:{w4.name}"] = {
        "fwd_ms": round(fwd, 4), "bwd_ms": round(bwd, 4),
        "fwd_tflops": round(4.0 * BH * G * n * 64 / (fwd * 1e-3) / 1e12, 2),
        "bwd_tflops": round(10.0 * BH * G * n * 64 / (bwd * 1e-3) / 1e12, 2),
        "bound": "hbm", "fwd_roofline_frac": round(fb / (peaks["hbm_gbs"] * 1e9) / (fwd * 1e-3), 4),
        "bwd_roofline_frac": round(bb / (peaks["hbm_gbs"] * 1e9) / (bwd * 1e-3), 4),
        "note": "tcgen05 kernels, one CTA per 128-key tile (keys as the M dimension)"}
    return out


def step_summary(wl, step, per_step, per_kernel, peaks):
    return {"ms_per_step": round(statistics.mean(per_step), 4),
            "ms_per_step_median": round(statistics.median(per_step), 4),
            "ms_per_step_p10": round(float(np.percentile(per_step, 10)), 4),
            "ms_per_step_p90": round(float(np.percentile(per_step, 90)), 4),
            "tflops": round(step_flops(wl) / (statistics.mean(per_step) * 1e-3) / 1e12, 3),
            "per_call_us": {f"{i}:{nm}": round(statistics.mean(t) * 1e3, 2)
                            for i, (nm, t) in enumerate(zip(step.NAMES, per_kernel))},
            "roofline": roofline(wl, step.NAMES, per_kernel, peaks),
            "step_roofline_frac": round(step_roofline_frac(wl, step.NAMES, per_kernel, peaks), 4)}


_FLUSH_SINK = None


def flush_l2(flush):
    """Evict L2 before a timed step: write a buffer twice the size of L2, then
    read it back, so that the lines left in L2 are clean and the timed kernels
    do not pay for writing the flush's own data back to HBM."""
    global _FLUSH_SINK
    flush.zero_()
    if _FLUSH_SINK is None or _FLUSH_SINK.device != flush.device:
        _FLUSH_SINK = torch.empty(1, dtype=flush.dtype, device=flush.device)
    _FLUSH_SINK.copy_(flush.sum().view(1))


def time_steps(step, steps, warmup, flush):
    """Per-step device times (ms) and per-call times (ms) over `steps` steps: the
    calls run eagerly for the warm-up, are captured once into CUDA graphs, and
    the timed steps replay them."""
    for _ in range(warmup):
        flush_l2(flush)
        step.run(eager=True)
    torch.cuda.synchronize()
    step.capture()
    nk = len(step.NAMES)
    per_step, per_kernel = [], [[] for _ in range(nk)]
    for _ in range(steps):
        flush_l2(flush)  # L2 flush outside the timed events
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(nk + 1)]
        step.run(ev)
        torch.cuda.synchronize()
        per_step.append(ev[0].elapsed_time(ev[-1]))
        for k in range(nk):
            per_kernel[k].append(ev[k].elapsed_time(ev[k + 1]))
    return per_step, per_kernel


def fused_forward(wl, device, steps, warmup, flush, peaks):
    """band_attention (scores on chip) on one workload: ms, TFLOP/s, roofline."""
    import sliding_window_attention_band_gb300 as swab

    d = swab.Desc.from_workload(wl)
    Q, K, V = (x.to(device) for x in workload_inputs(wl, count=3))
    O = torch.empty_like(Q)
    lse = torch.empty((wl.BH, wl.n), dtype=torch.float32, device=device)
    for _ in range(warmup):
        swab.band_attention(d, wl.scale, Q, K, V, O, lse)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()   # captured once, replayed in the timed runs
    with torch.cuda.graph(g, capture_error_mode="thread_local"):
        swab.band_attention(d, wl.scale, Q, K, V, O, lse)
    torch.cuda.synchronize()
    ts = []
    for _ in range(steps):
        flush_l2(flush)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        g.replay()
        b.record()
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b))
    ms = statistics.mean(ts)
    flops = 2 * 2.0 * wl.head_dim * valid_pairs(wl)
    e = torch.finfo(wl.dtype).bits // 8
    nbytes = 4 * wl.BH * wl.n * wl.head_dim * e + wl.BH * wl.n * 4
    t_roof = max(nbytes / (peaks["hbm_gbs"] * 1e9), flops / (peaks["bf16_tflops"] * 1e12))
    bound = "tensor" if flops / (peaks["bf16_tflops"] * 1e12) > nbytes / (peaks["hbm_gbs"] * 1e9) \
        else "hbm"
    return {"ms": round(ms, 4), "tflops": round(flops / (ms * 1e-3) / 1e12, 2),
            "gbs": round(nbytes / (ms * 1e-3) / 1e9, 1), "bound": bound,
            "roofline_frac": round(t_roof / (ms * 1e-3), 4), "flops": flops, "bytes": nbytes}


E2E_SETS = 6   # device buffer sets the end-to-end steps rotate over


def time_e2e(step, steps, warmup, flush, sets=E2E_SETS):
    """End-to-end time per step (ms) through the public API.  Every step copies
    its own inputs (Q, K, V, dO) in from pinned host memory, makes the API
    calls eagerly, and copies its results (O, dQ, dK, dV) back out.  The steps
    are pipelined the way a data loader feeds a training loop: the next step's
    inputs go in on one copy stream and the previous step's results come out
    on another while a step computes on the current stream.  The inputs sit
    side by side in one pinned buffer and the results in another (one copy
    each way a step; the calls take the tensors as views).  The device
    buffers rotate over `sets` sets (8 tensors each; 300 MB at the Longformer
    base shape, over twice the L2), so no step finds an earlier step's data in
    L2: its inputs are the ones its own copy just wrote.  The time runs from
    the first copy in to the last copy out of the timed steps."""
    names_in, names_out = ("Q", "K", "V", "dO"), ("O", "dQ", "dK", "dV")
    # the four inputs side by side in one pinned buffer and the four results
    # in another, so that each direction is one copy a step
    shape = tuple(step.Q.shape)
    host_in = torch.stack([x for x in step.host]).pin_memory()
    host_out = torch.empty((4,) + shape, dtype=step.Q.dtype).pin_memory()
    bufs = []
    for _ in range(sets):
        din = torch.empty((4,) + shape, dtype=step.Q.dtype, device=step.Q.device)
        dout = torch.empty_like(din)
        buf = {"in": din, "out": dout}
        buf.update({nm: din[k] for k, nm in enumerate(names_in)})
        buf.update({nm: dout[k] for k, nm in enumerate(names_out)})
        bufs.append(buf)
    cur = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(sets)]
    ev_comp = [torch.cuda.Event() for _ in range(sets)]
    ev_out = [torch.cuda.Event() for _ in range(sets)]

    def issue(i):
        b, buf = i % sets, bufs[i % sets]
        with torch.cuda.stream(s_in):
            s_in.wait_event(ev_comp[b])          # the set's last step has read its inputs
            buf["in"].copy_(host_in, non_blocking=True)
            ev_in[b].record(s_in)
        cur.wait_event(ev_in[b])
        cur.wait_event(ev_out[b])                # the set's last results are out
        for nm in names_in + names_out:
            setattr(step, nm, buf[nm])
        step.run(eager=True)                     # the calls a user makes, host work included
        ev_comp[b].record(cur)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_comp[b])
            host_out.copy_(buf["out"], non_blocking=True)
            ev_out[b].record(s_out)

    keep = {nm: getattr(step, nm) for nm in names_in + names_out}
    for i in range(warmup):
        issue(i)
    torch.cuda.synchronize()
    flush_l2(flush)
    a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(cur)
    s_in.wait_stream(cur)
    for i in range(warmup, warmup + steps):
        issue(i)
    cur.wait_stream(s_out)
    b_.record(cur)
    torch.cuda.synchronize()
    for nm, t in keep.items():
        setattr(step, nm, t)
    return a.elapsed_time(b_) / steps


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.path = tempfile.mktemp(suffix=".csv")
        self.proc = None
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.f,
                stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx = float(parts[2])
                except ValueError:
                    continue
                for nm, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(nm)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# roofline
# ---------------------------------------------------------------------------
def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def kernel_source_hash(kernel):
    files = {"band_qk": "k_band_qk.cu", "band_pv": "k_band_gather.cu", "band_t": "k_band_gather.cu",
             "band_softmax": "k_softmax.cu", "band_softmax_bwd": "k_softmax.cu",
             "band_attention": "k_attention.cu", "band_attention_bwd": "k_attention_bwd.cu"}
    path = os.path.join(ROOT, "sliding_window_attention_band_gb300", "csrc", files[kernel])
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def ncu_traffic(kernel, workload):
    """DRAM bytes per launch from the committed ncu summary, if the kernel source
    still matches the one profiled; else None."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        table = json.load(f)
    ent = table.get(workload, {}).get(kernel)
    if not ent or ent.get("source_sha256_16") != kernel_source_hash(kernel):
        return None
    return ent.get("dram_bytes_per_launch")


def roofline(wl, names, per_kernel_ms, peaks):
    """The kernel with the largest total time in the step."""
    tot = {}
    cnt = {}
    for name, ts in zip(names, per_kernel_ms):
        tot[name] = tot.get(name, 0.0) + sum(ts)
        cnt[name] = cnt.get(name, 0) + len(ts)
    top = max(tot, key=tot.get)
    avg_ms = tot[top] / cnt[top]
    nbytes = kernel_bytes(wl)[top]
    flops = kernel_flops(wl)[top]
    t_hbm = nbytes / (peaks["hbm_gbs"] * 1e9)
    t_tc = flops / (peaks["bf16_tflops"] * 1e12)
    if t_tc > t_hbm:
        ach, peak, unit, bound = flops / (avg_ms * 1e-3) / 1e12, peaks["bf16_tflops"], "TFLOP/s", "tensor"
    else:
        ach, peak, unit, bound = nbytes / (avg_ms * 1e-3) / 1e9, peaks["hbm_gbs"], "GB/s", "hbm"
    return {"kernel": top, "bound": bound, "achieved": round(ach, 1), "peak": peak,
            "unit": unit, "frac": round(ach / peak, 4), "traffic": ncu_traffic(top, wl.name),
            "algorithmic_bytes": nbytes, "avg_launch_us": round(avg_ms * 1e3, 2),
            "peak_source": peaks["source"]}


def step_roofline_frac(wl, names, per_kernel_ms, peaks):
    """sum over kernels of max(bytes/BW, flops/TC) / measured step time."""
    kb, kf = kernel_bytes(wl), kernel_flops(wl)
    ideal = sum(max(kb[nm] / (peaks["hbm_gbs"] * 1e9), kf[nm] / (peaks["bf16_tflops"] * 1e12))
                for nm in names)
    meas = sum(statistics.mean(ts) for ts in per_kernel_ms) * 1e-3
    return ideal / meas


# ---------------------------------------------------------------------------
# CPU oracle timing
# ---------------------------------------------------------------------------
def oracle_step(wl, slices):
    """The same fwd+bwd chain on the fp64 oracle for `slices` (b,h) slices."""
    import oracle

    Q, K, V, dO = workload_inputs(wl)
    q, k, v, go = (x[:slices].double().numpy() for x in (Q, K, V, dO))
    w, wu, dil, sc = wl.w, wl.w_upper, wl.dilation, wl.scale
    t0 = time.perf_counter()
    S = oracle.band_qk(q, k, w, wu, dil, sc, wl.padding)
    P, _ = oracle.band_softmax(S, w, wu, dil)
    oracle.band_pv(P, v, w, wu, dil, 1.0)
    dP = oracle.band_qk(go, v, w, wu, dil, 1.0, wl.padding)
    dS = oracle.band_softmax_bwd(P, dP, w, wu, dil)
    oracle.band_pv(dS, k, w, wu, dil, sc)
    oracle.band_t(dS, q, w, wu, dil, sc)
    oracle.band_t(P, go, w, wu, dil, 1.0)
    return time.perf_counter() - t0


def cpu_baseline(wl, budget_s=15.0):
    import oracle

    t1 = oracle_step(wl, 1)
    slices = int(max(1, min(wl.BH, budget_s // max(t1, 1e-3))))
    t = oracle_step(wl, slices) if slices > 1 else t1
    flops = step_flops(wl) * slices / wl.BH
    return {"value": round(flops / t / 1e12, 6), "unit": "TFLOP/s", "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": f"{slices} of {wl.BH} (b,h) slices of {wl.name}, full fwd+bwd chain in fp64, "
                      f"{t:.2f} s"}


def job_value(dev_ms, world, steps, flops_per_step, dist=None, device=None):
    """Whole-job throughput over N ranks that each run the same workload (weak
    scaling, replicas): the slowest rank's timed region (max over ranks) and
    the flops of all ranks divided by it, in TFLOP/s."""
    if dist is not None and world > 1:
        t = torch.tensor([float(dev_ms)], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        dev_ms = float(t.item())
    return dev_ms, world * flops_per_step * steps / (dev_ms * 1e-3) / 1e12


def run_reference(args):
    """The fp64 oracle as it stands, on the host cores: each step runs the full
    forward + backward chain on ONE (b, h) slice of the headline workload (a
    bounded sample; all 12 slices take about 12x as long), and the line reports
    the time of exactly that work."""
    import oracle

    wl = WORKLOADS[MAIN_CFG]
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    oracle.build()
    for _ in range(args.warmup):
        oracle_step(wl, 1)
    ts = [oracle_step(wl, 1) for _ in range(args.steps)]
    flops = step_flops(wl) / wl.BH
    val = flops * len(ts) / sum(ts) / 1e12
    sample = (f"each step: 1 of {wl.BH} (b,h) slices of {wl.name}, the full fwd+bwd chain in "
              f"fp64; ms_per_step is the time of that one slice")
    line = {"impl": "reference", "metric": METRIC, "value": round(val, 6), "unit": "TFLOP/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(statistics.mean(ts) * 1e3, 3),
            "ms_per_step_median": round(statistics.median(ts) * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {**wl.describe(), "parallelism": "none (host oracle)",
                       "slices_per_step": 1, "flops_per_step": flops},
            "cpu_baseline": {"value": round(val, 6), "unit": "TFLOP/s",
                             "cores": oracle.num_threads(), "kind": "oracle", "sample": sample},
            "e2e": {"value": round(val, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="swab", choices=["swab", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--step", default="fused", choices=["fused", "materialised"],
                    help="fused: band_attention + band_attention_bwd; materialised: the "
                         "eight band_qk / softmax / band_pv / band_t calls")
    ap.add_argument("--no-also", action="store_true",
                    help="skip the companion timings (other step variant, dilation 3, long "
                         "causal forward); used for short profiling runs")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl")

    from sliding_window_attention_band_gb300 import build as swab_build

    if rank == 0 or world == 1:
        swab_build.build()
    if dist:
        dist.barrier()
    import sliding_window_attention_band_gb300 as swab

    swab.load()
    device = torch.device("cuda", local)
    wl = WORKLOADS[MAIN_CFG]
    step_cls = FusedStep if args.step == "fused" else Step
    step = step_cls(wl, device)
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=device)
    peaks = measured_peaks()

    clocks = ClockSampler(local)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    per_step, per_kernel = time_steps(step, args.steps, args.warmup, flush)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    t_wall = time.perf_counter() - t_wall
    clk = clocks.stop()

    flops = step_flops(wl)
    dev_ms, value = job_value(sum(per_step), world, args.steps, flops, dist, device)
    ms_per_step = dev_ms / args.steps
    e2e_ms = time_e2e(step, max(10, args.steps), 3, flush)
    e2e_val = world * flops / (e2e_ms * 1e-3) / 1e12

    # companions, timed the same way: the other step variant, dilation 3, the
    # fused forward on the long causal workload
    also = {}
    n_also = max(3, args.steps // 2)
    for cls in (() if args.no_also else (FusedStep, Step)):
        for w_ in (WORKLOADS[MAIN_CFG], WORKLOADS[ALSO_CFG]):
            if cls is step_cls and w_ is wl:
                continue
            st = cls(w_, device)
            ps, pk = time_steps(st, n_also, 3, flush)
            also[f"{'fused' if cls is FusedStep else 'materialised'}:{w_.name}"] = \
                step_summary(w_, st, ps, pk, peaks)
            del st
    if not args.no_also:
        wl5 = WORKLOADS[5]
        also[f"band_attention:{wl5.name}"] = fused_forward(wl5, device, n_also, 3, flush, peaks)
        # the same workload with its [1, 12, 32768, 4097] scores materialised:
        # the forward calls alone (band_qk, band_softmax, band_pv) against the
        # fused forward above, then the whole eight-call step
        st = Step(wl5, device)
        ps, pk = time_steps(st, n_also, 3, flush)
        summ = step_summary(wl5, st, ps, pk, peaks)
        fwd_ms = sum(statistics.mean(t) for t in pk[:3])
        summ["forward_calls_ms"] = round(fwd_ms, 4)
        summ["forward_tflops"] = round(2 * 2.0 * wl5.head_dim * valid_pairs(wl5) / (fwd_ms * 1e-3) / 1e12, 2)
        also[f"materialised:{wl5.name}"] = summ
        del st
        for feature in ("dropout p=0.1", "dropout p=0.1 keep-bit cache", "key bias", "strided qkv"):
            st = FusedVariantStep(wl, device, feature)
            ps, pk = time_steps(st, n_also, 3, flush)
            also[f"fused+{feature.replace(' ', '_')}:{wl.name}"] = step_summary(wl, st, ps, pk, peaks)
            del st
        also.update(prologue_and_globals(device, n_also, flush, peaks))
        # the training workload with global tokens through the materialised calls
        w4 = WORKLOADS[4]
        st = GlobStep(w4, device)
        ps, pk = time_steps(st, max(3, n_also // 4), 3, flush)
        ms = statistics.mean(ps)
        fl = 6 * 2.0 * w4.head_dim * valid_pairs_globals(w4)
        also[f"materialised+globals:{w4.name}"] = {
            "ms_per_step": round(ms, 4), "tflops": round(fl / (ms * 1e-3) / 1e12, 2),
            "per_call_us": {f"{i}:{nm}": round(statistics.mean(t) * 1e3, 1)
                            for i, (nm, t) in enumerate(zip(st.NAMES, pk))},
            "note": "eight materialised calls with global tokens (16), bf16; flops = 6 contractions x "
                    "2 x head_dim over the attended pairs"}
        del st
    if swab.device_status(reset=True) != 0:
        raise SystemExit("a kernel raised the device status word during the benchmark")

    line = {
        "metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
        "ms_per_step_median": round(statistics.median(per_step), 4),
        "ms_per_step_p10": round(float(np.percentile(per_step, 10)), 4),
        "ms_per_step_p90": round(float(np.percentile(per_step, 90)), 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "data": "synthetic",
        "config": {**wl.describe(), "parallelism": f"replicas x{world}" if world > 1 else "none",
                   "l2": "flushed before every timed step (256 MB write, then read back so L2 holds clean lines)",
                   "step": step.DESCRIPTION, "flops_per_step": flops,
                   "launch": "each API call captured once into a CUDA graph and replayed in the "
                             "timed steps; e2e calls the API eagerly",
                   "flops_counted": "6 banded contractions x 2*head_dim per valid pair"},
        "per_call_us": {f"{i}:{nm}": round(statistics.mean(t) * 1e3, 2)
                        for i, (nm, t) in enumerate(zip(step.NAMES, per_kernel))},
        "roofline": roofline(wl, step.NAMES, per_kernel, peaks),
        "step_roofline_frac": round(step_roofline_frac(wl, step.NAMES, per_kernel, peaks), 4),
        "e2e": {"value": round(e2e_val, 3), "unit": "TFLOP/s",
                "h2d_bytes_per_step": step.h2d_bytes, "d2h_bytes_per_step": step.d2h_bytes,
                "ms_per_step": round(e2e_ms, 4),
                "pipeline": f"pinned-host copies in and out of every step on two copy streams "
                            f"(the four inputs packed in one buffer, the four results in "
                            f"another: one copy each way), overlapping the neighbouring steps' "
                            f"API calls; device buffers rotate over {E2E_SETS} sets (> 2x L2)"},
        "gpu_launches": step.LAUNCHES * args.steps,
        "clocks": clk,
        "wall_s_timed_region": round(t_wall, 3),
        "also": also,
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
