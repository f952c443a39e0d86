"""The strided [b, n, h, hd] layout of the fused calls and AddBiasTranspose
(ONNX Runtime issue "[WIP] Improve LongformerAttention performance", item (2)
and the merged QKV projection of conclusion (c)), against the fp64 oracle.

* add_bias_transpose: bit-exact against the oracle's fp64 sum rounded once to
  the dtype (the kernel's fp32 sum of two fp16 / bf16 values, rounded once, is
  the correctly rounded sum);
* band_attention / band_attention_bwd reading Q, K, V straight out of a merged
  [b, n, 3, h, 64] projection buffer and writing O, dQ, dK, dV into strided
  buffers: bitwise equal to the contiguous-layout call (the layout changes only
  addresses) for O, lse, dK, dV; dQ is summed by fp32 atomic additions in a
  run-dependent order, so it is compared with the oracle's tolerance; the
  unused columns of every strided buffer keep their sentinel.
"""
import numpy as np
import pytest
import torch

import oracle
import sliding_window_attention_band_gb300 as swab

from test_gpu_parity import F32_TOL, f64, normwise, within_abs

pytestmark = [pytest.mark.gpu, pytest.mark.usefixtures("device_status_guard")]

DTYPES = [torch.float16, torch.bfloat16, torch.float32]


def dname(dt):
    return str(dt).split(".")[-1]


@pytest.mark.parametrize("dtype", DTYPES, ids=dname)
@pytest.mark.parametrize("b,n,M,h,hd,with_bias", [(1, 4096, 3, 12, 64, True),
                                                    (2, 777, 3, 3, 64, True),
                                                    (3, 129, 1, 2, 64, False),
                                                    (2, 100, 2, 5, 32, True)])
def test_add_bias_transpose(dtype, b, n, M, h, hd, with_bias):
    g = torch.Generator().manual_seed(b * 1000 + n)
    X = (torch.randn(b, n, M, h, hd, generator=g) * 4).to(dtype)
    bias = (torch.randn(M, h, hd, generator=g)).to(dtype) if with_bias else None
    d = swab.Desc(b, h, n, hd, 1, 1, dtype=dtype)
    Y = torch.full((M, b, h, n, hd), float("nan"), dtype=dtype, device="cuda")
    swab.add_bias_transpose(d, X.cuda(), bias.cuda() if with_bias else None, Y)
    torch.cuda.synchronize()
    ref = oracle.add_bias_transpose(f64(X), f64(bias) if with_bias else None)
    want = torch.from_numpy(ref).to(dtype)   # one rounding of the exact fp64 sum
    assert torch.equal(Y.cpu(), want)


def strided_case(b, h, n, dtype, seed, pad_o=64):
    """Q, K, V views of a merged [b, n, 3, h, 64] buffer; O, dO in rows of
    h*64 + pad_o elements (the padding holds a sentinel)."""
    g = torch.Generator().manual_seed(seed)
    qkv = torch.randn(b, n, 3, h, 64, generator=g).to(dtype).cuda()
    ors = h * 64 + pad_o
    dOb = torch.full((b, n, ors), 7.0, dtype=dtype)
    dOb[:, :, :h * 64] = torch.randn(b, n, h * 64, generator=g).to(dtype)
    return qkv, dOb.cuda(), ors


def view_heads(buf, b, n, h, rs):
    return buf.as_strided((b, n, h, 64), (n * rs, rs, 64, 1))


def to_contig(v):
    """[b, n, h, 64] view -> contiguous [b*h, n, 64]."""
    b, n, h, hd = v.shape
    return v.permute(0, 2, 1, 3).reshape(b * h, n, hd).contiguous()


LAYOUT_CASES = [  # b, h, n, w, w_upper, dilation, dtype, dropout p, key bias
    (1, 12, 1024, 256, 256, 0, torch.float16, 0.0, False),
    (2, 3, 777, 100, 37, 2, torch.bfloat16, 0.0, False),
    (2, 2, 600, 64, 0, 0, torch.float16, 0.1, True),
    (2, 3, 333, 7, 30, 1, torch.float32, 0.0, False),
]


@pytest.mark.parametrize("case", LAYOUT_CASES,
                         ids=lambda c: f"b{c[0]}h{c[1]}-n{c[2]}-w{c[3]}-wu{c[4]}-d{c[5]}-"
                                       f"{dname(c[6])}-p{c[7]}{'-bias' if c[8] else ''}")
def test_fused_strided_layout(case):
    b, h, n, w, wu, dil, dtype, p, with_bias = case
    qkv, dOb, ors = strided_case(b, h, n, dtype, seed=n + 51)
    prs = 3 * h * 64
    bias = None
    if with_bias:
        bias = torch.where(torch.rand(b, n, generator=torch.Generator().manual_seed(3)) > 0.2,
                           0.0, -10000.0).cuda()
    kw = dict(key_bias=bias, dropout_p=p, dropout_seed=1234)
    ds = swab.Desc(b, h, n, 64, w, wu, dil, 0.0, dtype, qkv_row_stride=prs, out_row_stride=ors,
                   **kw)
    dc = swab.Desc(b, h, n, 64, w, wu, dil, 0.0, dtype, **kw)
    Q, K, V = (qkv[:, :, m] for m in range(3))   # [b, n, h, 64] views, row stride 3 h 64
    dO = view_heads(dOb, b, n, h, ors)
    # strided call: O into a padded buffer, dQ/dK/dV into a merged gradient buffer
    Ob = torch.full((b, n, ors), 7.0, dtype=dtype, device="cuda")
    O = view_heads(Ob, b, n, h, ors)
    lse_s = torch.empty(b * h, n, dtype=torch.float32, device="cuda")
    dqkv = torch.full((b, n, 3, h, 64), 5.0, dtype=dtype, device="cuda")
    ws = torch.empty(swab.band_attention_bwd_workspace(ds) // 4, dtype=torch.float32,
                     device="cuda")
    swab.band_attention(ds, 0.125, Q, K, V, O, lse_s)
    swab.band_attention_bwd(ds, 0.125, Q, K, V, O, dO, lse_s, dqkv[:, :, 0], dqkv[:, :, 1],
                            dqkv[:, :, 2], ws)
    # contiguous call on the same values
    Qc, Kc, Vc, dOc = (to_contig(x) for x in (Q, K, V, dO))
    Oc = torch.empty_like(Qc)
    lse_c = torch.empty_like(lse_s)
    dQc, dKc, dVc = (torch.empty_like(Qc) for _ in range(3))
    wsc = torch.empty_like(ws)
    swab.band_attention(dc, 0.125, Qc, Kc, Vc, Oc, lse_c)
    swab.band_attention_bwd(dc, 0.125, Qc, Kc, Vc, Oc, dOc, lse_c, dQc, dKc, dVc, wsc)
    torch.cuda.synchronize()
    # the padding of the strided buffers is untouched
    assert bool((Ob[:, :, h * 64:] == 7.0).all())
    assert torch.equal(to_contig(O), Oc)
    assert torch.equal(lse_s, lse_c)
    dQs, dKs, dVs = (to_contig(dqkv[:, :, m]) for m in range(3))
    assert torch.equal(dKs, dKc) and torch.equal(dVs, dVc)
    # against the oracle (dQ: atomics in a run-dependent order)
    kb = bias.cpu().repeat_interleave(h, dim=0).double().numpy() if with_bias else None
    args = dict(key_bias=kb, drop_t=ds.drop_t, seed=1234)
    q, k, v, go = (f64(x.cpu()) for x in (Qc, Kc, Vc, dOc))
    refO, _ = oracle.attention_fwd(q, k, v, w, wu, dil, 0.125, **args)
    refs = oracle.attention_bwd(q, k, v, go, w, wu, dil, 0.125, **args)
    for name, got, ref in (("O", Oc, refO), ("dQ", dQs, refs[0]), ("dK", dKs, refs[1]),
                           ("dV", dVs, refs[2])):
        if dtype == torch.float32:
            assert normwise(f64(got), ref) <= F32_TOL, name
        else:
            assert within_abs(f64(got), ref, dtype), name


def test_merged_projection_pipeline():
    """AddBiasTranspose then the contiguous fused forward equals the fused
    forward reading the biased merged buffer in place (bias added by the
    same kernel with no transpose: M = 1 over a [b*n*3, 1, h, 64] view)."""
    b, h, n = 2, 4, 512
    g = torch.Generator().manual_seed(8)
    X = torch.randn(b, n, 3, h, 64, generator=g).half().cuda()
    bias = torch.randn(3, h, 64, generator=g).half().cuda()
    d = swab.Desc(b, h, n, 64, 64, 64, 0, 0.0, torch.float16)
    Y = torch.empty(3, b, h, n, 64, dtype=torch.float16, device="cuda")
    swab.add_bias_transpose(d, X, bias, Y)
    O1 = torch.empty(b * h, n, 64, dtype=torch.float16, device="cuda")
    swab.band_attention(d, 0.125, Y[0], Y[1], Y[2], O1)
    Xb = (X.float() + bias.float()).half()   # the same correctly rounded sums
    ds = swab.Desc(b, h, n, 64, 64, 64, 0, 0.0, torch.float16, qkv_row_stride=3 * h * 64)
    O2 = torch.empty(b * h, n, 64, dtype=torch.float16, device="cuda")
    swab.band_attention(ds, 0.125, Xb[:, :, 0], Xb[:, :, 1], Xb[:, :, 2], O2)
    torch.cuda.synchronize()
    assert torch.equal(O1, O2)
