"""The bounds-checked build (libswab_bounds.so, SWAB_BOUNDS_CHECK=1).

In that build every plain global load, store and reduction of every kernel
is tested against the extents the host derives from the descriptor for the
call's buffers (and every tensor map's footprint against the same extents).
This file runs one call of every entry point -- fused forward and backward
in each of their variants (fp16 / bf16 / fp32, dilation, causal, key bias,
dropout with the keep-bit cache, the strided layout, global tokens), the
allocation-free backward, the materialised chain with and without global
tokens, the dropout softmax, the global-query calls and AddBiasTranspose --
at sizes that span several tiles and a ragged tail, in a child process that
loads the checked build, and requires

* no access outside the extents: the status word clear and nothing recorded;
* the same results as the regular build in this process: bit for bit, except
  the dQ outputs that are summed by fp32 atomic additions in a run-dependent
  order (compared within a few units of their last place);
* the checks themselves to work: the self-test's stores outside its extent
  refused and recorded with their site, the ones inside it landed.

No case addresses memory outside its buffers in either build: the checked
build would record such an access instead of making it.

The whole GPU suite can also run on the checked build (SWAB_BOUNDS_CHECK=1 in
the environment of pytest): every module's status-word guard then fails on an
out-of-bounds access.  The two tests here compare the two builds and are
skipped in that mode.
"""
import os
import subprocess
import sys

import pytest
import torch

import sliding_window_attention_band_gb300 as swab
from sliding_window_attention_band_gb300 import build as swab_build

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(os.environ.get("SWAB_BOUNDS_CHECK") == "1",
                                 reason="compares the checked build with the regular one in this process")]

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
BOUNDS_BIT = 1 << 6          # SWAB_ERR_BOUNDS in the device status word
API_FILE_ID = 10             # site id of the entry-point file (self-test kernel)
# outputs summed by fp32 atomic additions (run-dependent order)
ATOMIC = ("dQ",)


def rnd(shape, dtype, seed, scale=0.5):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(*shape, generator=g) * scale).to(dtype).cuda()


def bits(t):
    """The tensor's bit patterns (NaNs compare equal to themselves)."""
    return t.contiguous().view({1: torch.uint8, 2: torch.int16, 4: torch.int32}[t.element_size()])


def sentinel(shape, dtype):
    return torch.full(shape, 3.0, dtype=dtype, device="cuda")


def fused_pair(out, tag, d, seed, noalloc=False):
    """band_attention + band_attention_bwd (+ the allocation-free backward)."""
    shp = (d.BH, d.n, d.head_dim)
    Q, K, V, dO = (rnd(shp, d.dtype, seed + k) for k in range(4))
    O = sentinel(shp, d.dtype)
    lse = torch.zeros(d.BH, d.n, dtype=torch.float32, device="cuda")
    swab.band_attention(d, 0.125, Q, K, V, O, lse)
    dQ, dK, dV = (sentinel(shp, d.dtype) for _ in range(3))
    ws = torch.empty(swab.band_attention_bwd_workspace(d) // 4 + 1, dtype=torch.float32, device="cuda")
    swab.band_attention_bwd(d, 0.125, Q, K, V, O, dO, lse, dQ, dK, dV, ws)
    out.update({f"{tag}.O": O, f"{tag}.lse": lse, f"{tag}.dQ": dQ, f"{tag}.dK": dK, f"{tag}.dV": dV})
    if noalloc:
        nq, nk, nv = (sentinel(shp, d.dtype) for _ in range(3))
        swab.band_attention_bwd_noalloc(d, 0.125, Q, K, V, O, dO, lse, nq, nk, nv)
        out.update({f"{tag}.noalloc.dQ": nq, f"{tag}.noalloc.dK": nk, f"{tag}.noalloc.dV": nv})


def fused_strided(out, tag, b, h, n, dtype, seed):
    """Q, K, V (and dQ, dK, dV) in merged [b, n, 3, h, 64] buffers; O, dO in
    rows of h*64 + 64 elements."""
    qkv = rnd((b, n, 3, h, 64), dtype, seed)
    ors = h * 64 + 64
    dOb = rnd((b, n, ors), dtype, seed + 1)
    Ob = sentinel((b, n, ors), dtype)
    grads = sentinel((b, n, 3, h, 64), dtype)
    rs = 3 * h * 64
    d = swab.Desc(b, h, n, 64, 64, 32, 0, dtype=dtype, qkv_row_stride=rs, out_row_stride=ors)
    heads = lambda buf, k, stride: buf.view(-1)[k * h * 64:].as_strided((b, n, h, 64), (n * stride, stride, 64, 1))
    Q, K, V = (heads(qkv, k, rs) for k in range(3))
    O, dO = heads(Ob, 0, ors), heads(dOb, 0, ors)
    dQ, dK, dV = (heads(grads, k, rs) for k in range(3))
    lse = torch.zeros(b * h, n, dtype=torch.float32, device="cuda")
    swab.band_attention(d, 0.125, Q, K, V, O, lse)
    ws = torch.empty(swab.band_attention_bwd_workspace(d) // 4 + 1, dtype=torch.float32, device="cuda")
    swab.band_attention_bwd(d, 0.125, Q, K, V, O, dO, lse, dQ, dK, dV, ws)
    out.update({f"{tag}.O": Ob, f"{tag}.lse": lse, f"{tag}.dQ": grads[:, :, 0].contiguous(),
                f"{tag}.dKV": grads[:, :, 1:].contiguous()})


def chain(out, tag, d, seed):
    """The materialised forward and backward: eight calls."""
    shp, band = (d.BH, d.n, d.head_dim), (d.BH, d.n, d.D)
    Q, K, V, dO = (rnd(shp, d.dtype, seed + k) for k in range(4))
    G = d.G

    def glob():
        return (sentinel((d.BH, d.n, G), d.dtype), sentinel((d.BH, G, d.n), d.dtype)) if G else None

    S, P, dP, dS = (sentinel(band, d.dtype) for _ in range(4))
    Sg, Pg, dPg, dSg = glob(), glob(), glob(), glob()
    lse = torch.zeros(d.BH, d.n, dtype=torch.float32, device="cuda")
    O, dQ, dK, dV = (sentinel(shp, d.dtype) for _ in range(4))
    swab.band_qk(d, 0.125, Q, K, S, Sg)
    swab.band_softmax(d, S, P, lse, Sg, Pg)
    swab.band_pv(d, 1.0, P, V, O, Pg)
    swab.band_qk(d, 1.0, dO, V, dP, dPg)
    swab.band_softmax_bwd(d, P, dP, dS, Pg, dPg, dSg)
    swab.band_pv(d, 0.125, dS, K, dQ, dSg)
    swab.band_qk_bwd_t(d, 0.125, dS, Q, dK, dSg)
    swab.band_pv_bwd_t(d, 1.0, P, dO, dV, Pg)
    out.update({f"{tag}.S": S, f"{tag}.P": P, f"{tag}.lse": lse, f"{tag}.O": O, f"{tag}.dS": dS,
                f"{tag}.mdQ": dQ, f"{tag}.dK": dK, f"{tag}.dV": dV})
    if G:
        out.update({f"{tag}.Pc": Pg[0], f"{tag}.Pr": Pg[1], f"{tag}.dSc": dSg[0], f"{tag}.dSr": dSg[1]})


def battery():
    out = {}
    f16, b16, f32 = torch.float16, torch.bfloat16, torch.float32
    fused_pair(out, "f16", swab.Desc(1, 2, 1000, 64, 64, 64, 0, dtype=f16), 10, noalloc=True)
    fused_pair(out, "bf16.dil2", swab.Desc(1, 2, 777, 64, 100, 37, 2, dtype=b16), 20, noalloc=True)
    kb = torch.where(rnd((1, 1500), f32, 30) > 0.8, -10000.0, 0.0).contiguous()
    dp = swab.Desc(1, 2, 1500, 64, 256, 0, 0, dtype=f16, key_bias=kb, dropout_p=0.1, dropout_seed=7)
    mask = torch.zeros(swab.band_attention_dropout_mask_bytes(dp) // 4, dtype=torch.int32, device="cuda")
    dp = swab.Desc(1, 2, 1500, 64, 256, 0, 0, dtype=f16, key_bias=kb, dropout_p=0.1, dropout_seed=7,
                   dropout_mask=mask)
    fused_pair(out, "causal.bias.drop", dp, 40)
    out["causal.bias.drop.mask"] = mask
    fused_strided(out, "strided", 2, 2, 640, b16, 50)
    fused_pair(out, "f32", swab.Desc(1, 2, 300, 64, 20, 20, 1, dtype=f32), 60, noalloc=True)
    fused_pair(out, "glob", swab.Desc(1, 2, 1000, 64, 64, 64, 0, dtype=f16, global_idx=[0, 17, 500, 999]), 70)
    chain(out, "chain.f16.dil1.glob", swab.Desc(1, 2, 700, 64, 40, 40, 1, dtype=f16, global_idx=[3, 64, 650]), 80)
    chain(out, "chain.bf16", swab.Desc(2, 1, 513, 64, 33, 9, 0, dtype=b16), 90)
    chain(out, "chain.f32.glob", swab.Desc(1, 2, 300, 64, 12, 20, 0, dtype=f32, global_idx=[5, 299]), 100)
    # dropout softmax
    d = swab.Desc(1, 2, 600, 64, 64, 16, 0, dtype=f16, dropout_p=0.2, dropout_seed=3)
    S = rnd((d.BH, d.n, d.D), f16, 110)
    P, Pd = sentinel((d.BH, d.n, d.D), f16), sentinel((d.BH, d.n, d.D), f16)
    lse = torch.zeros(d.BH, d.n, dtype=f32, device="cuda")
    swab.band_softmax_dropout(d, S, Pd, P, lse)
    out.update({"sdrop.P": P, "sdrop.Pd": Pd, "sdrop.lse": lse})
    # global queries with their own projections
    for dt, tag in ((f16, "gproj.f16"), (f32, "gproj.f32")):
        d = swab.Desc(1, 2, 900, 64, 8, 8, 0, dtype=dt, global_idx=list(range(0, 900, 45)))
        gs, ns = (d.BH, d.G, 64), (d.BH, d.n, 64)
        Qg, Kg, Vg, dOg = rnd(gs, dt, 120), rnd(ns, dt, 121), rnd(ns, dt, 122), rnd(gs, dt, 123)
        Og, dQg = sentinel(gs, dt), sentinel(gs, dt)
        dKg, dVg = sentinel(ns, dt), sentinel(ns, dt)
        lseg = torch.zeros(d.BH, d.G, dtype=f32, device="cuda")
        ws = torch.empty(swab.global_attention_workspace(d) // 4 + 1, dtype=f32, device="cuda")
        swab.global_attention(d, 0.125, Qg, Kg, Vg, Og, lseg, ws)
        swab.global_attention_bwd(d, 0.125, Qg, Kg, Vg, Og, dOg, lseg, dQg, dKg, dVg, ws)
        out.update({f"{tag}.Og": Og, f"{tag}.lseg": lseg, f"{tag}.dQg": dQg, f"{tag}.dKg": dKg,
                    f"{tag}.dVg": dVg})
    # AddBiasTranspose
    d = swab.Desc(2, 3, 777, 64, 1, 1, dtype=b16)
    X, bias = rnd((2, 777, 3, 3, 64), b16, 130), rnd((3, 3, 64), b16, 131)
    Y = sentinel((3, 2, 3, 777, 64), b16)
    swab.add_bias_transpose(d, X, bias, Y)
    out["abt.Y"] = Y
    torch.cuda.synchronize()
    return {k: v.cpu() for k, v in out.items()}


def child(path):
    """Runs in a process that loads the checked build."""
    assert swab.bounds_checked(), "the checked build was not loaded"
    swab.device_status(reset=True)
    swab.bounds_report(reset=True)
    res = battery()
    status, report = swab.device_status(reset=True), swab.bounds_report(reset=True)
    swab.selftest_bounds()
    st_status, st_report = swab.device_status(reset=True), swab.bounds_report(reset=True)
    torch.save({"out": res, "status": status, "report": report, "selftest_status": st_status,
                "selftest_report": st_report}, path)


def test_bounds_checked_build_matches_regular_build_and_records_nothing(tmp_path):
    swab_build.build_all()
    swab.load()
    assert not swab.bounds_checked()
    path = str(tmp_path / "checked.pt")
    env = dict(os.environ, SWAB_BOUNDS_CHECK="1",
               PYTHONPATH=os.pathsep.join([ROOT, os.environ.get("PYTHONPATH", "")]).rstrip(os.pathsep))
    proc = subprocess.run([sys.executable, os.path.abspath(__file__), "--child", path], cwd=ROOT, env=env,
                          capture_output=True, text=True, timeout=900)
    assert proc.returncode == 0, proc.stdout[-3000:] + proc.stderr[-3000:]
    got = torch.load(path)
    assert got["report"] is None, f"out-of-bounds access recorded: {got['report']}"
    assert got["status"] == 0, f"status word {got['status']:#x}"
    # the self-test: refused stores recorded at the entry-point file's kernel
    assert got["selftest_status"] & BOUNDS_BIT
    site, _, nbytes = got["selftest_report"]
    assert (site - 1) >> 16 == API_FILE_ID and nbytes == 4
    ref = battery()
    assert swab.device_status(reset=True) == 0
    assert set(ref) == set(got["out"])
    for k, r in ref.items():
        g = got["out"][k]
        if k.split(".")[-1] in ATOMIC:
            assert torch.allclose(g.float(), r.float(), rtol=2e-2, atol=2e-3), k
        else:
            assert g.dtype == r.dtype and torch.equal(bits(g), bits(r)), k


def test_regular_build_has_no_bounds_selftest():
    swab_build.build()
    swab.load()
    with pytest.raises(swab.SwabError) as e:
        swab.selftest_bounds()
    assert e.value.status_name == "SWAB_ERR_UNSUPPORTED"
    assert swab.bounds_report(reset=True) is None


if __name__ == "__main__" and len(sys.argv) == 3 and sys.argv[1] == "--child":
    child(sys.argv[2])
