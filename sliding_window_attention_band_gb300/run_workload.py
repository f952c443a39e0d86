"""Run one API call on a named workload, a few times, for a profiler.

    python -m sliding_window_attention_band_gb300.run_workload \\
        --workload causal_fp16_n32768_w4096 --call band_attention --repeat 3

Builds the workload's seeded inputs on the current CUDA device, calls the
fused forward (``band_attention``) or the fused forward then its backward
(``band_attention_bwd``, only the backward repeated) ``--repeat`` times,
synchronises, checks the device status word and exits 0.  It prints nothing
but one line with the call and the status, so a profiler's launch list holds
only the library's kernels and torch's input copies.
"""
from __future__ import annotations

import argparse

import torch

import sliding_window_attention_band_gb300 as swab
from sliding_window_attention_band_gb300.inputs import WORKLOADS, workload_inputs


def main() -> int:
    names = {wl.name: wl for wl in WORKLOADS.values()}
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", required=True, choices=sorted(names))
    ap.add_argument("--call", default="band_attention", choices=["band_attention", "band_attention_bwd"])
    ap.add_argument("--repeat", type=int, default=3)
    args = ap.parse_args()
    wl = names[args.workload]
    swab.load()
    d = swab.Desc.from_workload(wl)
    Q, K, V, dO = (x.cuda() for x in workload_inputs(wl))
    O = torch.empty_like(Q)
    lse = torch.empty(wl.BH, wl.n, dtype=torch.float32, device="cuda")
    fwd = lambda: swab.band_attention(d, wl.scale, Q, K, V, O, lse)
    if args.call == "band_attention":
        for _ in range(args.repeat):
            fwd()
    else:
        fwd()
        dQ, dK, dV = (torch.empty_like(Q) for _ in range(3))
        ws = torch.empty(swab.band_attention_bwd_workspace(d) // 4, dtype=torch.float32, device="cuda")
        for _ in range(args.repeat):
            swab.band_attention_bwd(d, wl.scale, Q, K, V, O, dO, lse, dQ, dK, dV, ws)
    torch.cuda.synchronize()
    status = swab.device_status(reset=True)
    print(f"{args.call} {wl.name} x{args.repeat}: status {status}")
    return 0 if status == 0 else 1


if __name__ == "__main__":
    raise SystemExit(main())
