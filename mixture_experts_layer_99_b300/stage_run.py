"""Run the layer, or one of its entry points, on a workload's seeded inputs a
given number of times: a bounded program for a profiler to capture one kernel
of (``ncu -k regex:<kernel> ...``). It times nothing and checks nothing.

    python -m mixture_experts_layer_99_b300.stage_run --workload mixtral \
        [--E 2] [--T 4096] [--stage layer|router|dispatch|ffn|combine|backward] [--calls 4]

``backward`` runs moe_layer_backward (loss sum <dy, y> + 0.01 L_balance, dy
seeded) after the layer call it differentiates.

``--E`` / ``--T`` shrink the workload (a workload without drops, c = E/k,
keeps c = E'/k so that it still drops nothing); with the same T, d and k the
router, dispatch and combine move the same bytes as the full workload while
the expert weights on the device shrink by E/E'.
"""
from __future__ import annotations

import argparse
from fractions import Fraction

import torch

from mixture_experts_layer_99_b300 import moe, workloads as W


def reduced(w: W.Workload, E: int | None, T: int | None) -> W.Workload:
    kw = {}
    if E is not None and E != w.E:
        kw["E"] = E
        if w.c == Fraction(w.E, w.k):   # "no drops" workloads stay without drops
            kw["c"] = Fraction(E, w.k)
    if T is not None:
        kw["T"] = T
    if not kw:
        return w
    return w.with_(name=f"{w.name}[{','.join(f'{k}={v}' for k, v in kw.items())}]", **kw)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="mixtral", choices=sorted(W.WORKLOADS))
    ap.add_argument("--E", type=int, default=None)
    ap.add_argument("--T", type=int, default=None)
    ap.add_argument("--stage", default="layer",
                    choices=["layer", "router", "dispatch", "ffn", "combine", "backward"])
    ap.add_argument("--calls", type=int, default=4)
    args = ap.parse_args()
    w = reduced(W.WORKLOADS[args.workload], args.E, args.T)
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    inp = W.to_device(W.make_inputs(w), dev)
    cfg = moe.config_from_workload(w)
    ws = moe.workspace(cfg, dev)
    out = moe.alloc_outputs(cfg, dev, full=True)
    moe.layer_forward(cfg, inp, ws=ws, out=out)   # routing and packed rows for the stages
    torch.cuda.synchronize(dev)
    if args.stage in ("dispatch", "ffn", "combine"):
        d = moe.dispatch(cfg, out["topk_idx"], inp["x"], ws=ws)
        Y = moe.expert_ffn(cfg, d["xd"], d["offset"], inp["W1"], inp["W2"], inp.get("W3"),
                           inp.get("b1"), inp.get("b2"), ws=ws)
        torch.cuda.synchronize(dev)
    if args.stage == "backward":
        dy = torch.randn(w.T, w.d, generator=torch.Generator().manual_seed(5)).to(
            w.torch_dtype).to(dev)
        bws = moe.workspace_backward(cfg, dev)
        grads = moe.alloc_grads(cfg, inp, dev)
    for _ in range(args.calls):
        if args.stage == "layer":
            moe.layer_forward(cfg, inp, ws=ws, out=out)
        elif args.stage == "router":
            moe.router_topk(cfg, inp["x"], inp["Wg"], inp.get("bias"), inp.get("noise"), ws=ws)
        elif args.stage == "dispatch":
            moe.dispatch(cfg, out["topk_idx"], inp["x"], ws=ws)
        elif args.stage == "ffn":
            moe.expert_ffn(cfg, d["xd"], d["offset"], inp["W1"], inp["W2"], inp.get("W3"),
                           inp.get("b1"), inp.get("b2"), ws=ws, Y=Y)
        elif args.stage == "combine":
            moe.combine(cfg, Y, d["slot_of"], out["topk_gate"])
        else:
            moe.layer_backward(cfg, inp, out, dy, 0.01, ws=ws, bws=bws, grads=grads)
    torch.cuda.synchronize(dev)
    print(f"stage_run: {w.name} {args.stage} x{args.calls}, status {moe.device_status(ws)}")


if __name__ == "__main__":
    main()
