"""Small forward, backward and stage calls whose outputs are hashed, for the
comparison of the checked library (index checks in the kernels) with the
normal one. Run as a script (``python tests/checked_cases.py [corrupt]``) it
prints the digests and device statuses as one JSON line; the library it uses
is the one ``MOE_B300_CHECKED`` selects. With ``corrupt`` it instead runs one
backward whose forward outputs hold a slot past the packed rows."""
import hashlib
import json
import os
import sys
from fractions import Fraction

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from mixture_experts_layer_99_b300 import moe, workloads as W  # noqa: E402

DEV = "cuda"
WL = W.WORKLOADS
CASES = {
    "switch_k1": W.small(WL["switch_top1"], T=600, d=128, H=256),
    "longtail_drops": W.small(WL["longtail"], T=999, d=64, H=64, c=Fraction(1, 2)),
    "sweep_k4": W.small(WL["sweep_e16_k4"], T=512, d=128, H=128),
    "wide_e96": W.small(WL["longtail"], T=700, d=64, H=64, E=96, k=4),
}


def _h(t):
    return hashlib.sha256(t.detach().contiguous().cpu().view(torch.uint8).numpy()
                          .tobytes()).hexdigest()[:16]


def run_cases():
    res = {}
    for name, w in CASES.items():
        inp = W.to_device(W.make_inputs(w), DEV)
        cfg = moe.config_from_workload(w)
        ws = moe.workspace(cfg, DEV)
        out = moe.layer_forward(cfg, inp, ws=ws)
        dy = torch.randn(w.T, w.d, generator=torch.Generator().manual_seed(3)).to(
            w.torch_dtype).to(DEV)
        g = moe.layer_backward(cfg, inp, out, dy, 0.05, ws=ws)
        torch.cuda.synchronize()
        d = {k: _h(v) for k, v in out.items() if isinstance(v, torch.Tensor)}
        d.update({"d_" + k: _h(v) for k, v in g.items() if v is not None})
        d["status"] = list(moe.device_status(ws))
        # the stage calls on the same routing
        sd = moe.dispatch(cfg, out["topk_idx"], inp["x"], ws=ws)
        Y = moe.expert_ffn(cfg, sd["xd"], sd["offset"], inp["W1"], inp["W2"], inp.get("W3"),
                           inp.get("b1"), inp.get("b2"), ws=ws)
        y = moe.combine(cfg, Y, sd["slot_of"], out["topk_gate"])
        torch.cuda.synchronize()
        R = int(sd["offset"][-1].item())
        d.update(stage_xd=_h(sd["xd"][:R]), stage_slot_of=_h(sd["slot_of"]), stage_y=_h(y))
        d["stage_status"] = list(moe.device_status(ws))
        res[name] = d
    return res


def run_corrupt():
    """A backward whose forward slot_of holds one slot past the packed rows:
    the checked build skips that slot and reports it (the normal build must
    not be given this)."""
    w = CASES["longtail_drops"]
    inp = W.to_device(W.make_inputs(w), DEV)
    cfg = moe.config_from_workload(w)
    ws = moe.workspace(cfg, DEV)
    out = moe.layer_forward(cfg, inp, ws=ws)
    torch.cuda.synchronize()
    R = min(cfg.T * cfg.k, cfg.E * cfg.capacity)
    out["slot_of"].view(-1)[5] = R + 3
    dy = torch.randn(w.T, w.d, generator=torch.Generator().manual_seed(3)).to(
        w.torch_dtype).to(DEV)
    bws = moe.workspace_backward(cfg, DEV)
    moe.layer_backward(cfg, inp, out, dy, 0.05, ws=ws, bws=bws)
    torch.cuda.synchronize()
    return dict(backward_status=list(moe.device_status(bws)))


if __name__ == "__main__":
    if os.environ.get("MOE_B300_CHECKED") != "1" and "corrupt" in sys.argv:
        raise SystemExit("the corrupted case runs on the checked library only")
    print(json.dumps(run_corrupt() if "corrupt" in sys.argv else run_cases()))
