"""End-to-end parity of moe_layer_forward (the fused C-ABI call) against the
CPU oracle on the five workloads: small variants checked on every token,
and the full-size shapes checked with routing on every token and the expert
outputs on a seeded sample (plus every token of the least-loaded experts)."""
from fractions import Fraction

import numpy as np
import pytest
import torch

from mixture_experts_layer_99_b300 import moe, workloads as W
from oracle import moe_oracle as ORC
from parity_util import TOL_Y, check_layer, np_of, rel_err

pytestmark = pytest.mark.gpu
DEV = "cuda"
WL = W.WORKLOADS

SMALL = {
    "ref_fp32": WL["ref_fp32"],
    "switch_small": W.small(WL["switch_top1"], T=1500, d=256, H=512),
    "mixtral_small": W.small(WL["mixtral"], T=700, d=256, H=384),
    "longtail_small": W.small(WL["longtail"], T=2000, d=128, H=192),
    "decode_small": W.small(WL["decode"], T=64, d=512, H=256),
    "drops_heavy": W.small(WL["longtail"], T=999, d=64, H=64, c=Fraction(1, 3)),
    "single_expert": W.small(WL["switch_top1"], T=77, d=64, H=128, E=1, k=1),
    # >= 512 rows per expert on average: the grouped GEMM runs as CTA pairs
    "switch_pairs": W.small(WL["switch_top1"], T=4100, d=256, H=512, E=4),
    "mixtral_pairs": W.small(WL["mixtral"], T=2100, d=256, H=384, E=4),
    "longtail_pairs": W.small(WL["longtail"], T=6000, d=128, H=192, E=16),
    # 16 experts, top-4, Gaussian router noise
    "sweep_small": W.small(WL["sweep_e16_k4"], T=2048, d=256, H=512),
    "sweep_small_single_cta": W.small(WL["sweep_e16_k4"], T=1000, d=128, H=256),
    # std-scaled router noise (kwkr.cn MoE article, section 3.3)
    "std_noise_small": W.small(WL["sweep_std_noise"], T=2048, d=256, H=512),
    # 157 router tiles in two rounds over the 148 CTAs, with drops
    "tiles_two_rounds": W.small(WL["longtail"], T=20000, d=128, H=64),
    # fp32 beyond the reference layer: SwiGLU with router bias, Gumbel noise
    # and drops over 64 experts; 96 experts top-4 (the FMA router)
    "f32_swiglu_drops": W.small(WL["longtail"], T=700, d=64, H=96).with_(dtype="f32"),
    "f32_wide_e96_k4": W.small(WL["switch_top1"], T=500, d=64, H=64, E=96,
                               k=4).with_(dtype="f32"),
}


@pytest.mark.parametrize("name", sorted(SMALL))
def test_layer_small(name):
    res = check_layer(SMALL[name], DEV)
    assert res["tokens_checked"] == SMALL[name].T


@pytest.mark.parametrize("seed", [1, 2])
def test_layer_seeds(seed):
    check_layer(W.small(WL["longtail"], T=1024, d=128, H=128), DEV, seed=seed)


FULL = {"ref_fp32": None, "switch_top1": 2048, "decode": None, "longtail": 1024,
        "mixtral": 128, "sweep_e16_k4": 1024, "sweep_std_noise": 1024}


@pytest.mark.parametrize("name", list(FULL))
def test_layer_full_size(name):
    res = check_layer(WL[name], DEV, n_sample=FULL[name])
    print(name, {k: v for k, v in res.items() if k not in ("out", "r")})


@pytest.mark.parametrize("name,seed", [("switch_top1", 1), ("switch_top1", 2),
                                       ("longtail", 1), ("longtail", 2)])
def test_layer_full_size_other_seeds(name, seed):
    """The Switch and long-tail workloads at full size on two more seeds."""
    res = check_layer(WL[name].with_(seed=seed), DEV, n_sample=512)
    print(name, seed, {k: v for k, v in res.items() if k not in ("out", "r")})


@pytest.mark.parametrize("name", ["ref_fp32", "switch_small", "mixtral_small",
                                  "longtail_small", "drops_heavy", "sweep_small"])
def test_layer_reads_no_unwritten_workspace_bytes(name):
    """A workspace filled with NaN bytes (past its status header) gives the
    same outputs, bit for bit, as a zeroed one: the layer reads only what it
    wrote in the same call."""
    w = SMALL[name]
    cfg = moe.config_from_workload(w)
    dinp = W.to_device(W.make_inputs(w), DEV)
    outs = []
    for fill in (0, 255):
        ws = moe.workspace(cfg, DEV)
        ws[256:].fill_(fill)
        outs.append(moe.layer_forward(cfg, dinp, ws=ws))
        torch.cuda.synchronize()
        assert moe.device_status(ws)[0] == 0
    for key, t in outs[0].items():
        assert torch.equal(t, outs[1][key]), key


def test_layer_host_io_matches_device_call():
    w = W.small(WL["switch_top1"], T=512, d=128, H=256)
    cfg = moe.config_from_workload(w)
    inp = W.make_inputs(w)
    dinp = W.to_device(inp, DEV)
    out = moe.layer_forward(cfg, dinp)
    ws = moe.workspace(cfg, DEV, host_io=True)
    xh = inp["x"].pin_memory()
    yh = torch.empty_like(xh).pin_memory()
    Lh = torch.empty(1, dtype=torch.float32).pin_memory()
    moe.layer_forward_host(cfg, xh, dinp, yh, ws=ws, L_host=Lh)
    torch.cuda.synchronize()
    assert torch.equal(yh, out["y"].cpu())
    assert Lh.item() == out["L_balance"].item()


@pytest.mark.parametrize("name", ["switch_top1", "longtail"])
def test_pipelined_host_calls_match_device_calls(name):
    """moe_layer_forward_host_pipelined over six calls on two workspaces and
    three streams, with different inputs per call: each call's y and
    L_balance equal those of the device call on the same inputs, so the
    events keep every staging buffer from being reused too early."""
    w = W.small(WL[name], T=700, d=128, H=256)
    cfg = moe.config_from_workload(w)
    sets = [W.make_inputs(w, seed=s) for s in range(3)]
    dsets = [W.to_device(s, DEV) for s in sets]
    ref = [moe.layer_forward(cfg, d) for d in dsets]
    torch.cuda.synchronize()
    wss = [moe.workspace(cfg, DEV, host_io=True) for _ in range(2)]
    evs = [[torch.cuda.Event() for _ in range(3)] for _ in range(2)]
    s_in, s_c, s_out = (torch.cuda.Stream() for _ in range(3))
    xh = [s["x"].pin_memory() for s in sets]
    n = 6
    yh = [torch.empty_like(xh[0]).pin_memory() for _ in range(n)]
    Lh = [torch.empty(1, dtype=torch.float32).pin_memory() for _ in range(n)]
    for i in range(n):
        j = i % 3
        moe.layer_forward_host_pipelined(cfg, xh[j], dsets[j], yh[i], ws=wss[i % 2],
                                         events=evs[i % 2], copy_in=s_in, compute=s_c,
                                         copy_out=s_out, L_host=Lh[i])
    s_out.synchronize()
    torch.cuda.synchronize()
    for i in range(n):
        assert torch.equal(yh[i], ref[i % 3]["y"].cpu()), i
        assert Lh[i].item() == ref[i % 3]["L_balance"].item(), i
    for ws in wss:
        assert moe.device_status(ws) == (0, 0)


def test_layer_deterministic():
    w = W.small(WL["longtail"], T=3000, d=128, H=128)
    cfg = moe.config_from_workload(w)
    dinp = W.to_device(W.make_inputs(w), DEV)
    a = moe.layer_forward(cfg, dinp)
    b = moe.layer_forward(cfg, dinp)
    torch.cuda.synchronize()
    for k in a:
        assert torch.equal(a[k], b[k]), k


def test_layer_zero_router_closed_form():
    """W_g = 0: every token picks experts 0..k-1 with gates 1/k; tokens at or
    beyond C lose every slot and get y = 0; L_balance = 1."""
    w = W.small(WL["mixtral"], T=600, d=64, H=64, E=4, k=2, c=Fraction(1, 2))
    inp = W.make_inputs(w)
    inp["Wg"] = torch.zeros_like(inp["Wg"])
    cfg = moe.config_from_workload(w)
    C = cfg.capacity          # ceil(0.5 * 2 * 600 / 4) = 150
    assert C == 150
    out = moe.layer_forward(cfg, W.to_device(inp, DEV))
    torch.cuda.synchronize()
    assert (out["topk_idx"].cpu() == torch.tensor([0, 1], dtype=torch.int32)).all()
    assert (out["y"][C:] == 0).all()
    assert abs(out["L_balance"].item() - 1.0) < 1e-6
    assert out["dropped"].item() == 2 * (600 - C)
    r = ORC.moe_forward(inp, k=2, c=w.c, act=w.act, tokens=np.arange(C))
    assert rel_err(np_of(out["y"][:C]), r["y"]) <= TOL_Y["bf16"]


@pytest.mark.parametrize("name", ["switch_small", "longtail_small", "ref_fp32"])
def test_layer_profiled_matches_and_times(name):
    """moe_layer_forward_profiled gives the same results as moe_layer_forward
    and records six ordered stage events."""
    w = SMALL[name]
    cfg = moe.config_from_workload(w)
    dinp = W.to_device(W.make_inputs(w), DEV)
    a = moe.layer_forward(cfg, dinp)
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
    for e in evs:
        e.record()
    b = moe.layer_forward_profiled(cfg, dinp, evs, ws=moe.workspace(cfg, DEV),
                                   out=moe.alloc_outputs(cfg, DEV))
    torch.cuda.synchronize()
    for k in a:
        assert torch.equal(a[k], b[k]), k
    times = [evs[i].elapsed_time(evs[i + 1]) for i in range(5)]
    assert all(t >= 0 for t in times)
    assert evs[0].elapsed_time(evs[5]) > 0



SHARED = {
    "longtail_shared_small": W.small(WL["longtail_shared"], T=1500, d=128, H=192).with_(shared_H=256),
    "switch_shared_small": W.small(WL["switch_top1"], T=900, d=256, H=512).with_(shared_H=384),
    "ref_fp32_shared": WL["ref_fp32"].with_(shared_H=128),
    "heavy_drops_shared": W.small(WL["longtail"], T=777, d=64, H=64,
                                  c=Fraction(1, 4)).with_(shared_H=64),
}


@pytest.mark.parametrize("name", sorted(SHARED))
def test_layer_shared_expert_small(name):
    """moe_layer_forward_shared against the oracle with its shared expert:
    every token, dropped or not, gets the shared FFN with weight 1."""
    res = check_layer(SHARED[name], DEV)
    assert res["tokens_checked"] == SHARED[name].T


def test_layer_shared_expert_full_size():
    res = check_layer(WL["longtail_shared"], DEV, n_sample=512)
    print({k: v for k, v in res.items() if k not in ("out", "r")})
