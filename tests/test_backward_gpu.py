"""Parity of moe_layer_backward (the C-ABI backward call) with the fp64
backward oracle on the same seeded inputs, routing taken from the GPU's own
fp32 logits. Every gradient is compared on every element."""
from fractions import Fraction

import numpy as np
import pytest
import torch

from mixture_experts_layer_99_b300 import moe, workloads as W
from oracle import moe_backward as OB
from parity_util import np_of, rel_err

pytestmark = pytest.mark.gpu
DEV = "cuda"
WL = W.WORKLOADS

# max |err| / max |ref| per gradient. The GPU path rounds dY, the recomputed
# pre-activations, the activation gradients, dxd and the transposed operands
# to bf16 (relative spacing 2^-8) and accumulates in fp32; each gradient is a
# sum of such products, so a few bf16 ulps of the largest entry bound it.
TOL = dict(dx=2e-2, dWg=2e-2, dbias=2e-2, dW1=2e-2, dW3=2e-2, dW2=2e-2, db1=2e-2, db2=2e-2)
# fp32 layers run every step in fp32 (FMA) against the fp64 oracle: sums of at
# most a few thousand fp32 products, each rounded at 2^-24 relative
TOL_F32 = 1e-5

CASES = {
    "switch_small": (W.small(WL["switch_top1"], T=1500, d=256, H=512), 0.1, True),
    "switch_pairs": (W.small(WL["switch_top1"], T=4100, d=256, H=512, E=4), 0.1, False),
    "mixtral_small": (W.small(WL["mixtral"], T=700, d=256, H=384), 0.05, False),
    "mixtral_pairs": (W.small(WL["mixtral"], T=2100, d=256, H=384, E=4), 0.05, False),
    "longtail_small": (W.small(WL["longtail"], T=2000, d=128, H=192), 0.01, False),
    "sweep_small": (W.small(WL["sweep_e16_k4"], T=2048, d=256, H=512), 0.1, True),
    "drops_heavy": (W.small(WL["longtail"], T=999, d=64, H=64, c=Fraction(1, 3)), 0.2, False),
    "ragged_dims": (W.small(WL["switch_top1"], T=600, d=136, H=200, E=5, k=2), 0.3, True),
    # SwiGLU with H not a multiple of 64: dxd reads the transposed [W1^T | W3^T]
    "swiglu_ragged_h": (W.small(WL["mixtral"], T=640, d=136, H=200, E=5), 0.1, False),
    # std-scaled router noise: its strength carries no gradient
    "std_noise": (W.small(WL["sweep_std_noise"], T=1500, d=256, H=256), 0.1, False),
    # more than 64 experts: the FMA router forward, the warp-per-token router
    # backward (4 and 8 experts per lane), padded dz columns up to 128 and 256
    "wide_e96_k4": (W.small(WL["longtail"], T=1200, d=128, H=128, E=96, k=4), 0.05, False),
    "wide_e256_k8": (W.small(WL["sweep_e16_k4"], T=1024, d=64, H=128, E=256, k=8), 0.1, True),
    "wide_e65_k1": (W.small(WL["switch_top1"], T=700, d=64, H=64, E=65, k=1), 0.2, False),
    # fp32 (the fp32 FMA backward): the small reference layer itself (GELU, expert
    # biases, drops), SwiGLU, k = 1 with heavy drops, more than 64 experts, and
    # bias + Gumbel noise + temperature
    "f32_ref": (WL["ref_fp32"], 0.1, True),
    "f32_swiglu": (W.small(WL["mixtral"], T=300, d=64, H=96, E=4).with_(dtype="f32"), 0.05,
                   False),
    "f32_k1_drops": (W.small(WL["switch_top1"], T=400, d=64, H=128, E=4,
                             c=Fraction(1, 2)).with_(dtype="f32"), 0.1, True),
    "f32_wide_e96_k4": (W.small(WL["longtail"], T=300, d=32, H=64, E=96,
                                k=4).with_(dtype="f32"), 0.05, False),
    "f32_bias_noise_tau": (W.small(WL["longtail"], T=500, d=64, H=64).with_(dtype="f32",
                                                                           tau=0.7), 0.1, False),
    # fp32 dimensions that are not multiples of the 64-wide GEMM tiles
    "f32_ragged_dims": (W.small(WL["switch_top1"], T=333, d=36, H=52, E=5,
                                k=2).with_(dtype="f32"), 0.2, True),
    "f32_ragged_swiglu": (W.small(WL["mixtral"], T=211, d=44, H=28, E=3).with_(dtype="f32"),
                          0.2, False),
}


def _run(w, alpha, with_bias, seed=0, keep_preact=False):
    inp = W.make_inputs(w, seed)
    if with_bias:  # nonzero expert biases for the GELU bias gradients
        g = torch.Generator().manual_seed(seed + 99)
        inp["b1"] = (0.1 * torch.randn(w.E, w.H, generator=g)).to(w.torch_dtype)
        inp["b2"] = (0.1 * torch.randn(w.E, w.d, generator=g)).to(w.torch_dtype)
    gdy = torch.Generator().manual_seed(seed + 7)
    dy = torch.randn(w.T, w.d, generator=gdy).to(w.torch_dtype)
    cfg = moe.config_from_workload(w, keep_preact=keep_preact)
    dinp = W.to_device(inp, DEV)
    ws = moe.workspace(cfg, DEV)
    out = moe.layer_forward(cfg, dinp, ws=ws)
    grads = moe.layer_backward(cfg, dinp, out, dy.to(DEV), alpha, ws=ws)
    torch.cuda.synchronize()
    return inp, dy, cfg, out, grads


@pytest.mark.parametrize("name", ["switch_small", "switch_pairs", "mixtral_pairs",
                                  "longtail_small", "swiglu_ragged_h", "ragged_dims",
                                  "wide_e96_k4"])
def test_kept_preactivations_give_identical_results(name):
    """MOE_FLAG_KEEP_PREACT: GEMM1's epilogue stores the pre-activations it
    computes and the backward reads them instead of recomputing them with the
    same kernel, so the forward outputs and every gradient are bit-identical
    to the recomputing path."""
    w, alpha, with_bias = CASES[name]
    _, _, _, out0, g0 = _run(w, alpha, with_bias)
    _, _, cfg, out1, g1 = _run(w, alpha, with_bias, keep_preact=True)
    assert cfg.flags == moe.MOE_FLAG_KEEP_PREACT
    for key, v in out0.items():
        if isinstance(v, torch.Tensor):
            assert torch.equal(v, out1[key]), key
    for key, v in g0.items():
        if v is not None:
            assert torch.equal(v, g1[key]), key


@pytest.mark.parametrize("name", sorted(CASES))
def test_backward_matches_oracle(name):
    w, alpha, with_bias = CASES[name]
    inp, dy, cfg, out, grads = _run(w, alpha, with_bias)
    ref = OB.moe_backward(inp, w.k, w.c, w.act, dy, alpha, w.tau,
                          logits=out["logits"].cpu().numpy(), noise_scale=w.noise_scale)
    # the oracle followed the GPU's routing
    np.testing.assert_array_equal(ref["route"]["slot_of"], out["slot_of"].cpu().numpy())
    pairs = dict(dx=ref["dx"], dWg=ref["dWg"], dbias=ref["dbias"], dW1=ref["dW1"],
                 dW3=ref["dW3"], dW2=ref["dW2"], db1=ref["db1"], db2=ref["db2"])
    errs = {}
    for key, r in pairs.items():
        if r is None:
            assert grads.get(key) is None, key
            continue
        errs[key] = rel_err(np_of(grads[key]), r)
    print(name, {k: f"{v:.2e}" for k, v in errs.items()})
    for key, e in errs.items():
        assert e <= (TOL_F32 if w.dtype == "f32" else TOL[key]), (key, e)


SHARED_CASES = {
    # SwiGLU long tail plus a shared expert (drops, bias, Gumbel noise)
    "longtail_shared_small": W.small(WL["longtail_shared"], T=2000, d=128, H=192).with_(
        shared_H=256),
    # GELU, k = 2, with nonzero biases on the routed and the shared experts
    "gelu_shared_bias": W.small(WL["sweep_e16_k4"], T=1500, d=256, H=256, k=2).with_(
        shared_H=320, expert_bias=True),
    # SwiGLU shared expert whose H is not a multiple of 64 (transposed [W1; W3])
    "swiglu_shared_ragged_h": W.small(WL["mixtral"], T=700, d=136, H=128, E=4).with_(
        shared_H=200),
    # fp32: GELU with biases on the routed and the shared experts; SwiGLU
    "f32_gelu_shared_bias": W.small(WL["sweep_e16_k4"], T=500, d=64, H=96, k=2).with_(
        shared_H=100, expert_bias=True, dtype="f32"),
    "f32_swiglu_shared": W.small(WL["mixtral"], T=300, d=64, H=64, E=4).with_(
        shared_H=76, dtype="f32"),
}


@pytest.mark.parametrize("name", sorted(SHARED_CASES))
def test_backward_shared_expert_matches_oracle(name):
    """moe_layer_backward_shared: the routed gradients as without the shared
    expert, plus the shared expert's weight gradients and its term of dx
    (the shared expert of the lpnh.cn MoE guide, section 4.10)."""
    w = SHARED_CASES[name]
    inp = W.make_inputs(w)
    sh = inp["shared"]
    if w.expert_bias:  # nonzero biases everywhere
        g = torch.Generator().manual_seed(42)
        for key, shape in (("b1", (w.E, w.H)), ("b2", (w.E, w.d))):
            inp[key] = (0.1 * torch.randn(*shape, generator=g)).to(w.torch_dtype)
        sh["b1"] = (0.1 * torch.randn(w.shared_H, generator=g)).to(w.torch_dtype)
        sh["b2"] = (0.1 * torch.randn(w.d, generator=g)).to(w.torch_dtype)
    dy = torch.randn(w.T, w.d, generator=torch.Generator().manual_seed(8)).to(w.torch_dtype)
    cfg = moe.config_from_workload(w)
    dinp = W.to_device(inp, DEV)
    ws = moe.workspace_shared(cfg, w.shared_H, DEV)
    bws = moe.workspace_backward_shared(cfg, w.shared_H, DEV)
    ws[256:].fill_(255)    # NaN bytes: nothing may read what no kernel wrote
    bws[256:].fill_(255)
    out = moe.layer_forward_shared(cfg, dinp, dinp["shared"], ws=ws)
    grads, sgrads = moe.layer_backward_shared(cfg, dinp, dinp["shared"], out, dy.to(DEV), 0.05,
                                              ws=ws, bws=bws)
    torch.cuda.synchronize()
    assert moe.device_status(bws)[0] == 0
    for key, t in grads.items():
        bad = torch.isnan(t)
        if bad.any():
            idx = torch.nonzero(bad)[:8].tolist()
            raise AssertionError(f"{key}: {int(bad.sum())} NaN, first at {idx}; "
                                 f"offsets {out['expert_offset'].tolist()}")
    ref = OB.moe_backward(inp, w.k, w.c, w.act, dy, 0.05, w.tau,
                          logits=out["logits"].cpu().numpy(), shared=sh,
                          noise_scale=w.noise_scale)
    np.testing.assert_array_equal(ref["route"]["slot_of"], out["slot_of"].cpu().numpy())
    errs = {}
    for key in ("dx", "dWg", "dbias", "dW1", "dW3", "dW2", "db1", "db2"):
        if ref[key] is not None:
            errs[key] = rel_err(np_of(grads[key]), ref[key])
    for key in ("dW1", "dW3", "dW2", "db1", "db2"):
        if ref["shared"][key] is not None:
            errs["shared_" + key] = rel_err(np_of(sgrads[key]), ref["shared"][key])
        else:
            assert key not in sgrads, key
    print(name, {k: f"{v:.2e}" for k, v in errs.items()})
    for key, e in errs.items():
        assert e <= (TOL_F32 if w.dtype == "f32" else 2e-2), (key, e)
    assert moe.device_status(ws)[0] == 0


@pytest.mark.parametrize("name", ["longtail_small", "drops_heavy", "switch_small", "f32_ref",
                                  "f32_k1_drops", "f32_wide_e96_k4"])
def test_backward_reads_no_unwritten_workspace_bytes(name):
    """Both workspaces start filled with NaN bytes (past their status
    headers): the forward and the backward must read only what they wrote, so
    the gradients still match the oracle. (The last 64-row block of an expert
    that is not the last one can reach past the final kept row; its unwritten
    rows must be zeroed before the weight-gradient product reads them.)"""
    w, alpha, with_bias = CASES[name]
    inp = W.make_inputs(w)
    dy = torch.randn(w.T, w.d, generator=torch.Generator().manual_seed(11)).to(w.torch_dtype)
    cfg = moe.config_from_workload(w)
    dinp = W.to_device(inp, DEV)
    ws = moe.workspace(cfg, DEV)
    bws = moe.workspace_backward(cfg, DEV)
    ws[256:].fill_(255)
    bws[256:].fill_(255)
    out = moe.layer_forward(cfg, dinp, ws=ws)
    grads = moe.layer_backward(cfg, dinp, out, dy.to(DEV), alpha, ws=ws, bws=bws)
    torch.cuda.synchronize()
    assert moe.device_status(bws)[0] == 0
    ref = OB.moe_backward(inp, w.k, w.c, w.act, dy, alpha, w.tau,
                          logits=out["logits"].cpu().numpy())
    for key in ("dx", "dWg", "dbias", "dW1", "dW3", "dW2"):
        if ref[key] is None:
            continue
        assert not torch.isnan(grads[key]).any(), key
        tol = TOL_F32 if w.dtype == "f32" else TOL[key]
        assert rel_err(np_of(grads[key]), ref[key]) <= tol, key


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_backward_is_deterministic(dtype):
    w = W.small(WL["mixtral"], T=900, d=128, H=192).with_(dtype=dtype)
    cfg = moe.config_from_workload(w)
    dinp = W.to_device(W.make_inputs(w), DEV)
    dy = torch.randn(w.T, w.d, generator=torch.Generator().manual_seed(3)).to(w.torch_dtype).to(DEV)
    ws = moe.workspace(cfg, DEV)
    out = moe.layer_forward(cfg, dinp, ws=ws)
    a = moe.layer_backward(cfg, dinp, out, dy, 0.1, ws=ws)
    b = moe.layer_backward(cfg, dinp, out, dy, 0.1, ws=ws)
    torch.cuda.synchronize()
    for k in a:
        assert torch.equal(a[k], b[k]), k


def test_backward_status_is_clean():
    w = W.small(WL["switch_top1"], T=512, d=128, H=256)
    cfg = moe.config_from_workload(w)
    dinp = W.to_device(W.make_inputs(w), DEV)
    ws = moe.workspace(cfg, DEV)
    out = moe.layer_forward(cfg, dinp, ws=ws)
    bws = moe.workspace_backward(cfg, DEV)
    dy = torch.ones(w.T, w.d, dtype=torch.bfloat16, device=DEV)
    moe.layer_backward(cfg, dinp, out, dy, 0.0, ws=ws, bws=bws)
    assert moe.device_status(bws) == (0, 0)


@pytest.mark.slow
def test_backward_full_size_switch():
    """switch_top1 at full size: dWg, dx and the expert gradients on every
    element (the oracle's fp64 run takes tens of seconds)."""
    w = WL["switch_top1"]
    inp, dy, cfg, out, grads = _run(w, 0.01, False)
    ref = OB.moe_backward(inp, w.k, w.c, w.act, dy, 0.01, w.tau,
                          logits=out["logits"].cpu().numpy())
    for key in ("dx", "dWg", "dW1", "dW2"):
        assert rel_err(np_of(grads[key]), ref[key]) <= TOL[key], key
