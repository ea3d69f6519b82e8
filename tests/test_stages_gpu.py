"""Stage-by-stage parity of the CUDA path (through the C ABI) against the
CPU oracle on seeded inputs: router, dispatch, expert FFN, combine and the
load-balance statistics, at small and ragged sizes and their edge cases."""
from fractions import Fraction

import numpy as np
import pytest
import torch

from mixture_experts_layer_99_b300 import moe, workloads as W
from oracle import moe_oracle as ORC
from parity_util import TOL_GATE, TOL_LOGITS, TOL_STATS, TOL_Y, np_of, rel_err

pytestmark = pytest.mark.gpu
DEV = "cuda"

WL = W.WORKLOADS
ROUTER_CASES = {
    "ref_fp32": WL["ref_fp32"],
    "switch_ragged": W.small(WL["switch_top1"], T=1000, d=256, H=512),
    "mixtral_small": W.small(WL["mixtral"], T=300, d=512, H=256),
    "longtail_small": W.small(WL["longtail"], T=777, d=128, H=64),
    "decode_full_router": WL["decode"].with_(H=64),
    "one_token": W.small(WL["switch_top1"], T=1, d=64, H=64),
    "one_expert": W.small(WL["switch_top1"], T=100, d=64, H=64, E=1, k=1),
    "k_equals_E": W.small(WL["mixtral"], T=65, d=64, H=64, E=4, k=4, c=Fraction(1)),
    "E256_k8": W.small(WL["switch_top1"], T=200, d=64, H=64, E=256, k=8, c=Fraction(1)),
    "tau_half": W.small(WL["longtail"], T=90, d=64, H=64).with_(tau=0.5),
    "fp32_E64": W.small(WL["ref_fp32"], T=333, d=96, H=64, E=64, k=3),
    # 40 tiles on 40 CTAs; 157 tiles on the 148 CTAs (a second round)
    "tiles_one_round": W.small(WL["longtail"], T=5000, d=128, H=64),
    "tiles_two_rounds": W.small(WL["sweep_e16_k4"], T=20000, d=64, H=64),
    # std-scaled router noise (kwkr.cn MoE article, section 3.3) on every
    # router path: tensor cores (E = 16; E = 64 with a bias), the K-split
    # decode router, the FMA router (fp32; bf16 with E > 64)
    "std_noise_E16": W.small(WL["sweep_std_noise"], T=3000, d=256, H=64),
    "std_noise_E64_bias": W.small(WL["longtail"], T=600, d=128, H=64).with_(
        noise="gaussian_std", noise_std=0.3),
    "std_noise_split": WL["decode"].with_(H=64, noise="gaussian_std", noise_std=0.2),
    "std_noise_fp32": W.small(WL["ref_fp32"], T=300, d=64, H=64, E=12, k=3).with_(
        noise="gaussian_std", noise_std=0.2),
    "std_noise_E100": W.small(WL["switch_top1"], T=200, d=64, H=64, E=100, k=2).with_(
        noise="gaussian_std", noise_std=0.5),
    # keys formed while the accumulator leaves TMEM: bias only, noise only,
    # and an E that is not a multiple of 4 (scalar noise loads), over tiles
    # of one and of several column groups
    "bias_only_E64": W.small(WL["longtail"], T=700, d=128, H=64).with_(noise=None),
    "noise_only_E8": W.small(WL["mixtral"], T=500, d=256, H=64).with_(noise="gumbel"),
    "bias_noise_E6": W.small(WL["longtail"], T=400, d=64, H=64, E=6, k=2),
    "bias_noise_E50_k3": W.small(WL["longtail"], T=1300, d=128, H=64, E=50, k=3),
}


def test_router_noise_base_not_16_byte_aligned():
    # a [T, E] noise tensor that starts 4 bytes past a 16-byte boundary (E a
    # multiple of 4): the router must read it element by element
    w = W.small(WL["longtail"], T=300, d=128, H=64)
    inp = W.make_inputs(w)
    cfg = moe.config_from_workload(w)
    d = W.to_device(inp, DEV)
    buf = torch.zeros(w.T * w.E + 4, dtype=torch.float32, device=DEV)
    noise = buf[1:1 + w.T * w.E].view(w.T, w.E)
    noise.copy_(d["noise"])
    assert noise.data_ptr() % 16 == 4
    lg, idx, gate, psum = moe.router_topk(cfg, d["x"], d["Wg"], d["bias"], noise)
    lg0, idx0, gate0, psum0 = moe.router_topk(cfg, d["x"], d["Wg"], d["bias"], d["noise"])
    torch.cuda.synchronize()
    assert torch.equal(lg, lg0) and torch.equal(idx, idx0)
    assert torch.equal(gate, gate0) and torch.equal(psum, psum0)


@pytest.mark.parametrize("name", sorted(ROUTER_CASES))
def test_router_topk(name):
    w = ROUTER_CASES[name]
    inp = W.make_inputs(w)
    cfg = moe.config_from_workload(w)
    d = W.to_device(inp, DEV)
    lg, idx, gate, psum = moe.router_topk(cfg, d["x"], d["Wg"], d["bias"], d["noise"])
    torch.cuda.synchronize()
    lg = lg.cpu().numpy()
    ref_l = ORC.router_logits(inp["x"], inp["Wg"], inp["bias"], inp["noise"], w.tau,
                              w.noise_scale)
    assert rel_err(lg, ref_l) <= TOL_LOGITS[w.dtype]
    r = ORC.route_from_logits(lg, w.k, cfg.capacity)
    np.testing.assert_array_equal(idx.cpu().numpy(), r["ids"])
    assert np.abs(gate.cpu().numpy() - r["gates"]).max() <= TOL_GATE
    np.testing.assert_allclose(np_of(psum) / w.T, r["P"], rtol=TOL_STATS, atol=1e-9)


def test_router_zero_weights_ties_to_lowest_ids():
    w = W.small(WL["mixtral"], T=130, d=64, H=64, E=6, k=3)
    inp = W.make_inputs(w)
    inp["Wg"] = torch.zeros_like(inp["Wg"])
    cfg = moe.config_from_workload(w)
    d = W.to_device(inp, DEV)
    lg, idx, gate, psum = moe.router_topk(cfg, d["x"], d["Wg"])
    assert (idx.cpu() == torch.arange(3, dtype=torch.int32)).all()
    assert torch.allclose(gate.cpu(), torch.full((130, 3), 1 / 3), rtol=0, atol=1e-7)
    np.testing.assert_allclose(np_of(psum), np.full(6, 130 / 6), rtol=1e-6)


DISPATCH_CASES = [
    # (T, E, k, c, skew, d, dtype)
    (256, 4, 2, Fraction(5, 4), 0.0, 64, "f32"),
    (8192, 8, 1, Fraction(1), 0.3, 128, "bf16"),
    (1000, 16, 2, Fraction(1, 2), 2.0, 40, "bf16"),      # heavy drops, ragged T*k
    (32768, 64, 2, Fraction(2), 3.0, 64, "bf16"),         # long tail
    (1, 3, 2, Fraction(1), 0.0, 16, "bf16"),
    (3000, 5, 5, Fraction(1), 0.0, 8, "bf16"),             # k = E, every expert full
    (777, 7, 3, Fraction(1, 100), 0.0, 24, "bf16"),        # C = 1
    (513, 256, 8, Fraction(1), 1.0, 32, "f32"),
]


@pytest.mark.parametrize("T,E,k,c,skew,d,dt", DISPATCH_CASES)
def test_dispatch(T, E, k, c, skew, d, dt):
    ids = W.make_routing(T, E, k, seed=T + E, skew=skew)
    x = W.make_rows(T, d, torch.float32 if dt == "f32" else torch.bfloat16, seed=1)
    C = ORC.capacity(c, k, T, E)
    cfg = moe.make_config(T, d, E, k, 8, C, dt, "gelu")
    out = moe.dispatch(cfg, ids.to(DEV), x.to(DEV))
    torch.cuda.synchronize()
    r = ORC.dispatch(ids.numpy(), E, C)
    np.testing.assert_array_equal(out["count"].cpu().numpy(), r["count"])
    np.testing.assert_array_equal(out["offset"].cpu().numpy(), r["offset"])
    np.testing.assert_array_equal(out["slot_of"].cpu().numpy(), r["slot_of"])
    R = int(r["offset"][-1])
    np.testing.assert_array_equal(out["token_of_row"][:R].cpu().numpy(), r["token_of_row"])
    tor = torch.from_numpy(r["token_of_row"].astype(np.int64))
    assert torch.equal(out["xd"][:R].cpu(), x[tor])


def test_dispatch_all_tokens_one_expert():
    T, E, k, d = 5000, 8, 1, 64
    ids = torch.zeros(T, k, dtype=torch.int32)
    x = W.make_rows(T, d, torch.bfloat16, seed=3)
    C = 1234
    cfg = moe.make_config(T, d, E, k, 8, C, "bf16", "gelu")
    out = moe.dispatch(cfg, ids.to(DEV), x.to(DEV))
    torch.cuda.synchronize()
    cnt = out["count"].cpu()
    assert cnt[0] == T and (cnt[1:] == 0).all()
    off = out["offset"].cpu()
    assert (off[1:] == C).all() and off[0] == 0
    so = out["slot_of"].cpu()[:, 0]
    assert torch.equal(so[:C], torch.arange(C, dtype=torch.int32))
    assert (so[C:] == -1).all()
    assert torch.equal(out["xd"][:C].cpu(), x[:C])


def _ffn_case(E, d, H, act, dt, kept, seed):
    w = W.Workload("ffn", T=int(sum(kept)), d=d, E=E, k=1, H=H, act=act, dtype=dt,
                   c=Fraction(E), expert_bias=(act == "gelu"), seed=seed)
    inp = W.make_inputs(w)
    if w.expert_bias:   # nonzero biases so that the bias path is exercised
        g = torch.Generator().manual_seed(seed + 7)
        inp["b1"] = (0.1 * torch.randn(E, H, generator=g)).to(w.torch_dtype)
        inp["b2"] = (0.1 * torch.randn(E, d, generator=g)).to(w.torch_dtype)
    off = np.zeros(E + 1, dtype=np.int32)
    off[1:] = np.cumsum(kept)
    return w, inp, off


FFN_CASES = [
    # E, d, H, act, dtype, kept per expert
    (4, 64, 256, "gelu", "f32", [70, 0, 129, 1]),
    (8, 256, 512, "gelu", "bf16", [300, 129, 0, 64, 1, 250, 77, 128]),
    (3, 512, 384, "swiglu", "bf16", [257, 1, 190]),
    (5, 136, 200, "swiglu", "bf16", [33, 0, 0, 140, 9]),    # ragged d, H
    (2, 2048, 1408, "swiglu", "bf16", [300, 45]),
    (1, 64, 64, "gelu", "bf16", [1]),
    # 148 to 266 output tiles: a second wave under 90 % full
    (2, 2048, 1024, "gelu", "bf16", [2400, 2300]),
    (2, 512, 1024, "swiglu", "bf16", [1300, 1290]),
    # at least 512 rows per expert on average: CTA pairs with 256-row tiles;
    # experts ending inside the first or the second CTA's half, a one-row
    # expert (the second CTA has no valid row), an empty expert, ragged d, H
    (2, 256, 512, "gelu", "bf16", [700, 333]),
    (4, 512, 768, "swiglu", "bf16", [1, 1500, 0, 600]),
    (3, 136, 200, "gelu", "bf16", [900, 700, 2]),
    (3, 136, 200, "swiglu", "bf16", [900, 700, 2]),
    (1, 1024, 1024, "gelu", "bf16", [3000]),
]


@pytest.mark.parametrize("E,d,H,act,dt,kept", FFN_CASES)
def test_expert_ffn(E, d, H, act, dt, kept):
    w, inp, off = _ffn_case(E, d, H, act, dt, kept, seed=E * 100 + d)
    R = int(off[-1])
    cfg = moe.make_config(R, d, E, 1, H, R, dt, act)     # T = R rows, C = R
    dv = W.to_device(inp, DEV)
    Y = moe.expert_ffn(cfg, dv["x"], torch.from_numpy(off).to(DEV), dv["W1"], dv["W2"],
                       dv["W3"], dv["b1"], dv["b2"])
    torch.cuda.synchronize()
    ref = np.zeros((R, d))
    for e in range(E):
        if off[e + 1] > off[e]:
            ref[off[e]:off[e + 1]] = ORC.expert_ffn_rows(
                inp["x"][off[e]:off[e + 1]], inp["W1"][e], inp["W2"][e],
                None if inp["W3"] is None else inp["W3"][e],
                None if inp["b1"] is None else inp["b1"][e],
                None if inp["b2"] is None else inp["b2"][e], act)
    err = rel_err(np_of(Y), ref)
    assert err <= TOL_Y[dt], err
    # per-expert check too: a wrong expert's weights cannot hide behind a big one
    for e in range(E):
        if off[e + 1] > off[e]:
            assert rel_err(np_of(Y[off[e]:off[e + 1]]), ref[off[e]:off[e + 1]]) <= TOL_Y[dt]


@pytest.mark.parametrize("T,E,k,c,d,dt", [(300, 6, 2, Fraction(1, 2), 64, "bf16"),
                                         (256, 4, 2, Fraction(5, 4), 64, "f32"),
                                         (1000, 8, 1, Fraction(1), 1024, "bf16"),
                                         (70, 64, 8, Fraction(1, 4), 48, "bf16")])
def test_combine(T, E, k, c, d, dt):
    ids = W.make_routing(T, E, k, seed=5, skew=1.0)
    C = ORC.capacity(c, k, T, E)
    r = ORC.dispatch(ids.numpy(), E, C)
    R = max(int(r["offset"][-1]), 1)
    tdt = torch.float32 if dt == "f32" else torch.bfloat16
    Yrows = W.make_rows(R, d, tdt, seed=9)
    gates = W.make_gates(T, k, seed=4)
    cfg = moe.make_config(T, d, E, k, 8, C, dt, "gelu")
    y = moe.combine(cfg, Yrows.to(DEV), torch.from_numpy(r["slot_of"]).to(DEV),
                    gates.to(DEV))
    torch.cuda.synchronize()
    ref = ORC.combine_rows(Yrows, r["slot_of"], gates.numpy())
    # fp32 accumulate of exact inputs; only the final rounding to the output dtype
    tol = 1e-6 if dt == "f32" else 8e-3
    assert rel_err(np_of(y), ref) <= tol
    dropped = (r["slot_of"] < 0).all(axis=1)
    assert (y.cpu()[torch.from_numpy(dropped)] == 0).all()


@pytest.mark.parametrize("T,E,k,C", [(256, 4, 2, 160), (32768, 64, 2, 2048), (7, 3, 1, 1)])
def test_aux_stats(T, E, k, C):
    ids = W.make_routing(T, E, k, seed=2, skew=2.0)
    r = ORC.dispatch(ids.numpy(), E, C)
    g = torch.Generator().manual_seed(3)
    psum = (torch.rand(E, generator=g) * T / E).to(torch.float32)
    cfg = moe.make_config(T, 8, E, k, 8, C, "bf16", "gelu")
    f, P, L, dropped = moe.aux_stats(cfg, torch.from_numpy(r["count"]).to(DEV), psum.to(DEV))
    torch.cuda.synchronize()
    b = ORC.balance_from_sums(r["count"], psum.numpy(), T, k, r["kept"])
    np.testing.assert_allclose(np_of(f), b["f"], rtol=1e-6)
    np.testing.assert_allclose(np_of(P), b["P"], rtol=1e-6)
    assert abs(L.item() - b["L"]) <= 1e-6 * abs(b["L"])
    assert dropped.item() == b["dropped"]


def test_workspace_status_clean_after_calls():
    w = W.small(WL["switch_top1"], T=64, d=64, H=64)
    cfg = moe.config_from_workload(w)
    ws = moe.workspace(cfg, DEV)
    inp = W.to_device(W.make_inputs(w), DEV)
    moe.layer_forward(cfg, inp, ws=ws)
    assert moe.device_status(ws) == (0, 0)


def _bf16_ulp(v):
    """Spacing of bf16 numbers at |v| (8 significant bits)."""
    a = np.maximum(np.abs(v), 1e-30)
    return np.exp2(np.floor(np.log2(a)) - 7)


@pytest.mark.parametrize("act", ["gelu", "swiglu"])
def test_tensor_core_activation_accuracy(act):
    """Identity expert weights make Y = bf16(act(x)) exactly (fp32 sums of
    x * 1 are exact), so the device activation can be checked element by
    element against the exact one: the only allowed error is the final bf16
    rounding plus a slack far below it (4e-6 relative for the fast exp and
    division, 3e-7 absolute per unit of |u| for the erf approximation, whose
    bound is 1.5e-7). A tanh-form GELU (error ~1e-3) would fail."""
    d = H = 256
    R = 1024
    g = torch.Generator().manual_seed(21)
    xv = torch.linspace(-9.0, 9.0, R * d - 6, dtype=torch.float64)
    xv = torch.cat([xv, torch.tensor([0.0, 1e-6, -1e-6, 30.0, -30.0, -100.0],
                                     dtype=torch.float64)])
    xv = xv[torch.randperm(xv.numel(), generator=g)]
    x = xv.reshape(R, d).to(torch.bfloat16)
    eye = torch.eye(d, dtype=torch.bfloat16)
    W1 = eye[None].clone()
    W2 = eye[None].clone()
    W3 = eye[None].clone() if act == "swiglu" else None
    cfg = moe.make_config(R, d, 1, 1, H, R, "bf16", act)
    off = torch.tensor([0, R], dtype=torch.int32, device=DEV)
    Y = moe.expert_ffn(cfg, x.to(DEV), off, W1.to(DEV), W2.to(DEV),
                       None if W3 is None else W3.to(DEV))
    torch.cuda.synchronize()
    u = x.double().numpy()
    if act == "gelu":
        exact = ORC.gelu(u)
    else:
        exact = ORC.silu(u) * u
    y = Y.double().cpu().numpy()
    bound = 0.5 * _bf16_ulp(exact) + 4e-6 * np.abs(exact) + 3e-7 * np.maximum(1.0, np.abs(u))
    bad = np.abs(y - exact) > bound
    assert not bad.any(), (u[bad][:5], y[bad][:5], exact[bad][:5])


# ---------------------------------------------------------------------------
# device-resident inputs out of range: recorded in the workspace header, the
# rest of the call unaffected (ids) or nothing computed (offsets)
# ---------------------------------------------------------------------------
BAD_IDS = [-1, 1 << 30, -(1 << 31)]


@pytest.mark.parametrize("T,E,k,c,dt", [(1000, 16, 2, Fraction(1, 2), "bf16"),
                                        (257, 5, 3, Fraction(1), "f32")])
def test_dispatch_out_of_range_ids_are_left_out_and_reported(T, E, k, c, dt):
    ids = W.make_routing(T, E, k, seed=11, skew=1.0)
    g = torch.Generator().manual_seed(12)
    bad = torch.rand(T, k, generator=g) < 0.1
    vals = torch.tensor(BAD_IDS + [E, E + 3], dtype=torch.int32)
    ids_bad = torch.where(bad, vals[torch.randint(len(vals), (T, k), generator=g)], ids)
    x = W.make_rows(T, 32, torch.float32 if dt == "f32" else torch.bfloat16, seed=2)
    C = ORC.capacity(c, k, T, E)
    cfg = moe.make_config(T, 32, E, k, 8, C, dt, "gelu")
    ws = moe.workspace(cfg, DEV)
    out = moe.dispatch(cfg, ids_bad.to(DEV), x.to(DEV), ws=ws)
    assert moe.device_status(ws) == (1, 41)    # MOE_ERR_INVALID_ARG, the dispatch count
    # expected: every bad id as a choice of an extra last expert E, then
    # that expert removed (offsets of the first E experts are unchanged)
    r = ORC.dispatch(torch.where(bad, E, ids).numpy(), E + 1, C)
    np.testing.assert_array_equal(out["count"].cpu().numpy(), r["count"][:E])
    np.testing.assert_array_equal(out["offset"].cpu().numpy(), r["offset"][:E + 1])
    np.testing.assert_array_equal(out["slot_of"].cpu().numpy(),
                                  np.where(bad.numpy(), -1, r["slot_of"]))
    R = int(r["offset"][E])
    np.testing.assert_array_equal(out["token_of_row"][:R].cpu().numpy(), r["token_of_row"][:R])
    assert torch.equal(out["xd"][:R].cpu(), x[torch.from_numpy(r["token_of_row"][:R]).long()])
    # the status was cleared by the read; a valid call leaves it clean
    moe.dispatch(cfg, ids.to(DEV), x.to(DEV), ws=ws)
    assert moe.device_status(ws) == (0, 0)


def _bad_offsets(E, R):
    ok = np.linspace(0, R, E + 1).astype(np.int32)
    cases = {}
    o = ok.copy(); o[0] = 3; cases["first_not_zero"] = o
    o = ok.copy(); o[1], o[2] = o[2], o[1]; cases["decreasing"] = o
    o = ok.copy(); o[1] = -256; cases["negative"] = o
    o = ok.copy(); o[E] = R + 1; cases["past_rows"] = o
    o = ok.copy(); o[1:] = 2 ** 31 - 1; cases["huge"] = o
    return ok, cases


@pytest.mark.parametrize("E,d,H,act,dt,rows", [(3, 64, 128, "gelu", "bf16", 600),
                                                (2, 256, 256, "swiglu", "bf16", 2100),
                                                (3, 64, 128, "swiglu", "f32", 300)])
def test_expert_ffn_bad_offsets_compute_nothing_and_report(E, d, H, act, dt, rows):
    w, inp, _ = _ffn_case(E, d, H, act, dt, [rows // E] * (E - 1) + [rows - rows // E * (E - 1)],
                          seed=5)
    cfg = moe.make_config(rows, d, E, 1, H, rows, dt, act)     # rows bound: T k = rows
    dv = W.to_device(inp, DEV)
    ws = moe.workspace(cfg, DEV)
    ok, cases = _bad_offsets(E, rows)
    where = 43 if dt == "f32" else 42
    for name, o in cases.items():
        Y = torch.full((rows, d), 7.0, dtype=dv["x"].dtype, device=DEV)
        moe.expert_ffn(cfg, dv["x"], torch.from_numpy(o).to(DEV), dv["W1"], dv["W2"], dv["W3"],
                       dv["b1"], dv["b2"], ws=ws, Y=Y)
        assert moe.device_status(ws) == (1, where), name
        assert bool((Y == 7.0).all()), name
    Y = moe.expert_ffn(cfg, dv["x"], torch.from_numpy(ok).to(DEV), dv["W1"], dv["W2"], dv["W3"],
                       dv["b1"], dv["b2"], ws=ws)
    assert moe.device_status(ws) == (0, 0)
    assert bool(torch.isfinite(Y.float()).all())
