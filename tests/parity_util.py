"""Helpers shared by the GPU parity tests: run the CUDA path through the
binding and the CPU oracle on the same seeded inputs, and compare."""
from __future__ import annotations

import numpy as np
import torch

from mixture_experts_layer_99_b300 import moe, workloads as W
from oracle import moe_oracle as ORC

# Tolerances (max |err| / max |ref|), from the layer's precision contract:
# bf16 experts with fp32 accumulation 2e-2, the fp32 workload 1e-5; router
# logits 1e-3 (bf16 inputs) / 1e-5 (fp32); statistics 1e-5 relative.
TOL_Y = {"bf16": 2e-2, "f32": 1e-5}
TOL_LOGITS = {"bf16": 1e-3, "f32": 1e-5}
TOL_STATS = 1e-5
TOL_GATE = 2e-6


def rel_err(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = float(np.abs(ref).max()) if ref.size else 0.0
    num = float(np.abs(got - ref).max()) if ref.size else 0.0
    return num / den if den > 0 else num


def np_of(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64 if t.is_floating_point() else t.dtype).numpy()


def sample_tokens(r: dict, T: int, n: int, seed: int = 0, tail_experts: int = 3):
    """A seeded sample of n tokens plus every token routed (kept) to the
    `tail_experts` least-loaded experts that received any token."""
    rng = np.random.default_rng(seed)
    base = rng.choice(T, size=min(n, T), replace=False)
    kept = np.asarray(r["kept"])
    active = np.nonzero(kept > 0)[0]
    tail = active[np.argsort(kept[active], kind="stable")[:tail_experts]]
    ids, slot = np.asarray(r["ids"]), np.asarray(r["slot_of"])
    extra = np.nonzero(np.isin(ids, tail).any(axis=1) & (slot >= 0).any(axis=1))[0]
    return np.unique(np.concatenate([base, extra]))


def check_layer(w: W.Workload, device, n_sample=None, seed=None, inp=None):
    """End-to-end parity of moe_layer_forward against the oracle.

    Routing is compared bit-exactly with the oracle run on the GPU's own fp32
    logits; the logits themselves against the oracle's fp64 logits; y on all
    tokens (or a sample) with the workload's tolerance; f, P, L_balance and the
    drop count with 1e-5."""
    inp = W.make_inputs(w, seed) if inp is None else inp
    cfg = moe.config_from_workload(w)
    dinp = W.to_device(inp, device)
    shared = inp.get("shared")
    if shared is not None:
        out = moe.layer_forward_shared(cfg, dinp, dinp["shared"])
    else:
        out = moe.layer_forward(cfg, dinp)
    torch.cuda.synchronize()
    C = ORC.capacity(w.c, w.k, w.T, w.E)
    assert cfg.capacity == C
    lg = out["logits"].cpu().numpy()                     # fp32 keys
    ref_l = ORC.router_logits(inp["x"], inp["Wg"], inp["bias"], inp["noise"], w.tau,
                              w.noise_scale)
    e_l = rel_err(lg, ref_l)
    assert e_l <= TOL_LOGITS[w.dtype], f"logits rel err {e_l}"
    r = ORC.route_from_logits(lg, w.k, C)
    np.testing.assert_array_equal(out["topk_idx"].cpu().numpy(), r["ids"])
    np.testing.assert_array_equal(out["slot_of"].cpu().numpy(), r["slot_of"])
    np.testing.assert_array_equal(out["expert_count"].cpu().numpy(), r["count"])
    np.testing.assert_array_equal(out["expert_offset"].cpu().numpy(), r["offset"])
    g = out["topk_gate"].cpu().numpy()
    assert np.abs(g - r["gates"]).max() <= TOL_GATE
    assert int(out["dropped"].item()) == r["dropped"]
    np.testing.assert_allclose(np_of(out["f"]), r["f"], rtol=TOL_STATS, atol=0)
    np.testing.assert_allclose(np_of(out["P"]), r["P"], rtol=TOL_STATS, atol=1e-9)
    assert abs(float(out["L_balance"].item()) - r["L"]) <= TOL_STATS * abs(r["L"])
    tokens = (np.arange(w.T) if n_sample is None
              else sample_tokens(r, w.T, n_sample, seed=w.seed))
    ref_y = ORC.combine_tokens(tokens, inp["x"], r["ids"], r["gates"], r["slot_of"],
                               inp["W1"], inp["W2"], inp.get("W3"), inp.get("b1"),
                               inp.get("b2"), w.act)
    if shared is not None:
        ref_y = ref_y + ORC.shared_expert_rows(ORC.as_f64(inp["x"][tokens]), shared, w.act)
    y = np_of(out["y"])[tokens]
    e_y = rel_err(y, ref_y)
    assert e_y <= TOL_Y[w.dtype], f"y rel err {e_y}"
    # tokens with every slot dropped are exactly zero (without a shared expert)
    all_dropped = (r["slot_of"] < 0).all(axis=1)
    if all_dropped.any() and shared is None:
        assert (out["y"][torch.from_numpy(all_dropped).to(device)] == 0).all()
    flips = int((ORC.topk_ids(ref_l, w.k) != r["ids"]).any(axis=1).sum())
    return dict(logits_err=e_l, y_err=e_y, dropped=r["dropped"], L=r["L"],
                selection_flips_vs_fp64=flips, tokens_checked=len(tokens), out=out, r=r)
