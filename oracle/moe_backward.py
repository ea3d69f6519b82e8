"""CPU oracle for the backward pass of the top-k routed MoE FFN layer.

TEST INFRASTRUCTURE ONLY, like ``moe_oracle``: nothing in the product path
imports it; only ``tests/`` and the CPU legs of ``bench.py`` may call it. It
shares no code with the CUDA library.

The pages train this layer (the kwkr.cn article, "MoE sparse activation: from
the math to the code", section 2.2 adds alpha * L_balance to the task loss
and section 3.3 trains the router; the intelliparadigm tutorial, section 2.3,
does the same for k = 1) but print no gradient formulas. The gradients below
are the chain rule applied to the forward of ``moe_oracle`` step by step, in
fp64:

    loss = sum_t <dy_t, y_t> + alpha * L_balance

* combine  y_t = sum_{kept j} g_tj Y_tj:
      dY_tj = g_tj dy_t,   dg_tj = <dy_t, Y_tj>   (0 for a dropped slot)
* renormalised gates  g_j = p_{K_j} / S,  S = sum_m p_{K_m}:
      dp_{K_i} += (dg_i - sum_j g_j dg_j) / S
* load balance  L = E sum_i f_i P_i,  P_i = (1/T) sum_t p_ti,  f piecewise
  constant:  dp_ti += alpha E f_i / T
* softmax:  dl_t = p_t * (dp_t - <p_t, dp_t>);  keys l = z / tau:  dz = dl / tau
* router GEMM  z = x Wg^T + b + noise:  dx += dz Wg,  dWg = dz^T x,  db = sum_t dz_t
* expert e on its kept rows (xr -> Y):
      GELU    u = xr W1^T + b1, h = gelu(u), Y = h W2^T + b2
              dh = dY W2, du = dh * gelu'(u), dxr = du W1,
              dW2 = dY^T h, db2 = sum dY, dW1 = du^T xr, db1 = sum du
      SwiGLU  a = xr W1^T, v = xr W3^T, h = silu(a) * v, Y = h W2^T
              dh = dY W2, da = dh * v * silu'(a), dv = dh * silu(a),
              dxr = da W1 + dv W3, dW1 = da^T xr, dW3 = dv^T xr, dW2 = dY^T h
* dispatch:  dx_t += sum over the kept slots of t of dxr[slot]
* shared expert: an expert with dY = dy for every token.

Selection (top-k), capacity and drops are piecewise constant: they get no
gradient, and the derivative is taken with the routing held fixed.

Pinned in ``tests/test_oracle_backward.py`` by central finite differences of
the forward oracle's loss, by torch autograd through an independent dense
restatement of the forward, and by closed-form special cases.
"""
from __future__ import annotations

import math

import numpy as np
from scipy.special import erf as _erf

from oracle import moe_oracle as F


def gelu_grad(u):
    """d/du [u/2 (1 + erf(u/sqrt 2))] = Phi(u) + u phi(u)."""
    u = np.asarray(u, dtype=np.float64)
    return 0.5 * (1.0 + _erf(u / math.sqrt(2.0))) + u * np.exp(-0.5 * u * u) / math.sqrt(
        2.0 * math.pi)


def silu_grad(u):
    """d/du [u sigma(u)] = sigma(u) (1 + u (1 - sigma(u)))."""
    u = np.asarray(u, dtype=np.float64)
    s = 1.0 / (1.0 + np.exp(-u))
    return s * (1.0 + u * (1.0 - s))


def expert_ffn_backward_rows(xr, dYr, W1e, W2e, W3e=None, b1e=None, act="gelu"):
    """Gradients of one expert on its rows: returns dict(dx, dW1, dW2, dW3,
    db1, db2) for the upstream gradient dYr [n, d] of its outputs."""
    xr = F.as_f64(xr)
    dYr = F.as_f64(dYr)
    W1e = F.as_f64(W1e)
    W2e = F.as_f64(W2e)
    a = xr @ W1e.T
    out = {}
    if act == "gelu":
        if b1e is not None:
            a = a + F.as_f64(b1e)[None, :]
        h = F.gelu(a)
        dh = dYr @ W2e
        du = dh * gelu_grad(a)
        out["dx"] = du @ W1e
        out["dW1"] = du.T @ xr
        out["db1"] = du.sum(axis=0)
        out["dW3"] = None
    elif act == "swiglu":
        W3e = F.as_f64(W3e)
        v = xr @ W3e.T
        h = F.silu(a) * v
        dh = dYr @ W2e
        da = dh * v * silu_grad(a)
        dv = dh * F.silu(a)
        out["dx"] = da @ W1e + dv @ W3e
        out["dW1"] = da.T @ xr
        out["dW3"] = dv.T @ xr
        out["db1"] = None
    else:
        raise ValueError(act)
    out["dW2"] = dYr.T @ h
    out["db2"] = dYr.sum(axis=0) if act == "gelu" else None
    return out


def gate_logit_grads(p, ids, gates, dg, f, alpha: float, tau: float = 1.0):
    """Router part: dg [T,k] (upstream gradient of the gates) and the
    balance term alpha * L_balance -> dp -> dl (softmax) -> dz = dl / tau.
    Returns dict(dp, dl, dz), all [T, E] fp64."""
    p = np.asarray(p, dtype=np.float64)
    T, E = p.shape
    ids = np.asarray(ids).astype(np.int64)
    g = np.asarray(gates, dtype=np.float64)
    dg = np.asarray(dg, dtype=np.float64)
    S = np.take_along_axis(p, ids, axis=1).sum(axis=1, keepdims=True)     # [T,1]
    dsel = (dg - (g * dg).sum(axis=1, keepdims=True)) / S                  # [T,k]
    dp = np.zeros((T, E))
    np.put_along_axis(dp, ids, dsel, axis=1)   # the k chosen experts are distinct
    dp = dp + alpha * E * np.asarray(f, dtype=np.float64)[None, :] / T
    dl = p * (dp - (p * dp).sum(axis=1, keepdims=True))
    return dict(dp=dp, dl=dl, dz=dl / float(tau))


def moe_backward(inp: dict, k: int, c, act: str, dy, alpha: float = 0.0, tau: float = 1.0,
                 logits=None, shared=None, noise_scale: float = 0.0):
    """Gradients of loss = sum <dy, y> + alpha * L_balance with respect to x,
    Wg, the router bias (if present), W1, W3, W2, b1, b2 (if present) and the
    shared expert's weights (if present). Routing follows ``logits`` (the
    GPU's fp32 keys) when given, else the oracle's own fp64 logits.

    With std-scaled router noise (noise_scale > 0) the noise strength
    noise_scale * std_t is taken without gradient: it sets how far the router
    explores, it is not a path for training the router, so dz is the same as
    for that noise added as a fixed input.

    Returns dict(dx, dWg, dbias, dW1, dW3, dW2, db1, db2, dgates, dz,
    shared=dict(...) or None) plus the routing dict under "route"."""
    x = inp["x"]
    xf = F.as_f64(x)
    T, d = xf.shape
    E = inp["Wg"].shape[0]
    C = F.capacity(c, k, T, E)
    if logits is None:
        logits = F.router_logits(x, inp["Wg"], inp.get("bias"), inp.get("noise"), tau,
                                 noise_scale)
    r = F.route_from_logits(logits, k, C)
    ids, slot_of, g = r["ids"], r["slot_of"], r["gates"]
    dyf = F.as_f64(dy)
    W1, W2, W3 = inp["W1"], inp["W2"], inp.get("W3")
    b1, b2 = inp.get("b1"), inp.get("b2")
    H = W1.shape[1]
    dW1 = np.zeros((E, H, d))
    dW2 = np.zeros((E, d, H))
    dW3 = np.zeros((E, H, d)) if act == "swiglu" else None
    db1 = np.zeros((E, H)) if (act == "gelu" and b1 is not None) else None
    db2 = np.zeros((E, d)) if (act == "gelu" and b2 is not None) else None
    dx = np.zeros((T, d))
    dg = np.zeros((T, k))
    for e in range(E):
        t_idx, j_idx = np.nonzero((ids == e) & (slot_of >= 0))
        if len(t_idx) == 0:
            continue
        xr = xf[t_idx]
        Ye = F.expert_ffn_rows(xr, W1[e], W2[e], None if W3 is None else W3[e],
                               None if b1 is None else b1[e], None if b2 is None else b2[e],
                               act)
        dg[t_idx, j_idx] = (dyf[t_idx] * Ye).sum(axis=1)
        dYr = g[t_idx, j_idx][:, None] * dyf[t_idx]
        ge = expert_ffn_backward_rows(xr, dYr, W1[e], W2[e], None if W3 is None else W3[e],
                                      None if b1 is None else b1[e], act)
        np.add.at(dx, t_idx, ge["dx"])
        dW1[e] = ge["dW1"]
        dW2[e] = ge["dW2"]
        if dW3 is not None:
            dW3[e] = ge["dW3"]
        if db1 is not None:
            db1[e] = ge["db1"]
        if db2 is not None:
            db2[e] = ge["db2"]
    rg = gate_logit_grads(r["p"], ids, g, dg, r["f"], alpha, tau)
    dz = rg["dz"]
    dx += dz @ F.as_f64(inp["Wg"])
    dWg = dz.T @ xf
    dbias = dz.sum(axis=0) if inp.get("bias") is not None else None
    sh = None
    if shared is not None:
        gs = expert_ffn_backward_rows(xf, dyf, shared["W1"], shared["W2"], shared.get("W3"),
                                      shared.get("b1"), act)
        dx += gs["dx"]
        sh = dict(dW1=gs["dW1"], dW2=gs["dW2"], dW3=gs["dW3"], db1=gs["db1"], db2=gs["db2"])
    return dict(dx=dx, dWg=dWg, dbias=dbias, dW1=dW1, dW3=dW3, dW2=dW2, db1=db1, db2=db2,
                dgates=dg, dz=dz, shared=sh, route=r)


def layer_loss(inp: dict, k: int, c, act: str, dy, alpha: float = 0.0, tau: float = 1.0,
               shared=None):
    """The scalar the gradients above differentiate, from the forward oracle:
    sum <dy, y> + alpha * L_balance. Returns (loss, routing dict)."""
    r = F.moe_forward(inp, k, c, act, tau, shared=shared)
    return float((F.as_f64(dy) * r["y"]).sum() + alpha * r["L"]), r
