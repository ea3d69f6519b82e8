"""Pins of the backward oracle (CPU): central finite differences of the
forward oracle's loss, torch autograd through an independent dense
restatement of the forward, closed forms, and planted mistakes that the pins
must catch."""
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import moe_backward as B
from oracle import moe_oracle as F


def _tiny(act, seed, T=12, d=5, E=4, k=2, H=7, bias=True, noise=True, expert_bias=True,
          shared=False):
    rng = np.random.default_rng(seed)
    inp = dict(x=rng.standard_normal((T, d)),
               Wg=rng.standard_normal((E, d)),
               W1=rng.standard_normal((E, H, d)) / np.sqrt(d),
               W2=rng.standard_normal((E, d, H)) / np.sqrt(H),
               W3=rng.standard_normal((E, H, d)) / np.sqrt(d) if act == "swiglu" else None,
               b1=0.1 * rng.standard_normal((E, H)) if (expert_bias and act == "gelu") else None,
               b2=0.1 * rng.standard_normal((E, d)) if (expert_bias and act == "gelu") else None,
               bias=rng.standard_normal(E) if bias else None,
               noise=0.3 * rng.standard_normal((T, E)) if noise else None)
    sh = None
    if shared:
        Hs = 6
        sh = dict(W1=rng.standard_normal((Hs, d)) / np.sqrt(d),
                  W2=rng.standard_normal((d, Hs)) / np.sqrt(Hs),
                  W3=rng.standard_normal((Hs, d)) / np.sqrt(d) if act == "swiglu" else None,
                  b1=0.1 * rng.standard_normal(Hs) if act == "gelu" else None,
                  b2=0.1 * rng.standard_normal(d) if act == "gelu" else None)
    dy = rng.standard_normal((T, d))
    return inp, sh, dy


CASES = [
    # act, k, c (drops when c < E/k), alpha, tau, shared
    ("gelu", 2, Fraction(3, 4), 0.3, 0.8, False),
    ("swiglu", 2, Fraction(3, 4), 0.3, 1.0, False),
    ("gelu", 1, Fraction(1), 0.5, 1.0, False),
    ("swiglu", 3, Fraction(2), 0.0, 1.3, False),
    ("gelu", 2, Fraction(1), 0.2, 1.0, True),
    ("swiglu", 2, Fraction(1, 2), 0.7, 1.0, True),
]

PARAMS = ["x", "Wg", "bias", "W1", "W3", "W2", "b1", "b2"]


def _fd_check(act, k, c, alpha, tau, shared, seed=0, h=1e-6):
    inp, sh, dy = _tiny(act, seed, k=k, shared=shared)
    got = B.moe_backward(inp, k, c, act, dy, alpha, tau, shared=sh)
    ref_route = got["route"]
    grads = dict(x=got["dx"], Wg=got["dWg"], bias=got["dbias"], W1=got["dW1"],
                 W3=got["dW3"], W2=got["dW2"], b1=got["db1"], b2=got["db2"])
    targets = [(inp, name, grads[name]) for name in PARAMS if inp.get(name) is not None]
    if sh is not None:
        for name in ("W1", "W3", "W2", "b1", "b2"):
            if sh.get(name) is not None:
                targets.append((sh, name, got["shared"]["d" + name]))
    for holder, name, g in targets:
        base = holder[name]
        num = np.zeros_like(base)
        for i in np.ndindex(base.shape):
            vals = []
            for s in (+1.0, -1.0):
                pert = base.copy()
                pert[i] += s * h
                holder[name] = pert
                loss, r = B.layer_loss(inp, k, c, act, dy, alpha, tau, shared=sh)
                # the routing must not move under the perturbation
                assert np.array_equal(r["ids"], ref_route["ids"])
                assert np.array_equal(r["slot_of"], ref_route["slot_of"])
                vals.append(loss)
            holder[name] = base
            num[i] = (vals[0] - vals[1]) / (2 * h)
        err = np.abs(num - g).max()
        assert err <= 1e-6 * max(1.0, np.abs(num).max()), (name, err)


@pytest.mark.parametrize("act,k,c,alpha,tau,shared", CASES)
def test_backward_matches_finite_differences(act, k, c, alpha, tau, shared):
    _fd_check(act, k, c, alpha, tau, shared)


def _torch_dense_loss(inp, sh, dy, k, c, act, alpha, tau, route):
    """Independent restatement of the forward in torch (fp64, dense: every
    expert on every token, masked by the routing decisions held fixed), for
    autograd."""
    t = {n: (torch.tensor(v, dtype=torch.float64, requires_grad=True) if v is not None else None)
         for n, v in inp.items()}
    x = t["x"]
    z = x @ t["Wg"].T
    if t["bias"] is not None:
        z = z + t["bias"]
    if t["noise"] is not None:
        z = z + t["noise"].detach()
    p = torch.softmax(z / tau, dim=1)
    ids = torch.tensor(route["ids"], dtype=torch.int64)
    keep = torch.tensor(route["slot_of"] >= 0)
    sel = p.gather(1, ids)
    g = sel / sel.sum(dim=1, keepdim=True)
    E = t["Wg"].shape[0]
    y = torch.zeros_like(x)
    for e in range(E):
        u = x @ t["W1"][e].T
        if act == "gelu":
            if t["b1"] is not None:
                u = u + t["b1"][e]
            hh = torch.nn.functional.gelu(u)
        else:
            hh = torch.nn.functional.silu(u) * (x @ t["W3"][e].T)
        ye = hh @ t["W2"][e].T
        if act == "gelu" and t["b2"] is not None:
            ye = ye + t["b2"][e]
        w = ((ids == e) & keep).to(torch.float64) * g        # [T, k]
        y = y + w.sum(dim=1, keepdim=True) * ye
    ts = None
    if sh is not None:
        ts = {n: (torch.tensor(v, dtype=torch.float64, requires_grad=True) if v is not None
                  else None) for n, v in sh.items()}
        u = x @ ts["W1"].T
        if act == "gelu":
            hh = torch.nn.functional.gelu(u + ts["b1"]) if ts["b1"] is not None else \
                torch.nn.functional.gelu(u)
        else:
            hh = torch.nn.functional.silu(u) * (x @ ts["W3"].T)
        ye = hh @ ts["W2"].T
        if act == "gelu" and ts["b2"] is not None:
            ye = ye + ts["b2"]
        y = y + ye
    f = torch.tensor(route["f"], dtype=torch.float64)
    L = E * (f * p.mean(dim=0)).sum()
    loss = (torch.tensor(dy) * y).sum() + alpha * L
    return loss, t, ts


@pytest.mark.parametrize("act,k,c,alpha,tau,shared", CASES)
def test_backward_matches_torch_autograd(act, k, c, alpha, tau, shared):
    inp, sh, dy = _tiny(act, 11, T=40, d=8, E=5, H=9, k=k, shared=shared)
    got = B.moe_backward(inp, k, c, act, dy, alpha, tau, shared=sh)
    loss, t, ts = _torch_dense_loss(inp, sh, dy, k, c, act, alpha, tau, got["route"])
    names = [n for n in PARAMS if t.get(n) is not None and n != "noise"]
    leaves = [t[n] for n in names]
    snames = [n for n in ("W1", "W3", "W2", "b1", "b2") if ts is not None and ts.get(n) is not None]
    leaves += [ts[n] for n in snames]
    grads = torch.autograd.grad(loss, leaves)
    mine = dict(x=got["dx"], Wg=got["dWg"], bias=got["dbias"], W1=got["dW1"], W3=got["dW3"],
                W2=got["dW2"], b1=got["db1"], b2=got["db2"])
    for n, gr in zip(names, grads[:len(names)]):
        np.testing.assert_allclose(mine[n], gr.numpy(), rtol=1e-10, atol=1e-12, err_msg=n)
    for n, gr in zip(snames, grads[len(names):]):
        np.testing.assert_allclose(got["shared"]["d" + n], gr.numpy(), rtol=1e-10, atol=1e-12,
                                   err_msg="shared " + n)


def test_top1_gates_carry_no_router_gradient():
    """k = 1: every kept gate is exactly 1, so without the balance term the
    router receives no gradient at all."""
    inp, _, dy = _tiny("gelu", 3, k=1)
    got = B.moe_backward(inp, 1, Fraction(1), "gelu", dy, alpha=0.0)
    assert np.all(got["dz"] == 0.0)
    assert np.all(got["dWg"] == 0.0)


def test_std_scaled_noise_strength_carries_no_gradient():
    """With std-scaled router noise (kwkr.cn MoE article, section 3.3) the
    strength s * std_t is taken without gradient: the gradients equal those
    of the same noise frozen into a fixed input, s * std_t(z) * n, with std_t
    computed here by torch (population std of z = x W_g^T + b per token).
    The finite-difference and autograd pins cover the fixed-input case."""
    for act, k, tau in (("gelu", 2, 1.3), ("swiglu", 1, 1.0)):
        inp, _, dy = _tiny(act, 9, T=20, k=k)
        inp["noise"] = np.random.default_rng(19).standard_normal(inp["noise"].shape)
        s = 0.4
        got = B.moe_backward(inp, k, Fraction(3, 4), act, dy, alpha=0.1, tau=tau,
                             noise_scale=s)
        z = torch.nn.functional.linear(torch.from_numpy(inp["x"]), torch.from_numpy(inp["Wg"]),
                                       torch.from_numpy(inp["bias"]))
        frozen = (s * z.std(dim=1, unbiased=False)[:, None]).numpy() * inp["noise"]
        ref = B.moe_backward(dict(inp, noise=frozen), k, Fraction(3, 4), act, dy, alpha=0.1,
                             tau=tau)
        np.testing.assert_array_equal(got["route"]["ids"], ref["route"]["ids"])
        np.testing.assert_array_equal(got["route"]["slot_of"], ref["route"]["slot_of"])
        for key in ("dx", "dWg", "dbias", "dW1", "dW2", "dz"):
            np.testing.assert_allclose(got[key], ref[key], rtol=1e-10, atol=1e-12, err_msg=key)


def test_balance_gradient_closed_form_on_a_uniform_router():
    """W_g = 0, no bias or noise, dy = 0: p = 1/E everywhere and only the
    balance term acts, dl_ti = (alpha / T) (f_i - 1/E)."""
    inp, _, dy = _tiny("gelu", 4, T=30, k=2, bias=False, noise=False)
    inp["Wg"] = np.zeros_like(inp["Wg"])
    alpha = 0.25
    got = B.moe_backward(inp, 2, Fraction(2), "gelu", np.zeros_like(dy), alpha=alpha)
    T, E = 30, inp["Wg"].shape[0]
    f = got["route"]["f"]
    want = np.broadcast_to(alpha / T * (f - 1.0 / E), (T, E))
    np.testing.assert_allclose(got["dz"], want, rtol=0, atol=1e-15)
    np.testing.assert_allclose(got["dWg"], want.T @ inp["x"], rtol=1e-12, atol=1e-15)


def test_activation_derivatives_against_differences():
    u = np.linspace(-8, 8, 2001)
    h = 1e-6
    np.testing.assert_allclose(B.gelu_grad(u), (F.gelu(u + h) - F.gelu(u - h)) / (2 * h),
                               rtol=0, atol=1e-8)
    np.testing.assert_allclose(B.silu_grad(u), (F.silu(u + h) - F.silu(u - h)) / (2 * h),
                               rtol=0, atol=1e-8)


# planted mistakes: each must make the finite-difference pin fail
def _gelu_grad_no_density(u):
    return 0.5 * (1.0 + B._erf(np.asarray(u) / np.sqrt(2.0)))


def _gates_without_mean(p, ids, gates, dg, f, alpha, tau=1.0):
    p = np.asarray(p, dtype=np.float64)
    T, E = p.shape
    ids = np.asarray(ids).astype(np.int64)
    S = np.take_along_axis(p, ids, axis=1).sum(axis=1, keepdims=True)
    dp = np.zeros((T, E))
    np.put_along_axis(dp, ids, np.asarray(dg) / S, axis=1)
    dp = dp + alpha * E * np.asarray(f)[None, :] / T
    dl = p * (dp - (p * dp).sum(axis=1, keepdims=True))
    return dict(dp=dp, dl=dl, dz=dl / float(tau))


def _softmax_without_projection(p, ids, gates, dg, f, alpha, tau=1.0):
    p = np.asarray(p, dtype=np.float64)
    T, E = p.shape
    ids = np.asarray(ids).astype(np.int64)
    g = np.asarray(gates, dtype=np.float64)
    dg = np.asarray(dg, dtype=np.float64)
    S = np.take_along_axis(p, ids, axis=1).sum(axis=1, keepdims=True)
    dp = np.zeros((T, E))
    np.put_along_axis(dp, ids, (dg - (g * dg).sum(axis=1, keepdims=True)) / S, axis=1)
    dp = dp + alpha * E * np.asarray(f)[None, :] / T
    dl = p * dp
    return dict(dp=dp, dl=dl, dz=dl / float(tau))


def _silu_grad_wrong(u):
    s = 1.0 / (1.0 + np.exp(-np.asarray(u)))
    return s


MUTANTS = [
    ("gelu_grad", _gelu_grad_no_density, ("gelu", 2, Fraction(3, 4), 0.3, 0.8, False)),
    ("gate_logit_grads", _gates_without_mean, ("gelu", 2, Fraction(3, 4), 0.0, 1.0, False)),
    ("gate_logit_grads", _softmax_without_projection, ("swiglu", 2, Fraction(1), 0.3, 1.0, False)),
    ("silu_grad", _silu_grad_wrong, ("swiglu", 2, Fraction(3, 4), 0.0, 1.0, False)),
]


@pytest.mark.parametrize("name,fn,case", MUTANTS)
def test_pins_catch_planted_mistakes(monkeypatch, name, fn, case):
    monkeypatch.setattr(B, name, fn)
    with pytest.raises(AssertionError):
        _fd_check(*case)
