"""Pins of the CPU oracle against what the MoE pages and the mathematics fix.

Each ``pin_*`` takes the oracle module and asserts; the tests below run every
pin on the real oracle, and ``test_planted_mistakes_are_caught`` plants
plausible mistakes in the oracle (on the CPU, via monkeypatch) and checks that
at least one pin fails for each. Sources (page title, section):

* kwkr.cn MoE article ("MoE sparse activation: from the math to the code"),
  sections 2.1-2.3, 3.1-3.2.
* intelliparadigm.com "MoE模型：动态计算架构解析与实践指南", section 2.1
  (DenseExpert), section 2.3 (k=1 load-balancing loss) and section 3.1 (the
  dense-masked expert loop of MoELlama).
"""
import itertools
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import scipy.special
import torch
import torch.nn.functional as F

from oracle import moe_oracle as ORC

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _rng(seed):
    return np.random.default_rng(seed)


# ---------------------------------------------------------------- capacity
def pin_capacity_golden(o):
    """The hand-worked closed-form values of C = ceil(c k T / E)."""
    for case in _load("capacity.json")["cases"]:
        c = Fraction(case["c"])
        assert o.capacity(c, case["k"], case["T"], case["E"]) == case["C"], case
        assert o.capacity(float(c), case["k"], case["T"], case["E"]) == case["C"]


def pin_capacity_grid(o):
    """Integer ceiling division of (p k T) by (q E) for c = p/q."""
    for (p, q), k, T, E in itertools.product(
            [(1, 1), (5, 4), (3, 2), (2, 1), (1, 3), (7, 8), (32, 1)],
            [1, 2, 3], [1, 7, 64, 1000, 8191], [1, 3, 8, 64]):
        want = -(-(p * k * T) // (q * E))
        assert o.capacity(Fraction(p, q), k, T, E) == want


# ---------------------------------------------------------------- routing
def _brute_route(l, k, C):
    """Brute force: the chosen set maximises the descending list of keys
    (l_i, -i) over all k-subsets; positions by direct counting."""
    T, E = l.shape
    ids = []
    for t in range(T):
        best = None
        for S in itertools.combinations(range(E), k):
            keyed = sorted(((l[t, i], -i) for i in S), reverse=True)
            if best is None or keyed > best[0]:
                best = (keyed, [-ni for _, ni in keyed])
        ids.append(best[1])
    count = [sum(e in ids[t] for t in range(T)) for e in range(E)]
    kept = [min(cn, C) for cn in count]
    off = [sum(kept[:e]) for e in range(E + 1)]
    slot = []
    for t in range(T):
        row = []
        for e in ids[t]:
            pos = sum(e in ids[u] for u in range(t))
            row.append(off[e] + pos if pos < C else -1)
        slot.append(row)
    return np.array(ids), np.array(count), np.array(off), np.array(slot)


def pin_routing_hand(o):
    g = _load("routing_hand.json")
    l = np.array(g["logits"], dtype=np.float64)
    r = o.route_from_logits(l, g["k"], g["C"])
    assert o.capacity(Fraction(g["c"]), g["k"], l.shape[0], l.shape[1]) == g["C"]
    for key in ("ids", "count", "pos", "kept", "offset", "slot_of",
                "token_of_row"):
        np.testing.assert_array_equal(r[key], np.array(g[key]), err_msg=key)
    assert r["dropped"] == g["dropped"]
    e = math.e
    want_g = np.array([[e / (e + 1), 1 / (e + 1)], [.5, .5], [.5, .5], [.5, .5]])
    np.testing.assert_allclose(r["gates"], want_g, rtol=0, atol=1e-15)
    # P by closed forms per token
    s0 = e * e + e + 1
    s2 = e + 2 * e ** 3
    s3 = 2 * e ** 5 + 1
    p = np.array([[e * e / s0, e / s0, 1 / s0],
                  [1 / 3, 1 / 3, 1 / 3],
                  [e / s2, e ** 3 / s2, e ** 3 / s2],
                  [e ** 5 / s3, 1 / s3, e ** 5 / s3]])
    np.testing.assert_allclose(r["P"], p.mean(axis=0), rtol=1e-14)
    f = np.array([3 / 8, 3 / 8, 2 / 8])
    np.testing.assert_allclose(r["f"], f, rtol=0, atol=0)
    assert abs(r["L"] - 3 * float((f * p.mean(axis=0)).sum())) < 1e-14


def pin_routing_bruteforce(o):
    rng = _rng(1)
    for trial in range(60):
        T = int(rng.integers(1, 9))
        E = int(rng.integers(1, 7))
        k = int(rng.integers(1, E + 1))
        C = int(rng.integers(1, T + 2))
        # small integer logits force many ties
        l = rng.integers(-2, 3, size=(T, E)).astype(np.float32)
        ids, count, off, slot = _brute_route(l, k, C)
        r = o.route_from_logits(l, k, C)
        np.testing.assert_array_equal(r["ids"], ids)
        np.testing.assert_array_equal(r["count"], count)
        np.testing.assert_array_equal(r["offset"], off)
        np.testing.assert_array_equal(r["slot_of"], slot)
        # token_of_row inverts slot_of
        rows = r["token_of_row"]
        for t in range(T):
            for j in range(k):
                if slot[t, j] >= 0:
                    assert rows[slot[t, j]] == t
        assert (rows >= 0).all()


def pin_zero_router(o):
    """W_g = 0: every logit ties, so every token picks experts 0..k-1 with
    gates 1/k; expert e<k gets all T tokens in order; P = 1/E and L = 1."""
    for T, E, k, C in [(10, 4, 2, 6), (7, 3, 3, 7), (5, 8, 1, 2), (9, 5, 2, 20)]:
        x = _rng(T).standard_normal((T, 6))
        Wg = np.zeros((E, 6))
        l = o.router_logits(x, Wg)
        r = o.route_from_logits(l, k, C)
        np.testing.assert_array_equal(r["ids"], np.tile(np.arange(k), (T, 1)))
        np.testing.assert_array_equal(r["gates"], np.full((T, k), 1.0 / k))
        cnt = np.array([T if e < k else 0 for e in range(E)])
        np.testing.assert_array_equal(r["count"], cnt)
        kept = min(T, C)
        for t in range(T):
            for j in range(k):
                want = j * kept + t if t < C else -1
                assert r["slot_of"][t, j] == want
        np.testing.assert_allclose(r["P"], np.full(E, 1.0 / E), rtol=1e-15)
        assert abs(r["L"] - 1.0) < 1e-14
        assert r["dropped"] == k * T - k * kept


def pin_gates(o):
    rng = _rng(2)
    for k in (1, 2, 3, 5):
        l = rng.standard_normal((200, 7)) * 3
        r = o.route_from_logits(l, k, 200)
        s = r["gates"].sum(axis=1)
        np.testing.assert_allclose(s, 1.0, rtol=0, atol=1e-15)
        assert (np.diff(r["gates"], axis=1) <= 0).all()
        if k == 1:
            assert (r["gates"] == 1.0).all()
        # gates are the chosen softmax probabilities up to one common factor
        p = scipy.special.softmax(l, axis=1)
        chosen = np.take_along_axis(p, r["ids"].astype(np.int64), axis=1)
        np.testing.assert_allclose(r["gates"] * chosen.sum(axis=1, keepdims=True),
                                   chosen, rtol=1e-13)


def pin_topk_logits_equals_topk_probs(o):
    """Softmax is monotone, so top-k on logits = top-k on probabilities."""
    rng = _rng(3)
    l = rng.standard_normal((500, 16)) * 4
    p = scipy.special.softmax(l, axis=1)
    for k in (1, 2, 4):
        ids = o.topk_ids(l, k)
        by_p = np.argsort(-p, axis=1, kind="stable")[:, :k]
        np.testing.assert_array_equal(ids, by_p)


# ---------------------------------------------------------------- aux
def pin_uniform_balance(o):
    """Uniform counts and uniform probabilities give L_balance = 1."""
    for E, k, T in [(4, 2, 8), (8, 1, 64), (64, 2, 128)]:
        p = np.full((T, E), 1.0 / E)
        count = np.full(E, k * T // E)
        a = o.aux_stats(p, count, count, k)
        assert abs(a["L"] - 1.0) < 1e-13
        np.testing.assert_allclose(a["f"].sum(), 1.0, rtol=1e-15)
        np.testing.assert_allclose(a["P"].sum(), 1.0, rtol=1e-14)
        assert a["dropped"] == 0


def pin_k1_balance_matches_tutorial(o):
    """For k = 1 the statistic equals the tutorial's loss: E * sum over
    experts of (mean one-hot selection) * (mean softmax probability)."""
    rng = _rng(4)
    T, E = 300, 6
    l = rng.standard_normal((T, E))
    r = o.route_from_logits(l, 1, T)
    onehot = np.eye(E)[np.argmax(l, axis=1)]
    probs = scipy.special.softmax(l, axis=1)
    want = E * float((onehot.mean(axis=0) * probs.mean(axis=0)).sum())
    assert abs(r["L"] - want) < 1e-13
    np.testing.assert_allclose(r["P"], probs.mean(axis=0), rtol=1e-13)


# ---------------------------------------------------------------- experts
def _weights(rng, E, d, H, swiglu, bias):
    W1 = rng.standard_normal((E, H, d)) / math.sqrt(d)
    W3 = rng.standard_normal((E, H, d)) / math.sqrt(d) if swiglu else None
    W2 = rng.standard_normal((E, d, H)) / math.sqrt(H)
    b1 = rng.standard_normal((E, H)) * 0.1 if bias else None
    b2 = rng.standard_normal((E, d)) * 0.1 if bias else None
    return W1, W3, W2, b1, b2


def _torch_ffn(x, W1, W3, W2, b1, b2, act):
    xt = torch.from_numpy(x)
    t1 = torch.from_numpy(W1)
    if act == "gelu":
        h = F.gelu(F.linear(xt, t1, None if b1 is None else torch.from_numpy(b1)))
        return F.linear(h, torch.from_numpy(W2),
                        None if b2 is None else torch.from_numpy(b2)).numpy()
    h = F.silu(F.linear(xt, t1)) * F.linear(xt, torch.from_numpy(W3))
    return F.linear(h, torch.from_numpy(W2)).numpy()


def pin_single_expert_is_dense_ffn(o):
    """E = 1, k = 1, c >= 1: the layer is exactly the dense FFN."""
    rng = _rng(5)
    for act, bias in (("gelu", True), ("gelu", False), ("swiglu", False)):
        T, d, H = 37, 12, 20
        x = rng.standard_normal((T, d))
        Wg = rng.standard_normal((1, d))
        W1, W3, W2, b1, b2 = _weights(rng, 1, d, H, act == "swiglu", bias)
        inp = dict(x=x, Wg=Wg, W1=W1, W3=W3, W2=W2, b1=b1, b2=b2)
        r = o.moe_forward(inp, k=1, c=1, act=act)
        want = _torch_ffn(x, W1[0], None if W3 is None else W3[0], W2[0],
                          None if b1 is None else b1[0],
                          None if b2 is None else b2[0], act)
        np.testing.assert_allclose(r["y"], want, rtol=0, atol=1e-12)
        assert r["dropped"] == 0


def pin_dense_masked_loop(o):
    """No drops: y equals running every expert on every token and weighting
    by the gate where the expert was chosen, 0 elsewhere (the dense-masked
    loop of the tutorial's MoELlama, generalised to k)."""
    rng = _rng(6)
    for act, E, k in (("gelu", 4, 2), ("swiglu", 5, 3), ("gelu", 3, 1)):
        T, d, H = 23, 8, 16
        x = rng.standard_normal((T, d))
        Wg = rng.standard_normal((E, d))
        bias = rng.standard_normal(E)
        noise = rng.standard_normal((T, E))
        W1, W3, W2, b1, b2 = _weights(rng, E, d, H, act == "swiglu",
                                      act == "gelu")
        inp = dict(x=x, Wg=Wg, W1=W1, W3=W3, W2=W2, b1=b1, b2=b2, bias=bias,
                   noise=noise)
        tau = 0.7
        r = o.moe_forward(inp, k=k, c=Fraction(E, k), act=act, tau=tau)
        assert r["dropped"] == 0
        logits = (F.linear(torch.from_numpy(x), torch.from_numpy(Wg),
                           torch.from_numpy(bias)).numpy() + noise) / tau
        order = torch.sort(torch.from_numpy(logits), dim=1, descending=True,
                           stable=True).indices[:, :k].numpy()
        probs = scipy.special.softmax(logits, axis=1)
        G = np.zeros((T, E))
        for t in range(T):
            sel = probs[t, order[t]]
            G[t, order[t]] = sel / sel.sum()
        y = np.zeros((T, d))
        for e in range(E):
            ye = _torch_ffn(x, W1[e], None if W3 is None else W3[e], W2[e],
                            None if b1 is None else b1[e],
                            None if b2 is None else b2[e], act)
            y += G[:, e:e + 1] * ye
        np.testing.assert_allclose(r["y"], y, rtol=0, atol=1e-12)


def pin_sort_based_layer(o):
    """Restatement of the article's layer with a sort-based dispatch: flatten
    the token-major slots, stable-sort them by expert, keep the first C of
    each expert's run, run each expert on its run, scatter-add gate-weighted
    rows back. Capacity is the closed form and there is no epsilon."""
    rng = _rng(7)
    for act, E, k, c in (("gelu", 4, 2, Fraction(3, 4)),
                         ("swiglu", 6, 2, Fraction(1, 2)),
                         ("gelu", 5, 1, Fraction(1))):
        T, d, H = 41, 10, 14
        x = rng.standard_normal((T, d))
        Wg = rng.standard_normal((E, d))
        W1, W3, W2, b1, b2 = _weights(rng, E, d, H, act == "swiglu", False)
        inp = dict(x=x, Wg=Wg, W1=W1, W3=W3, W2=W2)
        r = o.moe_forward(inp, k=k, c=c, act=act)
        C = -(-(c.numerator * k * T) // (c.denominator * E))
        lg = torch.from_numpy(x) @ torch.from_numpy(Wg).T
        top = torch.sort(lg, dim=1, descending=True, stable=True).indices[:, :k]
        pr = torch.softmax(lg, dim=1)
        w = torch.gather(pr, 1, top)
        w = w / w.sum(dim=1, keepdim=True)
        flat_e = top.reshape(-1)
        flat_w = w.reshape(-1)
        flat_t = torch.arange(T).repeat_interleave(k)
        srt, order = torch.sort(flat_e, stable=True)
        out = torch.zeros(T, d, dtype=torch.float64)
        start = 0
        for e in range(E):
            n = int((srt == e).sum())
            seg = order[start:start + min(n, C)]
            start += n
            if len(seg) == 0:
                continue
            toks = flat_t[seg]
            ye = _torch_ffn(x[toks.numpy()], W1[e], None if W3 is None else W3[e],
                            W2[e], None, None, act)
            out.index_add_(0, toks, torch.from_numpy(ye) * flat_w[seg, None])
        np.testing.assert_allclose(r["y"], out.numpy(), rtol=0, atol=1e-12)


def pin_dropped_tokens_zero(o):
    """With W_g = 0 and C < T, tokens t >= C lose all k slots: y_t = 0 and
    they never appear among the packed rows."""
    rng = _rng(8)
    T, d, H, E, k = 12, 6, 10, 4, 2
    x = rng.standard_normal((T, d))
    W1, W3, W2, b1, b2 = _weights(rng, E, d, H, False, True)
    inp = dict(x=x, Wg=np.zeros((E, d)), W1=W1, W2=W2, b1=b1, b2=b2)
    c = Fraction(5, 6)            # C = ceil(5/6 * 2 * 12 / 4) = 5
    r = o.moe_forward(inp, k=k, c=c, act="gelu")
    assert r["C"] == 5
    assert (r["y"][5:] == 0).all()
    assert (np.abs(r["y"][:5]).sum(axis=1) > 0).all()
    assert set(r["token_of_row"].tolist()) == set(range(5))
    assert r["dropped"] == k * (T - 5)


def pin_combine_rows_is_layer_output(o):
    """The combine step alone, fed the packed expert outputs, equals the
    layer's y (y = sum_j g_j E_{K_j}(x) with dropped slots masked; kwkr.cn MoE
    article, sections 2.1 and 2.3). The layer's y is pinned independently by
    the dense-masked loop and the sort-based restatement, so a combine that
    ignores the gates, keeps dropped slots or reads the wrong packed row fails
    here. Cases with drops, k = 2 and k = 3, and one token-ordered tie so that
    dropped and kept slots sit side by side."""
    rng = _rng(12)
    for act, T, E, k, c in (("gelu", 37, 5, 2, Fraction(3, 5)),
                            ("swiglu", 29, 6, 3, Fraction(1, 2)),
                            ("gelu", 16, 4, 2, Fraction(1, 4))):
        d, H = 9, 13
        x = rng.standard_normal((T, d))
        Wg = rng.standard_normal((E, d))
        W1, W3, W2, b1, b2 = _weights(rng, E, d, H, act == "swiglu", act == "gelu")
        inp = dict(x=x, Wg=Wg, W1=W1, W3=W3, W2=W2, b1=b1, b2=b2)
        r = o.moe_forward(inp, k=k, c=c, act=act)
        assert r["dropped"] > 0 and (r["slot_of"] >= 0).any()
        off = r["offset"]
        Yrows = np.zeros((int(off[-1]), d))
        for e in range(E):
            a, b = int(off[e]), int(off[e + 1])
            if b > a:
                toks = r["token_of_row"][a:b]
                Yrows[a:b] = _torch_ffn(x[toks], W1[e], None if W3 is None else W3[e], W2[e],
                                        None if b1 is None else b1[e],
                                        None if b2 is None else b2[e], act)
        y = o.combine_rows(Yrows, r["slot_of"], r["gates"])
        np.testing.assert_allclose(y, r["y"], rtol=0, atol=1e-12)
        dead = (r["slot_of"] < 0).all(axis=1)
        assert (y[dead] == 0).all()


# ---------------------------------------------------------------- std-scaled router noise
# kwkr.cn MoE article, section 3.3: the router noise strength follows the
# standard deviation of the current logits instead of a fixed scale.
def pin_std_noise_two_experts_closed_form(o):
    """E = 2: the population std of a token's two logits is |z0 - z1| / 2, so
    the keys are (z + s |z0 - z1| / 2 n) / tau (z from F.linear, tau != 1)."""
    rng = _rng(21)
    T, d, s, tau = 50, 7, 0.3, 2.0
    x = rng.standard_normal((T, d))
    Wg = rng.standard_normal((2, d))
    b = rng.standard_normal(2)
    n = rng.standard_normal((T, 2))
    z = F.linear(torch.from_numpy(x), torch.from_numpy(Wg), torch.from_numpy(b)).numpy()
    half = np.abs(z[:, 0] - z[:, 1])[:, None] / 2.0
    want = (z + s * half * n) / tau
    got = o.router_logits(x, Wg, b, n, tau, noise_scale=s)
    np.testing.assert_allclose(got, want, rtol=1e-13, atol=1e-13)


def pin_std_noise_follows_logit_scale(o):
    """Scaling the tokens by a > 0 scales every key by a (bias 0, tau 1), so
    the routing does not change: the noise grows with the logits. A fixed-scale
    noise would not satisfy this."""
    rng = _rng(22)
    T, d, E, k = 64, 12, 6, 2
    x = rng.standard_normal((T, d))
    Wg = rng.standard_normal((E, d))
    n = rng.standard_normal((T, E))
    base = o.router_logits(x, Wg, None, n, 1.0, noise_scale=0.5)
    for a in (0.25, 3.0, 40.0):
        got = o.router_logits(a * x, Wg, None, n, 1.0, noise_scale=0.5)
        np.testing.assert_allclose(got, a * base, rtol=1e-12, atol=1e-12)
        assert np.array_equal(o.topk_ids(got, k), o.topk_ids(base, k))


def pin_std_noise_shift(o):
    """A common shift c of every expert's bias leaves each token's std
    unchanged, so every key moves by exactly c / tau."""
    rng = _rng(23)
    T, d, E, tau, c = 40, 9, 5, 1.5, 0.75
    x = rng.standard_normal((T, d))
    Wg = rng.standard_normal((E, d))
    b = rng.standard_normal(E)
    n = rng.standard_normal((T, E))
    k0 = o.router_logits(x, Wg, b, n, tau, noise_scale=0.2)
    k1 = o.router_logits(x, Wg, b + c, n, tau, noise_scale=0.2)
    np.testing.assert_allclose(k1 - k0, c / tau, rtol=0, atol=1e-12)


def pin_std_noise_flat_logits_get_none(o):
    """W_g = 0, no bias: every token's logits are equal, the std is 0, so
    the noise vanishes and every token takes experts 0..k-1 (ties to the lower
    index) with gates 1/k; with noise_scale = 0 the same noise would be added
    as given."""
    rng = _rng(24)
    T, d, E, k = 20, 5, 4, 2
    x = rng.standard_normal((T, d))
    n = rng.standard_normal((T, E))
    l = o.router_logits(x, np.zeros((E, d)), None, n, 1.0, noise_scale=0.7)
    assert (l == 0).all()
    r = o.route_from_logits(l, k, T)
    assert (r["ids"] == np.arange(k)[None, :]).all()
    np.testing.assert_allclose(r["gates"], 1.0 / k, rtol=0, atol=1e-15)
    l0 = o.router_logits(x, np.zeros((E, d)), None, n, 1.0, noise_scale=0.0)
    np.testing.assert_allclose(l0, n, rtol=0, atol=0)


def pin_activations_match_library(o):
    u = np.linspace(-8, 8, 1001)
    ut = torch.from_numpy(u)
    np.testing.assert_allclose(o.gelu(u), F.gelu(ut).numpy(), rtol=0, atol=1e-15)
    np.testing.assert_allclose(o.silu(u), F.silu(ut).numpy(), rtol=0, atol=1e-14)


def pin_router_logits(o):
    rng = _rng(9)
    x = rng.standard_normal((9, 7))
    Wg = rng.standard_normal((5, 7))
    b = rng.standard_normal(5)
    g = rng.standard_normal((9, 5))
    got = o.router_logits(x, Wg, b, g, tau=0.5)
    want = (F.linear(torch.from_numpy(x), torch.from_numpy(Wg),
                     torch.from_numpy(b)).numpy() + g) / 0.5
    np.testing.assert_allclose(got, want, rtol=1e-14, atol=1e-14)
    # bf16 inputs are taken at their exact values
    xb = torch.from_numpy(x).to(torch.bfloat16)
    got = o.router_logits(xb, Wg)
    want = xb.double().numpy() @ Wg.T
    np.testing.assert_allclose(got, want, rtol=1e-14, atol=1e-14)


def _shared(rng, d, Hs, act):
    W1 = rng.standard_normal((Hs, d)) / math.sqrt(d)
    W3 = rng.standard_normal((Hs, d)) / math.sqrt(d) if act == "swiglu" else None
    W2 = rng.standard_normal((d, Hs)) / math.sqrt(Hs)
    b1 = rng.standard_normal(Hs) * 0.1 if act == "gelu" else None
    b2 = rng.standard_normal(d) * 0.1 if act == "gelu" else None
    return dict(W1=W1, W3=W3, W2=W2, b1=b1, b2=b2)


def pin_shared_expert_alone(o):
    """Routed experts with W2 = 0 (and no b2) contribute nothing, so the layer
    is exactly the shared expert as a dense FFN."""
    rng = _rng(12)
    for act in ("gelu", "swiglu"):
        T, d, H, Hs, E, k = 29, 10, 12, 18, 4, 2
        x = rng.standard_normal((T, d))
        W1, W3, W2, _, _ = _weights(rng, E, d, H, act == "swiglu", False)
        inp = dict(x=x, Wg=rng.standard_normal((E, d)), W1=W1, W3=W3, W2=np.zeros_like(W2))
        sh = _shared(rng, d, Hs, act)
        r = o.moe_forward(inp, k=k, c=Fraction(1, 2), act=act, shared=sh)
        want = _torch_ffn(x, sh["W1"], sh["W3"], sh["W2"], sh["b1"], sh["b2"], act)
        np.testing.assert_allclose(r["y"], want, rtol=0, atol=1e-12)


def pin_shared_expert_equal_to_single_routed(o):
    """E = 1, k = 1, no drops and a shared expert with the routed expert's
    weights: y = 2 FFN(x). Fully dropped tokens (C < T) keep the shared term."""
    rng = _rng(13)
    T, d, H = 21, 8, 14
    x = rng.standard_normal((T, d))
    W1, W3, W2, b1, b2 = _weights(rng, 1, d, H, False, True)
    inp = dict(x=x, Wg=rng.standard_normal((1, d)), W1=W1, W2=W2, b1=b1, b2=b2)
    sh = dict(W1=W1[0], W2=W2[0], b1=b1[0], b2=b2[0])
    dense = _torch_ffn(x, W1[0], None, W2[0], b1[0], b2[0], "gelu")
    r = o.moe_forward(inp, k=1, c=1, act="gelu", shared=sh)
    np.testing.assert_allclose(r["y"], 2 * dense, rtol=0, atol=1e-12)
    r = o.moe_forward(inp, k=1, c=Fraction(1, 3), act="gelu", shared=sh)   # C = 7
    np.testing.assert_allclose(r["y"][:7], 2 * dense[:7], rtol=0, atol=1e-12)
    np.testing.assert_allclose(r["y"][7:], dense[7:], rtol=0, atol=1e-12)


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(ORC)


# ---------------------------------------------------------------- mutants
def _mutants():
    o = ORC
    m = {}
    m["capacity_floor"] = ("capacity", lambda c, k, T, E: math.floor(Fraction(c) * k * T / E))
    m["capacity_int_plus_one"] = ("capacity", lambda c, k, T, E: int(float(c) * T * k / E) + 1)

    def topk_high_tie(l, k, chunk=4096):
        l = np.asarray(l)
        rev = o.__dict__["_orig_topk"](l[:, ::-1].copy(), k)
        return (l.shape[1] - 1 - rev).astype(np.int32)
    m["topk_tie_to_higher"] = ("topk_ids", topk_high_tie)

    def topk_ascending(l, k, chunk=4096):
        return o.__dict__["_orig_topk"](l, k)[:, ::-1].copy()
    m["topk_slot_order_reversed"] = ("topk_ids", topk_ascending)
    m["gates_not_renormalised"] = ("renormalised_gates",
                                   lambda p, ids: np.take_along_axis(np.asarray(p), ids.astype(np.int64), 1))

    def gates_eps(p, ids):
        s = np.take_along_axis(np.asarray(p), ids.astype(np.int64), 1)
        return s / (s.sum(1, keepdims=True) + 1e-6)
    m["gates_epsilon"] = ("renormalised_gates", gates_eps)

    def disp_late_wins(ids, E, C):
        T = ids.shape[0]
        r = o.__dict__["_orig_dispatch"](ids[::-1], E, C)
        # map back: later tokens now have priority
        out = dict(r)
        out["slot_of"] = r["slot_of"][::-1]
        out["pos"] = r["pos"][::-1]
        out["token_of_row"] = np.where(r["token_of_row"] >= 0, T - 1 - r["token_of_row"], -1)
        return out
    m["dispatch_later_tokens_win"] = ("dispatch", disp_late_wins)

    def disp_inclusive(ids, E, C):
        r = o.__dict__["_orig_dispatch"](ids, E, C)
        out = dict(r)
        pos = r["pos"] + 1
        off = r["offset"]
        out["pos"] = pos
        out["slot_of"] = np.where(pos < C, off[ids] + pos, -1).astype(np.int32)
        return out
    m["dispatch_pos_inclusive"] = ("dispatch", disp_inclusive)

    def aux_f_over_T(p, count, kept, k):
        a = o.__dict__["_orig_aux"](p, count, kept, k)
        p = np.asarray(p)
        f = np.asarray(count, float) / p.shape[0]
        return dict(a, f=f, L=p.shape[1] * float((f * a["P"]).sum()))
    m["aux_f_over_T"] = ("aux_stats", aux_f_over_T)

    def aux_no_E(p, count, kept, k):
        a = o.__dict__["_orig_aux"](p, count, kept, k)
        return dict(a, L=a["L"] / np.asarray(p).shape[1])
    m["aux_missing_E"] = ("aux_stats", aux_no_E)

    def aux_f_after_drop(p, count, kept, k):
        a = o.__dict__["_orig_aux"](p, kept, kept, k)
        return a
    m["aux_f_after_drops"] = ("aux_stats", aux_f_after_drop)
    m["gelu_tanh"] = ("gelu", lambda u: 0.5 * u * (1 + np.tanh(math.sqrt(2 / math.pi) * (u + 0.044715 * u ** 3))))
    m["silu_sign"] = ("silu", lambda u: u / (1.0 + np.exp(u)))

    def ffn_swap13(xr, W1e, W2e, W3e=None, b1e=None, b2e=None, act="gelu"):
        if act == "swiglu":
            return o.__dict__["_orig_ffn"](xr, W3e, W2e, W1e, b1e, b2e, act)
        return o.__dict__["_orig_ffn"](xr, W1e, W2e, W3e, b1e, b2e, act)
    m["swiglu_W1_W3_swapped"] = ("expert_ffn_rows", ffn_swap13)

    def ffn_no_b2(xr, W1e, W2e, W3e=None, b1e=None, b2e=None, act="gelu"):
        return o.__dict__["_orig_ffn"](xr, W1e, W2e, W3e, b1e, None, act)
    m["ffn_drops_b2"] = ("expert_ffn_rows", ffn_no_b2)

    def logits_no_bias(x, Wg, bias=None, noise=None, tau=1.0, noise_scale=0.0):
        return o.__dict__["_orig_logits"](x, Wg, None, noise, tau, noise_scale)
    m["router_drops_bias"] = ("router_logits", logits_no_bias)

    def logits_tau_mul(x, Wg, bias=None, noise=None, tau=1.0, noise_scale=0.0):
        return o.__dict__["_orig_logits"](x, Wg, bias, noise, 1.0, noise_scale) * tau
    m["router_tau_multiplies"] = ("router_logits", logits_tau_mul)

    def combine_no_gate(tokens, x, ids, gates, slot_of, *a, **kw):
        return o.__dict__["_orig_combine"](tokens, x, ids, np.ones_like(np.asarray(gates, float)), slot_of, *a, **kw)
    m["combine_ignores_gates"] = ("combine_tokens", combine_no_gate)

    def combine_keeps_dropped(tokens, x, ids, gates, slot_of, *a, **kw):
        return o.__dict__["_orig_combine"](tokens, x, ids, gates, np.abs(np.asarray(slot_of)), *a, **kw)
    m["combine_keeps_dropped"] = ("combine_tokens", combine_keeps_dropped)

    def combine_rows_no_gate(Yrows, slot_of, gates):
        return o.__dict__["_orig_combine_rows"](Yrows, slot_of,
                                                np.ones_like(np.asarray(gates, float)))
    m["combine_rows_ignores_gates"] = ("combine_rows", combine_rows_no_gate)

    def combine_rows_keeps_dropped(Yrows, slot_of, gates):
        return o.__dict__["_orig_combine_rows"](Yrows, np.abs(np.asarray(slot_of)), gates)
    m["combine_rows_keeps_dropped"] = ("combine_rows", combine_rows_keeps_dropped)

    def combine_rows_next_row(Yrows, slot_of, gates):
        s = np.asarray(slot_of)
        n = np.asarray(Yrows).shape[0]
        return o.__dict__["_orig_combine_rows"](Yrows, np.where(s >= 0, (s + 1) % n, s), gates)
    m["combine_rows_wrong_row"] = ("combine_rows", combine_rows_next_row)

    def std_over_tokens(z):
        z = np.asarray(z, dtype=np.float64)
        return np.broadcast_to(z.std(axis=0).mean(), (z.shape[0],)).copy()
    m["noise_std_over_tokens"] = ("logit_std", std_over_tokens)
    m["noise_std_sample_ddof1"] = ("logit_std", lambda z: np.asarray(z, float).std(axis=1, ddof=1))
    m["noise_variance_not_std"] = ("logit_std", lambda z: np.asarray(z, float).var(axis=1))

    def logits_noise_not_over_tau(x, Wg, bias=None, noise=None, tau=1.0, noise_scale=0.0):
        l = o.__dict__["_orig_logits"](x, Wg, bias, None, tau, 0.0)
        if noise is None:
            return l
        if not noise_scale:
            return l + o.as_f64(noise) / tau
        z = l * tau
        return l + noise_scale * o.logit_std(z)[:, None] * o.as_f64(noise)
    m["noise_not_divided_by_tau"] = ("router_logits", logits_noise_not_over_tau)

    def softmax_no_max_over_wrong_axis(l):
        e = np.exp(np.asarray(l, float))
        return e / e.sum(axis=0, keepdims=True)
    m["softmax_wrong_axis"] = ("softmax", softmax_no_max_over_wrong_axis)

    def shared_missing(xr, shared, act):
        return 0.0 * o.__dict__["_orig_shared"](xr, shared, act)
    m["shared_expert_dropped"] = ("shared_expert_rows", shared_missing)

    def shared_halved(xr, shared, act):
        return 0.5 * o.__dict__["_orig_shared"](xr, shared, act)
    m["shared_expert_weight_half"] = ("shared_expert_rows", shared_halved)
    return m


MUTANTS = _mutants()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistakes_are_caught(name, monkeypatch):
    o = ORC
    originals = dict(_orig_topk=o.topk_ids, _orig_dispatch=o.dispatch,
                     _orig_aux=o.aux_stats, _orig_ffn=o.expert_ffn_rows,
                     _orig_logits=o.router_logits, _orig_combine=o.combine_tokens,
                     _orig_shared=o.shared_expert_rows, _orig_combine_rows=o.combine_rows)
    for k, v in originals.items():
        monkeypatch.setattr(o, k, v, raising=False)
    attr, bad = MUTANTS[name]
    monkeypatch.setattr(o, attr, bad)
    failed = []
    for pin in ALL_PINS:
        try:
            pin(o)
        except Exception:   # an assertion, or a shape error from a wrong operand
            failed.append(pin.__name__)
    assert failed, f"planted mistake {name} passed every pin"


def test_combine_rows_and_balance_helpers():
    """The stage-level helpers agree with the layer-level functions."""
    rng = _rng(11)
    T, E, k, d = 30, 5, 2, 4
    l = rng.standard_normal((T, E))
    r = ORC.route_from_logits(l, k, 10)
    Yrows = rng.standard_normal((int(r["offset"][-1]), d))
    y = ORC.combine_rows(Yrows, r["slot_of"], r["gates"])
    for t in range(T):
        want = np.zeros(d)
        for j in range(k):
            if r["slot_of"][t, j] >= 0:
                want += r["gates"][t, j] * Yrows[r["slot_of"][t, j]]
        np.testing.assert_allclose(y[t], want, rtol=0, atol=1e-14)
    b = ORC.balance_from_sums(r["count"], r["p"].sum(axis=0), T, k, r["kept"])
    assert abs(b["L"] - r["L"]) < 1e-15 and b["dropped"] == r["dropped"]
