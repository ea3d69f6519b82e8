"""CPU oracle for the forward pass of one top-k routed MoE FFN layer.

TEST INFRASTRUCTURE ONLY. Nothing in the product path imports this module:
only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` call it. It shares no code with the
CUDA library and never reads anything the CUDA path produced except where a
function says so (``route_from_logits`` takes the GPU's fp32 logits, so that
routing decisions are compared on the same keys).

Every step is written out from its definition in fp64 (numpy; scipy's
``erf`` for GELU). Source of the method - the pages are cited by title and
section:

* [MoE-math] kwkr.cn, "MoE sparse activation: from the math to the code"
  (the page's title was lost in extraction), sections 2.1-2.3 and 3.1-3.2:
  the gate softmax, top-k on the logits, renormalisation of the k chosen
  probabilities, y = sum_{i in K(x)} g_i(x) E_i(x), the load-balance statistic
  L_balance = E * sum_i f_i P_i and the capacity C = ceil(c k T / E).
* [MoE-tutorial] intelliparadigm.com, "MoE模型：动态计算架构解析与实践指南",
  section 2.1 (DenseExpert: Linear -> GELU -> Linear) and section 2.3
  (the k=1 load-balancing loss).
* [MoE-guide] lpnh.cn, "Mixture of Experts（MoE）原理与工程落地全指南",
  sections 2.2 and 3.3 (Gumbel noise added to the logits before the softmax,
  temperature division).

Readings where the pages are silent or disagree (the section each reading
rests on is named with it):

* Selection is on the logits, ties go to the lower expert index, and the k
  chosen experts are ordered by descending logit ([MoE-math] 2.1 says to pick
  on logits; no page states a tie rule).
* No epsilon in the renormalisation denominator (the text says the k weights
  sum to one; the denominator is >= 1/E > 0).
* One key l = (x W_g^T + b + g) / tau drives selection, gates and P_i.
* Capacity is the closed form of [MoE-math] 2.3, evaluated in exact rational
  arithmetic.
* Std-scaled router noise ([MoE-math] 3.3: the noise strength follows the
  logits' standard deviation rather than a fixed scale) uses each token's own
  population standard deviation over its E pre-noise logits (bias included).
* Drop priority is token order (the stable sort of [MoE-math] 3.2): a slot
  (t, j) of expert e is kept iff fewer than C earlier tokens chose e. Dropped
  slots are not re-routed and the surviving gates are not renormalised again.
* f_i = count_i / (k T) with count_i taken before drops, so sum_i f_i = 1 and
  uniform routing gives L_balance = 1, as [MoE-math] 2.2 states.
* A token whose k slots are all dropped gets y = 0 (the layer adds no residual).
* GELU is the exact erf form; SwiGLU is W2 (silu(W1 x) * (W3 x)), no biases.
* A shared expert (the lpnh.cn guide, section 4.10, routes out-of-distribution
  tokens to one) is read as an expert of the same FFN form that every token
  passes through with weight 1, added to the routed sum and untouched by
  capacity and drops.

Parity status of each function is stated in its docstring; all are pinned by
the CPU tests in ``tests/test_oracle.py``.
"""
from __future__ import annotations

import math
from fractions import Fraction

import numpy as np
from scipy.special import erf as _erf


def as_f64(a):
    """Marshal an input (numpy array or CPU torch tensor of any float type,
    bf16 included) to a float64 numpy array. Conversion only, no arithmetic."""
    if a is None:
        return None
    if hasattr(a, "detach"):  # torch tensor
        import torch
        return a.detach().to("cpu", torch.float64).numpy()
    return np.asarray(a, dtype=np.float64)


# --------------------------------------------------------------------------
# capacity  ([MoE-math] 2.3)
# --------------------------------------------------------------------------
def capacity(c, k: int, T: int, E: int) -> int:
    """C = ceil(c * k * T / E), exact: c is taken as the rational value of
    the given number (a float's exact binary value, or a Fraction).
    Pinned: the five workload values and a rational grid (tests)."""
    q = Fraction(c) * k * T / E
    return math.ceil(q)


# --------------------------------------------------------------------------
# router  ([MoE-math] 2.1, 3.2; [MoE-guide] 3.3 for bias/noise/temperature)
# --------------------------------------------------------------------------
def router_logits(x, Wg, bias=None, noise=None, tau: float = 1.0,
                  noise_scale: float = 0.0):
    """l[t,i] = (z[t,i] + g[t,i]) / tau with z[t,i] = sum_j x[t,j] Wg[i,j] + b_i,
    fp64. Wg is stored [E, d] (nn.Linear convention of the gate in
    [MoE-math] 3.2).

    The noise: with noise_scale == 0 it is added as given, g = noise (a fixed
    strength, or Gumbel noise: [MoE-guide] 3.3). With noise_scale > 0 its
    strength follows the token's own logits, as [MoE-math] 3.3 recommends
    over a fixed scale: g[t,i] = noise_scale * std_t * noise[t,i], where std_t
    is the population standard deviation of z[t, :] over the E experts (the
    logits before the noise; bias included)."""
    x = as_f64(x)
    Wg = as_f64(Wg)
    z = x @ Wg.T
    if bias is not None:
        z = z + as_f64(bias)[None, :]
    if noise is not None:
        n = as_f64(noise)
        if noise_scale:
            z = z + float(noise_scale) * logit_std(z)[:, None] * n
        else:
            z = z + n
    return z / float(tau)


def logit_std(z):
    """Population standard deviation of each row: sqrt(mean_i (z_i - mean z)^2).
    Pinned: the two-expert closed form |z_0 - z_1| / 2 and the scale and
    shift behaviour of the std-scaled router noise (tests)."""
    z = np.asarray(z, dtype=np.float64)
    m = z.mean(axis=1, keepdims=True)
    return np.sqrt(((z - m) ** 2).mean(axis=1))


def softmax(l):
    """p[t,i] = exp(l_i - max_j l_j) / sum_m exp(l_m - max_j l_j)."""
    l = np.asarray(l, dtype=np.float64)
    m = l.max(axis=1, keepdims=True)
    e = np.exp(l - m)
    return e / e.sum(axis=1, keepdims=True)


def topk_ids(l, k: int, chunk: int = 4096):
    """Top-k on the keys l by rank: rank_i = #{j : l_j > l_i or (l_j == l_i and
    j < i)}; expert i is chosen iff rank_i < k and sits in slot rank_i.

    ``l`` may be fp32 (the GPU's logits) or fp64: comparisons are exact in
    either. Returns ids [T,k] int32."""
    l = np.asarray(l)
    T, E = l.shape
    ids = np.empty((T, k), dtype=np.int32)
    idx = np.arange(E)
    lower = idx[None, :] < idx[:, None]          # [i, j]: j < i
    for s in range(0, T, chunk):
        lc = l[s:s + chunk]                      # [t, E]
        li = lc[:, :, None]                      # l_i
        lj = lc[:, None, :]                      # l_j
        beats = (lj > li) | ((lj == li) & lower[None, :, :])
        rank = beats.sum(axis=2)                 # [t, E]
        t_idx, i_idx = np.nonzero(rank < k)
        ids[s + t_idx, rank[t_idx, i_idx]] = i_idx
    return ids


def renormalised_gates(p, ids):
    """g[t,j] = p[t, K_j] / sum_m p[t, K_m] ("second normalisation",
    [MoE-math] 2.1)."""
    p = np.asarray(p, dtype=np.float64)
    sel = np.take_along_axis(p, ids.astype(np.int64), axis=1)
    return sel / sel.sum(axis=1, keepdims=True)


# --------------------------------------------------------------------------
# dispatch  ([MoE-math] 2.3 and the stable sort of 3.2)
# --------------------------------------------------------------------------
def dispatch(ids, E: int, C: int):
    """Capacity-limited, token-order dispatch.

    count_e = #{(t,j): K_j(t) = e}; pos(t,j) = #{t' < t : K_j(t) in K(t')};
    keep iff pos < C; kept_e = min(count_e, C); off_e = sum_{e'<e} kept_e';
    slot_of[t,j] = off_e + pos or -1; token_of_row[off_e + pos] = t.
    Returns a dict of int arrays."""
    ids = np.asarray(ids)
    T, k = ids.shape
    chosen = np.zeros((T, E), dtype=np.int64)          # chosen[t,e] in {0,1}
    np.put_along_axis(chosen, ids.astype(np.int64), 1, axis=1)
    count = chosen.sum(axis=0)                          # [E]
    before = np.cumsum(chosen, axis=0) - chosen         # earlier tokens, [T,E]
    pos = np.take_along_axis(before, ids.astype(np.int64), axis=1)   # [T,k]
    kept = np.minimum(count, C)
    offset = np.zeros(E + 1, dtype=np.int64)
    offset[1:] = np.cumsum(kept)
    keep = pos < C
    slot_of = np.where(keep, offset[ids] + pos, -1)
    token_of_row = np.full(int(offset[E]), -1, dtype=np.int64)
    t_idx, j_idx = np.nonzero(keep)
    token_of_row[slot_of[t_idx, j_idx]] = t_idx
    return dict(count=count.astype(np.int32), kept=kept.astype(np.int32),
                offset=offset.astype(np.int32), pos=pos.astype(np.int32),
                slot_of=slot_of.astype(np.int32),
                token_of_row=token_of_row.astype(np.int32))


# --------------------------------------------------------------------------
# experts  ([MoE-math] 3.1; [MoE-tutorial] 2.1; SwiGLU by its usual definition)
# --------------------------------------------------------------------------
def gelu(u):
    """Exact GELU: u/2 * (1 + erf(u / sqrt 2))."""
    return 0.5 * u * (1.0 + _erf(u / math.sqrt(2.0)))


def silu(u):
    """u / (1 + exp(-u))."""
    return u / (1.0 + np.exp(-u))


def expert_ffn_rows(xr, W1e, W2e, W3e=None, b1e=None, b2e=None, act="gelu"):
    """One expert on rows xr [n, d]:
    GELU   : W2 gelu(W1 x + b1) + b2
    SwiGLU : W2 (silu(W1 x) * (W3 x))
    Weights in [out, in] storage. fp64."""
    xr = as_f64(xr)
    W1e = as_f64(W1e)
    W2e = as_f64(W2e)
    u = xr @ W1e.T
    if act == "gelu":
        if b1e is not None:
            u = u + as_f64(b1e)[None, :]
        h = gelu(u)
    elif act == "swiglu":
        v = xr @ as_f64(W3e).T
        h = silu(u) * v
    else:
        raise ValueError(act)
    yr = h @ W2e.T
    if act == "gelu" and b2e is not None:
        yr = yr + as_f64(b2e)[None, :]
    return yr


def combine_tokens(tokens, x, ids, gates, slot_of, W1, W2, W3=None, b1=None,
                   b2=None, act="gelu"):
    """y_t = sum over kept slots j of g[t,j] * E_{K_j(t)}(x_t), for the listed
    tokens only (rows in the order of ``tokens``); y_t = 0 if all slots of t
    were dropped ([MoE-math] 2.1 and 2.3). Expert weights are converted to
    fp64 one expert at a time."""
    tokens = np.asarray(tokens, dtype=np.int64)
    d = x.shape[1]
    y = np.zeros((len(tokens), d), dtype=np.float64)
    sub_ids = np.asarray(ids)[tokens]
    sub_keep = np.asarray(slot_of)[tokens] >= 0
    sub_g = np.asarray(gates, dtype=np.float64)[tokens]
    for e in np.unique(sub_ids[sub_keep]):
        r, j = np.nonzero((sub_ids == e) & sub_keep)
        xr = as_f64(x[tokens[r]])
        ye = expert_ffn_rows(
            xr, W1[e], W2[e], None if W3 is None else W3[e],
            None if b1 is None else b1[e], None if b2 is None else b2[e], act)
        # accumulate in slot order j = 0..k-1 for each token
        for jj in range(sub_ids.shape[1]):
            m = j == jj
            y[r[m]] += sub_g[r[m], jj][:, None] * ye[m]
    return y


# --------------------------------------------------------------------------
# load-balance statistics  ([MoE-math] 2.2; drop count per [MoE-math] 6.2)
# --------------------------------------------------------------------------
def aux_stats(p, count, kept, k: int):
    """f_i = count_i / (k T) (before drops), P_i = (1/T) sum_t p[t,i],
    L_balance = E * sum_i f_i P_i, dropped = k T - sum_i kept_i."""
    p = np.asarray(p, dtype=np.float64)
    T = p.shape[0]
    return balance_from_sums(count, p.sum(axis=0), T, k, kept)


def balance_from_sums(count, prob_sum, T: int, k: int, kept):
    """The same statistics from per-expert sums: f_i = count_i / (k T),
    P_i = prob_sum_i / T, L_balance = E sum_i f_i P_i, dropped = kT - sum kept."""
    f = np.asarray(count, dtype=np.float64) / float(k * T)
    P = np.asarray(prob_sum, dtype=np.float64) / float(T)
    E = f.shape[0]
    L = float(E) * float((f * P).sum())
    dropped = int(k * T - int(np.asarray(kept, dtype=np.int64).sum()))
    return dict(f=f, P=P, L=L, dropped=dropped)


def combine_rows(Yrows, slot_of, gates):
    """Combine step alone: y_t = sum over j with slot_of[t,j] >= 0 of
    g[t,j] * Yrows[slot_of[t,j]] (fp64), y_t = 0 if no slot was kept.
    Pinned: fed the packed outputs of each expert on its kept rows, it
    reproduces the layer's y, which the dense-masked loop and the sort-based
    restatement pin on their own (tests)."""
    Yrows = as_f64(Yrows)
    slot_of = np.asarray(slot_of)
    gates = np.asarray(gates, dtype=np.float64)
    T, k = slot_of.shape
    y = np.zeros((T, Yrows.shape[1]), dtype=np.float64)
    for j in range(k):
        keep = slot_of[:, j] >= 0
        y[keep] += gates[keep, j][:, None] * Yrows[slot_of[keep, j]]
    return y


# --------------------------------------------------------------------------
# whole layer
# --------------------------------------------------------------------------
def route_from_logits(l, k: int, C: int):
    """Routing steps from given keys (fp32 GPU logits or fp64 oracle logits):
    softmax, top-k, renormalised gates, dispatch, aux statistics."""
    l = np.asarray(l)
    T, E = l.shape
    p = softmax(l.astype(np.float64))
    ids = topk_ids(l, k)
    g = renormalised_gates(p, ids)
    disp = dispatch(ids, E, C)
    aux = aux_stats(p, disp["count"], disp["kept"], k)
    return dict(logits=l, p=p, ids=ids, gates=g, **disp, **aux)


def shared_expert_rows(xr, shared: dict, act: str):
    """The shared expert on rows xr: the same FFN form as a routed expert
    (weights W1 [Hs, d], W3 [Hs, d] for SwiGLU, W2 [d, Hs], optional b1, b2
    for GELU), applied to every token with weight 1."""
    return expert_ffn_rows(xr, shared["W1"], shared["W2"], shared.get("W3"),
                           shared.get("b1"), shared.get("b2"), act)


def moe_forward(inp: dict, k: int, c, act: str, tau: float = 1.0,
                tokens=None, logits=None, shared=None, noise_scale: float = 0.0):
    """The layer: router -> softmax -> top-k -> gates -> dispatch -> experts ->
    combine -> aux statistics.

    ``inp`` holds x, Wg, W1, W3, W2, b1, b2, bias, noise (workload inputs).
    ``logits``: if given (the GPU's fp32 logits), routing follows them;
    otherwise the oracle's own fp64 logits are used.
    ``tokens``: if given, y is computed only for those tokens (routing is
    always computed for the whole batch, since capacity couples tokens).
    ``shared``: optional shared-expert weights (see shared_expert_rows),
    added with weight 1 to every token's output.
    ``noise_scale``: > 0 scales the router noise by each token's logit
    standard deviation (see router_logits).
    Returns the routing dict plus y [len(tokens) or T, d]."""
    x = inp["x"]
    T = x.shape[0]
    E = inp["Wg"].shape[0]
    C = capacity(c, k, T, E)
    if logits is None:
        logits = router_logits(x, inp["Wg"], inp.get("bias"), inp.get("noise"),
                               tau, noise_scale)
    r = route_from_logits(logits, k, C)
    r["C"] = C
    tok = np.arange(T) if tokens is None else np.asarray(tokens)
    r["tokens"] = tok
    r["y"] = combine_tokens(tok, x, r["ids"], r["gates"], r["slot_of"],
                            inp["W1"], inp["W2"], inp.get("W3"), inp.get("b1"),
                            inp.get("b2"), act)
    if shared is not None:
        r["y"] = r["y"] + shared_expert_rows(as_f64(x[tok]), shared, act)
    return r
