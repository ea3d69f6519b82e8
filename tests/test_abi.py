"""CPU checks of the C-ABI library: it loads, exports every call that
include/moe.h declares, computes the capacity closed form, and rejects bad
arguments on the host before touching a GPU (no compute call is made)."""
import ctypes
import os
import re
from fractions import Fraction

import pytest

from mixture_experts_layer_99_b300 import moe
from oracle import moe_oracle as ORC

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    syms = set()
    for name in os.listdir(os.path.join(ROOT, "include")):
        if name.endswith(".h"):
            text = open(os.path.join(ROOT, "include", name)).read()
            syms |= set(re.findall(r"MOE_API[^;(]*?\b(moe_\w+)\s*\(", text))
    return syms


def test_library_exports_every_declared_symbol():
    L = moe.lib()
    syms = declared_symbols()
    assert "moe_layer_forward" in syms and len(syms) >= 14
    for s in sorted(syms):
        assert hasattr(L, s), s
    assert set(moe.EXPORTED) <= syms


def test_checked_library_exports_the_same_symbols():
    """The checked build (index checks in the kernels) has the same ABI."""
    import ctypes as ct
    from mixture_experts_layer_99_b300 import build as B
    if B.stale(B.LIB_CHECK):   # missing, or built before the current sources
        B.build(check=True)
    L = ct.CDLL(B.LIB_CHECK)
    for s in sorted(declared_symbols()):
        assert hasattr(L, s), s
    L.moe_abi_version.restype = ct.c_int32
    assert L.moe_abi_version() == moe.lib().moe_abi_version()
    L.moe_status_string.restype = ct.c_char_p
    L.moe_status_string.argtypes = [ct.c_int32]
    assert b"check" in L.moe_status_string(6)


def test_abi_version_and_status_strings():
    L = moe.lib()
    # 1.01: moe_config_t carries noise_scale (std-scaled router noise);
    # 1.02: and flags (MOE_FLAG_KEEP_PREACT)
    assert L.moe_abi_version() == 102
    assert ctypes.sizeof(moe.Config) == 11 * 4
    for code in range(6):
        assert L.moe_status_string(code)
    assert L.moe_status_string(99) == b"unknown status"


@pytest.mark.parametrize("c,k,T,E", [(Fraction(5, 4), 2, 256, 4), (1, 1, 8192, 8),
                                     (4, 2, 16384, 8), (2, 2, 32768, 64), (32, 2, 64, 64),
                                     (Fraction(7, 3), 3, 1001, 17), (Fraction(1, 9), 1, 5, 3)])
def test_capacity_matches_oracle(c, k, T, E):
    assert moe.capacity(c, k, T, E) == ORC.capacity(c, k, T, E)


def test_capacity_rejects_bad_args():
    L = moe.lib()
    assert L.moe_capacity(0, 1, 1, 1, 1) == -1
    assert L.moe_capacity(1, 1, 1, 1, 0) == -1
    assert L.moe_capacity(1 << 40, 1, 8, 1 << 20, 1) == -1


def _cfg(**kw):
    base = dict(T=64, d=64, E=4, k=2, H=128, capacity_=40, dtype="bf16", act="gelu", tau=1.0)
    base.update(kw)
    return moe.make_config(**base)


@pytest.mark.parametrize("bad", [dict(T=0), dict(E=0), dict(k=0), dict(k=5), dict(d=60),
                                 dict(H=100), dict(capacity_=0), dict(tau=0.0),
                                 dict(tau=float("nan")), dict(d=63, dtype="f32"),
                                 dict(noise_scale=-0.1), dict(noise_scale=float("inf"))])
def test_invalid_config_rejected(bad):
    with pytest.raises(moe.MoEError) as ei:
        moe.workspace_size(_cfg(**bad))
    assert ei.value.status == 1


@pytest.mark.parametrize("bad", [dict(E=300, k=2), dict(E=16, k=9),
                                 dict(dtype="f32", keep_preact=True)])
def test_unsupported_config(bad):
    with pytest.raises(moe.MoEError) as ei:
        moe.workspace_size(_cfg(**bad))
    assert ei.value.status == 2


def test_unknown_flags_rejected():
    for bad in (2, 4, 1 << 30, -1):
        cfg = _cfg()
        cfg.flags = bad
        with pytest.raises(moe.MoEError) as ei:
            moe.workspace_size(cfg)
        assert ei.value.status == 1


@pytest.mark.parametrize("act,mult", [("gelu", 1), ("swiglu", 2)])
def test_keep_preact_workspace(act, mult):
    """The forward workspace grows by the kept pre-activations (bf16 rows of
    H, or 2H for SwiGLU); the backward workspace loses its copy of them."""
    a, b = _cfg(act=act), _cfg(act=act, keep_preact=True)
    R = min(a.T * a.k, a.E * a.capacity)
    grow = moe.workspace_size(b) - moe.workspace_size(a)
    # (regions are 256-byte aligned, and an empty one still takes 256 bytes)
    assert R * a.H * mult * 2 - 256 <= grow <= R * a.H * mult * 2 + 256
    L = moe.lib()
    na, nb = ctypes.c_size_t(0), ctypes.c_size_t(0)
    assert L.moe_workspace_size_backward(ctypes.byref(a), ctypes.byref(na)) == 0
    assert L.moe_workspace_size_backward(ctypes.byref(b), ctypes.byref(nb)) == 0
    assert na.value - nb.value >= R * a.H * mult * 2 - 256


def test_workspace_size_grows_with_shape():
    a = moe.workspace_size(_cfg())
    b = moe.workspace_size(_cfg(T=128))
    assert 0 < a < b
    assert moe.workspace_size(_cfg(), host_io=True) > a


def test_null_pointers_rejected_before_any_launch():
    L = moe.lib()
    cfg = _cfg()
    r = ctypes.byref(cfg)
    fake = ctypes.c_void_p(4096)
    # required pointers missing -> invalid argument, nothing enqueued
    assert L.moe_router_topk(r, None, fake, None, None, None, fake, fake, fake, fake, 1 << 30,
                             None) == 1
    assert L.moe_dispatch(r, fake, fake, None, fake, fake, fake, fake, fake, 1 << 30, None) == 1
    assert L.moe_combine(r, fake, None, fake, fake, None) == 1
    assert L.moe_aux_stats(r, fake, fake, fake, fake, None, fake, None) == 1
    # SwiGLU without W3, GELU with W3
    sw = _cfg(act="swiglu")
    assert L.moe_expert_ffn(ctypes.byref(sw), fake, fake, fake, None, fake, None, None, fake,
                            fake, 1 << 30, None) == 1
    assert L.moe_expert_ffn(r, fake, fake, fake, fake, fake, None, None, fake, fake, 1 << 30,
                            None) == 1
    inp = moe.LayerInputs(None, 4096, None, None, 4096, None, 4096, None, None)
    out = moe.LayerOutputs(*([4096] + [None] * 10))
    assert L.moe_layer_forward(r, ctypes.byref(inp), ctypes.byref(out), fake, 1 << 30,
                               None) == 1
    # the pipelined host call needs its three events
    full = moe.LayerInputs(None, 4096, None, None, 4096, None, 4096, None, None)
    no_ev = (ctypes.c_void_p * 3)(None, None, None)
    assert L.moe_layer_forward_host_pipelined(r, fake, ctypes.byref(full), fake, None, fake,
                                              1 << 30, None, None, None, no_ev) == 1
    assert L.moe_layer_forward_host_pipelined(r, fake, ctypes.byref(full), fake, None, fake,
                                              1 << 30, None, None, None, None) == 1


def test_workspace_checks():
    L = moe.lib()
    cfg = _cfg()
    r = ctypes.byref(cfg)
    fake = ctypes.c_void_p(4096)
    need = moe.workspace_size(cfg)
    inp = moe.LayerInputs(4096, 4096, None, None, 4096, None, 4096, None, None)
    out = moe.LayerOutputs(*([4096] + [None] * 10))
    assert L.moe_layer_forward(r, ctypes.byref(inp), ctypes.byref(out), fake, need - 1,
                               None) == 3
    assert L.moe_layer_forward(r, ctypes.byref(inp), ctypes.byref(out), ctypes.c_void_p(4100),
                               need, None) == 3
    assert L.moe_layer_forward(r, ctypes.byref(inp), ctypes.byref(out), None, need, None) == 3
    assert L.moe_router_topk(r, fake, fake, None, None, None, fake, fake, fake, fake, 16,
                             None) == 3


def test_launch_count_matches_path():
    """Kernels per moe_layer_forward: 5 (tensor-core router, k = 1: GEMM2
    writes y), 6 (tensor-core router, k > 1), +1 when the router's K range is
    split (at most 16 tiles of 128 tokens), 10 (fp32 or E > 64)."""
    from mixture_experts_layer_99_b300 import workloads as W
    L = moe.lib()
    cases = [(W.WORKLOADS["switch_top1"], 5), (W.WORKLOADS["longtail"], 6),
             (W.WORKLOADS["mixtral"], 6), (W.WORKLOADS["decode"], 6),
             (W.WORKLOADS["ref_fp32"], 10), (W.WORKLOADS["sweep_e16_k4"], 6),
             (W.small(W.WORKLOADS["switch_top1"], T=64, d=64, H=64, E=128, k=2), 10)]
    for w, want in cases:
        cfg = moe.config_from_workload(w)
        assert L.moe_layer_forward_launch_count(ctypes.byref(cfg)) == want, w.name
    bad = _cfg(T=0)
    assert L.moe_layer_forward_launch_count(ctypes.byref(bad)) == 0


def test_shared_expert_validation():
    L = moe.lib()
    cfg = _cfg(act="swiglu")
    r = ctypes.byref(cfg)
    fake = 4096
    inp = moe.LayerInputs(fake, fake, None, None, fake, fake, fake, None, None)
    out = moe.LayerOutputs(*([fake] + [None] * 10))
    ok = moe.SharedExpert(64, fake, fake, fake, None, None)
    need = moe.c_size_t(0)
    assert L.moe_workspace_size_shared(r, 64, ctypes.byref(need)) == 0
    assert need.value > moe.workspace_size(cfg)
    for bad in (moe.SharedExpert(0, fake, fake, fake, None, None),      # H = 0
                moe.SharedExpert(60, fake, fake, fake, None, None),     # H not a multiple of 8
                moe.SharedExpert(64, fake, None, fake, None, None),     # SwiGLU without W3
                moe.SharedExpert(64, fake, fake, fake, fake, None)):    # bias with SwiGLU
        assert L.moe_layer_forward_shared(r, ctypes.byref(inp), ctypes.byref(bad),
                                          ctypes.byref(out), ctypes.c_void_p(4096),
                                          need.value, None) == 1
    assert L.moe_layer_forward_shared(r, ctypes.byref(inp), ctypes.byref(ok), ctypes.byref(out),
                                      ctypes.c_void_p(4096), need.value - 1, None) == 3


def test_backward_validation_without_a_gpu():
    """The backward's host-side checks: unsupported shapes and missing
    pointers are refused before anything is enqueued."""
    from mixture_experts_layer_99_b300 import workloads as W
    L = moe.lib()
    n = ctypes.c_size_t(0)
    # fp32 (on FMA) and E > 64 have a backward
    assert L.moe_workspace_size_backward(ctypes.byref(moe.config_from_workload(
        W.WORKLOADS["ref_fp32"])), ctypes.byref(n)) == 0
    assert n.value > 0
    big = W.small(W.WORKLOADS["switch_top1"], T=64, d=64, H=64, E=128, k=2)
    assert L.moe_workspace_size_backward(ctypes.byref(moe.config_from_workload(big)),
                                         ctypes.byref(n)) == 0
    cfg = moe.config_from_workload(W.WORKLOADS["switch_top1"])
    assert L.moe_workspace_size_backward(ctypes.byref(cfg), ctypes.byref(n)) == 0
    assert n.value > 0
    li = moe.LayerInputs()
    lo = moe.LayerOutputs()
    lg = moe.LayerGrads()
    # missing inputs, outputs and gradients: INVALID_ARG (1)
    assert L.moe_layer_backward(ctypes.byref(cfg), ctypes.byref(li), ctypes.byref(lo), None,
                                ctypes.c_float(0.0), ctypes.byref(lg), None, 0, None, 0,
                                None) == 1
