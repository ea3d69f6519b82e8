"""Python binding of the C ABI in ``include/moe.h`` (ctypes).

Argument marshalling only: every step of the layer runs in the CUDA library.
PyTorch supplies device memory (``torch.empty``) and the current stream. The
library must be built (``python -m mixture_experts_layer_99_b300.build``);
without it every call raises, there is no fallback.

Names follow the C calls: ``router_topk``, ``dispatch``, ``expert_ffn``,
``combine``, ``aux_stats``, ``layer_forward``, ``layer_forward_host``.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_float, c_int32, c_int64, c_size_t, c_void_p
from fractions import Fraction
from typing import Optional

import torch

# MOE_B300_CHECKED=1 loads the checked build (index checks in the kernels,
# MOE_ERR_DEVICE_CHECK on a failure; the same ABI)
LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)),
                        "libmoe_b300_check.so" if os.environ.get("MOE_B300_CHECKED") == "1"
                        else "libmoe_b300.so")

MOE_F32, MOE_BF16 = 0, 1
MOE_ACT_GELU, MOE_ACT_SWIGLU = 0, 1
STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED",
          3: "MOE_ERR_WORKSPACE", 4: "MOE_ERR_CUDA", 5: "MOE_ERR_DEVICE_TIMEOUT",
          6: "MOE_ERR_DEVICE_CHECK"}

EXPORTED = ["moe_abi_version", "moe_status_string", "moe_capacity", "moe_workspace_size",
            "moe_workspace_size_host", "moe_workspace_init", "moe_device_status",
            "moe_router_topk", "moe_dispatch", "moe_expert_ffn", "moe_combine",
            "moe_aux_stats", "moe_layer_forward", "moe_layer_forward_host",
            "moe_layer_forward_host_pipelined",
            "moe_layer_forward_launch_count", "moe_layer_forward_profiled",
            "moe_workspace_size_shared", "moe_layer_forward_shared", "moe_dispatch_static_scratch",
            "moe_workspace_size_backward", "moe_layer_backward",
            "moe_workspace_size_backward_shared", "moe_layer_backward_shared"]


class MoEError(RuntimeError):
    def __init__(self, call, status):
        self.status = status
        super().__init__(f"{call} failed: {STATUS.get(status, status)} "
                         f"({lib().moe_status_string(status).decode()})")


class Config(ctypes.Structure):
    _fields_ = [("T", c_int32), ("d", c_int32), ("E", c_int32), ("k", c_int32),
                ("H", c_int32), ("capacity", c_int32), ("dtype", c_int32),
                ("act", c_int32), ("tau", c_float), ("noise_scale", c_float),
                ("flags", c_int32)]

    def __repr__(self):
        return (f"Config(T={self.T}, d={self.d}, E={self.E}, k={self.k}, H={self.H}, "
                f"C={self.capacity}, dtype={self.dtype}, act={self.act}, tau={self.tau}, "
                f"noise_scale={self.noise_scale}, flags={self.flags})")


MOE_FLAG_KEEP_PREACT = 1


class LayerInputs(ctypes.Structure):
    _fields_ = [("x", c_void_p), ("Wg", c_void_p), ("bias", c_void_p), ("noise", c_void_p),
                ("W1", c_void_p), ("W3", c_void_p), ("W2", c_void_p), ("b1", c_void_p),
                ("b2", c_void_p)]


class SharedExpert(ctypes.Structure):
    _fields_ = [("H", c_int32), ("W1", c_void_p), ("W3", c_void_p), ("W2", c_void_p),
                ("b1", c_void_p), ("b2", c_void_p)]


class LayerOutputs(ctypes.Structure):
    _fields_ = [("y", c_void_p), ("logits", c_void_p), ("topk_idx", c_void_p),
                ("topk_gate", c_void_p), ("slot_of", c_void_p), ("expert_count", c_void_p),
                ("expert_offset", c_void_p), ("f", c_void_p), ("P", c_void_p),
                ("L_balance", c_void_p), ("dropped", c_void_p)]


class LayerGrads(ctypes.Structure):
    _fields_ = [("dx", c_void_p), ("dWg", c_void_p), ("dbias", c_void_p), ("dW1", c_void_p),
                ("dW3", c_void_p), ("dW2", c_void_p), ("db1", c_void_p), ("db2", c_void_p)]


class SharedGrads(ctypes.Structure):
    _fields_ = [("dW1", c_void_p), ("dW3", c_void_p), ("dW2", c_void_p), ("db1", c_void_p),
                ("db2", c_void_p)]


_LIB = None


def lib():
    """Load the CUDA library (raises if it has not been built)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                           "`python -m mixture_experts_layer_99_b300.build`")
    L = ctypes.CDLL(LIB_PATH)
    cfgp = POINTER(Config)
    vp = c_void_p
    sig = {
        "moe_abi_version": (c_int32, []),
        "moe_status_string": (ctypes.c_char_p, [c_int32]),
        "moe_capacity": (c_int32, [c_int64, c_int64, c_int32, c_int32, c_int32]),
        "moe_workspace_size": (c_int32, [cfgp, POINTER(c_size_t)]),
        "moe_workspace_size_host": (c_int32, [cfgp, POINTER(c_size_t)]),
        "moe_workspace_init": (c_int32, [vp, c_size_t, vp]),
        "moe_device_status": (c_int32, [vp, POINTER(c_int32), POINTER(c_int32), vp]),
        "moe_router_topk": (c_int32, [cfgp, vp, vp, vp, vp, vp, vp, vp, vp, vp, c_size_t, vp]),
        "moe_dispatch": (c_int32, [cfgp, vp, vp, vp, vp, vp, vp, vp, vp, c_size_t, vp]),
        "moe_expert_ffn": (c_int32, [cfgp, vp, vp, vp, vp, vp, vp, vp, vp, vp, c_size_t, vp]),
        "moe_combine": (c_int32, [cfgp, vp, vp, vp, vp, vp]),
        "moe_aux_stats": (c_int32, [cfgp, vp, vp, vp, vp, vp, vp, vp]),
        "moe_layer_forward": (c_int32, [cfgp, POINTER(LayerInputs), POINTER(LayerOutputs),
                                        vp, c_size_t, vp]),
        "moe_layer_forward_launch_count": (c_int32, [cfgp]),
        "moe_workspace_size_shared": (c_int32, [cfgp, c_int32, POINTER(c_size_t)]),
        "moe_layer_forward_shared": (c_int32, [cfgp, POINTER(LayerInputs),
                                               POINTER(SharedExpert), POINTER(LayerOutputs),
                                               vp, c_size_t, vp]),
        "moe_layer_forward_profiled": (c_int32, [cfgp, POINTER(LayerInputs),
                                                 POINTER(LayerOutputs), vp, c_size_t, vp,
                                                 POINTER(c_void_p)]),
        "moe_layer_forward_host": (c_int32, [cfgp, vp, POINTER(LayerInputs), vp, vp, vp,
                                             c_size_t, vp]),
        "moe_layer_forward_host_pipelined": (c_int32, [cfgp, vp, POINTER(LayerInputs), vp, vp,
                                                       vp, c_size_t, vp, vp, vp,
                                                       POINTER(c_void_p)]),
        "moe_workspace_size_backward": (c_int32, [cfgp, POINTER(c_size_t)]),
        "moe_layer_backward": (c_int32, [cfgp, POINTER(LayerInputs), POINTER(LayerOutputs), vp,
                                         ctypes.c_float, POINTER(LayerGrads), vp, c_size_t, vp,
                                         c_size_t, vp]),
        "moe_workspace_size_backward_shared": (c_int32, [cfgp, c_int32, POINTER(c_size_t)]),
        "moe_layer_backward_shared": (c_int32, [cfgp, POINTER(LayerInputs), POINTER(SharedExpert),
                                                POINTER(LayerOutputs), vp, ctypes.c_float,
                                                POINTER(LayerGrads), POINTER(SharedGrads), vp,
                                                c_size_t, vp, c_size_t, vp]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    _LIB = L
    return L


# ------------------------------------------------------------------ helpers
def capacity(c, k: int, T: int, E: int) -> int:
    """C = ceil(c k T / E) computed by the library in integer arithmetic."""
    q = Fraction(c)
    v = lib().moe_capacity(q.numerator, q.denominator, k, T, E)
    if v < 0:
        raise ValueError("invalid capacity arguments")
    return v


def make_config(T, d, E, k, H, capacity_, dtype="bf16", act="gelu", tau=1.0,
                noise_scale=0.0, keep_preact=False) -> Config:
    """keep_preact: the forward keeps the experts' pre-activations in its
    workspace for the backward (MOE_FLAG_KEEP_PREACT)."""
    return Config(T, d, E, k, H, capacity_, MOE_F32 if dtype == "f32" else MOE_BF16,
                  MOE_ACT_GELU if act == "gelu" else MOE_ACT_SWIGLU, float(tau),
                  float(noise_scale), MOE_FLAG_KEEP_PREACT if keep_preact else 0)


def config_from_workload(w, T: Optional[int] = None, keep_preact: bool = False) -> Config:
    T = w.T if T is None else T
    return make_config(T, w.d, w.E, w.k, w.H, capacity(w.c, w.k, T, w.E), w.dtype, w.act,
                       w.tau, w.noise_scale, keep_preact)


def _dt(cfg):
    return torch.float32 if cfg.dtype == MOE_F32 else torch.bfloat16


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(device=None):
    return torch.cuda.current_stream(device).cuda_stream


def _need(t, name, dtype, shape, device=None):
    if t is None:
        raise ValueError(f"{name} is required")
    if t.dtype != dtype:
        raise TypeError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if device is not None and t.device != device:
        raise ValueError(f"{name} on {t.device}, expected {device}")
    return t


def _opt(t, name, dtype, shape, device=None):
    return None if t is None else _need(t, name, dtype, shape, device)


def _call(name, *args):
    st = getattr(lib(), name)(*args)
    if st != 0:
        raise MoEError(name, st)


def workspace_size(cfg: Config, host_io: bool = False) -> int:
    n = c_size_t(0)
    _call("moe_workspace_size_host" if host_io else "moe_workspace_size",
          ctypes.byref(cfg), ctypes.byref(n))
    return n.value


def workspace(cfg: Config, device="cuda", host_io: bool = False) -> torch.Tensor:
    """Allocate (torch) and initialise a workspace for ``cfg``."""
    n = workspace_size(cfg, host_io)
    ws = torch.empty(n + 256, dtype=torch.uint8, device=device)
    off = (-ws.data_ptr()) % 256
    ws = ws[off:off + n]
    _call("moe_workspace_init", c_void_p(ws.data_ptr()), n, c_void_p(_stream(ws.device)))
    return ws


def device_status(ws: torch.Tensor):
    code, where = c_int32(0), c_int32(0)
    _call("moe_device_status", c_void_p(ws.data_ptr()), ctypes.byref(code),
          ctypes.byref(where), c_void_p(_stream(ws.device)))
    return code.value, where.value


# ------------------------------------------------------------------ the calls
def router_topk(cfg, x, Wg, bias=None, noise=None, *, ws=None, logits=True):
    """Returns (logits or None, topk_idx [T,k] int32, topk_gate [T,k] fp32,
    prob_sum [E] fp32)."""
    dev = x.device
    dt = _dt(cfg)
    _need(x, "x", dt, (cfg.T, cfg.d), dev)
    _need(Wg, "Wg", dt, (cfg.E, cfg.d), dev)
    _opt(bias, "bias", torch.float32, (cfg.E,), dev)
    _opt(noise, "noise", torch.float32, (cfg.T, cfg.E), dev)
    lg = torch.empty(cfg.T, cfg.E, dtype=torch.float32, device=dev) if logits else None
    idx = torch.empty(cfg.T, cfg.k, dtype=torch.int32, device=dev)
    gate = torch.empty(cfg.T, cfg.k, dtype=torch.float32, device=dev)
    psum = torch.empty(cfg.E, dtype=torch.float32, device=dev)
    ws = workspace(cfg, dev) if ws is None else ws
    _call("moe_router_topk", ctypes.byref(cfg), _ptr(x), _ptr(Wg), _ptr(bias), _ptr(noise),
          _ptr(lg), _ptr(idx), _ptr(gate), _ptr(psum), _ptr(ws), ws.numel(), _stream(dev))
    return lg, idx, gate, psum


def dispatch(cfg, topk_idx, x, *, ws=None):
    """Returns dict(count [E], offset [E+1], slot_of [T,k], token_of_row [T*k],
    xd [T*k, d]); only the first offset[E] rows of token_of_row and xd are set."""
    dev = x.device
    _need(topk_idx, "topk_idx", torch.int32, (cfg.T, cfg.k), dev)
    _need(x, "x", _dt(cfg), (cfg.T, cfg.d), dev)
    R = cfg.T * cfg.k
    out = dict(count=torch.empty(cfg.E, dtype=torch.int32, device=dev),
               offset=torch.empty(cfg.E + 1, dtype=torch.int32, device=dev),
               slot_of=torch.empty(cfg.T, cfg.k, dtype=torch.int32, device=dev),
               token_of_row=torch.empty(R, dtype=torch.int32, device=dev),
               xd=torch.empty(R, cfg.d, dtype=_dt(cfg), device=dev))
    ws = workspace(cfg, dev) if ws is None else ws
    _call("moe_dispatch", ctypes.byref(cfg), _ptr(topk_idx), _ptr(x), _ptr(out["count"]),
          _ptr(out["offset"]), _ptr(out["slot_of"]), _ptr(out["token_of_row"]),
          _ptr(out["xd"]), _ptr(ws), ws.numel(), _stream(dev))
    return out


def expert_ffn(cfg, xd, expert_offset, W1, W2, W3=None, b1=None, b2=None, *, ws=None,
               Y=None):
    """Y [rows, d] for the packed rows xd [rows, d] (rows >= offset[E])."""
    dev = xd.device
    dt = _dt(cfg)
    rows = xd.shape[0]
    _need(xd, "xd", dt, (rows, cfg.d), dev)
    _need(expert_offset, "expert_offset", torch.int32, (cfg.E + 1,), dev)
    _need(W1, "W1", dt, (cfg.E, cfg.H, cfg.d), dev)
    _need(W2, "W2", dt, (cfg.E, cfg.d, cfg.H), dev)
    _opt(W3, "W3", dt, (cfg.E, cfg.H, cfg.d), dev)
    _opt(b1, "b1", dt, (cfg.E, cfg.H), dev)
    _opt(b2, "b2", dt, (cfg.E, cfg.d), dev)
    if rows < min(cfg.T * cfg.k, cfg.E * cfg.capacity):
        raise ValueError("xd must hold min(T*k, E*C) rows")
    Y = torch.empty(rows, cfg.d, dtype=dt, device=dev) if Y is None else Y
    ws = workspace(cfg, dev) if ws is None else ws
    _call("moe_expert_ffn", ctypes.byref(cfg), _ptr(xd), _ptr(expert_offset), _ptr(W1),
          _ptr(W3), _ptr(W2), _ptr(b1), _ptr(b2), _ptr(Y), _ptr(ws), ws.numel(), _stream(dev))
    return Y


def combine(cfg, Y, slot_of, topk_gate):
    dev = Y.device
    _need(slot_of, "slot_of", torch.int32, (cfg.T, cfg.k), dev)
    _need(topk_gate, "topk_gate", torch.float32, (cfg.T, cfg.k), dev)
    if Y.dtype != _dt(cfg) or Y.shape[1] != cfg.d or not Y.is_contiguous():
        raise ValueError("Y must be contiguous [rows, d] of the config dtype")
    y = torch.empty(cfg.T, cfg.d, dtype=_dt(cfg), device=dev)
    _call("moe_combine", ctypes.byref(cfg), _ptr(Y), _ptr(slot_of), _ptr(topk_gate), _ptr(y),
          _stream(dev))
    return y


def aux_stats(cfg, expert_count, prob_sum):
    """Returns (f [E], P [E], L_balance [1], dropped [1])."""
    dev = expert_count.device
    _need(expert_count, "expert_count", torch.int32, (cfg.E,), dev)
    _need(prob_sum, "prob_sum", torch.float32, (cfg.E,), dev)
    f = torch.empty(cfg.E, dtype=torch.float32, device=dev)
    P = torch.empty(cfg.E, dtype=torch.float32, device=dev)
    L = torch.empty(1, dtype=torch.float32, device=dev)
    dropped = torch.empty(1, dtype=torch.int32, device=dev)
    _call("moe_aux_stats", ctypes.byref(cfg), _ptr(expert_count), _ptr(prob_sum), _ptr(f),
          _ptr(P), _ptr(L), _ptr(dropped), _stream(dev))
    return f, P, L, dropped


def _layer_inputs(cfg, inp, dev, with_x=True):
    dt = _dt(cfg)
    x = inp.get("x") if with_x else None
    if with_x:
        _need(x, "x", dt, (cfg.T, cfg.d), dev)
    _need(inp["Wg"], "Wg", dt, (cfg.E, cfg.d), dev)
    _opt(inp.get("bias"), "bias", torch.float32, (cfg.E,), dev)
    _opt(inp.get("noise"), "noise", torch.float32, (cfg.T, cfg.E), dev)
    _need(inp["W1"], "W1", dt, (cfg.E, cfg.H, cfg.d), dev)
    _opt(inp.get("W3"), "W3", dt, (cfg.E, cfg.H, cfg.d), dev)
    _need(inp["W2"], "W2", dt, (cfg.E, cfg.d, cfg.H), dev)
    _opt(inp.get("b1"), "b1", dt, (cfg.E, cfg.H), dev)
    _opt(inp.get("b2"), "b2", dt, (cfg.E, cfg.d), dev)
    return LayerInputs(_ptr(x), _ptr(inp["Wg"]), _ptr(inp.get("bias")),
                       _ptr(inp.get("noise")), _ptr(inp["W1"]), _ptr(inp.get("W3")),
                       _ptr(inp["W2"]), _ptr(inp.get("b1")), _ptr(inp.get("b2")))


def alloc_outputs(cfg, device, full=True):
    dev = torch.device(device)
    o = dict(y=torch.empty(cfg.T, cfg.d, dtype=_dt(cfg), device=dev))
    if full:
        o.update(
            logits=torch.empty(cfg.T, cfg.E, dtype=torch.float32, device=dev),
            topk_idx=torch.empty(cfg.T, cfg.k, dtype=torch.int32, device=dev),
            topk_gate=torch.empty(cfg.T, cfg.k, dtype=torch.float32, device=dev),
            slot_of=torch.empty(cfg.T, cfg.k, dtype=torch.int32, device=dev),
            expert_count=torch.empty(cfg.E, dtype=torch.int32, device=dev),
            expert_offset=torch.empty(cfg.E + 1, dtype=torch.int32, device=dev),
            f=torch.empty(cfg.E, dtype=torch.float32, device=dev),
            P=torch.empty(cfg.E, dtype=torch.float32, device=dev),
            L_balance=torch.empty(1, dtype=torch.float32, device=dev),
            dropped=torch.empty(1, dtype=torch.int32, device=dev))
    return o


def layer_forward(cfg, inp: dict, *, ws=None, out: Optional[dict] = None, full=True):
    """The fused layer. ``inp``: x, Wg, W1, W2 and optional W3, b1, b2, bias,
    noise (device tensors). Returns the output dict (``y`` plus, if ``full``,
    logits, topk_idx, topk_gate, slot_of, expert_count, expert_offset, f, P,
    L_balance, dropped)."""
    dev = inp["x"].device
    li = _layer_inputs(cfg, inp, dev)
    out = alloc_outputs(cfg, dev, full) if out is None else out
    lo = LayerOutputs(*[_ptr(out.get(n)) for n, _ in LayerOutputs._fields_])
    ws = workspace(cfg, dev) if ws is None else ws
    _call("moe_layer_forward", ctypes.byref(cfg), ctypes.byref(li), ctypes.byref(lo),
          _ptr(ws), ws.numel(), _stream(dev))
    return out


def workspace_shared(cfg: Config, H_shared: int, device="cuda") -> torch.Tensor:
    n = c_size_t(0)
    _call("moe_workspace_size_shared", ctypes.byref(cfg), H_shared, ctypes.byref(n))
    ws = torch.empty(n.value + 256, dtype=torch.uint8, device=device)
    off = (-ws.data_ptr()) % 256
    ws = ws[off:off + n.value]
    _call("moe_workspace_init", c_void_p(ws.data_ptr()), n.value,
          c_void_p(_stream(ws.device)))
    return ws


def layer_forward_shared(cfg, inp: dict, shared: dict, *, ws=None, out=None, full=True):
    """The fused layer plus a shared expert (every token, weight 1). ``shared``
    holds W1 [Hs, d], W2 [d, Hs], and W3 [Hs, d] (SwiGLU) or optional b1 [Hs],
    b2 [d] (GELU)."""
    dev = inp["x"].device
    dt = _dt(cfg)
    li = _layer_inputs(cfg, inp, dev)
    Hs = shared["W1"].shape[0]
    _need(shared["W1"], "shared W1", dt, (Hs, cfg.d), dev)
    _need(shared["W2"], "shared W2", dt, (cfg.d, Hs), dev)
    _opt(shared.get("W3"), "shared W3", dt, (Hs, cfg.d), dev)
    _opt(shared.get("b1"), "shared b1", dt, (Hs,), dev)
    _opt(shared.get("b2"), "shared b2", dt, (cfg.d,), dev)
    se = SharedExpert(Hs, _ptr(shared["W1"]), _ptr(shared.get("W3")), _ptr(shared["W2"]),
                      _ptr(shared.get("b1")), _ptr(shared.get("b2")))
    out = alloc_outputs(cfg, dev, full) if out is None else out
    lo = LayerOutputs(*[_ptr(out.get(n)) for n, _ in LayerOutputs._fields_])
    ws = workspace_shared(cfg, Hs, dev) if ws is None else ws
    _call("moe_layer_forward_shared", ctypes.byref(cfg), ctypes.byref(li), ctypes.byref(se),
          ctypes.byref(lo), _ptr(ws), ws.numel(), _stream(dev))
    return out


def layer_forward_profiled(cfg, inp: dict, events, *, ws, out: dict):
    """moe_layer_forward that records six torch.cuda.Event (timing enabled,
    already recorded once so that they exist) at the stage boundaries."""
    dev = inp["x"].device
    li = _layer_inputs(cfg, inp, dev)
    lo = LayerOutputs(*[_ptr(out.get(n)) for n, _ in LayerOutputs._fields_])
    arr = (c_void_p * 6)(*[c_void_p(e.cuda_event) for e in events])
    _call("moe_layer_forward_profiled", ctypes.byref(cfg), ctypes.byref(li), ctypes.byref(lo),
          _ptr(ws), ws.numel(), _stream(dev), arr)
    return out


def layer_forward_host(cfg, x_host, weights: dict, y_host, *, ws, L_host=None):
    """The fused layer with host (page-locked) x and y; weights on the device.
    Enqueues the copies and the layer on the current stream; synchronise the
    stream before reading y_host."""
    dev = weights["Wg"].device
    li = _layer_inputs(cfg, weights, dev, with_x=False)
    _need(x_host, "x_host", _dt(cfg), (cfg.T, cfg.d), torch.device("cpu"))
    _need(y_host, "y_host", _dt(cfg), (cfg.T, cfg.d), torch.device("cpu"))
    _call("moe_layer_forward_host", ctypes.byref(cfg), _ptr(x_host), ctypes.byref(li),
          _ptr(y_host), _ptr(L_host), _ptr(ws), ws.numel(), _stream(dev))


def layer_forward_host_pipelined(cfg, x_host, weights: dict, y_host, *, ws, events,
                                 copy_in, compute, copy_out, L_host=None):
    """moe_layer_forward_host_pipelined: the copy in on ``copy_in``, the layer
    on ``compute``, the copies out on ``copy_out`` (torch.cuda.Stream each);
    ``events`` are three torch.cuda.Event objects that belong to ``ws`` and
    go with it to every call. Synchronise ``copy_out`` (or wait on
    events[2]) before reading y_host."""
    dev = weights["Wg"].device
    li = _layer_inputs(cfg, weights, dev, with_x=False)
    _need(x_host, "x_host", _dt(cfg), (cfg.T, cfg.d), torch.device("cpu"))
    _need(y_host, "y_host", _dt(cfg), (cfg.T, cfg.d), torch.device("cpu"))
    if len(events) != 3:
        raise ValueError("three events per workspace")
    for e in events:  # torch creates the CUDA event on its first record
        if not e.cuda_event:
            e.record(compute)
    evs = (c_void_p * 3)(*[c_void_p(e.cuda_event) for e in events])
    _call("moe_layer_forward_host_pipelined", ctypes.byref(cfg), _ptr(x_host), ctypes.byref(li),
          _ptr(y_host), _ptr(L_host), _ptr(ws), ws.numel(), c_void_p(copy_in.cuda_stream),
          c_void_p(compute.cuda_stream), c_void_p(copy_out.cuda_stream), evs)


def workspace_backward(cfg: Config, device="cuda") -> torch.Tensor:
    """The backward pass's own workspace (256-byte aligned, header zeroed)."""
    n = c_size_t(0)
    _call("moe_workspace_size_backward", ctypes.byref(cfg), ctypes.byref(n))
    ws = torch.empty(n.value + 256, dtype=torch.uint8, device=device)
    off = (-ws.data_ptr()) % 256
    ws = ws[off:off + n.value]
    _call("moe_workspace_init", c_void_p(ws.data_ptr()), n.value,
          c_void_p(_stream(ws.device)))
    return ws


def alloc_grads(cfg, inp: dict, device):
    """Gradient buffers matching the inputs: dx in the layer dtype, fp32 weight
    gradients; dbias, dW3, db1, db2 only where the inputs have them."""
    E, d, H, T = cfg.E, cfg.d, cfg.H, cfg.T
    f32 = dict(dtype=torch.float32, device=device)
    g = dict(dx=torch.empty(T, d, dtype=_dt(cfg), device=device),
             dWg=torch.empty(E, d, **f32), dW1=torch.empty(E, H, d, **f32),
             dW2=torch.empty(E, d, H, **f32))
    if inp.get("bias") is not None:
        g["dbias"] = torch.empty(E, **f32)
    if inp.get("W3") is not None:
        g["dW3"] = torch.empty(E, H, d, **f32)
    if inp.get("b1") is not None:
        g["db1"] = torch.empty(E, H, **f32)
    if inp.get("b2") is not None:
        g["db2"] = torch.empty(E, d, **f32)
    return g


def layer_backward(cfg, inp: dict, fwd: dict, dy, alpha: float = 0.0, *, ws, bws=None,
                   grads: Optional[dict] = None):
    """Gradients of sum <dy, y> + alpha * L_balance for the forward call that
    produced ``fwd`` (the output dict of layer_forward with full=True) with
    workspace ``ws``. Returns the gradient dict (see alloc_grads)."""
    dev = inp["x"].device
    li = _layer_inputs(cfg, inp, dev)
    _need(dy, "dy", _dt(cfg), (cfg.T, cfg.d), dev)
    lo = LayerOutputs(*[_ptr(fwd.get(n)) for n, _ in LayerOutputs._fields_])
    g = alloc_grads(cfg, inp, dev) if grads is None else grads
    lg = LayerGrads(*[_ptr(g.get(n)) for n, _ in LayerGrads._fields_])
    bws = workspace_backward(cfg, dev) if bws is None else bws
    _call("moe_layer_backward", ctypes.byref(cfg), ctypes.byref(li), ctypes.byref(lo),
          _ptr(dy), ctypes.c_float(alpha), ctypes.byref(lg), _ptr(ws), ws.numel(), _ptr(bws),
          bws.numel(), _stream(dev))
    return g


def _shared_expert(cfg, shared: dict, dev) -> SharedExpert:
    dt = _dt(cfg)
    Hs = shared["W1"].shape[0]
    _need(shared["W1"], "shared W1", dt, (Hs, cfg.d), dev)
    _need(shared["W2"], "shared W2", dt, (cfg.d, Hs), dev)
    _opt(shared.get("W3"), "shared W3", dt, (Hs, cfg.d), dev)
    _opt(shared.get("b1"), "shared b1", dt, (Hs,), dev)
    _opt(shared.get("b2"), "shared b2", dt, (cfg.d,), dev)
    return SharedExpert(Hs, _ptr(shared["W1"]), _ptr(shared.get("W3")), _ptr(shared["W2"]),
                        _ptr(shared.get("b1")), _ptr(shared.get("b2")))


def workspace_backward_shared(cfg: Config, H_shared: int, device="cuda") -> torch.Tensor:
    """The backward workspace of a layer with a shared expert (256-byte
    aligned, header zeroed)."""
    n = c_size_t(0)
    _call("moe_workspace_size_backward_shared", ctypes.byref(cfg), H_shared, ctypes.byref(n))
    ws = torch.empty(n.value + 256, dtype=torch.uint8, device=device)
    off = (-ws.data_ptr()) % 256
    ws = ws[off:off + n.value]
    _call("moe_workspace_init", c_void_p(ws.data_ptr()), n.value, c_void_p(_stream(ws.device)))
    return ws


def alloc_shared_grads(cfg, shared: dict, device):
    """fp32 gradient buffers for the shared expert's weights (dW3, db1, db2
    only where the shared expert has them)."""
    Hs, d = shared["W1"].shape[0], cfg.d
    f32 = dict(dtype=torch.float32, device=device)
    g = dict(dW1=torch.empty(Hs, d, **f32), dW2=torch.empty(d, Hs, **f32))
    if shared.get("W3") is not None:
        g["dW3"] = torch.empty(Hs, d, **f32)
    if shared.get("b1") is not None:
        g["db1"] = torch.empty(Hs, **f32)
    if shared.get("b2") is not None:
        g["db2"] = torch.empty(d, **f32)
    return g


def layer_backward_shared(cfg, inp: dict, shared: dict, fwd: dict, dy, alpha: float = 0.0, *,
                          ws, bws=None, grads: Optional[dict] = None,
                          shared_grads: Optional[dict] = None):
    """Backward of a layer_forward_shared call (workspace ``ws``, outputs
    ``fwd``). Returns (gradient dict, shared-expert gradient dict)."""
    dev = inp["x"].device
    li = _layer_inputs(cfg, inp, dev)
    se = _shared_expert(cfg, shared, dev)
    _need(dy, "dy", _dt(cfg), (cfg.T, cfg.d), dev)
    lo = LayerOutputs(*[_ptr(fwd.get(n)) for n, _ in LayerOutputs._fields_])
    g = alloc_grads(cfg, inp, dev) if grads is None else grads
    sg = alloc_shared_grads(cfg, shared, dev) if shared_grads is None else shared_grads
    lg = LayerGrads(*[_ptr(g.get(n)) for n, _ in LayerGrads._fields_])
    lsg = SharedGrads(*[_ptr(sg.get(n)) for n, _ in SharedGrads._fields_])
    bws = workspace_backward_shared(cfg, se.H, dev) if bws is None else bws
    _call("moe_layer_backward_shared", ctypes.byref(cfg), ctypes.byref(li), ctypes.byref(se),
          ctypes.byref(lo), _ptr(dy), ctypes.c_float(alpha), ctypes.byref(lg), ctypes.byref(lsg),
          _ptr(ws), ws.numel(), _ptr(bws), bws.numel(), _stream(dev))
    return g, sg
