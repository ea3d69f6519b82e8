"""The allocation-free dispatch entry point against the regular one.

moe_dispatch_static_scratch serves callers that cannot allocate a workspace
(an op interface that passes only the op's own tensors, or a runtime that
forbids device allocation after start-up); it keeps its scratch in a fixed
array inside the library. Its results must equal moe_dispatch's exactly, on
two calls in a row (the second call must not see leftovers of the first).
This file is collected last on purpose."""
import ctypes
from fractions import Fraction

import pytest
import torch

from mixture_experts_layer_99_b300 import moe, workloads as W
from oracle import moe_oracle as ORC

pytestmark = pytest.mark.gpu


def _static_call(cfg, ids, x, out):
    L = moe.lib()
    fn = L.moe_dispatch_static_scratch
    fn.restype = ctypes.c_int32
    fn.argtypes = [ctypes.POINTER(moe.Config)] + [ctypes.c_void_p] * 8
    return fn(ctypes.byref(cfg), ids.data_ptr(), x.data_ptr(), out["count"].data_ptr(),
              out["offset"].data_ptr(), out["slot_of"].data_ptr(),
              out["token_of_row"].data_ptr(), out["xd"].data_ptr(),
              torch.cuda.current_stream().cuda_stream)


def _empty_outputs(cfg, dt):
    R = cfg.T * cfg.k
    return dict(count=torch.full((cfg.E,), -7, dtype=torch.int32, device="cuda"),
                offset=torch.full((cfg.E + 1,), -7, dtype=torch.int32, device="cuda"),
                slot_of=torch.full((cfg.T, cfg.k), -7, dtype=torch.int32, device="cuda"),
                token_of_row=torch.full((R,), -7, dtype=torch.int32, device="cuda"),
                xd=torch.zeros(R, cfg.d, dtype=dt, device="cuda"))


@pytest.mark.parametrize("T,E,k,c,skew,d", [(32768, 64, 2, Fraction(2), 3.0, 128),
                                            (8192, 8, 1, Fraction(1), 0.3, 1024),
                                            (1000, 16, 2, Fraction(1, 2), 2.0, 40)])
def test_static_scratch_dispatch_matches_workspace_dispatch(T, E, k, c, skew, d):
    C = ORC.capacity(c, k, T, E)
    cfg = moe.make_config(T, d, E, k, 8, C, "bf16", "gelu")
    for call in range(2):     # two calls in a row, different routings
        ids = W.make_routing(T, E, k, seed=100 + call, skew=skew).to("cuda")
        x = W.make_rows(T, d, torch.bfloat16, seed=200 + call).to("cuda")
        ref = moe.dispatch(cfg, ids, x)
        got = _empty_outputs(cfg, torch.bfloat16)
        assert _static_call(cfg, ids, x, got) == 0
        torch.cuda.synchronize()
        R = int(ref["offset"][-1].item())
        for key in ("count", "offset", "slot_of"):
            assert torch.equal(got[key], ref[key]), key
        assert torch.equal(got["token_of_row"][:R], ref["token_of_row"][:R])
        assert torch.equal(got["xd"][:R], ref["xd"][:R])
    # after those calls (the first one looked the scratch address up), a
    # further call changes neither torch's allocations nor the device's free
    # memory: it allocates nothing
    got = _empty_outputs(cfg, torch.bfloat16)
    torch.cuda.synchronize()
    alloc0, free0 = torch.cuda.memory_allocated(), torch.cuda.mem_get_info()[0]
    assert _static_call(cfg, ids, x, got) == 0
    torch.cuda.synchronize()
    assert torch.cuda.memory_allocated() == alloc0
    assert torch.cuda.mem_get_info()[0] == free0


def test_static_scratch_rejects_oversize():
    # ceil(T*k/1024) * E = 1025 * 64 > 65536 entries of static scratch
    cfg = moe.make_config(1025 * 1024, 8, 64, 1, 8, 1, "bf16", "gelu")
    L = moe.lib()
    fn = L.moe_dispatch_static_scratch
    fn.restype = ctypes.c_int32
    fn.argtypes = [ctypes.POINTER(moe.Config)] + [ctypes.c_void_p] * 8
    fake = ctypes.c_void_p(4096)
    assert fn(ctypes.byref(cfg), fake, fake, fake, fake, fake, fake, fake, None) == 2
