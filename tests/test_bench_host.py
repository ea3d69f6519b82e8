"""Host-side arithmetic of bench.py (no GPU): the algorithmic work behind the
roofline fractions, written out for the mixtral and long-tail shapes from the
closed forms of the method's data movement, and the rotating input sets."""
import bench
from mixture_experts_layer_99_b300 import workloads as W


def test_mixtral_algorithmic_work():
    w = W.WORKLOADS["mixtral"]           # T=16384, d=4096, E=8, k=2, SwiGLU H=14336, bf16
    T, d, E, k, H = 16384, 4096, 8, 2, 14336
    kept = T * k                         # no drops
    a = bench.algorithmic(w, kept, E)
    # router: x, W_g, ids + gates (4 + 4 bytes per slot), the E probability sums
    assert a["router_bytes"] == T * d * 2 + E * d * 2 + T * k * 8 + E * 4 == 134545440
    assert a["router_flops"] == 2 * T * d * E
    # dispatch: ids read, slot_of written, every kept row read and written, counts
    assert a["dispatch_bytes"] == 2 * T * k * 4 + 2 * kept * d * 2 + 8 * E == 537133120
    # combine: kept expert rows read, slots and gates read, y written
    assert a["combine_bytes"] == kept * d * 2 + T * k * 8 + T * d * 2 == 402915328
    # three d x H products per kept row for SwiGLU
    assert a["gemm_flops"] == kept * 2 * 3 * d * H
    assert abs(a["gemm_flops"] / 1e12 - 11.545) < 1e-3
    # every active expert's three matrices once, plus the packed rows in and out
    assert a["gemm_bytes"] == E * 3 * d * H * 2 + 2 * kept * d * 2
    assert a["tc_router"]


def test_longtail_router_bytes_include_the_noise():
    w = W.WORKLOADS["longtail"]          # Gumbel noise [T, E] fp32 is an input
    a = bench.algorithmic(w, 23500, 64)
    T, d, E, k = 32768, 2048, 64, 2
    assert a["router_bytes"] == T * d * 2 + E * d * 2 + T * E * 4 + T * k * 8 + E * 4
    assert a["gemm_flops"] == 23500 * 2 * 3 * d * 1408


def test_gelu_has_two_matrices():
    w = W.WORKLOADS["switch_top1"]
    a = bench.algorithmic(w, 8000, 8)
    assert a["gemm_flops"] == 8000 * 2 * 2 * 1024 * 4096


def test_rotating_sets_exceed_three_l2():
    for fp in (10 * 2**20, 200 * 2**20, 3 * 2**30):
        n = bench.rotating_sets(fp)
        assert n >= 2 and n * fp > 3 * bench.L2_BYTES


def test_extrapolated_sample_label():
    w = W.WORKLOADS["mixtral"]
    assert bench.sample_label(w, 1000, 2.0).startswith("extrapolated (1000 of 16384 tokens)")
    assert not bench.sample_label(w, w.T, 2.0).startswith("extrapolated")
