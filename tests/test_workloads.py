"""The seeded input generators (CPU): shapes, draw order stability and the
router-noise distributions the workloads declare."""
import math

import torch

from mixture_experts_layer_99_b300 import workloads as W


def test_gaussian_noise_has_the_declared_std():
    w = W.WORKLOADS["sweep_e16_k4"]
    inp = W.make_inputs(W.small(w, T=4096, d=64, H=64))
    n = inp["noise"].double()
    assert n.shape == (4096, w.E) and inp["noise"].dtype == torch.float32
    # 65536 draws: the sample mean and std lie within a few standard errors
    assert abs(n.mean().item()) < 5 * w.noise_std / math.sqrt(n.numel())
    assert abs(n.std().item() / w.noise_std - 1.0) < 0.02


def test_std_scaled_noise_is_drawn_unscaled():
    """std-scaled router noise: the tensor is N(0, 1); the router applies the
    strength noise_std times each token's logit standard deviation."""
    w = W.WORKLOADS["sweep_std_noise"]
    inp = W.make_inputs(W.small(w, T=4096, d=64, H=64))
    n = inp["noise"].double()
    assert n.shape == (4096, w.E) and inp["noise"].dtype == torch.float32
    assert abs(n.mean().item()) < 5 / math.sqrt(n.numel())
    assert abs(n.std().item() - 1.0) < 0.02
    assert w.noise_scale == w.noise_std > 0
    assert W.WORKLOADS["sweep_e16_k4"].noise_scale == 0.0


def test_gumbel_noise_matches_its_moments():
    w = W.small(W.WORKLOADS["longtail"], T=4096, d=64, H=64)
    n = W.make_inputs(w)["noise"].double()
    # standard Gumbel: mean = Euler-Mascheroni constant, variance = pi^2 / 6
    assert abs(n.mean().item() - 0.5772156649) < 0.02
    assert abs(n.var().item() / (math.pi ** 2 / 6) - 1.0) < 0.03


def test_noise_is_drawn_after_the_weights():
    """Adding noise to a workload leaves x and every weight unchanged."""
    base = W.small(W.WORKLOADS["switch_top1"], T=64, d=32, H=48)
    noisy = base.with_(noise="gaussian", noise_std=0.05)
    a, b = W.make_inputs(base), W.make_inputs(noisy)
    for key in ("x", "Wg", "W1", "W2"):
        assert torch.equal(a[key], b[key]), key
    assert a["noise"] is None and b["noise"] is not None


def test_seeds_give_distinct_reproducible_draws():
    w = W.small(W.WORKLOADS["mixtral"], T=16, d=32, H=48)
    assert torch.equal(W.make_inputs(w, 3)["x"], W.make_inputs(w, 3)["x"])
    assert not torch.equal(W.make_inputs(w, 3)["x"], W.make_inputs(w, 4)["x"])
