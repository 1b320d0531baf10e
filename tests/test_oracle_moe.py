"""Pins of the MoE forward oracle: the Part 3 worked example, loop == token view,
the dense SwiGLU special case, and linearity in the route weights."""
import json

import numpy as np
import torch

from conftest import GOLDEN
from oracle import moe
import synth


def test_part3_gather_projection_example():
    fx = json.loads((GOLDEN / "fused_moe_part3_example.json").read_text())
    w = np.stack([np.full((fx["N"], fx["K"]), v) for v in fx["weight_fill"]])
    out = moe.expert_projection(np.array(fx["x"], float), w, np.array(fx["topk_ids"]))
    assert out.tolist() == fx["expected_output"]


def _rand_layer(T=13, H=24, I=10, E=5, k=2, seed=0):
    rng = np.random.default_rng(seed)
    x = rng.normal(size=(T, H))
    w1 = rng.normal(0, 0.3, size=(E, 2 * I, H))
    w2 = rng.normal(0, 0.3, size=(E, H, I))
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)])
    tw = rng.uniform(0.1, 1.0, size=(T, k))
    return x, w1, w2, tw, ids


def test_expert_loop_equals_token_view():
    for seed in range(3):
        x, w1, w2, tw, ids = _rand_layer(seed=seed)
        a = moe.expert_loop_forward(x, w1, w2, tw, ids)
        b = moe.token_view_forward(x, w1, w2, tw, ids)
        np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-12)


def test_dense_swiglu_special_case():
    # E = 1, k = 1, weight 1: the layer is one dense SwiGLU MLP, written here as explicit loops.
    rng = np.random.default_rng(5)
    T, H, I = 3, 6, 4
    x = rng.normal(size=(T, H))
    w1 = rng.normal(size=(1, 2 * I, H))
    w2 = rng.normal(size=(1, H, I))
    y = moe.expert_loop_forward(x, w1, w2, np.ones((T, 1)), np.zeros((T, 1), dtype=np.int64))
    import math
    for t in range(T):
        h = []
        for i in range(I):
            g = sum(w1[0, i, c] * x[t, c] for c in range(H))
            u = sum(w1[0, I + i, c] * x[t, c] for c in range(H))
            h.append(g / (1 + math.exp(-g)) * u)
        for c in range(H):
            ref = sum(w2[0, c, i] * h[i] for i in range(I))
            assert abs(y[t, c] - ref) <= 1e-12 * max(1.0, abs(ref))


def test_gate_is_first_half():
    # Swapping gate and up halves changes the result (silu is not symmetric): pins the order.
    x, w1, w2, tw, ids = _rand_layer(seed=9)
    a = moe.expert_loop_forward(x, w1, w2, tw, ids)
    I = w1.shape[1] // 2
    swapped = np.concatenate([w1[:, I:], w1[:, :I]], axis=1)
    b = moe.expert_loop_forward(x, swapped, w2, tw, ids)
    assert np.abs(a - b).max() > 1e-3
    # and the first half goes through silu: zero up rows -> zero output
    z = w1.copy(); z[:, I:] = 0
    assert np.abs(moe.expert_loop_forward(x, z, w2, tw, ids)).max() == 0


def test_linear_in_route_weights():
    x, w1, w2, tw, ids = _rand_layer(seed=11)
    a = moe.expert_loop_forward(x, w1, w2, tw, ids)
    b = moe.expert_loop_forward(x, w1, w2, 2 * tw, ids)
    np.testing.assert_allclose(b, 2 * a, rtol=1e-12, atol=1e-14)
    t0 = moe.expert_loop_forward(x, w1, w2, np.where(np.arange(2) == 0, tw, 0), ids)
    t1 = moe.expert_loop_forward(x, w1, w2, np.where(np.arange(2) == 1, tw, 0), ids)
    np.testing.assert_allclose(t0 + t1, a, rtol=1e-12, atol=1e-12)


def test_token_outputs_matches_loop():
    x, w1, w2, tw, ids = _rand_layer(seed=13)
    y = moe.expert_loop_forward(x, w1, w2, tw, ids)
    for t in (0, 5, 12):
        yt = moe.token_outputs(x[t], [w1[e] for e in ids[t]], [w2[e] for e in ids[t]], tw[t])
        np.testing.assert_allclose(yt, y[t], rtol=1e-12, atol=1e-12)


def test_tiny_workload_routes_and_runs():
    cfg = synth.tiny_config()
    acts = synth.moe_activations(cfg, "cpu")
    W = synth.moe_weights(cfg, "cpu")
    y, tw, ids = moe.fused_forward(acts["x"].float().numpy(), acts["gating"].numpy(),
                                   W["w1"].float().numpy(), W["w2"].float().numpy(),
                                   cfg.topk, cfg.renormalize)
    assert y.shape == (cfg.T, cfg.H) and np.all(np.isfinite(y))
    np.testing.assert_allclose(tw.astype(np.float64).sum(1), 1.0, rtol=1e-6)
