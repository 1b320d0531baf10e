"""GPU moe_fused_forward (routing -> align -> gate_up GEMM + SwiGLU -> down GEMM
+ weighted combine) vs the float64 oracle.

Small layers are compared element by element on the whole output; the full
prefill and decode workloads on sampled tokens (each sampled token's output is
recomputed by the oracle from its own experts), plus exact routing on all tokens.
"""
import numpy as np
import pytest
import torch

from gpu_util import assert_moe_close, assert_weights_close, require_gpu
from oracle import moe as omoe
from oracle import routing
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _fused(cfg, acts, W, ws=None):
    import mixture_experts_routing_grouped_gb300 as moe
    out = moe.moe_fused_forward(acts["x"], acts["gating"], W["w1"], W["w2"], cfg.topk, cfg.renormalize,
                                cfg.num_expert_group, cfg.topk_group, cfg.scoring, cfg.routed_scaling_factor, ws=ws)
    torch.cuda.synchronize()
    return out


def _full_check(cfg):
    import mixture_experts_routing_grouped_gb300 as moe
    acts = synth.moe_activations(cfg, "cuda")
    W = synth.moe_weights(cfg, "cuda")
    ws = torch.zeros(moe.moe_fused_forward_workspace_size(cfg.T, cfg.H, cfg.I, cfg.E, cfg.topk),
                     dtype=torch.uint8, device="cuda")
    y, tw, ids = _fused(cfg, acts, W, ws)
    ry, rw, rids = omoe.fused_forward(acts["x"].float().cpu().numpy(), acts["gating"].cpu().numpy(),
                                      W["w1"].float().cpu().numpy(), W["w2"].float().cpu().numpy(), cfg.topk,
                                      cfg.renormalize, cfg.num_expert_group, cfg.topk_group, cfg.scoring,
                                      cfg.routed_scaling_factor)
    assert np.array_equal(ids.cpu().numpy(), rids)
    assert_weights_close(tw.cpu().numpy(), rw)
    assert_moe_close(y.float().cpu().numpy(), ry)
    assert moe.moe_check_device_error(ws) == 0
    # a second call on the same workspace gives the same routing and a close output
    y2, _, ids2 = _fused(cfg, acts, W, ws)
    assert torch.equal(ids2, ids)
    assert_moe_close(y2.float().cpu().numpy(), ry)


def test_tiny_layer():
    _full_check(synth.tiny_config())


@pytest.mark.parametrize("cfg", [
    synth.MoEConfig("ragged_T1000_H768_I384_E16_top4_grouped", T=1000, H=768, I=384, E=16, topk=4,
                    num_expert_group=4, topk_group=2, scoring="sigmoid", routed_scaling_factor=2.5,
                    logit_sigma=2.0, seed=11),
    synth.MoEConfig("ragged_T37_H256_I128_E8_top2", T=37, H=256, I=128, E=8, topk=2, seed=12),
    synth.MoEConfig("one_token_H512_I256_E64_top8", T=1, H=512, I=256, E=64, topk=8, num_expert_group=8,
                    topk_group=4, scoring="sigmoid", routed_scaling_factor=2.5, seed=13),
    synth.MoEConfig("skewed_T600_H512_I256_E4_top1_norenorm", T=600, H=512, I=256, E=4, topk=1, renormalize=False,
                    seed=14, logit_sigma=3.0),
], ids=lambda c: c.name)
def test_small_layers(cfg):
    _full_check(cfg)


def _sampled_check(cfg, n_samples=12):
    import mixture_experts_routing_grouped_gb300 as moe
    acts = synth.moe_activations(cfg, "cuda")
    W = synth.moe_weights(cfg, "cuda")
    ws = torch.zeros(moe.moe_fused_forward_workspace_size(cfg.T, cfg.H, cfg.I, cfg.E, cfg.topk),
                     dtype=torch.uint8, device="cuda")
    y, tw, ids = _fused(cfg, acts, W, ws)
    g = acts["gating"].cpu().numpy()
    rw, rids = routing.grouped_topk(g, cfg.topk, cfg.renormalize, cfg.num_expert_group, cfg.topk_group,
                                    cfg.scoring, cfg.routed_scaling_factor)
    assert np.array_equal(ids.cpu().numpy(), rids)
    assert_weights_close(tw.cpu().numpy(), rw)
    rng = np.random.default_rng(cfg.T)
    toks = sorted(set([0, cfg.T - 1] + rng.integers(0, cfg.T, size=n_samples).tolist()))
    x = acts["x"].float().cpu().numpy()
    got = y[toks].float().cpu().numpy()
    ref = np.stack([omoe.token_outputs(x[t], [W["w1"][e].float().cpu().numpy() for e in rids[t]],
                                       [W["w2"][e].float().cpu().numpy() for e in rids[t]], rw[t]) for t in toks])
    assert_moe_close(got, ref)
    assert moe.moe_check_device_error(ws) == 0
    yf = y.float()
    assert torch.isfinite(yf).all()


def test_prefill_workload_sampled():
    _sampled_check(synth.prefill_config())


@pytest.mark.parametrize("T", [1, 8, 32, 128])
def test_decode_workload_sampled(T):
    _sampled_check(synth.decode_config(T), n_samples=6)


def test_T0_is_a_no_op():
    import mixture_experts_routing_grouped_gb300 as moe
    cfg = synth.tiny_config()
    W = synth.moe_weights(cfg, "cuda")
    x = torch.empty((0, cfg.H), dtype=torch.bfloat16, device="cuda")
    g = torch.empty((0, cfg.E), dtype=torch.float32, device="cuda")
    y, tw, ids = moe.moe_fused_forward(x, g, W["w1"], W["w2"], cfg.topk)
    assert y.shape == (0, cfg.H)
