"""GPU moe_fused_forward (routing -> align -> gate_up GEMM + SwiGLU -> down GEMM
+ weighted combine) vs the float64 oracle.

Every test compares the whole output element by element: small layers against the
oracle's whole-layer function, the full prefill and decode workloads against its
expert loop fed one expert's weights at a time; routing ids bit-exact on all tokens.
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
    # from 8192 tokens the streaming routing kernel, which also writes each 32-token tile's
    # expert counts for align
    synth.MoEConfig("streamed_routing_T8192_H256_I128_E128_top8", T=8192, H=256, I=128, E=128, topk=8, seed=17),
    synth.MoEConfig("streamed_routing_T8192_H256_I128_E256_G8_top8", T=8192, H=256, I=128, E=256, topk=8,
                    num_expert_group=8, topk_group=4, scoring="sigmoid", seed=18),
    # 256 experts on the 128-row kernels: the seven-slot bf16 gate_up instance at its table's limit
    synth.MoEConfig("experts_at_limit_T2048_H256_I128_E256_top8", T=2048, H=256, I=128, E=256, topk=8,
                    num_expert_group=8, topk_group=4, scoring="sigmoid", seed=16),
    # more than 256 experts on the 128-row kernels: the six-slot bf16 gate_up instance
    synth.MoEConfig("many_experts_T4096_H256_I128_E512_top8", T=4096, H=256, I=128, E=512, topk=8,
                    num_expert_group=8, topk_group=4, seed=15),
], ids=lambda c: c.name)
def test_small_layers(cfg):
    _full_check(cfg)


def _host_f64(t):
    """One expert's bf16 matrix as float64 on the host (the exact conversion happens on the device)."""
    return t.double().cpu().numpy()


def _workload_check(cfg, rel_above_one=False):
    """The whole output of a full-size workload against the oracle's expert loop, every element.

    The oracle fetches each active expert's weights from the device copy (made by the seeded
    generator, never by the library) one expert at a time, so the layer never has to be held
    in float64 on the host at once."""
    import mixture_experts_routing_grouped_gb300 as moe
    acts = synth.moe_activations(cfg, "cuda")
    W = synth.moe_weights(cfg, "cuda")
    ws = torch.zeros(moe.moe_fused_forward_workspace_size(cfg.T, cfg.H, cfg.I, cfg.E, cfg.topk),
                     dtype=torch.uint8, device="cuda")
    y, tw, ids = _fused(cfg, acts, W, ws)
    assert moe.moe_check_device_error(ws) == 0
    g = acts["gating"].cpu().numpy()
    rw, rids = routing.grouped_topk(g, cfg.topk, cfg.renormalize, cfg.num_expert_group, cfg.topk_group,
                                    cfg.scoring, cfg.routed_scaling_factor)
    assert np.array_equal(ids.cpu().numpy(), rids)
    assert_weights_close(tw.cpu().numpy(), rw)
    x = acts["x"].double().cpu().numpy()
    ry = omoe.expert_loop_forward(x, lambda e: _host_f64(W["w1"][e]), lambda e: _host_f64(W["w2"][e]), rw, rids)
    assert_moe_close(y.float().cpu().numpy(), ry, rel_above_one=rel_above_one)
    # a second call on the same workspace: the kernels leave their scratch (counters,
    # tickets) as they found it
    y2, _, ids2 = _fused(cfg, acts, W, ws)
    assert torch.equal(ids2, ids)
    assert_moe_close(y2.float().cpu().numpy(), ry, rel_above_one=rel_above_one)


def test_prefill_workload_whole():
    _workload_check(synth.prefill_config())


@pytest.mark.parametrize("T", [1, 8, 32, 128])
def test_decode_workload_whole(T):
    # outputs scaled by 2.5 reach |y| >= 8, where one bf16 rounding exceeds 2e-2 absolute
    _workload_check(synth.decode_config(T), rel_above_one=True)


def test_T0_is_a_no_op():
    import mixture_experts_routing_grouped_gb300 as moe
    cfg = synth.tiny_config()
    W = synth.moe_weights(cfg, "cuda")
    x = torch.empty((0, cfg.H), dtype=torch.bfloat16, device="cuda")
    g = torch.empty((0, cfg.E), dtype=torch.float32, device="cuda")
    y, tw, ids = moe.moe_fused_forward(x, g, W["w1"], W["w2"], cfg.topk)
    assert y.shape == (0, cfg.H)
