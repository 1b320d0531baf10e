"""GPU moe_fused_forward_fp8 (routing -> align -> per-token e4m3 x -> FP8 gate_up +
SwiGLU -> per-row e4m3 h -> FP8 down + weighted combine) vs the float64 oracle
``oracle.moe.fused_forward_fp8``.

The e4m3 weight codes and their per-channel scales are made on the CPU by the
oracle's quantiser and uploaded, so every input both sides see is the same and
none of the oracle's inputs comes from the CUDA path. Small layers and the full
prefill workload are compared on the whole output (the prefill workload through
the oracle's expert loop, every expert's codes quantised on the CPU and checked
against the device copy). The decode workload (E=256, H=7168, I=2048, T=1..128:
the swap-AB kernels with e4m3 weights) is compared on the whole output too, its
weight codes made on the device by torch's e4m3 cast (the same rounding; checked
against the oracle's quantiser on sampled experts) and fed to the oracle's expert
loop, one active expert at a time.
Tolerance as for the bf16 layer: |dy| <= 2e-2 per element and a
relative Frobenius error <= 1e-2 (the two sides quantise the same x codes; h is
computed in fp32 on the GPU and float64 in the oracle before its bf16 rounding
and e4m3 quantisation, so a rare code of h may differ by one step).
"""
import numpy as np
import pytest
import torch

from gpu_util import assert_moe_close, assert_weights_close, require_gpu
from oracle import moe as omoe
from oracle import quant, routing
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _quant_weights_cpu(w):
    """[E, R, K] bf16 weights -> (codes uint8 [E, R, K], scales fp32 [E, R]) by the oracle's quantiser."""
    E, R, K = w.shape
    q, s = quant.quant_rows_e4m3(w.float().cpu().numpy().reshape(E * R, K))
    return q.reshape(E, R, K), s.reshape(E, R)


def _fp8(cfg, acts, q1, s1, q2, s2, ws=None):
    import mixture_experts_routing_grouped_gb300 as moe
    dev = acts["x"].device
    out = moe.moe_fused_forward_fp8(acts["x"], acts["gating"], torch.from_numpy(q1).to(dev),
                                    torch.from_numpy(s1).to(dev), torch.from_numpy(q2).to(dev),
                                    torch.from_numpy(s2).to(dev), cfg.topk, cfg.renormalize, cfg.num_expert_group,
                                    cfg.topk_group, cfg.scoring, cfg.routed_scaling_factor, ws=ws)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("cfg", [
    synth.tiny_config(),
    synth.MoEConfig("ragged_T1000_H768_I384_E16_top4_grouped", T=1000, H=768, I=384, E=16, topk=4,
                    num_expert_group=4, topk_group=2, scoring="sigmoid", routed_scaling_factor=2.5,
                    logit_sigma=2.0, seed=11),
    synth.MoEConfig("ragged_T37_H256_I128_E8_top2", T=37, H=256, I=128, E=8, topk=2, seed=12),
    synth.MoEConfig("one_token_H512_I256_E64_top8", T=1, H=512, I=256, E=64, topk=8, num_expert_group=8,
                    topk_group=4, scoring="sigmoid", routed_scaling_factor=2.5, seed=13),
], ids=lambda c: c.name)
def test_fp8_small_layers(cfg):
    import mixture_experts_routing_grouped_gb300 as moe
    acts = synth.moe_activations(cfg, "cuda")
    W = synth.moe_weights(cfg, "cuda")
    q1, s1 = _quant_weights_cpu(W["w1"])
    q2, s2 = _quant_weights_cpu(W["w2"])
    ws = torch.zeros(moe.moe_fused_forward_fp8_workspace_size(cfg.T, cfg.H, cfg.I, cfg.E, cfg.topk),
                     dtype=torch.uint8, device="cuda")
    y, tw, ids = _fp8(cfg, acts, q1, s1, q2, s2, ws)
    ry, rw, rids = omoe.fused_forward_fp8(acts["x"].float().cpu().numpy(), acts["gating"].cpu().numpy(),
                                          q1, s1, q2, s2, cfg.topk, cfg.renormalize, cfg.num_expert_group,
                                          cfg.topk_group, cfg.scoring, cfg.routed_scaling_factor)
    assert np.array_equal(ids.cpu().numpy(), rids)
    assert_weights_close(tw.cpu().numpy(), rw)
    assert_moe_close(y.float().cpu().numpy(), ry)
    assert moe.moe_check_device_error(ws) == 0
    # a second call on the same workspace gives the same result up to accumulation order
    y2, _, ids2 = _fp8(cfg, acts, q1, s1, q2, s2, ws)
    assert torch.equal(ids2, ids)
    assert_moe_close(y2.float().cpu().numpy(), ry)


def _dev_quant(w, chunk=16):
    """Device-side weight codes: torch's float8_e4m3fn cast (nearest, ties to even) of w / (absmax / 448)
    in fp32, per output channel, a few experts at a time (tensor / tensor divisions: torch on CUDA
    multiplies by the reciprocal of a Python scalar divisor)."""
    E, R, K = w.shape
    q = torch.empty((E, R, K), dtype=torch.uint8, device=w.device)
    sc = torch.empty((E, R), dtype=torch.float32, device=w.device)
    for e0 in range(0, E, chunk):
        w32 = w[e0:e0 + chunk].float()
        amax = w32.abs().amax(dim=2)
        s = amax / torch.full_like(amax, 448.0)
        s = torch.where(s == 0, torch.ones_like(s), s)
        q[e0:e0 + chunk] = (w32 / s[:, :, None]).to(torch.float8_e4m3fn).view(torch.uint8)
        sc[e0:e0 + chunk] = s
        del w32
    return q, sc


def test_fp8_prefill_workload_whole():
    import mixture_experts_routing_grouped_gb300 as moe
    cfg = synth.prefill_config()
    acts = synth.moe_activations(cfg, "cuda")
    W = synth.moe_weights(cfg, "cuda")
    dq1, ds1 = _dev_quant(W["w1"])
    dq2, ds2 = _dev_quant(W["w2"])
    ws = torch.zeros(moe.moe_fused_forward_fp8_workspace_size(cfg.T, cfg.H, cfg.I, cfg.E, cfg.topk),
                     dtype=torch.uint8, device="cuda")
    y, tw, ids = moe.moe_fused_forward_fp8(acts["x"], acts["gating"], dq1, ds1, dq2, ds2, cfg.topk, cfg.renormalize,
                                           cfg.num_expert_group, cfg.topk_group, cfg.scoring,
                                           cfg.routed_scaling_factor, ws=ws)
    torch.cuda.synchronize()
    rw, rids = routing.grouped_topk(acts["gating"].cpu().numpy(), cfg.topk, cfg.renormalize, cfg.num_expert_group,
                                    cfg.topk_group, cfg.scoring, cfg.routed_scaling_factor)
    assert np.array_equal(ids.cpu().numpy(), rids)
    assert_weights_close(tw.cpu().numpy(), rw)
    assert moe.moe_check_device_error(ws) == 0
    # every expert's codes, quantised on the CPU by the oracle; the device copy must hold the same codes,
    # and the oracle sums with its own
    host = {}
    for e in range(cfg.E):
        q1, s1 = _quant_weights_cpu(W["w1"][e:e + 1])
        q2, s2 = _quant_weights_cpu(W["w2"][e:e + 1])
        assert np.array_equal(dq1[e].cpu().numpy(), q1[0]) and np.array_equal(ds1[e].cpu().numpy(), s1[0])
        assert np.array_equal(dq2[e].cpu().numpy(), q2[0]) and np.array_equal(ds2[e].cpu().numpy(), s2[0])
        host[e] = (q1[0], s1[0], q2[0], s2[0])
    x = acts["x"].float().cpu().numpy()
    ry = omoe.expert_loop_forward_fp8(x, lambda e: host[e][0], lambda e: host[e][1], lambda e: host[e][2],
                                      lambda e: host[e][3], rw, rids)
    assert_moe_close(y.float().cpu().numpy(), ry)


@pytest.fixture(scope="module")
def decode_fp8_weights():
    """The decode workload's weights (E=256, H=7168, I=2048) and their device-made e4m3 codes; the codes
    of a few experts are checked against the oracle's quantiser."""
    cfg = synth.decode_config(1)
    W = synth.moe_weights(cfg, "cuda")
    dq1, ds1 = _dev_quant(W["w1"])
    dq2, ds2 = _dev_quant(W["w2"])
    for e in (0, 137, cfg.E - 1):
        q1, s1 = _quant_weights_cpu(W["w1"][e:e + 1])
        q2, s2 = _quant_weights_cpu(W["w2"][e:e + 1])
        assert np.array_equal(dq1[e].cpu().numpy(), q1[0]) and np.array_equal(ds1[e].cpu().numpy(), s1[0])
        assert np.array_equal(dq2[e].cpu().numpy(), q2[0]) and np.array_equal(ds2[e].cpu().numpy(), s2[0])
    del W
    torch.cuda.empty_cache()
    return dq1, ds1, dq2, ds2


@pytest.mark.parametrize("T", [1, 8, 32, 128])
def test_fp8_decode_workload_whole(decode_fp8_weights, T):
    # decode sizes (T * topk <= 32 * E) run the swap-AB kernels with e4m3 weights
    import mixture_experts_routing_grouped_gb300 as moe
    cfg = synth.decode_config(T)
    dq1, ds1, dq2, ds2 = decode_fp8_weights
    acts = synth.moe_activations(cfg, "cuda")
    ws = torch.zeros(moe.moe_fused_forward_fp8_workspace_size(cfg.T, cfg.H, cfg.I, cfg.E, cfg.topk),
                     dtype=torch.uint8, device="cuda")
    y, tw, ids = moe.moe_fused_forward_fp8(acts["x"], acts["gating"], dq1, ds1, dq2, ds2, cfg.topk, cfg.renormalize,
                                           cfg.num_expert_group, cfg.topk_group, cfg.scoring,
                                           cfg.routed_scaling_factor, ws=ws)
    torch.cuda.synchronize()
    assert moe.moe_check_device_error(ws) == 0
    rw, rids = routing.grouped_topk(acts["gating"].cpu().numpy(), cfg.topk, cfg.renormalize, cfg.num_expert_group,
                                    cfg.topk_group, cfg.scoring, cfg.routed_scaling_factor)
    assert np.array_equal(ids.cpu().numpy(), rids)
    assert_weights_close(tw.cpu().numpy(), rw)
    x = acts["x"].float().cpu().numpy()
    ry = omoe.expert_loop_forward_fp8(x, lambda e: dq1[e].cpu().numpy(), lambda e: ds1[e].cpu().numpy(),
                                      lambda e: dq2[e].cpu().numpy(), lambda e: ds2[e].cpu().numpy(), rw, rids)
    # outputs scaled by 2.5 reach |y| >= 8, where one bf16 rounding exceeds 2e-2 absolute
    assert_moe_close(y.float().cpu().numpy(), ry, rel_above_one=True)


def test_fp8_T0_is_a_no_op():
    import mixture_experts_routing_grouped_gb300 as moe
    cfg = synth.tiny_config()
    W = synth.moe_weights(cfg, "cuda")
    q1, s1 = _quant_weights_cpu(W["w1"])
    q2, s2 = _quant_weights_cpu(W["w2"])
    x = torch.empty((0, cfg.H), dtype=torch.bfloat16, device="cuda")
    g = torch.empty((0, cfg.E), dtype=torch.float32, device="cuda")
    y, tw, ids = moe.moe_fused_forward_fp8(x, g, torch.from_numpy(q1).cuda(), torch.from_numpy(s1).cuda(),
                                           torch.from_numpy(q2).cuda(), torch.from_numpy(s2).cuda(), cfg.topk)
    assert y.shape == (0, cfg.H)
