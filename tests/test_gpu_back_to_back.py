"""Calls enqueued back to back on one stream, with no host synchronisation between them.

Every kernel of the library is launched as a programmatic dependent of the kernel before it
in the stream: it may start while that kernel finishes and waits in-kernel for its
completion before touching global memory. These tests queue several calls (different
layers, the same workspace twice, gmm_lowp's task counters, routing) before a single
synchronisation and check every result against the oracle, so that a kernel reading or
writing memory before its predecessor had finished would show up as a wrong result."""
import numpy as np
import pytest
import torch

from gpu_util import assert_moe_close, assert_weights_close, require_gpu
from oracle import gmm as ogmm
from oracle import moe as omoe
from oracle import quant
from oracle import routing
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


LAYERS = [
    synth.tiny_config(),
    # 16-row-block (decode) kernels
    synth.MoEConfig("one_token_H512_I256_E64_top8", T=1, H=512, I=256, E=64, topk=8, num_expert_group=8,
                    topk_group=4, scoring="sigmoid", routed_scaling_factor=2.5, seed=13),
    # 128-row-block kernels
    synth.MoEConfig("ragged_T1000_H768_I384_E16_top4_grouped", T=1000, H=768, I=384, E=16, topk=4,
                    num_expert_group=4, topk_group=2, scoring="sigmoid", routed_scaling_factor=2.5,
                    logit_sigma=2.0, seed=11),
]


def _layer_inputs(cfg):
    return synth.moe_activations(cfg, "cuda"), synth.moe_weights(cfg, "cuda")


def _oracle(cfg, acts, W):
    return omoe.fused_forward(acts["x"].float().cpu().numpy(), acts["gating"].cpu().numpy(),
                              W["w1"].float().cpu().numpy(), W["w2"].float().cpu().numpy(), cfg.topk,
                              cfg.renormalize, cfg.num_expert_group, cfg.topk_group, cfg.scoring,
                              cfg.routed_scaling_factor)


def _call(moe, cfg, acts, W, ws):
    return moe.moe_fused_forward(acts["x"], acts["gating"], W["w1"], W["w2"], cfg.topk, cfg.renormalize,
                                 cfg.num_expert_group, cfg.topk_group, cfg.scoring, cfg.routed_scaling_factor,
                                 ws=ws)


def test_layers_back_to_back():
    """Three layers (both kernel families), each twice on its own workspace, all queued first."""
    import mixture_experts_routing_grouped_gb300 as moe
    data = [(cfg, *_layer_inputs(cfg)) for cfg in LAYERS]
    torch.cuda.synchronize()
    outs = []
    for cfg, acts, W in data + data:
        ws = torch.zeros(moe.moe_fused_forward_workspace_size(cfg.T, cfg.H, cfg.I, cfg.E, cfg.topk),
                         dtype=torch.uint8, device="cuda")
        outs.append((cfg, acts, W, ws, _call(moe, cfg, acts, W, ws)))
    torch.cuda.synchronize()
    for cfg, acts, W, ws, (y, tw, ids) in outs:
        ry, rw, rids = _oracle(cfg, acts, W)
        assert np.array_equal(ids.cpu().numpy(), rids), cfg.name
        assert_weights_close(tw.cpu().numpy(), rw)
        assert_moe_close(y.float().cpu().numpy(), ry, rel_above_one=True)
        assert moe.moe_check_device_error(ws) == 0


@pytest.mark.parametrize("cfg", LAYERS[1:], ids=lambda c: c.name)
def test_same_workspace_back_to_back(cfg):
    """One workspace, four calls queued: each call's kernels start while the previous call's
    last kernels finish, and read the workspace only after them."""
    import mixture_experts_routing_grouped_gb300 as moe
    acts, W = _layer_inputs(cfg)
    ws = torch.zeros(moe.moe_fused_forward_workspace_size(cfg.T, cfg.H, cfg.I, cfg.E, cfg.topk),
                     dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    outs = [_call(moe, cfg, acts, W, ws) for _ in range(4)]
    torch.cuda.synchronize()
    ry, rw, rids = _oracle(cfg, acts, W)
    for y, tw, ids in outs:
        assert np.array_equal(ids.cpu().numpy(), rids)
        assert_weights_close(tw.cpu().numpy(), rw)
        assert_moe_close(y.float().cpu().numpy(), ry, rel_above_one=True)
    assert moe.moe_check_device_error(ws) == 0


@pytest.mark.parametrize("dt", ["i8", "e4m3"])
def test_gmm_lowp_back_to_back(dt):
    """gmm_lowp on one workspace with different group layouts, queued without a sync: each
    call's task counters must be back at zero when the next call's kernel reads them."""
    import mixture_experts_routing_grouped_gb300 as moe
    rng = np.random.default_rng(21)
    K, N, E = 256, 384, 5
    ws = torch.zeros(moe.gmm_lowp_workspace_size(700, K, N, E), dtype=torch.uint8, device="cuda")
    tdt = torch.int8 if dt == "i8" else torch.float8_e4m3fn
    cases = []
    for sizes in ([100, 0, 300, 1, 299], [700, 0, 0, 0, 0], [1, 2, 3, 4, 5], [0, 0, 0, 0, 129], [64] * 5):
        M = sum(sizes)
        x = rng.standard_normal((M, K))
        w = 0.05 * rng.standard_normal((E * N, K))
        qfn = quant.quant_rows_int8 if dt == "i8" else quant.quant_rows_e4m3
        qx, sx = qfn(x)
        qw, sw = qfn(w)
        off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
        dev = lambda c: (torch.from_numpy(np.ascontiguousarray(c.astype(np.int8))).cuda() if dt == "i8" else
                         torch.from_numpy(np.ascontiguousarray(c.astype(np.uint8))).cuda().view(tdt))
        args = (dev(qx), dev(qw).view(E, N, K), torch.from_numpy(sx.astype(np.float32)).cuda(),
                torch.from_numpy(sw.astype(np.float32)).cuda().view(E, N), torch.from_numpy(off).cuda(),
                torch.from_numpy(np.asarray(sizes, dtype=np.int32)).cuda())
        cases.append((qx, qw.reshape(E, N, K), sx, sw.reshape(E, N), off, sizes, args))
    torch.cuda.synchronize()
    outs = [moe.gmm_lowp(*c[6], out_dtype=torch.float32, ws=ws) for c in cases]
    torch.cuda.synchronize()
    assert moe.moe_check_device_error(ws) == 0
    assert torch.count_nonzero(ws[4:12]).item() == 0
    for (qx, qw, sx, sw, off, sizes, _), out in zip(cases, outs):
        ref = ogmm.gmm(qx, qw, sx, sw, off, sizes, dt)
        got = out.cpu().numpy().astype(np.float64)
        assert np.linalg.norm(got - ref) <= 1e-3 * np.linalg.norm(ref)
        assert np.abs(got - ref).max() <= 1e-3 * np.abs(ref).max()


def test_routing_back_to_back():
    """Routing calls of both kernels (segmented below 8192 tokens, streaming from 8192 on)
    queued without a sync."""
    import mixture_experts_routing_grouped_gb300 as moe
    cases = []
    for T, scoring in ((4096, "softmax"), (16384, "sigmoid"), (128, "sigmoid"), (16384, "softmax")):
        cfg = synth.routing_config(T, scoring)
        cases.append((cfg, synth.gating_logits(cfg, "cuda")))
    torch.cuda.synchronize()
    outs = [moe.moe_grouped_topk(g, cfg.topk, True, cfg.num_expert_group, cfg.topk_group, cfg.scoring,
                                 cfg.routed_scaling_factor) for cfg, g in cases]
    torch.cuda.synchronize()
    for (cfg, g), (w, ids) in zip(cases, outs):
        rw, rids = routing.grouped_topk(g.cpu().numpy(), cfg.topk, True, cfg.num_expert_group, cfg.topk_group,
                                        cfg.scoring, cfg.routed_scaling_factor)
        assert np.array_equal(ids.cpu().numpy(), rids)
        assert_weights_close(w.cpu().numpy(), rw)
