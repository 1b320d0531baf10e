"""The fused layers captured into a CUDA graph: every call of the boundary is
asynchronous on the caller's stream and makes no host synchronisation, so a
captured call replays the whole layer. The FP8 forward forks the quantisation of x
onto a second stream and joins it back, which the capture must carry as a branch.

Each layer is called once eagerly first (kernel loading and the library's stream and
events are set up outside the capture), then captured with preallocated outputs and
workspace, then replayed on new inputs copied into the captured input buffers; the
replay is compared with an eager call on the same inputs (ids exactly; y within the
layer tolerance, the fp32 combine's summation order being free)."""
import pytest
import torch

from gpu_util import assert_moe_close, require_gpu
from oracle import quant
import synth

pytestmark = pytest.mark.gpu

CFG = synth.MoEConfig("ragged_T1000_H768_I384_E16_top4_grouped", T=1000, H=768, I=384, E=16, topk=4,
                      num_expert_group=4, topk_group=2, scoring="sigmoid", routed_scaling_factor=2.5,
                      logit_sigma=2.0, seed=11)


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _outputs(cfg, dev):
    return (torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16, device=dev),
            torch.empty((cfg.T, cfg.topk), dtype=torch.float32, device=dev),
            torch.empty((cfg.T, cfg.topk), dtype=torch.int32, device=dev))


def _replay_matches_eager(call, x, g, x_new, g_new, outs, fresh_outs):
    call(x, g, *outs)                                  # eager: loads kernels, sets up streams
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call(x, g, *outs)
    x.copy_(x_new)
    g.copy_(g_new)
    graph.replay()
    torch.cuda.synchronize()
    call(x_new, g_new, *fresh_outs)
    torch.cuda.synchronize()
    y, tw, ids = outs
    ry, rtw, rids = fresh_outs
    assert torch.equal(ids, rids)
    assert torch.equal(tw, rtw)
    assert_moe_close(y.float().cpu().numpy(), ry.float().cpu().numpy())


def _inputs(cfg, seed_shift):
    c = synth.MoEConfig(**{**cfg.__dict__, "seed": cfg.seed + seed_shift})
    a = synth.moe_activations(c, "cuda")
    return a["x"].contiguous(), a["gating"].contiguous()


def test_bf16_layer_replays_from_a_cuda_graph():
    import mixture_experts_routing_grouped_gb300 as moe
    cfg = CFG
    W = synth.moe_weights(cfg, "cuda")
    ws = torch.zeros(moe.moe_fused_forward_workspace_size(cfg.T, cfg.H, cfg.I, cfg.E, cfg.topk), dtype=torch.uint8,
                     device="cuda")
    ws2 = torch.zeros_like(ws)

    def call(x, g, y, tw, ids):
        moe.moe_fused_forward(x, g, W["w1"], W["w2"], cfg.topk, cfg.renormalize, cfg.num_expert_group,
                              cfg.topk_group, cfg.scoring, cfg.routed_scaling_factor,
                              ws=ws if y.data_ptr() == outs[0].data_ptr() else ws2, y=y, topk_weights=tw,
                              topk_ids=ids)

    x, g = _inputs(cfg, 0)
    x_new, g_new = _inputs(cfg, 100)
    outs = _outputs(cfg, "cuda")
    _replay_matches_eager(call, x, g, x_new, g_new, outs, _outputs(cfg, "cuda"))


def test_fp8_layer_replays_from_a_cuda_graph():
    import mixture_experts_routing_grouped_gb300 as moe
    cfg = CFG
    W = synth.moe_weights(cfg, "cuda")
    E, I, H = cfg.E, cfg.I, cfg.H
    q1, s1 = quant.quant_rows_e4m3(W["w1"].float().cpu().numpy().reshape(E * 2 * I, H))
    q2, s2 = quant.quant_rows_e4m3(W["w2"].float().cpu().numpy().reshape(E * H, I))
    q1 = torch.from_numpy(q1).view(E, 2 * I, H).cuda()
    q2 = torch.from_numpy(q2).view(E, H, I).cuda()
    s1 = torch.from_numpy(s1).view(E, 2 * I).cuda()
    s2 = torch.from_numpy(s2).view(E, H).cuda()
    ws = torch.zeros(moe.moe_fused_forward_fp8_workspace_size(cfg.T, H, I, E, cfg.topk), dtype=torch.uint8,
                     device="cuda")
    ws2 = torch.zeros_like(ws)

    def call(x, g, y, tw, ids):
        moe.moe_fused_forward_fp8(x, g, q1, s1, q2, s2, cfg.topk, cfg.renormalize, cfg.num_expert_group,
                                  cfg.topk_group, cfg.scoring, cfg.routed_scaling_factor,
                                  ws=ws if y.data_ptr() == outs[0].data_ptr() else ws2, y=y, topk_weights=tw,
                                  topk_ids=ids)

    x, g = _inputs(cfg, 0)
    x_new, g_new = _inputs(cfg, 100)
    outs = _outputs(cfg, "cuda")
    _replay_matches_eager(call, x, g, x_new, g_new, outs, _outputs(cfg, "cuda"))
    assert moe.moe_check_device_error(ws) == 0
