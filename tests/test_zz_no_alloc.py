"""moe_fused_forward_noalloc: the layer forward for callers that cannot allocate
device memory (a plug-in inside a framework that owns all device memory, or a
latency-critical caller that cannot afford cudaMalloc). Its scratch is a fixed
array inside the library instead of a caller workspace.

Checked through the C ABI against moe_fused_forward on the same inputs, on two
calls in a row (the shared array keeps the previous call's contents), plus the
rejection of a problem too large for the array, and the read-and-clear of the
array's device error word. This file is collected last so
that a run stopping at the first failure has already run every other test."""
import ctypes

import pytest
import torch

import synth
from gpu_util import assert_moe_close, assert_weights_close, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


CONFIGS = [
    synth.tiny_config(),
    synth.MoEConfig("ragged_T1000_H768_I384_E16_top4_grouped", T=1000, H=768, I=384, E=16, topk=4,
                    num_expert_group=4, topk_group=2, scoring="sigmoid", routed_scaling_factor=2.5,
                    logit_sigma=2.0, seed=11),
    # decode-shaped: 256 experts, grouped sigmoid top-8, T * topk <= 32 * E selects the 16-row-block kernels,
    # whose scratch is far below that of the 128-row layout
    synth.MoEConfig("decode_like_T32_H1024_I512_E256_top8", T=32, H=1024, I=512, E=256, topk=8,
                    num_expert_group=8, topk_group=4, scoring="sigmoid", routed_scaling_factor=2.5,
                    logit_sigma=2.0, seed=15),
]


@pytest.mark.parametrize("cfg", CONFIGS, ids=lambda c: c.name)
def test_noalloc_matches_workspace_entry_point(cfg):
    import mixture_experts_routing_grouped_gb300 as moe
    acts = synth.moe_activations(cfg, "cuda")
    W = synth.moe_weights(cfg, "cuda")
    args = (acts["x"], acts["gating"], W["w1"], W["w2"], cfg.topk, cfg.renormalize, cfg.num_expert_group,
            cfg.topk_group, cfg.scoring, cfg.routed_scaling_factor)
    ref_y, ref_w, ref_ids = moe.moe_fused_forward(*args)
    torch.cuda.synchronize()
    for _ in range(2):
        y, w, ids = moe.moe_fused_forward_noalloc(*args)
        torch.cuda.synchronize()
        assert torch.equal(ids, ref_ids)
        assert_weights_close(w.cpu().numpy(), ref_w.cpu().numpy())
        # both are GPU results whose fp32 reductions may run in different orders (atomics),
        # so a bf16 output can differ by one rounding step, which exceeds 2e-2 once |y| >= 4
        # (the decode-like layer is scaled by 2.5)
        assert_moe_close(y.float().cpu().numpy(), ref_y.float().cpu().numpy(), rel_above_one=True)
    # nothing went wrong on the device, and reading the scratch's error word clears it
    assert moe.moe_fused_forward_noalloc_check_error() == 0


def test_noalloc_rejects_problems_beyond_the_scratch():
    import mixture_experts_routing_grouped_gb300 as moe
    L = moe.lib()
    limit = 64 * 1024 * 1024
    T, H, I, E, k = 4096, 2048, 768, 128, 8
    assert moe.moe_fused_forward_workspace_size(T, H, I, E, k) > limit
    fake = ctypes.c_void_p(0x10000)   # rejected on the host before any pointer is used
    st = L.moe_fused_forward_noalloc(fake, fake, fake, fake, T, H, I, E, 1, 1, k, 0, 1, 1.0, fake, fake, fake, None)
    assert st == 3   # MOE_ERR_WORKSPACE


def test_noalloc_accepts_the_decode_workload_sizes():
    """The decode workload (E=256, H=7168, I=2048, top-8) runs the 16-row-block kernels at
    T <= 128, whose scratch fits the array; the size check follows the selected kernels."""
    import mixture_experts_routing_grouped_gb300 as moe
    limit = 64 * 1024 * 1024
    for T in (1, 8, 32, 128):
        assert 0 < moe.moe_fused_forward_workspace_size(T, 7168, 2048, 256, 8) <= limit
