"""Failure detection on the device, without a fault: the bounded wait of the GEMM kernels
(an mbarrier wait with a time limit, which raises the CTA's abort flag and reports
MOE_DEVERR_TIMEOUT instead of hanging) made to run out by moe_wait_timeout_probe on a
barrier that nothing completes; the host reads the error word, and the context stays
usable: a layer forward right after is correct."""
import time

import numpy as np
import pytest
import torch

from gpu_util import assert_moe_close, require_gpu
from oracle import moe as omoe
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


@pytest.mark.parametrize("limit_ns", [100_000, 5_000_000])
def test_bounded_wait_runs_out_and_reports_timeout(limit_ns):
    import mixture_experts_routing_grouped_gb300 as moe
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    moe.moe_wait_timeout_probe(ws, limit_ns)
    code = moe.moe_check_device_error(ws)          # synchronises the stream
    elapsed = time.perf_counter() - t0
    assert code == moe.DEVERR_TIMEOUT
    assert elapsed >= limit_ns * 1e-9              # the wait lasted at least its limit ...
    assert elapsed < 1.5                           # ... and the second warp left through the abort flag
    assert moe.moe_check_device_error(ws) == 0     # the read cleared the word


def test_layer_is_correct_after_a_timeout():
    import mixture_experts_routing_grouped_gb300 as moe
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    moe.moe_wait_timeout_probe(ws, 1_000_000)
    assert moe.moe_check_device_error(ws) == moe.DEVERR_TIMEOUT
    cfg = synth.tiny_config()
    acts = synth.moe_activations(cfg, "cuda")
    W = synth.moe_weights(cfg, "cuda")
    y, tw, ids = moe.moe_fused_forward(acts["x"], acts["gating"], W["w1"], W["w2"], cfg.topk, cfg.renormalize)
    torch.cuda.synchronize()
    ry, _, rids = omoe.fused_forward(acts["x"].float().cpu().numpy(), acts["gating"].cpu().numpy(),
                                     W["w1"].float().cpu().numpy(), W["w2"].float().cpu().numpy(), cfg.topk,
                                     cfg.renormalize)
    assert np.array_equal(ids.cpu().numpy(), rids)
    assert_moe_close(y.float().cpu().numpy(), ry)


def test_probe_rejects_bad_limits():
    import mixture_experts_routing_grouped_gb300 as moe
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    for bad in (0, 3_000_000_000):
        with pytest.raises(moe.MoeError):
            moe.moe_wait_timeout_probe(ws, bad)
