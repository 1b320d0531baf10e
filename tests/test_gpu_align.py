"""GPU moe_align_block_size vs the oracle: every output buffer bit-exact."""
import numpy as np
import pytest
import torch

from gpu_util import require_gpu
from oracle import align, routing
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _check(ids_np, E, bm):
    import mixture_experts_routing_grouped_gb300 as moe
    ids = torch.from_numpy(np.ascontiguousarray(ids_np, dtype=np.int32)).cuda()
    ws = torch.zeros(moe.lib().moe_align_workspace_size(ids.numel(), E, bm), dtype=torch.uint8, device="cuda")
    s, eids, off, ntpp = moe.moe_align_block_size(ids, bm, E, ws=ws)
    s2, _, _, _ = moe.moe_align_block_size(ids, bm, E, ws=ws)   # the workspace is reusable as left
    assert torch.equal(s, s2)
    torch.cuda.synchronize()
    rs, reids, roff, rtotal = align.moe_align_block_size(ids_np, bm, E)
    assert int(ntpp.item()) == rtotal
    assert np.array_equal(off.cpu().numpy(), roff)
    assert np.array_equal(s.cpu().numpy(), rs)
    assert np.array_equal(eids.cpu().numpy(), reids)
    assert moe.moe_check_device_error(ws) == 0


@pytest.mark.parametrize("n", [0, 1, 5, 31, 33, 1000, 1024, 32768, 131072])
@pytest.mark.parametrize("E,bm", [(8, 4), (128, 128), (256, 16), (1000, 64), (1024, 256), (3, 1)])
def test_align_random(n, E, bm):
    rng = np.random.default_rng(n * 31 + E)
    _check(rng.integers(0, E, size=n), E, bm)


def test_align_skewed_and_single_expert():
    rng = np.random.default_rng(9)
    z = np.minimum(rng.zipf(1.3, size=20000) - 1, 255)
    _check(z, 256, 128)
    _check(np.full(5000, 17), 64, 32)


@pytest.mark.parametrize("cfg", [synth.tiny_config(), synth.prefill_config(), synth.decode_config(32)],
                         ids=lambda c: c.name)
def test_align_of_routed_workloads(cfg):
    g = synth.gating_logits(cfg, "cpu").numpy()
    _, ids = routing.grouped_topk(g, cfg.topk, cfg.renormalize, cfg.num_expert_group, cfg.topk_group, cfg.scoring,
                                  cfg.routed_scaling_factor)
    for bm in (16, 128):
        _check(ids.reshape(-1), cfg.E, bm)


def test_align_out_of_range_ids_are_skipped_and_reported():
    import mixture_experts_routing_grouped_gb300 as moe
    ids_np = np.array([3, 9, 1, -1, 3, 0, 7], dtype=np.int32)   # 9 and -1 are outside [0, 8)
    ids = torch.from_numpy(ids_np).cuda()
    ws = torch.zeros(moe.lib().moe_align_workspace_size(7, 8, 4), dtype=torch.uint8, device="cuda")
    s, eids, off, ntpp = moe.moe_align_block_size(ids, 4, 8, ws=ws)
    code = moe.moe_check_device_error(ws)
    assert code & moe.DEVERR_EXPERT_ID
    valid = np.array([p for p in range(7) if 0 <= ids_np[p] < 8])
    placed = s.cpu().numpy()[: int(ntpp.item())]
    assert sorted(placed[placed < 7].tolist()) == valid.tolist()
    assert moe.moe_check_device_error(ws) == 0   # reading clears the word
