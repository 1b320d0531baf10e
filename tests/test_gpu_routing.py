"""GPU routing (moe_grouped_topk through the C ABI) vs the oracle: ids bit-exact,
weights within 1e-6 relative."""
import numpy as np
import pytest
import torch

from gpu_util import assert_weights_close, require_gpu
from oracle import routing
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _run(logits_np, k, renorm, G, kg, scoring, rsf):
    import mixture_experts_routing_grouped_gb300 as moe
    g = torch.from_numpy(np.ascontiguousarray(logits_np, dtype=np.float32)).cuda()
    w, ids = moe.moe_grouped_topk(g, k, renorm, G, kg, scoring, rsf)
    torch.cuda.synchronize()
    rw, rids = routing.grouped_topk(logits_np, k, renorm, G, kg, scoring, rsf)
    got_ids = ids.cpu().numpy()
    assert np.array_equal(got_ids, rids), f"{(got_ids != rids).any(1).sum()} rows differ"
    assert_weights_close(w.cpu().numpy(), rw)


@pytest.mark.parametrize("T", [1, 128, 4096, 16384, 65536])
@pytest.mark.parametrize("scoring", ["softmax", "sigmoid"])
def test_routing_workload(T, scoring):
    cfg = synth.routing_config(T, scoring)
    g = synth.gating_logits(cfg, "cuda").cpu().numpy()
    _run(g, cfg.topk, True, cfg.num_expert_group, cfg.topk_group, scoring, cfg.routed_scaling_factor)


@pytest.mark.parametrize("cfg", [synth.tiny_config(), synth.prefill_config(), synth.decode_config(128)],
                         ids=lambda c: c.name)
def test_routing_of_layer_workloads(cfg):
    g = synth.gating_logits(cfg, "cuda").cpu().numpy()
    _run(g, cfg.topk, cfg.renormalize, cfg.num_expert_group, cfg.topk_group, cfg.scoring, cfg.routed_scaling_factor)


@pytest.mark.parametrize("E,G,kg,k", [(8, 4, 2, 2), (40, 5, 3, 24), (96, 4, 1, 24), (64, 32, 3, 6), (1024, 16, 4, 32),
                                      (256, 8, 8, 32), (6, 1, 1, 1), (160, 8, 2, 8), (512, 1, 1, 8)])
@pytest.mark.parametrize("scoring", ["softmax", "sigmoid"])
@pytest.mark.parametrize("renorm", [True, False])
def test_routing_shapes(E, G, kg, k, scoring, renorm):
    rng = np.random.default_rng(E * 7 + k)
    x = rng.normal(0, 2, size=(257, E)).astype(np.float32)
    _run(x, k, renorm, G, kg, scoring, 1.7)


def test_routing_ties_and_special_rows():
    rng = np.random.default_rng(5)
    E = 256
    rows = [np.zeros(E), np.full(E, 3.0), np.tile([5.0, 5.0, 1.0, 1.0], E // 4),
            rng.integers(-3, 4, size=E).astype(float), rng.integers(-3, 4, size=E).astype(float),
            np.where(np.arange(E) % 2 == 0, 30.0, -30.0), np.linspace(-20, 20, E), -np.linspace(-20, 20, E),
            rng.normal(0, 1e-3, size=E), np.full(E, -0.0)]
    x = np.array(rows, dtype=np.float32)
    x[-1, 7] = 0.0
    for scoring in ("softmax", "sigmoid"):
        for renorm in (True, False):
            _run(x, 8, renorm, 8, 4, scoring, 2.5)


def test_routing_T0_is_a_no_op():
    import mixture_experts_routing_grouped_gb300 as moe
    g = torch.empty((0, 256), dtype=torch.float32, device="cuda")
    w, ids = moe.moe_grouped_topk(g, 8, True, 8, 4, "softmax", 1.0)
    assert w.shape == (0, 8) and ids.shape == (0, 8)


def _special_rows(E, rng):
    rows = [np.zeros(E), np.full(E, 3.0), np.tile([5.0, 5.0, 1.0, 1.0], E // 4),
            rng.integers(-3, 4, size=E).astype(float), rng.integers(-1, 2, size=E).astype(float),
            np.where(np.arange(E) % 2 == 0, 30.0, -30.0), np.linspace(-20, 20, E), -np.linspace(-20, 20, E),
            rng.normal(0, 1e-3, size=E), np.full(E, -0.0), np.repeat(rng.normal(0, 2, size=E // 8), 8),
            np.where(np.arange(E) < 16, 7.0, rng.normal(0, 1, size=E))]
    return np.array(rows, dtype=np.float32)


@pytest.mark.parametrize("E,G,kg", [(256, 8, 4), (256, 1, 1), (128, 1, 1)])
@pytest.mark.parametrize("T", [2048, 4095, 20000])
@pytest.mark.parametrize("scoring", ["softmax", "sigmoid"])
@pytest.mark.parametrize("renorm", [True, False])
def test_routing_streaming_shapes_with_special_rows(E, G, kg, T, scoring, renorm):
    # T >= 2048 with topk = 8 selects the thread-per-token streaming kernel for these (E, G, topk_group);
    # every 5th row is one of the tie-heavy special rows (the list of candidates overflows on several)
    rng = np.random.default_rng(E + T + G)
    x = rng.normal(0, 2, size=(T, E)).astype(np.float32)
    sp = _special_rows(E, rng)
    idx = np.arange(0, T, 5)
    x[idx] = sp[np.arange(idx.size) % len(sp)]
    _run(x, 8, renorm, G, kg, scoring, 2.5)
