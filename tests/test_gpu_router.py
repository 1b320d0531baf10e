"""GPU moe_router_topk (router projection x @ W_g^T, then grouped top-k) vs the oracle.

Checks, through the C ABI:
1. the fp32 logits against the oracle's float64 projection, within the bound of a
   fixed-order fp32 sum of H products: |d| <= (H + 1) * 2^-24 * sum_k |x w|;
2. the routing of those logits: ids bit-exact and weights within 1e-6 relative of
   the oracle's grouped top-k applied to the same (GPU) logits;
3. the ids against the oracle end to end (oracle logits, oracle routing) on every
   row whose selection no change of its logits as large as that row's measured
   error (plus the oracle's own rounding to fp32) could alter; on the tiny workload
   every row is such a row.
The logits are deterministic: a second call gives the same bits.
"""
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


def _decided(logits64, bound, E, G, kg, k):
    """Rows whose group choice and top-k (with its order) hold under any change <= bound[t] per logit."""
    T = logits64.shape[0]
    P = E // G
    ok = np.ones(T, dtype=bool)
    for t in range(T):
        row = logits64[t]
        gmax = np.sort(row.reshape(G, P).max(axis=1))[::-1]
        if kg < G and gmax[kg - 1] - gmax[kg] <= 2 * bound[t]:
            ok[t] = False
            continue
        sel = np.argsort(-row.reshape(G, P).max(axis=1), kind="stable")[:kg]
        cand = np.sort(np.concatenate([row[g * P:(g + 1) * P] for g in sel]))[::-1]
        top = cand[:min(k + 1, cand.size)]
        if np.any(np.diff(top)[:k] >= -2 * bound[t]):
            ok[t] = False
    return ok


def _check(cfg, x, wg, expect_all_decided):
    import mixture_experts_routing_grouped_gb300 as moe
    logits, w, ids = moe.moe_router_topk(x, wg, cfg.topk, cfg.renormalize, cfg.num_expert_group, cfg.topk_group,
                                         cfg.scoring, cfg.routed_scaling_factor)
    torch.cuda.synchronize()
    xh = x.double().cpu().numpy()
    wh = wg.double().cpu().numpy()
    ref64 = xh @ wh.T
    bound = (cfg.H + 1) * 2.0 ** -24 * (np.abs(xh) @ np.abs(wh).T)
    got = logits.double().cpu().numpy()
    assert np.all(np.abs(got - ref64) <= bound), f"worst excess {(np.abs(got - ref64) - bound).max():.3e}"
    # routing of the GPU's own logits
    rw, rids = routing.grouped_topk(logits.cpu().numpy(), cfg.topk, cfg.renormalize, cfg.num_expert_group,
                                    cfg.topk_group, cfg.scoring, cfg.routed_scaling_factor)
    assert np.array_equal(ids.cpu().numpy(), rids)
    assert_weights_close(w.cpu().numpy(), rw)
    # end to end against the oracle where the selection is decided
    _, ow, oids = routing.router_topk(xh, wg.cpu().numpy(), cfg.topk, cfg.renormalize, cfg.num_expert_group,
                                      cfg.topk_group, cfg.scoring, cfg.routed_scaling_factor)
    err = np.abs(got - ref64).max(axis=1) + 2.0 ** -24 * np.abs(ref64).max(axis=1)
    dec = _decided(ref64, err, cfg.E, cfg.num_expert_group, cfg.topk_group, cfg.topk)
    if expect_all_decided:
        assert dec.all()
    assert dec.mean() > 0.99
    assert np.array_equal(ids.cpu().numpy()[dec], oids[dec])
    # deterministic: the same bits again
    logits2, _, ids2 = moe.moe_router_topk(x, wg, cfg.topk, cfg.renormalize, cfg.num_expert_group,
                                           cfg.topk_group, cfg.scoring, cfg.routed_scaling_factor)
    torch.cuda.synchronize()
    assert torch.equal(logits2, logits) and torch.equal(ids2, ids)


def _inputs(cfg, router_sigma):
    x = synth.normal((cfg.T, cfg.H), cfg.seed, synth.TAG_X, cfg.x_sigma, torch.bfloat16, "cuda")
    wg = synth.normal((cfg.E, cfg.H), cfg.seed, synth.TAG_WG, router_sigma, torch.float32, "cuda")
    return x, wg


def test_router_tiny_workload():
    cfg = synth.tiny_config()
    x, wg = _inputs(cfg, cfg.router_sigma)
    # the tiny layer's logits are this projection (the layer tests feed them precomputed)
    np.testing.assert_allclose(synth.gating_logits(cfg, "cpu").numpy(),
                               routing.router_logits(x.double().cpu().numpy(), wg.cpu().numpy()), rtol=1e-6,
                               atol=1e-6)
    _check(cfg, x, wg, expect_all_decided=True)


@pytest.mark.parametrize("cfg,sigma", [
    (synth.MoEConfig("router_T37_H256_E96_G8_top6", T=37, H=256, I=0, E=96, topk=6, num_expert_group=8,
                     topk_group=3, scoring="sigmoid", routed_scaling_factor=2.5, seed=31), 0.05),
    (synth.MoEConfig("router_T1_H7168_E256_G8_top8", T=1, H=7168, I=0, E=256, topk=8, num_expert_group=8,
                     topk_group=4, scoring="sigmoid", routed_scaling_factor=2.5, seed=32), 0.02),
    (synth.MoEConfig("router_T128_H7168_E256_G8_top8", T=128, H=7168, I=0, E=256, topk=8, num_expert_group=8,
                     topk_group=4, scoring="sigmoid", routed_scaling_factor=2.5, seed=33), 0.02),
    (synth.MoEConfig("router_T4096_H2048_E128_top8", T=4096, H=2048, I=0, E=128, topk=8, seed=34), 0.02),
    (synth.MoEConfig("router_T300_H96_E1024_G32_top32", T=300, H=96, I=0, E=1024, topk=32, num_expert_group=32,
                     topk_group=8, seed=35), 0.1),
], ids=lambda v: v.name if hasattr(v, "name") else str(v))
def test_router_shapes(cfg, sigma):
    x, wg = _inputs(cfg, sigma)
    _check(cfg, x, wg, expect_all_decided=False)


def test_router_rejects_unsupported_hidden_size():
    import mixture_experts_routing_grouped_gb300 as moe
    x = torch.zeros((4, 48), dtype=torch.bfloat16, device="cuda")
    wg = torch.zeros((8, 48), dtype=torch.float32, device="cuda")
    with pytest.raises(moe.MoeError):
        moe.moe_router_topk(x, wg, 2)
