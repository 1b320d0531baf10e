"""Pins of the routing oracle to the GroupedTopK blog and the mini-sglang chapter."""
import itertools
import json
import math

import numpy as np
import pytest
import torch

from conftest import GOLDEN
from oracle import routing


def _load(name):
    return json.loads((GOLDEN / name).read_text())


def test_blog_worked_example_ids_and_groups():
    fx = _load("groupedtopk_worked_example.json")
    x = np.array([fx["scores"]], dtype=np.float32)
    P = fx["E"] // fx["num_expert_group"]
    gs = x.reshape(fx["num_expert_group"], P).max(axis=1)
    np.testing.assert_allclose(gs, fx["expected_group_scores"], rtol=0, atol=1e-7)
    for scoring in ("softmax", "sigmoid"):
        w, ids = routing.grouped_topk(x, fx["topk"], True, fx["num_expert_group"], fx["topk_group"], scoring)
        assert ids[0].tolist() == fx["expected_topk_ids"]
        assert set(i // P for i in ids[0]) <= set(fx["expected_groups"])


def test_blog_worked_example_weights_closed_form():
    # Two selected experts with logits a > b, renormalised:
    # softmax -> w0 = 1 / (1 + e^(b - a)); sigmoid -> w0 = s(a) / (s(a) + s(b)).
    fx = _load("groupedtopk_worked_example.json")
    x = np.array([fx["scores"]], dtype=np.float32)
    a, b = float(np.float32(0.9)), float(np.float32(0.8))
    w, _ = routing.grouped_topk(x, 2, True, 4, 2, "softmax")
    ws = 1.0 / (1.0 + math.exp(b - a))
    np.testing.assert_allclose(w[0], [ws, 1 - ws], rtol=1e-6)
    assert abs(ws - 0.524979) < 1e-6
    w, _ = routing.grouped_topk(x, 2, True, 4, 2, "sigmoid", 2.5)
    sa, sb = 1 / (1 + math.exp(-a)), 1 / (1 + math.exp(-b))
    np.testing.assert_allclose(w[0], [2.5 * sa / (sa + sb), 2.5 * sb / (sa + sb)], rtol=1e-6)


def test_minisgl_seed0_example():
    fx = _load("minisgl_seed0_routing.json")
    g = np.array([[float.fromhex(v) for v in row] for row in fx["gating_hex"]], dtype=np.float32)
    w, ids = routing.select_experts(g, fx["topk"], fx["renormalize"])
    assert ids.tolist() == fx["expected_topk_ids"]
    np.testing.assert_allclose(np.round(w.astype(np.float64), 3), fx["expected_topk_weights_3dp"], atol=1e-9)


def test_single_group_is_plain_softmax_topk_library():
    # G = 1 reduces to softmax -> torch.topk -> renormalise (mini-sglang select_experts),
    # checked against torch's own softmax/topk on continuous random logits.
    rng = np.random.default_rng(1)
    x = rng.normal(0, 2, size=(64, 40)).astype(np.float32)
    for k in (1, 3, 8):
        for renorm in (True, False):
            w, ids = routing.grouped_topk(x, k, renorm, 1, 1, "softmax")
            p = torch.softmax(torch.from_numpy(x).double(), -1)
            tw, ti = p.topk(k, dim=-1)
            if renorm:
                tw = tw / tw.sum(-1, keepdim=True)
            assert np.array_equal(ids, ti.numpy())
            np.testing.assert_allclose(w, tw.numpy(), rtol=1e-6)


def test_sigmoid_single_group_library():
    rng = np.random.default_rng(2)
    x = rng.normal(0, 2, size=(50, 24)).astype(np.float32)
    w, ids = routing.grouped_topk(x, 5, False, 1, 1, "sigmoid", 1.5)
    p = torch.sigmoid(torch.from_numpy(x).double())
    tw, ti = p.topk(5, dim=-1)
    assert np.array_equal(ids, ti.numpy())
    np.testing.assert_allclose(w, 1.5 * tw.numpy(), rtol=1e-6)


def _brute(x_row, E, G, kg, k):
    """Enumerate every group subset and every candidate subset; keep the best sorted key list."""
    P = E // G
    gkey = [max(x_row[g * P:(g + 1) * P]) for g in range(G)]
    def key_list(items, keyf):
        return sorted(((keyf(i), -i) for i in items), reverse=True)
    best_groups = max(itertools.combinations(range(G), kg), key=lambda s: key_list(s, lambda g: gkey[g]))
    cand = [e for g in best_groups for e in range(g * P, (g + 1) * P)]
    best = max(itertools.combinations(cand, k), key=lambda s: key_list(s, lambda e: x_row[e]))
    return [i for _, i in ((kv, -ni) for kv, ni in key_list(best, lambda e: x_row[e]))]


@pytest.mark.parametrize("E,G,kg,k", [(8, 4, 2, 2), (12, 3, 2, 4), (12, 4, 1, 3), (10, 5, 3, 6), (6, 1, 1, 6)])
def test_brute_force_tiny(E, G, kg, k):
    rng = np.random.default_rng(E * 100 + G * 10 + k)
    for trial in range(30):
        if trial % 3 == 0:       # heavy ties: few distinct values
            x = rng.integers(-2, 3, size=(1, E)).astype(np.float32)
        else:
            x = rng.normal(0, 1.5, size=(1, E)).astype(np.float32)
        _, ids = routing.grouped_topk(x, k, True, G, kg, "softmax")
        assert ids[0].tolist() == _brute([float(v) for v in x[0]], E, G, kg, k)


def test_ranking_on_double_scores_matches_logit_order():
    # Reading check: for moderate logits, ranking the float64 scores themselves
    # (the literal section 3.3/3.5 steps) selects exactly the same experts.
    rng = np.random.default_rng(3)
    x = rng.normal(0, 2, size=(256, 256)).astype(np.float32)
    for scoring in ("softmax", "sigmoid"):
        _, ids = routing.grouped_topk(x, 8, True, 8, 4, scoring)
        s = routing.scores(x, scoring)
        for t in range(x.shape[0]):
            gsc = s[t].reshape(8, 32).max(axis=1)
            groups = np.argsort(-gsc, kind="stable")[:4]
            masked = np.full(256, -np.inf)
            for g in groups:
                masked[g * 32:(g + 1) * 32] = s[t, g * 32:(g + 1) * 32]
            assert np.argsort(-masked, kind="stable")[:8].tolist() == ids[t].tolist()


@pytest.mark.parametrize("scoring", ["softmax", "sigmoid"])
@pytest.mark.parametrize("renorm", [True, False])
def test_invariants(scoring, renorm):
    # Blog section 九 invariants: exactly topk distinct ids, in range, from the
    # selected groups; renormalised weights sum to the scaling factor; weights descend.
    rng = np.random.default_rng(4)
    x = rng.normal(0, 2, size=(300, 256)).astype(np.float32)
    rsf = 2.5
    w, ids = routing.grouped_topk(x, 8, renorm, 8, 4, scoring, rsf)
    assert ids.dtype == np.int32 and w.dtype == np.float32
    assert ids.min() >= 0 and ids.max() < 256
    for t in range(x.shape[0]):
        assert len(set(ids[t].tolist())) == 8
        assert len(set((ids[t] // 32).tolist())) <= 4
        assert np.all(np.diff(w[t].astype(np.float64)) <= 0)
    if renorm:
        np.testing.assert_allclose(w.astype(np.float64).sum(1), rsf, rtol=1e-6)
    else:
        s = routing.scores(x, scoring)
        np.testing.assert_allclose(w, rsf * np.take_along_axis(s, ids, 1), rtol=1e-6)


def test_special_values():
    # All-equal rows, all zeros, tied group maxima, large magnitudes (blog section 九).
    E, G = 16, 4
    rows = [np.zeros(E), np.full(E, 3.0), np.array([5.0, 5.0, 1, 1] * 4),
            np.array([1e30, -1e30] * 8), np.linspace(-40, 40, E)]
    x = np.array(rows, dtype=np.float32)
    w, ids = routing.grouped_topk(x, 4, True, G, 2, "sigmoid")
    assert ids[0].tolist() == [0, 1, 2, 3]           # all equal -> lowest indices
    assert ids[1].tolist() == [0, 1, 2, 3]
    assert ids[2].tolist() == [0, 1, 4, 5]           # tied groups -> lower group index
    assert ids[3].tolist() == [0, 2, 4, 6]
    assert ids[4].tolist() == [15, 14, 13, 12]       # sigmoid saturates; logit order still decides
    assert np.all(np.isfinite(w))
    np.testing.assert_allclose(w.astype(np.float64).sum(1), 1.0, rtol=1e-6)


def test_hidden_states_not_an_input():
    # The routing output depends on the gating logits only (blog section 九, last invariant):
    # the oracle's interface has no hidden_states argument at all.
    import inspect
    assert "hidden_states" not in inspect.signature(routing.grouped_topk).parameters


# --------------------------------------------------------------------------- router projection
def test_router_hand_worked_example():
    # Two tokens, H = 4, E = 3 (non-square, so a transposed operand cannot pass), values
    # chosen so that every product and sum is exact:
    #   token 0: e0 = 1*1 = 1; e1 = 2*0.25 + (-1)*1 = -0.5; e2 = 1*2 + 2*(-1) + 0*0.5 = 0
    #   token 1: e0 = 0.5;     e1 = 4*1 = 4;                e2 = 0.5*2 = 1
    x = np.array([[1.0, 2.0, 0.0, -1.0], [0.5, 0.0, 0.0, 4.0]])
    wg = np.array([[1.0, 0.0, 0.0, 0.0], [0.0, 0.25, 0.0, 1.0], [2.0, -1.0, 0.5, 0.0]], dtype=np.float32)
    logits = routing.router_logits(x, wg)
    assert logits.dtype == np.float32
    assert logits.tolist() == [[1.0, -0.5, 0.0], [0.5, 4.0, 1.0]]
    _, w, ids = routing.router_topk(x, wg, 2, True)
    assert ids.tolist() == [[0, 2], [1, 2]]
    # renormalised softmax of two logits a > b: 1 / (1 + e^(b - a)) and the rest
    e = np.e
    np.testing.assert_allclose(w, [[e / (e + 1), 1 / (e + 1)], [1 / (1 + e ** -3), e ** -3 / (1 + e ** -3)]],
                               rtol=1e-7)


def test_router_logits_exact_sum_rounded_once():
    # Against the exact rational dot product (fractions): float64 accumulation then one
    # rounding to float32 lands within one float32 ulp of the exact value.
    from fractions import Fraction
    rng = np.random.default_rng(17)
    T, H, E = 5, 96, 7
    x = rng.normal(size=(T, H)).astype(np.float32).astype(np.float64)
    x = np.round(x * 256) / 256                                  # bfloat16-like short values
    wg = rng.normal(0, 0.05, size=(E, H)).astype(np.float32)
    logits = routing.router_logits(x, wg)
    for t in range(T):
        for e in range(E):
            exact = sum(Fraction(float(x[t, h])) * Fraction(float(wg[e, h])) for h in range(H))
            got = Fraction(float(logits[t, e]))
            ulp = Fraction(float(np.spacing(np.float32(abs(float(exact))))))
            assert abs(got - exact) <= ulp


def test_router_rejects_mismatched_hidden_size():
    with pytest.raises(ValueError):
        routing.router_logits(np.zeros((2, 4)), np.zeros((3, 5), dtype=np.float32))
