"""Pins of the align oracle: the mini-sglang worked example, invariants, brute force."""
import json

import numpy as np
import pytest

from conftest import GOLDEN
from oracle import align, routing


def test_minisgl_worked_example():
    fx = json.loads((GOLDEN / "minisgl_seed0_routing.json").read_text())
    ids = np.array(fx["expected_topk_ids"], dtype=np.int32)
    sorted_ids, expert_ids, offsets, total = align.moe_align_block_size(ids, fx["block_m"], fx["E"])
    n = len(fx["expected_sorted_ids"])
    assert total == n
    assert sorted_ids[:n].tolist() == fx["expected_sorted_ids"]
    assert np.all(sorted_ids[n:] == ids.size)
    nb = len(fx["expected_expert_ids"])
    assert expert_ids[:nb].tolist() == fx["expected_expert_ids"]
    assert np.all(expert_ids[nb:] == -1)
    assert offsets.tolist() == [0, 0, 4, 4, 8, 12, 16, 20, 24]


def test_end_to_end_example_from_logits():
    fx = json.loads((GOLDEN / "minisgl_seed0_routing.json").read_text())
    g = np.array([[float.fromhex(v) for v in row] for row in fx["gating_hex"]], dtype=np.float32)
    _, ids = routing.select_experts(g, 2, True)
    sorted_ids, _, _, total = align.moe_align_block_size(ids, 4, 8)
    assert sorted_ids[:total].tolist() == fx["expected_sorted_ids"]


def _brute(flat, E, bm):
    # Python's sort is stable: sorting the pair indices by their expert keeps equal
    # experts in pair order. Then cut the sorted list into per-expert runs and pad each.
    order = sorted(range(len(flat)), key=lambda p: flat[p])
    out, blocks, i = [], [], 0
    for e in range(E):
        j = i
        while j < len(order) and flat[order[j]] == e:
            j += 1
        seg = order[i:j] + [len(flat)] * ((-(j - i)) % bm)
        out += seg
        blocks += [e] * (len(seg) // bm)
        i = j
    return out, blocks


@pytest.mark.parametrize("bm", [1, 4, 16, 128])
@pytest.mark.parametrize("E", [1, 3, 8, 33])
def test_brute_force_random(bm, E):
    rng = np.random.default_rng(bm * 1000 + E)
    for n in (0, 1, 7, 100, 513):
        flat = rng.integers(0, E, size=n).astype(np.int32)
        s, eids, off, total = align.moe_align_block_size(flat, bm, E)
        exp_s, exp_b = _brute(flat.tolist(), E, bm)
        assert total == len(exp_s)
        assert s[:total].tolist() == exp_s
        assert eids[:len(exp_b)].tolist() == exp_b
        assert len(s) == align.max_padded(n, E, bm) >= total
        assert np.all(s[total:] == n) and np.all(eids[len(exp_b):] == -1)


def test_invariants():
    rng = np.random.default_rng(7)
    T, k, E, bm = 97, 8, 128, 16
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    s, eids, off, total = align.moe_align_block_size(ids, bm, E)
    n = T * k
    real = s[:total][s[:total] < n]
    assert sorted(real.tolist()) == list(range(n))        # a permutation of the pairs
    assert np.all(np.diff(off) % bm == 0) and off[-1] == total
    flat = ids.reshape(-1)
    for e in range(E):
        seg = s[off[e]:off[e + 1]]
        r = seg[seg < n]
        assert np.all(flat[r] == e)
        assert np.all(np.diff(r) > 0)                     # stable: increasing pair index
        assert np.all(seg[len(r):] == n)                  # padding only at the segment end
        assert np.all(eids[off[e] // bm:off[e + 1] // bm] == e)
