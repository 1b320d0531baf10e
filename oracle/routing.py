"""Grouped top-k routing, plainly (test infrastructure; see ``oracle/__init__``).

Follows "GroupedTopK 算子优化入门" (blog.freezetheflame.cc), section 三
(3.1 scores, 3.2 per-group max, 3.3 top groups, 3.4 mask, 3.5 top-k, 3.6
renormalise and scale) and section 七 (monotonicity of the score functions),
and the ``select_experts`` routine of the mini-sglang MoE chapter (plain
softmax -> top-k -> optional renormalisation, i.e. one group).

Readings where the pages leave a step open:

* Selection order. Both selections take "the largest scores". Softmax and the
  logistic sigmoid are strictly increasing, so the order of the exact scores
  is the order of the logits (section 七). The oracle ranks on the logits, which
  are exact, rather than on rounded scores, which can collide (a double
  sigmoid is exactly 1.0 for every logit above ~37). Equal keys go to the lower
  index, for groups and for experts.
* Group score is the maximum over the group (3.2), not a top-2 sum.
* ``routed_scaling_factor`` multiplies the weights whether or not they were
  renormalised (3.6 lists it after the renormalisation without a condition).
* Output order is the ranking order (descending weight, ties by index).
* Inputs are finite; NaN and infinities are outside the contract.
* Router logits (``router_logits``): the mini-sglang chapter's ``MoEMLP`` computes
  them with ``gate = LinearReplicated(H, E)``, i.e. ``x @ W_g^T``; the blog's
  ``gating_output`` is that output. The pages give no precision for it; the
  reading here is the dot product of the bfloat16 hidden state and the float32
  router weights accumulated in float64 and rounded once to float32 (the
  routing's input dtype).
"""
from __future__ import annotations

import numpy as np


def scores(logits: np.ndarray, scoring_func: str) -> np.ndarray:
    """Section 3.1: per-token softmax (max-subtracted) or elementwise sigmoid, in float64."""
    x = np.asarray(logits, dtype=np.float64)
    if scoring_func == "softmax":
        m = x.max(axis=-1, keepdims=True)
        ex = np.exp(x - m)
        return ex / ex.sum(axis=-1, keepdims=True)
    if scoring_func == "sigmoid":
        # exp(-x) overflows to inf for x below about -709, which gives the limit 0 exactly.
        with np.errstate(over="ignore"):
            return 1.0 / (1.0 + np.exp(-x))
    raise ValueError(f"unknown scoring_func {scoring_func!r}")


def _rank_desc(keys: np.ndarray) -> np.ndarray:
    """Indices sorted by key descending, equal keys by ascending index (stable sort of -key)."""
    return np.argsort(-keys, axis=-1, kind="stable")


def grouped_topk(gating_output: np.ndarray, topk: int, renormalize: bool,
                 num_expert_group: int, topk_group: int, scoring_func: str = "softmax",
                 routed_scaling_factor: float = 1.0):
    """GroupedTopK forward: (topk_weights float32 [T, topk], topk_ids int32 [T, topk]).

    ``gating_output`` is [T, E] float32 logits; experts form ``num_expert_group``
    contiguous groups of E / G experts. ``hidden_states`` of the blog's
    interface is not an input: only its row count is ever used.
    """
    x = np.asarray(gating_output)
    T, E = x.shape
    G = num_expert_group
    if E % G != 0:
        raise ValueError("E must be divisible by num_expert_group")
    P = E // G
    if not (1 <= topk_group <= G) or not (1 <= topk <= topk_group * P):
        raise ValueError("invalid topk_group / topk")
    xd = x.astype(np.float64)
    s = scores(xd, scoring_func)                                # 3.1

    # 3.2: group score = max over each group of P experts (ranked on logits, see module doc)
    group_key = xd.reshape(T, G, P).max(axis=2)                 # [T, G]
    # 3.3: top-`topk_group` groups per token
    sel_groups = _rank_desc(group_key)[:, :topk_group]          # [T, topk_group]
    group_selected = np.zeros((T, G), dtype=bool)
    np.put_along_axis(group_selected, sel_groups, True, axis=1)
    # 3.4: experts of unselected groups are masked to -inf
    group_of_expert = np.arange(E) // P
    masked = np.where(group_selected[:, group_of_expert], xd, -np.inf)
    # 3.5: top-`topk` experts among the candidates
    ids = _rank_desc(masked)[:, :topk]                          # [T, topk]

    w = np.take_along_axis(s, ids, axis=1)                      # weights are the scores
    if renormalize:                                             # 3.6
        w = w / w.sum(axis=1, keepdims=True)
    w = w * routed_scaling_factor
    return w.astype(np.float32), ids.astype(np.int32)


def select_experts(gating_output: np.ndarray, topk: int, renormalize: bool):
    """mini-sglang ``select_experts``: softmax over all experts, top-k, optional renormalise.

    This is grouped top-k with a single group.
    """
    return grouped_topk(gating_output, topk, renormalize, num_expert_group=1, topk_group=1,
                        scoring_func="softmax", routed_scaling_factor=1.0)


def router_logits(hidden_states: np.ndarray, w_gate: np.ndarray) -> np.ndarray:
    """Router projection ``x @ W_g^T`` (mini-sglang MoE chapter, ``MoEMLP.gate``).

    ``hidden_states`` [T, H] (bfloat16 values, exact in float64), ``w_gate`` [E, H]
    float32 -> logits float32 [T, E], summed in float64 and rounded once.
    """
    x = np.asarray(hidden_states, dtype=np.float64)
    w = np.asarray(w_gate, dtype=np.float64)
    if x.ndim != 2 or w.ndim != 2 or x.shape[1] != w.shape[1]:
        raise ValueError("hidden_states [T, H] and w_gate [E, H] must share H")
    return (x @ w.T).astype(np.float32)


def router_topk(hidden_states: np.ndarray, w_gate: np.ndarray, topk: int, renormalize: bool,
                num_expert_group: int = 1, topk_group: int = 1, scoring_func: str = "softmax",
                routed_scaling_factor: float = 1.0):
    """The router followed by grouped top-k: (logits float32 [T, E], topk_weights, topk_ids)."""
    logits = router_logits(hidden_states, w_gate)
    w, ids = grouped_topk(logits, topk, renormalize, num_expert_group, topk_group, scoring_func,
                          routed_scaling_factor)
    return logits, w, ids
