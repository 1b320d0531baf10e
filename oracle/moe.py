"""MoE layer forward, plainly (test infrastructure; see ``oracle/__init__``).

Two independent formulations of the same sum, both in float64 with no
intermediate rounding:

* ``expert_loop_forward`` -- the "expert view" that the mini-sglang MoE chapter
  contrasts with the token view: the (token, slot) pairs are grouped by the
  expert they chose, each expert's SwiGLU MLP runs once over its pairs' tokens,
  and every pair's weighted result is added into its token's row;
* ``token_view_forward`` -- the "token view" of "Fused MoE Part 3" (section
  01, ``selected_weights = weight[topk_ids]``): every token is projected by the
  weights of its own selected experts, one (token, slot) pair at a time.

Weight layout follows the mini-sglang ``MoELayer``: ``w1`` (gate_up_proj) is
[E, 2I, H] with the gate rows first ([0, I)) and the up rows second ([I, 2I));
``w2`` (down_proj) is [E, H, I]. SwiGLU is ``silu(gate) * up`` (the chapter's
``silu_and_mul`` and its third exercise). The route weights stay in float64
(the page casts them to the activation dtype; the reading here keeps them
exact).
"""
from __future__ import annotations

import numpy as np

from . import routing


def silu(v: np.ndarray) -> np.ndarray:
    return v / (1.0 + np.exp(-v))


def expert_projection(x: np.ndarray, weight: np.ndarray, topk_ids: np.ndarray) -> np.ndarray:
    """Fused MoE Part 3, section 03 task: output[m, j, :] = x[m] @ weight[topk_ids[m, j]]^T.

    x [M, K], weight [E, N, K], topk_ids [M, topk] -> [M, topk, N] (float64).
    """
    x = np.asarray(x, dtype=np.float64)
    weight = np.asarray(weight, dtype=np.float64)
    ids = np.asarray(topk_ids)
    M, topk = ids.shape
    out = np.zeros((M, topk, weight.shape[1]))
    for m in range(M):
        for j in range(topk):
            out[m, j] = weight[ids[m, j]] @ x[m]
    return out


def _expert_matrix(w, e: int) -> np.ndarray:
    """Expert e's matrix from an [E, ...] array, or from a callable e -> matrix (so that the
    experts of a large layer can be fetched and converted one at a time)."""
    return np.asarray(w(e) if callable(w) else w[e], dtype=np.float64)


def expert_loop_forward(x, w1, w2, topk_weights, topk_ids) -> np.ndarray:
    """The layer summed one expert at a time (the chapter's expert view): y [T, H] float64.

    y[t] = sum over slots j of w[t, j] * W2_e (silu(G_e x_t) * U_e x_t), e = ids[t, j].
    The (token, slot) pairs are grouped by the expert they chose, so that each
    expert's matrices are read once for all of its pairs; each pair's contribution
    is then added into its token's row. ``w1`` [E, 2I, H] (gate rows [0, I), up rows
    [I, 2I)) and ``w2`` [E, H, I] are arrays or callables e -> that expert's matrix.
    """
    x = np.asarray(x, dtype=np.float64)
    ids = np.asarray(topk_ids)
    tw = np.asarray(topk_weights, dtype=np.float64)
    y = np.zeros_like(x)
    for e in sorted(set(ids.reshape(-1).tolist())):
        pair_tok, pair_slot = np.nonzero(ids == e)      # the pairs routed to e, token by token
        W1e = _expert_matrix(w1, e)
        I = W1e.shape[0] // 2
        xs = x[pair_tok]
        gate_proj = xs @ W1e[:I].T
        up_proj = xs @ W1e[I:].T
        act = silu(gate_proj) * up_proj                 # [pairs of e, I]
        contrib = (act @ _expert_matrix(w2, e).T) * tw[pair_tok, pair_slot][:, None]
        for r, t in enumerate(pair_tok):
            y[t] += contrib[r]
    return y


def token_view_forward(x, w1, w2, topk_weights, topk_ids) -> np.ndarray:
    """Token view: for every token t and slot j, y[t] += w[t,j] * down(swiglu(gate_up(x_t))).

    Uses ``expert_projection`` for the gathered gate_up projection. Python loops
    over (token, slot): small cases only.
    """
    x = np.asarray(x, dtype=np.float64)
    w2 = np.asarray(w2, dtype=np.float64)
    ids = np.asarray(topk_ids)
    tw = np.asarray(topk_weights, dtype=np.float64)
    I = np.asarray(w1).shape[1] // 2
    gu = expert_projection(x, w1, ids)                  # [T, topk, 2I]
    h = silu(gu[:, :, :I]) * gu[:, :, I:]               # [T, topk, I]
    T, topk = ids.shape
    out = np.zeros((T, w2.shape[1]))
    for t in range(T):
        for j in range(topk):
            out[t] += tw[t, j] * (w2[ids[t, j]] @ h[t, j])
    return out


def fused_forward(x, gating_output, w1, w2, topk: int, renormalize: bool,
                  num_expert_group: int = 1, topk_group: int = 1, scoring_func: str = "softmax",
                  routed_scaling_factor: float = 1.0):
    """The whole layer: grouped top-k routing, then the expert-loop MoE.

    Returns (y float64 [T, H], topk_weights float32, topk_ids int32). The float32
    route weights (the routing output) are the ones the MoE sums with.
    """
    tw, ids = routing.grouped_topk(gating_output, topk, renormalize, num_expert_group,
                                   topk_group, scoring_func, routed_scaling_factor)
    y = expert_loop_forward(x, w1, w2, tw, ids)
    return y, tw, ids


def token_outputs(x_rows, w1_experts, w2_experts, weights) -> np.ndarray:
    """One token's output from its own experts: sum_j w_j * W2_j (silu(G_j x) * U_j x).

    ``x_rows`` [H]; ``w1_experts`` list of [2I, H]; ``w2_experts`` list of [H, I];
    ``weights`` [topk]. Used to check sampled tokens of workloads too large for
    the full oracle.
    """
    x = np.asarray(x_rows, dtype=np.float64)
    out = 0.0
    for w1e, w2e, wj in zip(w1_experts, w2_experts, weights):
        w1e = np.asarray(w1e, dtype=np.float64)
        I = w1e.shape[0] // 2
        h = silu(w1e[:I] @ x) * (w1e[I:] @ x)
        out = out + float(wj) * (np.asarray(w2e, dtype=np.float64) @ h)
    return out


def _bf16_round(v: np.ndarray) -> np.ndarray:
    """float64 -> float32 -> bfloat16 (round to nearest even) -> float64."""
    import torch
    t = torch.from_numpy(np.asarray(v, dtype=np.float32))
    return t.to(torch.bfloat16).to(torch.float64).numpy()


def fused_forward_fp8(x, gating_output, qw1, sw1, qw2, sw2, topk: int, renormalize: bool,
                      num_expert_group: int = 1, topk_group: int = 1, scoring_func: str = "softmax",
                      routed_scaling_factor: float = 1.0):
    """The layer with FP8-e4m3 GEMM operands (low-precision GMM article: sections 2.3, 3.1, 3.2, 4.3).

    Per the article, weights carry one scale per output channel, activations one
    scale per token computed from the activation itself, products accumulate at
    full precision and only the operands of the matrix instructions are 8-bit:

    1. routing as in ``fused_forward``;
    2. ``(qx, sx) = quant_rows_e4m3(x)`` (one scale per token);
    3. for every (token t, slot j) pair with expert e:
       ``g = sx[t] * sw1[e, :I] * (deq(qx[t]) @ deq(qw1[e, :I])^T)``, ``u`` likewise
       with rows ``[I, 2I)``; ``h = silu(g) * u`` (float64);
    4. ``h`` is held in the layer's activation dtype (rounded to bfloat16) and
       quantised per pair row: ``(qh, sh) = quant_rows_e4m3(h)``;
    5. ``y[t] += w[t, j] * sh * sw2[e] * (deq(qh) @ deq(qw2[e])^T)``.

    ``qw1`` uint8 e4m3 codes [E, 2I, H] with ``sw1`` [E, 2I]; ``qw2`` [E, H, I] with
    ``sw2`` [E, H]. Returns (y float64 [T, H], topk_weights float32, topk_ids int32).
    """
    tw, ids = routing.grouped_topk(gating_output, topk, renormalize, num_expert_group,
                                   topk_group, scoring_func, routed_scaling_factor)
    x = np.asarray(x, dtype=np.float32)
    T, k = ids.shape
    y = np.zeros((T, np.asarray(qw2).shape[1]))
    for t in range(T):
        es = ids[t]
        y[t] = token_outputs_fp8(x[t], [qw1[e] for e in es], [sw1[e] for e in es], [qw2[e] for e in es],
                                 [sw2[e] for e in es], tw[t])
    return y, tw, ids


def token_outputs_fp8(x_row, qw1_experts, sw1_experts, qw2_experts, sw2_experts, weights) -> np.ndarray:
    """One token's output of the FP8 layer (steps 2-5 of ``fused_forward_fp8``) from its own
    experts: ``qw1_experts`` list of e4m3 codes [2I, H] with ``sw1_experts`` [2I], ``qw2_experts``
    list of [H, I] with ``sw2_experts`` [H], ``weights`` [topk] route weights."""
    from . import quant
    qx, sx = quant.quant_rows_e4m3(np.asarray(x_row, dtype=np.float32)[None, :])
    dx = quant.dequant(qx[0], "e4m3") * float(sx[0])                        # sx[t] * deq(qx[t])
    out = 0.0
    for q1, s1, q2, s2, wj in zip(qw1_experts, sw1_experts, qw2_experts, sw2_experts, weights):
        w1 = quant.dequant(q1, "e4m3") * np.asarray(s1, dtype=np.float64)[:, None]
        w2 = quant.dequant(q2, "e4m3") * np.asarray(s2, dtype=np.float64)[:, None]
        I = w1.shape[0] // 2
        h = _bf16_round(silu(w1[:I] @ dx) * (w1[I:] @ dx))
        qh, sh = quant.quant_rows_e4m3(h[None, :])
        out = out + float(wj) * (w2 @ (quant.dequant(qh[0], "e4m3") * float(sh[0])))
    return out


def expert_loop_forward_fp8(x, qw1, sw1, qw2, sw2, topk_weights, topk_ids) -> np.ndarray:
    """Steps 2-5 of ``fused_forward_fp8`` summed one expert at a time: y float64 [T, H].

    The same arithmetic as the token loop (``token_outputs_fp8``), grouped by expert
    so that each expert's codes are decoded once for all of its (token, slot) pairs:
    x is quantised per token; for expert e and each of its pairs, g and u are the
    scaled products of the decoded codes, h = silu(g) * u is held in bfloat16 and
    quantised per pair row, and the down product scaled by both scales and the route
    weight is added into the pair's token row. ``qw1`` / ``sw1`` / ``qw2`` / ``sw2``
    are arrays indexed by expert ([E, 2I, H], [E, 2I], [E, H, I], [E, H]) or callables
    e -> that expert's slice.
    """
    from . import quant
    x = np.asarray(x, dtype=np.float32)
    ids = np.asarray(topk_ids)
    tw = np.asarray(topk_weights, dtype=np.float64)
    qx, sx = quant.quant_rows_e4m3(x)                                       # one scale per token
    dx = quant.dequant(qx, "e4m3") * sx.astype(np.float64)[:, None]
    y = np.zeros((x.shape[0], x.shape[1]))

    def part(w, e):
        return np.asarray(w(e) if callable(w) else w[e])

    for e in sorted(set(ids.reshape(-1).tolist())):
        pair_tok, pair_slot = np.nonzero(ids == e)
        w1 = quant.dequant(part(qw1, e), "e4m3") * part(sw1, e).astype(np.float64)[:, None]
        I = w1.shape[0] // 2
        xs = dx[pair_tok]
        hs = _bf16_round(silu(xs @ w1[:I].T) * (xs @ w1[I:].T))            # held in bfloat16
        qh, sh = quant.quant_rows_e4m3(hs)                                  # one scale per pair row
        w2 = quant.dequant(part(qw2, e), "e4m3") * part(sw2, e).astype(np.float64)[:, None]
        dh = quant.dequant(qh, "e4m3") * sh.astype(np.float64)[:, None]
        contrib = (dh @ w2.T) * tw[pair_tok, pair_slot][:, None]
        for r, t in enumerate(pair_tok):
            y[t] += contrib[r]
    return y
