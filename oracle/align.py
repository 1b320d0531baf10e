"""``moe_align_block_size`` plainly (test infrastructure; see ``oracle/__init__``).

Follows the mini-sglang MoE chapter ("fused MoE", ``moe_align_block_size``):
stably sort the flat (token, expert) pair indices by expert, pad every
expert's segment to a multiple of ``block_m`` with the sentinel ``num_pairs``,
and give every block of ``block_m`` entries its expert.

Reading of the output buffers (the page returns exactly-sized tensors): the
buffers here have the fixed capacity ``max_padded(num_pairs, E, block_m)`` so
that a device implementation can size them without a host sync; entries
beyond ``num_tokens_post_padded`` hold the sentinel and trailing block
experts hold -1. ``expert_offsets`` is the exclusive prefix sum of the padded
segment lengths followed by the total.
"""
from __future__ import annotations

import numpy as np


def max_padded(num_pairs: int, E: int, block_m: int) -> int:
    """Capacity that holds every padded layout: each non-empty expert adds < block_m pad entries."""
    cap = num_pairs + min(E, num_pairs) * (block_m - 1)
    return (cap + block_m - 1) // block_m * block_m


def moe_align_block_size(topk_ids: np.ndarray, block_m: int, num_experts: int):
    """Returns (sorted_token_ids, expert_ids, expert_offsets, num_tokens_post_padded)."""
    flat = np.asarray(topk_ids).reshape(-1).astype(np.int64)
    num_pairs = flat.size
    E = num_experts
    counts = np.bincount(flat, minlength=E)                       # pairs per expert
    padded = (counts + block_m - 1) // block_m * block_m          # segment length
    seg_start = np.cumsum(padded) - padded                        # exclusive prefix sum
    order = np.argsort(flat, kind="stable")                       # pairs ordered by expert
    sorted_expert = flat[order]
    first_of_expert = np.cumsum(counts) - counts
    rank = np.arange(num_pairs) - first_of_expert[sorted_expert]  # rank within its expert
    total = int(padded.sum())

    cap = max_padded(num_pairs, E, block_m)
    sorted_ids = np.full(cap, num_pairs, dtype=np.int32)
    sorted_ids[seg_start[sorted_expert] + rank] = order.astype(np.int32)
    expert_ids = np.full(cap // block_m, -1, dtype=np.int32)
    expert_ids[:total // block_m] = np.repeat(np.arange(E), padded // block_m)
    expert_offsets = np.concatenate([seg_start, [total]]).astype(np.int32)
    return sorted_ids, expert_ids, expert_offsets, total
