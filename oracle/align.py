"""``moe_align_block_size`` plainly (test infrastructure; see ``oracle/__init__``).

Follows the mini-sglang MoE chapter ("fused MoE", ``moe_align_block_size``),
whose result is fixed by its description: the flat (token, expert) pair indices
stably sorted by expert, every expert's segment padded to a multiple of
``block_m`` with the sentinel ``num_pairs``, and every block of ``block_m``
entries labelled with its expert.

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
    """Returns (sorted_token_ids, expert_ids, expert_offsets, num_tokens_post_padded).

    Written as a counting sort with one write cursor per expert:

    1. count the pairs that chose each expert;
    2. lay the experts' segments out back to back, each segment its count rounded
       up to a multiple of ``block_m``;
    3. visit the pairs in increasing pair index and write each into the next free
       slot of its expert's segment (visiting in index order is what makes the
       sort stable);
    4. every block of ``block_m`` slots gets the expert whose segment holds it.
    """
    pair_expert = [int(e) for e in np.asarray(topk_ids).reshape(-1)]
    num_pairs = len(pair_expert)
    E = num_experts

    count = [0] * E                                               # 1.
    for e in pair_expert:
        count[e] += 1

    seg_begin, seg_len, pos = [], [], 0                           # 2.
    for e in range(E):
        length = -(-count[e] // block_m) * block_m
        seg_begin.append(pos)
        seg_len.append(length)
        pos += length
    total = pos

    cap = max_padded(num_pairs, E, block_m)
    sorted_ids = np.full(cap, num_pairs, dtype=np.int32)          # padding holds the sentinel
    cursor = list(seg_begin)                                      # 3.
    for p, e in enumerate(pair_expert):
        sorted_ids[cursor[e]] = p
        cursor[e] += 1

    expert_ids = np.full(cap // block_m, -1, dtype=np.int32)      # 4.
    for e in range(E):
        first_block = seg_begin[e] // block_m
        expert_ids[first_block:first_block + seg_len[e] // block_m] = e
    expert_offsets = np.array(seg_begin + [total], dtype=np.int32)
    return sorted_ids, expert_ids, expert_offsets, total
