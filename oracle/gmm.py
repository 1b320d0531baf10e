"""Low-precision grouped GEMM, dequantise-then-matmul (test infrastructure).

Follows the low-precision GMM article (pwwt.cn): section 2.1 defines
``Y_e = X[S_e] @ W_e^T`` for every expert e, with X pre-sorted by expert so
that S_e is the contiguous row range [offsets[e], offsets[e] + sizes[e]);
section 3.1 gives the interface ``gmm(input, weights, scales_x, scales_w,
expert_offsets, expert_sizes, output, M, K, N, E)`` with per-token activation
scales [M] and per-expert output-channel weight scales [E, N]; section 2.3
accumulates in high precision. The oracle dequantises every code exactly and
sums in float64:

    Y[m, n] = scales_x[m] * scales_w[e, n] * sum_k deq(q_x[m, k]) * deq(q_w[e, n, k])

Rows that belong to no expert are left at zero.
"""
from __future__ import annotations

import numpy as np

from .quant import dequant


def gmm(qx, qw, scales_x, scales_w, expert_offsets, expert_sizes, dtype: str) -> np.ndarray:
    """qx [M, K], qw [E, N, K] codes of ``dtype`` ("i8" | "e4m3") -> Y float64 [M, N]."""
    xq = dequant(qx, dtype)
    M = xq.shape[0]
    E, N, _ = np.asarray(qw).shape
    sx = np.asarray(scales_x, dtype=np.float64)
    sw = np.asarray(scales_w, dtype=np.float64)
    off = np.asarray(expert_offsets)
    size = np.asarray(expert_sizes)
    y = np.zeros((M, N))
    for e in range(E):
        lo, hi = int(off[e]), int(off[e]) + int(size[e])
        if hi == lo:
            continue
        we = dequant(np.asarray(qw)[e], dtype)                 # [N, K]
        acc = xq[lo:hi] @ we.T                                 # [M_e, N]
        y[lo:hi] = sx[lo:hi, None] * sw[e][None, :] * acc
    return y
