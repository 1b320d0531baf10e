"""Pins of the FP8-e4m3 layer forward oracle (oracle.moe.fused_forward_fp8).

1. Exact case: every operand on the e4m3 grid times a per-row power of two, and
   gate projections >= 40 so that silu(g) == g exactly in float64; then every
   quantiser in the path is exact and the FP8 forward must equal the exact
   expert-loop forward on the dequantised weights bit for bit. This checks that
   each scale (per token, per gate/up channel, per h row, per down channel) is
   applied to the right index.
2. Quantisation error: on random layers the FP8 result stays within the error
   that 3-bit-mantissa operands allow of the exact forward.
3. Power-of-two equivariance: doubling the scale of one down-projection output
   channel doubles that output column exactly and leaves the others unchanged.
4. A hand-worked token whose h row is held in bfloat16 before its per-row e4m3
   quantisation: the bf16 rounding moves one value onto an e4m3 midpoint (ties to
   even), so the output differs from the one without the bf16 step or without the
   quantisation of h.
"""
import numpy as np

from oracle import moe, quant


def test_fp8_forward_exact_when_every_quantiser_is_exact():
    # x rows: [448 * 2^a, 0, ...] (scale 2^a, codes exact). Weight rows: the row
    # absmax 448 * 2^b sits in a column x does not touch; the column x touches
    # holds c * 2^b with c in {1, 2, 4} (gate) or +-{1, 2, 4} (up, down). Then
    # g = 7 * 2^m >= 112, silu(g) == g in float64, u = +-7 * 2^m', h = +-49 * 2^m''
    # (exact in bf16), and h / (absmax(h) / 448) = 448 * 2^p lies on the e4m3 grid.
    rng = np.random.default_rng(3)
    T, H, I, E, k = 6, 4, 3, 3, 2
    a = rng.integers(0, 2, size=T)
    x = np.zeros((T, H))
    x[:, 0] = 448.0 * 2.0 ** a

    def rows(n, used_vals, b):
        m = np.zeros((n, H))
        m[:, 1] = 448.0
        m[:, 0] = rng.choice(used_vals, size=n)
        return m * 2.0 ** b[:, None]

    b1 = rng.integers(-2, 1, size=E * 2 * I)
    gate_up = np.concatenate([rows(E * I, [1.0, 2.0, 4.0], b1[:E * I]).reshape(E, I, H),
                              rows(E * I, [1.0, -2.0, 4.0, -1.0], b1[E * I:]).reshape(E, I, H)], axis=1)
    b2 = rng.integers(-6, -2, size=E * H)
    w2 = np.zeros((E * H, I))
    w2[:, 0] = 448.0
    w2[:, 1:] = rng.choice([1.0, -2.0, 4.0, -0.5], size=(E * H, I - 1))
    w2 = (w2 * 2.0 ** b2[:, None]).reshape(E, H, I)
    q1, s1 = quant.quant_rows_e4m3(gate_up.reshape(E * 2 * I, H))
    q2, s2 = quant.quant_rows_e4m3(w2.reshape(E * H, I))
    # the quantisers reproduce every operand exactly
    assert np.array_equal(quant.dequant(q1, "e4m3") * s1[:, None], gate_up.reshape(E * 2 * I, H))
    assert np.array_equal(quant.dequant(q2, "e4m3") * s2[:, None], w2.reshape(E * H, I))
    qx, sx = quant.quant_rows_e4m3(x)
    assert np.array_equal(quant.dequant(qx, "e4m3") * sx[:, None], x)
    gating = rng.normal(0, 1, size=(T, E)).astype(np.float32)
    y, tw, ids = moe.fused_forward_fp8(x, gating, q1.reshape(E, 2 * I, H), s1.reshape(E, 2 * I),
                                       q2.reshape(E, H, I), s2.reshape(E, H), k, True)
    g = np.stack([gate_up[ids[t, j], :I] @ x[t] for t in range(T) for j in range(k)])
    assert g.min() >= 40.0
    ref = moe.expert_loop_forward(x, gate_up, w2, tw, ids)
    assert np.array_equal(y, ref)
    assert np.count_nonzero(ref) > 0


def test_fp8_forward_within_quantisation_error_of_exact():
    rng = np.random.default_rng(11)
    T, H, I, E, k = 24, 64, 32, 4, 2
    x = rng.normal(0, 1, size=(T, H)).astype(np.float32)
    w1 = rng.normal(0, 0.1, size=(E, 2 * I, H)).astype(np.float32)
    w2 = rng.normal(0, 0.1, size=(E, H, I)).astype(np.float32)
    q1, s1 = quant.quant_rows_e4m3(w1.reshape(E * 2 * I, H))
    q2, s2 = quant.quant_rows_e4m3(w2.reshape(E * H, I))
    gating = rng.normal(0, 1, size=(T, E)).astype(np.float32)
    y, tw, ids = moe.fused_forward_fp8(x, gating, q1.reshape(E, 2 * I, H), s1.reshape(E, 2 * I),
                                       q2.reshape(E, H, I), s2.reshape(E, H), k, True)
    ref = moe.expert_loop_forward(x, w1, w2, tw, ids)
    rel = np.linalg.norm(y - ref) / np.linalg.norm(ref)
    # four quantised operands with relative rounding error <= 2^-4 each; random signs average out
    assert 1e-3 < rel < 0.1, rel
    # a dropped scale (x's is ~absmax/448) would be off by orders of magnitude
    assert np.abs(y).max() < 10 * np.abs(ref).max()


def test_fp8_forward_down_channel_scale_equivariance():
    rng = np.random.default_rng(5)
    T, H, I, E, k = 8, 32, 16, 3, 2
    x = rng.normal(0, 1, size=(T, H)).astype(np.float32)
    q1, s1 = quant.quant_rows_e4m3(rng.normal(0, 0.2, size=(E * 2 * I, H)).astype(np.float32))
    q2, s2 = quant.quant_rows_e4m3(rng.normal(0, 0.2, size=(E * H, I)).astype(np.float32))
    gating = rng.normal(0, 1, size=(T, E)).astype(np.float32)
    args = (q1.reshape(E, 2 * I, H), s1.reshape(E, 2 * I), q2.reshape(E, H, I))
    y0, _, _ = moe.fused_forward_fp8(x, gating, *args, s2.reshape(E, H), k, True)
    s2b = s2.reshape(E, H).copy()
    s2b[:, 5] *= 2.0
    y1, _, _ = moe.fused_forward_fp8(x, gating, *args, s2b, k, True)
    assert np.array_equal(y1[:, 5], 2.0 * y0[:, 5])
    assert np.array_equal(np.delete(y1, 5, axis=1), np.delete(y0, 5, axis=1))


E4M3_ONE, E4M3_448 = 0x38, 0x7E   # codes of 1.0 (0 0111 000) and 448 (0 1111 110)


def test_fp8_token_with_h_held_in_bf16_worked_by_hand():
    # x = [448, 1, 0, 0]: scale 1, dequantised x exactly [448, 1, 0, 0]. Only column 1 of
    # the gate_up weights is non-zero (code 1.0), so g and u are the channel scales:
    # gate channels 64, 64 (silu(64) == 64 in float64); up channels 6.125 and
    # 3809/2^18, giving h = [392, 3809/4096] exactly.
    # bf16(h) = [392, 238/256]; its row scale is 392/448 = 0.875 (exact), the quotients
    # are 448 and 1.0625, the midpoint of the e4m3 values 1 and 1.125: ties to even
    # give code 1.0, i.e. h dequantised [392, 0.875]. The down weights pick h[1] for
    # output 0 (code 1.0, scale 1) with route weight 1: y[0] = 0.875 exactly.
    # Without the bf16 step the quotient is 1.06278 -> 1.125 -> y[0] = 0.984375; without
    # quantising h, y[0] = 3809/4096.
    H, I = 4, 2
    x = np.array([448.0, 1.0, 0.0, 0.0], dtype=np.float32)
    q1 = np.zeros((2 * I, H), dtype=np.uint8)
    q1[:, 1] = E4M3_ONE
    s1 = np.array([64.0, 64.0, 6.125, 3809.0 / 2 ** 18], dtype=np.float32)
    q2 = np.zeros((H, I), dtype=np.uint8)
    q2[0, 1] = E4M3_ONE
    s2 = np.ones(H, dtype=np.float32)
    y = moe.token_outputs_fp8(x, [q1], [s1], [q2], [s2], np.array([1.0], dtype=np.float32))
    assert y.tolist() == [0.875, 0.0, 0.0, 0.0]


def test_e4m3_zero_row_gets_scale_one():
    x = np.zeros((2, 64), dtype=np.float32)
    x[1, 5] = -3.0
    c, s = quant.quant_rows_e4m3(x)
    assert s[0] == 1.0 and np.all(c[0] == 0)
    assert s[1] == np.float32(3.0) / np.float32(448.0) and c[1, 5] == 0x80 | E4M3_448


def test_fp8_expert_loop_equals_token_loop():
    # The expert-grouped form (used for layers too large for the token loop) sums the
    # same per-pair terms: it equals the token loop to float64 rounding on random layers,
    # with ties and repeats of experts across tokens.
    rng = np.random.default_rng(21)
    for T, H, I, E, k in ((9, 32, 16, 5, 2), (17, 64, 32, 8, 3)):
        x = rng.normal(size=(T, H)).astype(np.float32)
        q1, s1 = quant.quant_rows_e4m3(rng.normal(0, 0.1, size=(E * 2 * I, H)))
        q2, s2 = quant.quant_rows_e4m3(rng.normal(0, 0.1, size=(E * H, I)))
        gating = rng.normal(size=(T, E)).astype(np.float32)
        args = (q1.reshape(E, 2 * I, H), s1.reshape(E, 2 * I), q2.reshape(E, H, I), s2.reshape(E, H))
        y, tw, ids = moe.fused_forward_fp8(x, gating, *args, k, True)
        y2 = moe.expert_loop_forward_fp8(x, *args, tw, ids)
        np.testing.assert_allclose(y2, y, rtol=1e-12, atol=1e-12)
        # per-expert callables give the same sum as the arrays
        y3 = moe.expert_loop_forward_fp8(x, *(lambda e, a=a: a[e] for a in args), tw, ids)
        assert np.array_equal(y3, y2)
