"""Pins of the quantisers and the low-precision GMM oracle."""
import numpy as np
import pytest
import torch

from oracle import gmm, quant
import synth


def test_e4m3_codebook_spec_points():
    v = quant.E4M3_VALUES
    assert v[0x7E] == 448.0 and v[0xFE] == -448.0          # largest finite
    assert v[0x38] == 1.0                                   # exponent field 7 = bias
    assert v[0x08] == 2.0 ** -6                             # smallest normal
    assert v[0x01] == 2.0 ** -9                             # smallest subnormal
    assert v[0x07] == 7 * 2.0 ** -9                         # largest subnormal
    assert np.isnan(v[0x7F]) and np.isnan(v[0xFF])
    assert np.count_nonzero(np.isnan(v)) == 2               # no infinities, two NaNs
    fin = v[:0x7F]
    assert np.all(np.diff(fin) > 0)                         # codes 0..126 increase


def test_e4m3_round_trip_all_codes():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)])
    assert np.array_equal(quant.e4m3_encode(quant.E4M3_VALUES[codes]), codes.astype(np.uint8))


def test_e4m3_encode_matches_torch_cast_in_range():
    # Inside [-448, 448] the encoder is round-to-nearest-even, like torch's float8_e4m3fn cast.
    rng = np.random.default_rng(0)
    v = np.concatenate([rng.normal(0, 50, 20000), rng.uniform(-448, 448, 20000),
                        rng.normal(0, 0.01, 5000)]).astype(np.float32)
    mids = (quant.E4M3_VALUES[1:0x7E] + quant.E4M3_VALUES[2:0x7F]) / 2   # exact ties
    v = np.concatenate([v, mids.astype(np.float32), -mids.astype(np.float32)])
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(quant.e4m3_encode(v), ref)
    assert np.all(quant.e4m3_encode(np.array([500.0, 1e9, -460.0])) == [0x7E, 0x7E, 0xFE])


def test_int8_quant_error_bound_and_range():
    rng = np.random.default_rng(1)
    x = rng.normal(0, 0.02, size=(64, 300)).astype(np.float32)
    x[3] = 0.0
    q, s = quant.quant_rows_int8(x)
    assert q.dtype == np.int8 and np.abs(q.astype(int)).max() <= 127
    assert s[3] == 1.0 and np.all(q[3] == 0)
    err = np.abs(x.astype(np.float64) - s[:, None].astype(np.float64) * q)
    assert np.all(err <= s[:, None] * (0.5 + 1e-6))
    rows = [r for r in range(64) if r != 3]
    assert np.all(np.abs(q[rows]).max(axis=1) == 127)       # absmax maps to +-127


def test_int8_quant_matches_article_recipe_in_torch():
    # The article's torch recipe: scale = amax/127; clamp(round(w/scale), -127, 127).
    rng = np.random.default_rng(2)
    w = torch.from_numpy(rng.normal(0, 0.02, size=(32, 256)).astype(np.float32))
    scale = w.abs().amax(dim=1, keepdim=True) / 127.0
    ref = torch.clamp(torch.round(w / scale), -127, 127).to(torch.int8)
    q, s = quant.quant_rows_int8(w.numpy())
    assert np.array_equal(q, ref.numpy())
    assert np.array_equal(s, scale.squeeze(1).numpy())


def test_int8_ties_round_half_to_even():
    # absmax 127 gives the scale 1 exactly (254 gives 2): every quotient below is an exact
    # half-integer, and the article's torch.round sends it to the even neighbour, which is
    # also what Python's round() does.
    halves = [0.5, 1.5, 2.5, -2.5, -3.5, 63.5, 126.5, -126.5]
    x = np.array([[127.0] + halves, [254.0] + [2 * h for h in halves]], dtype=np.float32)
    q, s = quant.quant_rows_int8(x)
    assert list(s) == [1.0, 2.0]
    want = [127] + [round(h) for h in halves]
    assert q[0].tolist() == want and q[1].tolist() == want


def test_int8_quotient_is_rounded_to_fp32_first():
    # The article's recipe divides in float32: where the exact quotient lies just off a
    # half-integer but its float32 rounding lands on it (or across it), the code follows
    # the float32 quotient. Rows are built from such values, and the torch recipe decides.
    rng = np.random.default_rng(4)
    rows, n_differ = [], 0
    while len(rows) < 8:
        amax = np.float32(rng.uniform(1.0, 2.0))
        s32 = np.float32(amax / np.float32(127.0))
        vals = []
        for k in range(127):
            base = np.float32((k + 0.5) * np.float64(s32))
            for d in (-2, -1, 0, 1, 2):
                v = base
                for _ in range(abs(d)):
                    v = np.nextafter(v, np.float32(np.inf if d > 0 else -np.inf), dtype=np.float32)
                exact = np.float64(v) / np.float64(s32)
                if np.rint(np.float32(v / s32)) != np.rint(exact):
                    vals.append(v)
        if vals:
            n_differ += len(vals)
            rows.append(np.array([amax] + vals[:63] + [0.0] * (63 - len(vals[:63])), dtype=np.float32))
    x = np.stack(rows)
    w = torch.from_numpy(x)
    scale = w.abs().amax(dim=1, keepdim=True) / 127.0
    ref = torch.clamp(torch.round(w / scale), -127, 127).to(torch.int8)
    q, s = quant.quant_rows_int8(x)
    assert n_differ > 0
    assert np.array_equal(s, scale.squeeze(1).numpy())
    assert np.array_equal(q, ref.numpy())


def test_e4m3_quotient_is_rounded_to_fp32_first():
    # As for INT8: values placed a few float32 ulps from (midpoint between two e4m3
    # values) x scale, kept where the float32 quotient and the exact one fall on
    # different codes; the recipe (float32 division, then torch's e4m3 cast) decides.
    rng = np.random.default_rng(5)
    pos = np.sort(np.unique(np.abs(quant.E4M3_VALUES[np.isfinite(quant.E4M3_VALUES)])))
    mids = (pos[:-1] + pos[1:]) / 2.0
    rows, n_differ = [], 0
    while len(rows) < 8:
        amax = np.float32(rng.uniform(1.0, 2.0))
        s32 = np.float32(amax / np.float32(448.0))
        vals = []
        for m in mids:
            base = np.float32(m * np.float64(s32))
            for d in (-2, -1, 0, 1, 2):
                v = base
                for _ in range(abs(d)):
                    v = np.nextafter(v, np.float32(np.inf if d > 0 else -np.inf), dtype=np.float32)
                if abs(v) >= amax:
                    continue
                exact = np.float64(v) / np.float64(s32)
                if quant.e4m3_encode(np.float32(v / s32)) != quant.e4m3_encode(exact):
                    vals.append(v)
        if vals:
            n_differ += len(vals)
            vals = vals[:127]
            rows.append(np.array([amax] + vals + [0.0] * (127 - len(vals)), dtype=np.float32))
    x = np.stack(rows)
    w = torch.from_numpy(x)
    scale = w.abs().amax(dim=1, keepdim=True) / 448.0
    ref = (w / scale).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    c, s = quant.quant_rows_e4m3(x)
    assert n_differ > 0
    assert np.array_equal(s, scale.squeeze(1).numpy())
    assert np.array_equal(c, ref)


def test_e4m3_quant_bound():
    rng = np.random.default_rng(3)
    x = rng.normal(size=(16, 128)).astype(np.float32)
    c, s = quant.quant_rows_e4m3(x)
    deq = quant.dequant(c, "e4m3") * s[:, None]
    # relative spacing of e4m3 normals is 2^-3: rounding error <= half a spacing (+ subnormal floor)
    assert np.all(np.abs(deq - x) <= np.maximum(np.abs(x) * 2.0 ** -4, s[:, None] * 2.0 ** -10) + 1e-12)
    assert np.all(np.abs(quant.dequant(c, "e4m3")).max(axis=1) == 448.0)


def _groups(sizes):
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    return off, np.array(sizes, dtype=np.int32)


@pytest.mark.parametrize("dt", ["i8", "e4m3"])
def test_gmm_k1_closed_form(dt):
    rng = np.random.default_rng(4)
    sizes = [3, 0, 1, 4]
    off, sz = _groups(sizes)
    M, N, E = off[-1], 5, 4
    if dt == "i8":
        qx = rng.integers(-127, 128, size=(M, 1)).astype(np.int8)
        qw = rng.integers(-127, 128, size=(E, N, 1)).astype(np.int8)
        vx, vw = qx.astype(float), qw.astype(float)
    else:
        qx = rng.integers(0, 0x7F, size=(M, 1)).astype(np.uint8)
        qw = rng.integers(0x80, 0xFF, size=(E, N, 1)).astype(np.uint8)
        vx, vw = quant.E4M3_VALUES[qx], quant.E4M3_VALUES[qw]
    sx = rng.uniform(0.5, 2, M)
    sw = rng.uniform(0.5, 2, (E, N))
    y = gmm.gmm(qx, qw, sx, sw, off, sz, dt)
    for e in range(E):
        for m in range(off[e], off[e + 1]):
            for n in range(N):
                assert y[m, n] == pytest.approx(sx[m] * sw[e, n] * vx[m, 0] * vw[e, n, 0], rel=1e-15)


def test_gmm_exact_integers_and_groups():
    rng = np.random.default_rng(5)
    sizes = [5, 0, 1, 17, 2]
    off, sz = _groups(sizes)
    M, K, N, E = int(off[-1]), 64, 12, len(sizes)
    qx = rng.integers(-127, 128, size=(M, K)).astype(np.int8)
    qw = rng.integers(-127, 128, size=(E, N, K)).astype(np.int8)
    y = gmm.gmm(qx, qw, np.ones(M), np.ones((E, N)), off, sz, "i8")
    for e in range(E):
        ref = qx[off[e]:off[e + 1]].astype(np.int64) @ qw[e].astype(np.int64).T
        assert np.array_equal(y[off[e]:off[e + 1]], ref.astype(np.float64))
    # the size-1 group is a GEMV
    m = off[2]
    assert np.array_equal(y[m], (qw[2].astype(np.int64) @ qx[m].astype(np.int64)).astype(float))


def test_zipf_sizes_recipe():
    cfg = synth.lowp_config()
    s = synth.zipf_group_sizes(cfg.M, cfg.E, cfg.zipf_s, cfg.seed)
    assert sum(s) == cfg.M and len(s) == cfg.E
    assert 0 in s and 1 in s and max(s) > 256
