"""GPU gmm_lowp (INT8 / FP8-e4m3 grouped GEMM, scales fused) vs the float64
dequantise-then-matmul oracle. Codes and scales come from the oracle's
quantisers on the host, so both sides read identical inputs."""
import numpy as np
import pytest
import torch

from gpu_util import require_gpu
from oracle import gmm as ogmm
from oracle import quant
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


TORCH_DT = {"i8": torch.int8, "e4m3": torch.float8_e4m3fn}


def _to_dev(codes, dt):
    if dt == "i8":
        return torch.from_numpy(np.ascontiguousarray(codes.astype(np.int8))).cuda()
    return torch.from_numpy(np.ascontiguousarray(codes.astype(np.uint8))).cuda().view(torch.float8_e4m3fn)


def _run(qx, qw, sx, sw, sizes, dt, out_dtype):
    import mixture_experts_routing_grouped_gb300 as moe
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    M, K = qx.shape
    E, N, _ = qw.shape
    ws = torch.zeros(moe.gmm_lowp_workspace_size(M, K, N, E), dtype=torch.uint8, device="cuda")
    out = moe.gmm_lowp(_to_dev(qx, dt), _to_dev(qw, dt), torch.from_numpy(sx.astype(np.float32)).cuda(),
                       torch.from_numpy(sw.astype(np.float32)).cuda(), torch.from_numpy(off).cuda(),
                       torch.from_numpy(np.asarray(sizes, dtype=np.int32)).cuda(), out_dtype=out_dtype, ws=ws)
    torch.cuda.synchronize()
    assert moe.moe_check_device_error(ws) == 0
    return out.float().cpu().numpy().astype(np.float64), off


def _assert_close(got, ref, out_dtype):
    d = np.abs(got - ref)
    m = np.abs(ref).max() if ref.size else 0.0
    if out_dtype == torch.float32:
        assert np.linalg.norm(got - ref) <= 1e-3 * np.linalg.norm(ref)
        assert d.max() <= 1e-3 * m
    else:  # bf16 rounding of the fp32 result
        assert (d <= 2.0 ** -8 * np.abs(ref) + 1e-4 * m).all(), f"max dev {d.max()}"


def _random_codes(rng, shape, dt):
    if dt == "i8":
        return rng.integers(-127, 128, size=shape).astype(np.int8)
    c = rng.integers(0, 256, size=shape).astype(np.uint8)
    c[(c & 0x7F) == 0x7F] = 0x3A      # no NaN codes
    return c


@pytest.mark.parametrize("dt", ["i8", "e4m3"])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("sizes,K,N", [([37, 0, 1, 200, 130, 5], 256, 256), ([128], 128, 128),
                                       ([0, 0, 300, 0], 384, 128), ([1, 1, 1], 128, 384)])
def test_gmm_small_full(dt, out_dtype, sizes, K, N):
    rng = np.random.default_rng(len(sizes) * 1000 + K + N)
    M, E = sum(sizes), len(sizes)
    qx = _random_codes(rng, (M, K), dt)
    qw = _random_codes(rng, (E, N, K), dt)
    sx = rng.uniform(0.01, 0.1, M)
    sw = rng.uniform(0.001, 0.01, (E, N))
    got, off = _run(qx, qw, sx, sw, sizes, dt, out_dtype)
    ref = ogmm.gmm(qx, qw, sx.astype(np.float32), sw.astype(np.float32), off, sizes, dt)
    _assert_close(got, ref, out_dtype)


def test_gmm_int8_exact_integers():
    # unit scales and K = 256: every partial sum stays below 2^24, so fp32 accumulation is exact
    rng = np.random.default_rng(3)
    sizes = [70, 1, 0, 129]
    M, K, N, E = sum(sizes), 256, 128, len(sizes)
    qx = rng.integers(-127, 128, size=(M, K)).astype(np.int8)
    qw = rng.integers(-127, 128, size=(E, N, K)).astype(np.int8)
    got, off = _run(qx, qw, np.ones(M), np.ones((E, N)), sizes, "i8", torch.float32)
    for e in range(E):
        ref = qx[off[e]:off[e + 1]].astype(np.int64) @ qw[e].astype(np.int64).T
        assert np.array_equal(got[off[e]:off[e + 1]], ref.astype(np.float64))


@pytest.mark.parametrize("dt", ["i8", "e4m3"])
def test_gmm_workspace_reused_across_calls(dt):
    """The task counters live in the workspace: consecutive calls on one workspace (different
    group layouts and sizes) each compute every row, and leave the counters zero."""
    import mixture_experts_routing_grouped_gb300 as moe
    rng = np.random.default_rng(11)
    K, N, E = 256, 384, 5
    ws = torch.zeros(moe.gmm_lowp_workspace_size(700, K, N, E), dtype=torch.uint8, device="cuda")
    for sizes in ([100, 0, 300, 1, 299], [700, 0, 0, 0, 0], [1, 2, 3, 4, 5], [0, 0, 0, 0, 129]):
        M = sum(sizes)
        qx = _random_codes(rng, (M, K), dt)
        qw = _random_codes(rng, (E, N, K), dt)
        sx = rng.uniform(0.01, 0.1, M)
        sw = rng.uniform(0.001, 0.01, (E, N))
        off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
        out = moe.gmm_lowp(_to_dev(qx, dt), _to_dev(qw, dt), torch.from_numpy(sx.astype(np.float32)).cuda(),
                           torch.from_numpy(sw.astype(np.float32)).cuda(), torch.from_numpy(off).cuda(),
                           torch.from_numpy(np.asarray(sizes, dtype=np.int32)).cuda(), out_dtype=torch.float32,
                           ws=ws)
        torch.cuda.synchronize()
        assert moe.moe_check_device_error(ws) == 0
        assert torch.count_nonzero(ws[4:12]).item() == 0
        ref = ogmm.gmm(qx, qw, sx.astype(np.float32), sw.astype(np.float32), off, sizes, dt)
        _assert_close(out.cpu().numpy().astype(np.float64), ref, torch.float32)


def test_gmm_inconsistent_metadata_is_reported_and_skipped():
    import mixture_experts_routing_grouped_gb300 as moe
    rng = np.random.default_rng(4)
    M, K, N, E = 64, 128, 128, 2
    qx = torch.from_numpy(rng.integers(-127, 128, size=(M, K)).astype(np.int8)).cuda()
    qw = torch.from_numpy(rng.integers(-127, 128, size=(E, N, K)).astype(np.int8)).cuda()
    off = torch.tensor([0, 32, 64], dtype=torch.int32, device="cuda")
    sizes = torch.tensor([32, 40], dtype=torch.int32, device="cuda")   # expert 1 does not add up
    out = torch.full((M, N), 7.0, dtype=torch.float32, device="cuda")
    ws = torch.zeros(moe.gmm_lowp_workspace_size(M, K, N, E), dtype=torch.uint8, device="cuda")
    moe.gmm_lowp(qx, qw, torch.ones(M, device="cuda"), torch.ones(E, N, device="cuda"), off, sizes,
                 out_dtype=torch.float32, out=out, ws=ws)
    code = moe.moe_check_device_error(ws)
    assert code & moe.DEVERR_GROUP_META
    o = out.cpu().numpy()
    assert np.all(o[32:] == 7.0)                     # skipped expert's rows untouched
    ref = qx[:32].cpu().numpy().astype(np.int64) @ qw[0].cpu().numpy().astype(np.int64).T
    assert np.array_equal(o[:32], ref.astype(np.float32))


@pytest.fixture(scope="module", params=[synth.lowp_config(), synth.lowp_small_k_config()], ids=lambda c: c.name)
def lowp_workload(request):
    cfg = request.param
    d = synth.gmm_inputs(cfg, "cuda")
    x = d["x"].cpu().numpy()
    w = d["w"].cpu().numpy().reshape(cfg.E * cfg.N, cfg.K)
    del d["w"], d["x"]
    torch.cuda.empty_cache()
    return cfg, x, w, d["expert_sizes"].cpu().numpy()


@pytest.mark.parametrize("dt", ["i8", "e4m3"])
def test_gmm_lowp_workload_whole(lowp_workload, dt):
    """Every element of the full workload's output, with fp32 output (1e-3 relative: Frobenius
    and max) and with bf16 output (the bf16 rounding of the fp32 result)."""
    cfg, x, w, sizes = lowp_workload
    qfn = quant.quant_rows_int8 if dt == "i8" else quant.quant_rows_e4m3
    qx, sx = qfn(x)
    qw, sw = qfn(w)
    qw = qw.reshape(cfg.E, cfg.N, cfg.K)
    sw = sw.reshape(cfg.E, cfg.N)
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    ref = ogmm.gmm(qx, qw, sx, sw, off, sizes, dt)
    for out_dtype in (torch.float32, torch.bfloat16):
        got, _ = _run(qx, qw, sx, sw, sizes, dt, out_dtype)
        _assert_close(got, ref, out_dtype)
