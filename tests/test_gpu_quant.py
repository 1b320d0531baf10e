"""GPU per-row quantisation vs the oracle: codes bit-exact, scales bit-exact."""
import numpy as np
import pytest
import torch

from gpu_util import require_gpu
from oracle import quant
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


@pytest.mark.parametrize("qdt", [torch.int8, torch.float8_e4m3fn])
@pytest.mark.parametrize("xdt", [torch.float32, torch.bfloat16])
# (20000, 768) and (5000, 2048): several rows per warp of the persistent bf16 kernel
@pytest.mark.parametrize("M,K", [(1, 8), (37, 264), (2048, 4096), (20000, 768), (5000, 2048)])
def test_quant_rows(qdt, xdt, M, K):
    import mixture_experts_routing_grouped_gb300 as moe
    x = synth.normal((M, K), 99, M + K, 1.0, xdt, "cuda")
    x[M // 2] = 0                                      # an all-zero row
    q, s = moe.moe_quant_per_token(x, qdt)
    torch.cuda.synchronize()
    xn = x.float().cpu().numpy()
    if qdt == torch.int8:
        rq, rs = quant.quant_rows_int8(xn)
        assert np.array_equal(q.cpu().numpy(), rq)
    else:
        rq, rs = quant.quant_rows_e4m3(xn)
        assert np.array_equal(q.view(torch.uint8).cpu().numpy(), rq)
    assert np.array_equal(s.cpu().numpy(), rs)


def _hard_rows(M, K, seed):
    """Rows built to stress the quotient x / scale: per-row magnitudes 2^-60 .. 2^60, exact powers
    of two, small integers, repeated absmax values, and values on and next to the e4m3 rounding
    midpoints and the INT8 half-integers times the row scale (where a quotient one ulp off would
    change the code). The large kinds are placed first and the row's absmax taken after them, so
    that the boundary values sit on boundaries of the scale the row actually gets."""
    rng = np.random.default_rng(seed)
    x = rng.normal(0, 1, size=(M, K)).astype(np.float32)
    mag = np.float32(2.0) ** rng.integers(-60, 61, size=(M, 1)).astype(np.float32)
    x *= mag
    kind = rng.integers(0, 5, size=(M, K))
    x = np.where(kind == 2, np.float32(2.0) ** rng.integers(-8, 8, size=(M, K)).astype(np.float32) * mag, x)
    x = np.where(kind == 3, rng.integers(-300, 300, size=(M, K)).astype(np.float32) * mag, x)
    amax = np.abs(x).max(axis=1, keepdims=True)
    scale = (amax / np.float32(448.0)).astype(np.float32)
    mids = ((quant.E4M3_VALUES[1:0x7E] + quant.E4M3_VALUES[2:0x7F]) / 2).astype(np.float32)
    pick = rng.integers(0, len(mids), size=(M, K))
    nudge = rng.integers(-3, 4, size=(M, K)).astype(np.int32)
    on_mid = (mids[pick] * scale).astype(np.float32)
    on_mid = (on_mid.view(np.int32) + nudge).view(np.float32)             # a few ulps either side
    x = np.where(kind == 1, on_mid, x)
    # half-integers times the INT8 row scale (absmax / 127), a few ulps either side: INT8 rounding ties
    s8 = (amax / np.float32(127.0)).astype(np.float32)
    half = ((rng.integers(-127, 127, size=(M, K)) + 0.5).astype(np.float32) * s8).astype(np.float32)
    half = (half.view(np.int32) + rng.integers(-3, 4, size=(M, K)).astype(np.int32)).view(np.float32)
    x = np.where(kind == 4, half, x)
    x[:, 0] = amax[:, 0]
    x[:, 1] = -amax[:, 0]
    return x.astype(np.float32)


@pytest.mark.parametrize("qdt", [torch.int8, torch.float8_e4m3fn])
@pytest.mark.parametrize("xdt", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("M,K", [(4096, 1024), (1024, 2048), (128, 4104), (12000, 768)])
def test_quant_rows_hard_values(qdt, xdt, M, K):
    import mixture_experts_routing_grouped_gb300 as moe
    xt = torch.from_numpy(_hard_rows(M, K, M + K)).to(xdt)
    q, s = moe.moe_quant_per_token(xt.cuda(), qdt)
    torch.cuda.synchronize()
    xn = xt.float().numpy()
    if qdt == torch.int8:
        rq, rs = quant.quant_rows_int8(xn)
        got = q.cpu().numpy()
    else:
        rq, rs = quant.quant_rows_e4m3(xn)
        got = q.view(torch.uint8).cpu().numpy()
    assert np.array_equal(s.cpu().numpy(), rs)
    bad = np.argwhere(got != rq)
    assert bad.size == 0, f"{len(bad)} codes differ, first at {bad[:3].tolist()}"
