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
@pytest.mark.parametrize("M,K", [(1, 8), (37, 264), (2048, 4096)])
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
