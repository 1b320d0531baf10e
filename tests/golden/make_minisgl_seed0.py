"""Writes minisgl_seed0_routing.json: the input of the mini-sglang MoE chapter's example.

The chapter's example program (section "在 CPU 上运行 Triton", examples/ch20_moe.py)
seeds torch with 0, draws x = randn(5, 64) and then gating = randn(5, 8), routes
with top-2 softmax + renormalise, and aligns with block_m = 4. This script
re-draws those gating logits with torch's CPU generator and stores them with
the outputs the chapter prints (its "运行结果" block), typed in from the page.
It calls neither the oracle nor the CUDA library.
"""
import json
import pathlib

import torch

torch.manual_seed(0)
_x = torch.randn(5, 64)
gating = torch.randn(5, 8)

fixture = {
    "source": "mini-sglang MoE chapter (anrans.github.io/ai-infra-handbooks/minisgl/perf/moe/), "
              "example examples/ch20_moe.py and its printed results",
    "T": 5, "E": 8, "topk": 2, "renormalize": True, "block_m": 4,
    "gating_hex": [[float(v).hex() for v in row] for row in gating.tolist()],
    "expected_topk_ids": [[4, 3], [6, 1], [1, 7], [6, 4], [5, 4]],
    "expected_topk_weights_3dp": [[0.692, 0.308], [0.545, 0.455], [0.93, 0.07],
                                  [0.711, 0.289], [0.809, 0.191]],
    "expected_sorted_ids": [3, 4, 10, 10, 1, 10, 10, 10, 0, 7, 9, 10, 8, 10, 10, 10,
                            2, 6, 10, 10, 5, 10, 10, 10],
    "expected_expert_ids": [1, 3, 4, 5, 6, 7],
}
out = pathlib.Path(__file__).with_name("minisgl_seed0_routing.json")
out.write_text(json.dumps(fixture, indent=1) + "\n")
print("wrote", out)
