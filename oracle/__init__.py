"""CPU oracle for the fused, grouped-routed MoE layer forward.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import it. The
product path (the CUDA library and its Python binding) never calls it and
shares no code with it.

Plain, slow, obviously correct numpy in float64, each function written from the
pages it cites:

* ``routing``  grouped top-k routing (GroupedTopK blog, sections 3.1-3.6 and 7;
  mini-sglang MoE chapter, ``select_experts``);
* ``align``    ``moe_align_block_size`` (mini-sglang MoE chapter, "fused MoE");
* ``moe``      the expert-loop MoE forward (mini-sglang ``TorchMoeBackend``),
  the token-view form and the per-pair gathered projection (Fused MoE Part 3,
  sections 01 and 03), and the layer with FP8-e4m3 GEMM operands (per-token
  activation and per-channel weight scales, low-precision GMM article,
  sections 2.3, 3.2 and 4.3);
* ``quant``    symmetric per-row INT8 / FP8-e4m3 quantisation (low-precision
  GMM article, section 3.2) and the OCP E4M3 code book;
* ``gmm``      the dequantise-then-matmul grouped GEMM (low-precision GMM
  article, sections 2.1 and 3.1).

Every function is pinned by ``tests/test_oracle_*.py`` to the pages' worked
examples, closed forms, invariants or brute force; none is "parity unpinned".
"""
from . import align, gmm, moe, quant, routing  # noqa: F401
