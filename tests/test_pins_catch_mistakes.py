"""The oracle's pins catch plausible mistakes.

Each case plants one mistake in a copy of ``oracle/`` (a dropped term, a wrong sign
or index, a swapped operand, another rounding or tie rule, a wrong constant) and runs
the oracle pin tests (``tests/test_oracle_*.py``) against that copy: every case must
make at least one of them fail, and the unmodified copy must pass. Runs on the CPU;
nothing outside the temporary copy is changed.

One plausible edit is left out because it is not a mistake on valid inputs: taking
a group's end from ``expert_offsets[e + 1]`` instead of ``expert_offsets[e] +
expert_sizes[e]`` in the grouped GEMM, which agree whenever the metadata is
consistent (inconsistent metadata is a device-reported error, not an oracle case).
"""
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

import pytest

from conftest import ROOT

MISTAKES = [
    # routing (GroupedTopK blog; mini-sglang select_experts)
    ("routing.py", "group_key = xd.reshape(T, G, P).max(axis=2)", "group_key = xd.reshape(T, G, P).sum(axis=2)",
     "group score is a sum"),
    ("routing.py", 'return np.argsort(-keys, axis=-1, kind="stable")',
     'return (keys.shape[-1] - 1 - np.argsort(-keys[..., ::-1], axis=-1, kind="stable"))', "ties to the higher index"),
    ("routing.py", "        w = w / w.sum(axis=1, keepdims=True)", "        w = w", "no renormalisation"),
    ("routing.py", "    w = w * routed_scaling_factor", "    w = w * (routed_scaling_factor if renormalize else 1.0)",
     "scaling factor only with renormalisation"),
    ("routing.py", "return 1.0 / (1.0 + np.exp(-x))", "return 1.0 / (1.0 + np.exp(x))", "sigmoid sign"),
    ("routing.py", "ex = np.exp(x - m)", "ex = np.exp(x - m) + 1e-3", "softmax perturbed"),
    ("routing.py", "ids = _rank_desc(masked)[:, :topk]", "ids = _rank_desc(xd)[:, :topk]", "group mask ignored"),
    ("routing.py", "sel_groups = _rank_desc(group_key)[:, :topk_group]",
     "sel_groups = _rank_desc(-group_key)[:, :topk_group]", "worst groups kept"),
    ("routing.py", "    return (x @ w.T).astype(np.float32)", "    return (x @ w.T).astype(np.float16).astype(np.float32)",
     "router logits rounded to half precision"),
    ("routing.py", "    return (x @ w.T).astype(np.float32)",
     "    return (x.astype(np.float32) @ w.T.astype(np.float32)).astype(np.float32)", "router summed in float32"),
    ("routing.py", "    logits = router_logits(hidden_states, w_gate)\n",
     "    logits = -router_logits(hidden_states, w_gate)\n", "router logits negated"),
    # align (mini-sglang moe_align_block_size)
    ("align.py", "sorted_ids = np.full(cap, num_pairs, dtype=np.int32)",
     "sorted_ids = np.full(cap, num_pairs - 1, dtype=np.int32)", "sentinel off by one"),
    ("align.py", "length = -(-count[e] // block_m) * block_m", "length = (count[e] // block_m + 1) * block_m",
     "over-padding"),
    ("align.py", "    for p, e in enumerate(pair_expert):\n        sorted_ids",
     "    for p, e in reversed(list(enumerate(pair_expert))):\n        sorted_ids", "unstable within an expert"),
    ("align.py", "expert_ids = np.full(cap // block_m, -1, dtype=np.int32)",
     "expert_ids = np.full(cap // block_m, 0, dtype=np.int32)", "trailing block experts 0"),
    ("align.py", "expert_offsets = np.array(seg_begin + [total], dtype=np.int32)",
     "expert_offsets = np.array(seg_begin + [num_pairs], dtype=np.int32)", "offsets end at the pair count"),
    # MoE forward (mini-sglang TorchMoeBackend; Fused MoE Part 3)
    ("moe.py", "        act = silu(gate_proj) * up_proj", "        act = silu(up_proj) * gate_proj",
     "gate and up swapped (expert loop)"),
    ("moe.py", "        contrib = (act @ _expert_matrix(w2, e).T) * tw[pair_tok, pair_slot][:, None]",
     "        contrib = act @ _expert_matrix(w2, e).T", "route weight dropped"),
    ("moe.py", "        contrib = (act @ _expert_matrix(w2, e).T) * tw[pair_tok, pair_slot][:, None]",
     "        contrib = (act @ _expert_matrix(w2, e).T) * tw[pair_tok, 0][:, None]", "route weight of slot 0"),
    ("moe.py", "    return v / (1.0 + np.exp(-v))", "    return np.maximum(v, 0.0)", "relu instead of silu"),
    ("moe.py", "    h = silu(gu[:, :, :I]) * gu[:, :, I:]", "    h = silu(gu[:, :, I:]) * gu[:, :, :I]",
     "gate and up swapped (token view)"),
    ("moe.py", "        h = silu(w1e[:I] @ x) * (w1e[I:] @ x)", "        h = silu(w1e[I:] @ x) * (w1e[:I] @ x)",
     "gate and up swapped (one token)"),
    ("moe.py", "        h = _bf16_round(silu(w1[:I] @ dx) * (w1[I:] @ dx))", "        h = silu(w1[:I] @ dx) * (w1[I:] @ dx)",
     "FP8 layer: h not held in bf16"),
    ("moe.py", '    dx = quant.dequant(qx[0], "e4m3") * float(sx[0])', '    dx = quant.dequant(qx[0], "e4m3")',
     "FP8 layer: token scale dropped"),
    ("moe.py", '        w2 = quant.dequant(q2, "e4m3") * np.asarray(s2, dtype=np.float64)[:, None]',
     '        w2 = quant.dequant(q2, "e4m3")', "FP8 layer: down channel scale dropped"),
    ("moe.py", '        out = out + float(wj) * (w2 @ (quant.dequant(qh[0], "e4m3") * float(sh[0])))',
     "        out = out + float(wj) * (w2 @ h)", "FP8 layer: h not quantised"),
    ("moe.py", "        h = _bf16_round(silu(w1[:I] @ dx) * (w1[I:] @ dx))",
     "        h = _bf16_round(silu(w1[I:] @ dx) * (w1[:I] @ dx))", "FP8 layer: gate and up swapped"),
    ("moe.py", "        hs = _bf16_round(silu(xs @ w1[:I].T) * (xs @ w1[I:].T))",
     "        hs = silu(xs @ w1[:I].T) * (xs @ w1[I:].T)", "FP8 expert loop: h not held in bf16"),
    ("moe.py", '    dx = quant.dequant(qx, "e4m3") * sx.astype(np.float64)[:, None]',
     '    dx = quant.dequant(qx, "e4m3")', "FP8 expert loop: token scale dropped"),
    ("moe.py", "        contrib = (dh @ w2.T) * tw[pair_tok, pair_slot][:, None]",
     "        contrib = (hs @ w2.T) * tw[pair_tok, pair_slot][:, None]", "FP8 expert loop: h not quantised"),
    # quantisers and the E4M3 code book (low-precision GMM article; OCP FP8)
    ("quant.py", "INT8_QMAX = 127.0", "INT8_QMAX = 128.0", "INT8 range 128"),
    ("quant.py", "q = np.clip(np.rint(quot), -INT8_QMAX, INT8_QMAX)",
     "q = np.clip(np.trunc(quot + np.copysign(0.5, quot)), -INT8_QMAX, INT8_QMAX)", "INT8 ties away from zero"),
    ("quant.py", "    quot = (x32 / scale[:, None]).astype(np.float32)             # float32 division",
     "    quot = (x32.astype(np.float64) / scale[:, None])", "INT8 quotient in double"),
    ("quant.py", "    quot = (x32 / scale[:, None]).astype(np.float32)\n    return e4m3_encode(quot), scale",
     "    quot = (x32.astype(np.float64) / scale[:, None])\n    return e4m3_encode(quot), scale",
     "e4m3 quotient in double"),
    ("quant.py", "    scale = np.where(amax == 0, np.float32(1.0), scale).astype(np.float32)\n"
                 "    quot = (x32 / scale[:, None]).astype(np.float32)\n    return",
     "    scale = np.where(amax == 0, np.float32(0.0), scale).astype(np.float32)\n"
     "    quot = (x32 / scale[:, None]).astype(np.float32)\n    return", "e4m3 zero row scale 0"),
    ("quant.py", "E4M3_MAX = 448.0", "E4M3_MAX = 240.0", "e4m3 maximum 240"),
    ("quant.py", "        return sign * (man / 8.0) * 2.0 ** -6", "        return sign * (man / 8.0) * 2.0 ** -7",
     "e4m3 subnormal exponent"),
    ("quant.py", "    return sign * (1.0 + man / 8.0) * 2.0 ** (exp - 7)",
     "    return sign * (1.0 + man / 8.0) * 2.0 ** (exp - 8)", "e4m3 exponent bias 8"),
    ("quant.py", "    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (pos_codes[hi] % 2 == 0))",
     "    pick_hi = (d_hi <= d_lo)", "e4m3 ties up instead of to even"),
    # grouped GEMM (low-precision GMM article)
    ("gmm.py", "        y[lo:hi] = sx[lo:hi, None] * sw[e][None, :] * acc", "        y[lo:hi] = sx[lo:hi, None] * acc",
     "weight scale dropped"),
    ("gmm.py", "        y[lo:hi] = sx[lo:hi, None] * sw[e][None, :] * acc",
     "        y[lo:hi] = sx[lo:hi, None] * sw[min(e + 1, E - 1)][None, :] * acc", "next expert's weight scale"),
]

PIN_TESTS = sorted(p.name for p in (ROOT / "tests").glob("test_oracle_*.py"))


def _copy(dst):
    for d in ("oracle", "tests", "synth"):
        shutil.copytree(ROOT / d, dst / d, ignore=shutil.ignore_patterns("__pycache__"))
    shutil.copy(ROOT / "pytest.ini", dst)


def _run_pins(root):
    env = dict(os.environ, PYTHONDONTWRITEBYTECODE="1")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        *[f"tests/{t}" for t in PIN_TESTS]], cwd=root, capture_output=True, text=True,
                       env=env, timeout=600)
    return r.returncode, r.stdout[-2000:]


def test_every_planted_mistake_fails_a_pin(tmp_path):
    base = tmp_path / "base"
    _copy(base)
    rc, out = _run_pins(base)
    assert rc == 0, out

    def one(i):
        f, old, new, what = MISTAKES[i]
        root = tmp_path / f"m{i}"
        _copy(root)
        src = (root / "oracle" / f).read_text()
        assert src.count(old) >= 1, f"{what}: the line to change is not in oracle/{f}"
        (root / "oracle" / f).write_text(src.replace(old, new))
        rc, out = _run_pins(root)
        shutil.rmtree(root, ignore_errors=True)
        return what, rc, out

    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 2)) as ex:
        results = list(ex.map(one, range(len(MISTAKES))))
    missed = [what for what, rc, _ in results if rc == 0]
    assert not missed, f"mistakes no pin catches: {missed}"
