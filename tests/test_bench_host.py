"""Host logic of bench.py that needs no GPU: the clock sampler's parsing of
nvidia-smi's CSV and its selection of the samples inside a time window (the timed
steps, and the sustained window after them), and the max-over-ranks timing of
replicas, run as two gloo ranks on CPU."""
import datetime

import bench


class _Done:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        pass


def _sampler_with(tmp_path, lines):
    cs = bench.ClockSampler(0)
    cs.path = tmp_path / "clocks.csv"
    cs.path.write_text("\n".join(lines) + "\n")
    cs.proc = _Done()
    cs.fh = open(cs.path, "a")
    return cs


def _line(t, sm, power_cap=False, thermal=False):
    ts = t.strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
    na, act = "Not Active", "Active"
    return (f"{ts}, 0, {sm}, 2070, 900.00, 0x0, {na}, {na}, {act if thermal else na}, "
            f"{act if power_cap else na}")


def test_samples_are_selected_by_window(tmp_path):
    t0 = datetime.datetime(2026, 1, 1, 12, 0, 0)
    ms = lambda k: t0 + datetime.timedelta(milliseconds=k)
    lines = [_line(ms(10 * i), 2070 if i < 5 else 1800, power_cap=(i == 7)) for i in range(10)]
    lines.insert(3, "garbage line")
    lines.append("2026/01/01 12:00:01.000, 0, [N/A], 2070, 0, 0x0, x, x, x, x")
    rows = _sampler_with(tmp_path, lines).stop()
    assert len(rows) == 10                                  # malformed lines skipped
    first = bench.ClockSampler.summary(rows, ms(0), ms(45))
    assert first == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 5}
    late = bench.ClockSampler.summary(rows, ms(50), ms(95))
    assert late["sm_mhz"] == 1800.0 and late["reasons"] == ["sw_power_cap"] and late["samples"] == 5
    assert bench.ClockSampler.summary(rows, ms(500), ms(600))["samples"] == 0


def test_thermal_reasons_are_reported(tmp_path):
    t0 = datetime.datetime(2026, 1, 1, 12, 0, 0)
    rows = _sampler_with(tmp_path, [_line(t0, 1500, thermal=True)]).stop()
    s = bench.ClockSampler.summary(rows, t0, t0)
    assert s["reasons"] == ["sw_thermal_slowdown"] and s["sm_mhz"] == 1500.0


def test_no_sampler_gives_no_rows():
    assert bench.ClockSampler(0).stop() is None


def _rank_main(rank, world, port, step_ms, out):
    import os
    import torch
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(torch, step_ms[rank], torch.device("cpu"))
        out[rank] = (ms, bench.job_tokens_per_s(4096, world, ms))
    finally:
        dist.destroy_process_group()


def test_replica_timing_takes_the_slowest_rank():
    """Two gloo ranks on CPU with different step times: both see the slower one, and the job's
    throughput counts both ranks' tokens over it (the N > 1 bookkeeping of the bench)."""
    import socket
    import torch.multiprocessing as mp
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    step_ms = [0.35, 0.5]
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, step_ms, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    for r in range(2):
        ms, tps = out[r]
        assert ms == 0.5
        assert abs(tps - 2 * 4096 / 0.5e-3) < 1e-6 * tps


def test_single_process_timing_is_unchanged():
    import torch
    assert bench.max_over_ranks(torch, 0.25, torch.device("cpu")) == 0.25
    assert bench.job_tokens_per_s(4096, 1, 0.25) == 4096 / 0.25e-3


_CONTRACT = {
    "metric": str, "value": float, "unit": str, "n_gpus": int, "steps": int, "warmup": int,
    "ms_per_step": float, "higher_is_better": bool, "scaling": str, "dtype": str, "data": str,
    "config": dict, "cpu_baseline": dict, "e2e": dict,
}


def test_reference_arm_prints_the_contract_line():
    """The reference arm (the oracle on host cores) runs without a GPU: its JSON line carries
    every key of the bench contract, on a small workload here."""
    import argparse
    import json
    import synth
    args = argparse.Namespace(steps=2, warmup=3)
    line = json.loads(json.dumps(bench.run_reference(args, 0, 1, cfg=synth.tiny_config(), n=16)))
    for key, typ in _CONTRACT.items():
        assert isinstance(line[key], typ), key
    assert line["impl"] == "reference" and line["vs_baseline"] is None
    assert line["config"]["workload"] == synth.tiny_config().name
    assert line["metric"] == bench.METRIC and line["unit"] == "tokens/s" and line["higher_is_better"]
    assert line["value"] > 0 and line["ms_per_step"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["cpu_baseline"]["cores"] >= 1 and "16 of 64 tokens" in line["cpu_baseline"]["sample"]
    assert line["e2e"] == {"value": line["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}


def test_fp32_score_collisions_counts_rows_that_rounding_would_tie():
    import numpy as np
    a = np.float32(20.0)
    b = np.nextafter(a, np.float32(0.0), dtype=np.float32)   # distinct logit, same fp32 sigmoid (1.0)
    x = np.array([[a, b, 0.0, -1.0], [3.0, 2.0, 1.0, 0.0], [0.5, 0.5, 0.0, 0.0]], dtype=np.float32)
    assert bench.fp32_score_collisions(x, "sigmoid", 2) == 1   # equal logits are not counted
    assert bench.fp32_score_collisions(x, "softmax", 2) == 0   # softmax keeps 20 and its neighbour apart
    y = np.array([[0.0, -100.0, -100.00001, -200.0]], dtype=np.float32)
    assert bench.fp32_score_collisions(y, "softmax", 3) == 1   # both underflow to 0 in float32
    assert bench.fp32_score_collisions(y, "softmax", 2) == 0
