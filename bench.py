#!/usr/bin/env python
"""Benchmark of the GB300 fused MoE layer forward.

Default workload: the prefill layer T=4096, H=2048, I=768, E=128, top-8 softmax
routing with renormalisation (bf16 activations and weights). A step is one full
pass of the hot path through the C ABI (moe_fused_forward: routing, align,
gate_up grouped GEMM + SwiGLU, down grouped GEMM + weighted combine, cast).
Inputs are resident in HBM when the timed region starts; L2 is flushed (256 MiB
write) between timed steps, outside the per-step CUDA-event windows.

Also reported: the decode layer (E=256, H=7168, I=2048, grouped sigmoid routing)
as weight-stream GB/s at T in {1, 8, 32, 128}, and grouped top-k routing alone
at T=16384 as GB/s. `--impl reference` times the CPU oracle instead.

Prints one JSON line (rank 0).
"""
from __future__ import annotations

import argparse
import hashlib
import datetime
import json
import os
import pathlib
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = pathlib.Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

METRIC = "MoE layer tokens/s + % BF16 tensor peak; decode weight-stream GB/s vs HBM"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 256 << 20
E2E_STREAMS = 4  # streams (each with its own buffers) that the end-to-end steps rotate over


def load_peaks():
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        d = json.loads(p.read_text())
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("LOCAL_RANK", "0"))


# --------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons every 10 ms, timestamped, so
    that the samples inside a window (the timed steps) can be told from the rest."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        # The raw samples go to $MOE_BENCH_CLOCKS_DIR when it is set (to keep them), else
        # to the system's temporary directory.
        out = os.environ.get("MOE_BENCH_CLOCKS_DIR") or tempfile.gettempdir()
        self.path = pathlib.Path(out) / f"moe_bench_clocks_gpu{gpu_index}_{os.getpid()}.csv"

    def start(self, wait_s: float = 3.0):
        """Starts the sampler and returns once it has written its first sample (or after wait_s)."""
        try:
            self.path.parent.mkdir(parents=True, exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "10"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        t0 = time.time()
        while time.time() - t0 < wait_s and self.proc.poll() is None:
            self.fh.flush()
            if self.path.stat().st_size > 0:
                break
            time.sleep(0.01)

    @staticmethod
    def now():
        return datetime.datetime.now()

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        rows = []
        for line in self.path.read_text().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f")
                rows.append((ts, float(parts[2]), float(parts[3]),
                             {n for n, v in zip(self.REASONS, parts[6:10]) if v.lower().startswith("active")}))
            except ValueError:
                continue
        return rows

    @staticmethod
    def summary(rows, t0, t1):
        """Median SM clock, the clock limit and the throttle reasons of the samples in [t0, t1]."""
        sel = [r for r in rows if t0 <= r[0] <= t1]
        if not sel:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(r[1] for r in sel), "sm_max_mhz": max(r[2] for r in sel),
                "reasons": sorted(set().union(*(r[3] for r in sel))), "samples": len(sel)}


# --------------------------------------------------------------------------- helpers
def max_over_ranks(torch, value: float, device) -> float:
    """The largest `value` over the ranks of the default process group (`value` itself when
    no group is initialised). Every rank must call it: it is a collective."""
    dist = torch.distributed
    if not (dist.is_available() and dist.is_initialized()):
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(tokens_per_rank: int, world: int, ms: float) -> float:
    """Whole-job throughput: the tokens every rank processed over the slowest rank's step time."""
    return world * tokens_per_rank / (ms * 1e-3)


def kernel_traffic(kernel: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the current source."""
    p = ROOT / "profiles" / "traffic.json"
    if not p.exists():
        return None
    d = json.loads(p.read_text()).get(kernel)
    if not d:
        return None
    src = ROOT / d["source"]
    if not src.exists() or hashlib.sha256(src.read_bytes()).hexdigest() != d["source_sha256"]:
        return None
    return d["bytes_per_launch"]


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return max(n)
    except Exception:
        pass
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(var, "").isdigit():
            return int(os.environ[var])
    return os.cpu_count() or 1


def oracle_layer_step(cfg, x64, g32, w1_64, w2_64):
    from oracle import moe as omoe
    return omoe.fused_forward(x64, g32, w1_64, w2_64, cfg.topk, cfg.renormalize, cfg.num_expert_group,
                              cfg.topk_group, cfg.scoring, cfg.routed_scaling_factor)


def oracle_inputs(cfg, n_tokens):
    """float64 copies of the workload's first n_tokens tokens and all expert weights (generated on the host)."""
    import numpy as np
    import synth
    import torch
    acts = synth.moe_activations(synth.MoEConfig(**{**cfg.__dict__, "T": n_tokens}), "cpu")
    W = synth.moe_weights(cfg, "cuda" if torch.cuda.is_available() else "cpu")
    w1 = W["w1"].float().cpu().numpy().astype(np.float64)
    w2 = W["w2"].float().cpu().numpy().astype(np.float64)
    del W
    return acts["x"].float().numpy().astype(np.float64), acts["gating"].numpy(), w1, w2


# --------------------------------------------------------------------------- our arm
def run_ours(args, peaks, peaks_kind, rank, world, local_rank):
    import torch
    import mixture_experts_routing_grouped_gb300 as moe
    import synth

    from mixture_experts_routing_grouped_gb300 import build as _b
    _b.build()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    cfg = synth.prefill_config()
    acts = synth.moe_activations(cfg, dev)
    W = synth.moe_weights(cfg, dev)
    ws = torch.zeros(moe.moe_fused_forward_workspace_size(cfg.T, cfg.H, cfg.I, cfg.E, cfg.topk), dtype=torch.uint8,
                     device=dev)
    y = torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16, device=dev)
    tw = torch.empty((cfg.T, cfg.topk), dtype=torch.float32, device=dev)
    ids = torch.empty((cfg.T, cfg.topk), dtype=torch.int32, device=dev)
    flush = L2Flush(torch, dev)

    def step(x, g, yy, w_, i_):
        moe.moe_fused_forward(x, g, W["w1"], W["w2"], cfg.topk, cfg.renormalize, cfg.num_expert_group,
                              cfg.topk_group, cfg.scoring, cfg.routed_scaling_factor, ws=ws, y=yy, topk_weights=w_,
                              topk_ids=i_)

    n_stage = 6
    for _ in range(args.warmup):
        step(acts["x"], acts["gating"], y, tw, ids)
    torch.cuda.synchronize()

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(n_stage)] for _ in range(K)]
    s = torch.cuda.current_stream()
    for row in ev:                    # create the event handles before handing them to the library
        for e in row:
            e.record(s)
    torch.cuda.synchronize()
    clocks = ClockSampler(local_rank)
    clocks.start()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_begin = ClockSampler.now()
    # timed steps: one event before and one after each layer call (no instrumentation inside)
    step_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for k in range(K):
        flush(k)
        step_ev[k][0].record()
        step(acts["x"], acts["gating"], y, tw, ids)
        step_ev[k][1].record()
    torch.cuda.synchronize()
    t_end = ClockSampler.now()
    if world > 1:
        torch.distributed.barrier()
    step_ms = [a.elapsed_time(b) for a, b in step_ev]
    # A few timed steps last only milliseconds, less than the sampler's period allows
    # much of: the same steps (flush + layer) then run untimed for about 0.4 s more, and
    # their samples are reported beside the timed window's as `sustained`.
    t_sus0 = ClockSampler.now()
    n_sus = max(1, min(5000, int(400.0 / max(statistics.median(step_ms), 1e-3))))
    for k in range(n_sus):
        flush(k)
        step(acts["x"], acts["gating"], y, tw, ids)
    torch.cuda.synchronize()
    t_sus1 = ClockSampler.now()
    rows = clocks.stop()
    if rows is None:
        clk = {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
    else:
        clk = ClockSampler.summary(rows, t_begin, t_end)
        sus = ClockSampler.summary(rows, t_sus0, t_sus1)
        clk["sustained"] = dict(sus, steps=n_sus)
        clk["reasons"] = sorted(set(clk["reasons"]) | set(sus["reasons"]))
        if clk["sm_mhz"] is None:
            clk["sm_mhz"], clk["sm_max_mhz"] = sus["sm_mhz"], sus["sm_max_mhz"]
            clk["note"] = "no sample fell inside the timed steps; sm_mhz from the sustained window"
    # stage breakdown: a second pass with the library recording an event between its kernels
    for k in range(K):
        flush(k)
        moe.moe_set_stage_events(ev[k])
        step(acts["x"], acts["gating"], y, tw, ids)
        moe.moe_set_stage_events(None)
    torch.cuda.synchronize()
    stage_names = ["routing", "align", "gemm_gate_up", "gemm_down", "cast"]
    stage_ms = {n: statistics.mean(ev[k][i].elapsed_time(ev[k][i + 1]) for k in range(K))
                for i, n in enumerate(stage_names)}
    ms = max_over_ranks(torch, statistics.mean(step_ms), dev)
    err = moe.moe_check_device_error(ws)
    if err:
        raise RuntimeError(f"device error word {err:#x}")

    # ---- end to end through the C ABI with host buffers (pinned), copies inside the timed region
    xh = acts["x"].cpu().pin_memory()
    gh = acts["gating"].cpu().pin_memory()
    yh = torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16).pin_memory()
    twh = torch.empty((cfg.T, cfg.topk), dtype=torch.float32).pin_memory()
    idh = torch.empty((cfg.T, cfg.topk), dtype=torch.int32).pin_memory()
    xd, gd = torch.empty_like(acts["x"]), torch.empty_like(acts["gating"])
    e2e = []
    for k in range(args.warmup + K):
        flush(k)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        xd.copy_(xh, non_blocking=True)
        gd.copy_(gh, non_blocking=True)
        step(xd, gd, y, tw, ids)
        yh.copy_(y, non_blocking=True)
        twh.copy_(tw, non_blocking=True)
        idh.copy_(ids, non_blocking=True)
        b.record()
        b.synchronize()
        if k >= args.warmup:
            e2e.append(a.elapsed_time(b))
    e2e_serial_ms = max_over_ranks(torch, statistics.mean(e2e), dev)
    h2d = xh.numel() * 2 + gh.numel() * 4
    d2h = yh.numel() * 2 + twh.numel() * 4 + idh.numel() * 4

    # ---- the same, as a stream of steps: every step still copies its inputs from pinned host
    # memory and its outputs back, but steps rotate over E2E_STREAMS CUDA streams with their
    # own device buffers and workspaces, so that a step's copies (copy engines) overlap the
    # other steps' kernels (SMs). With two streams a stream's output copy and next input copy
    # (~90 + ~85 us) had to fit in one other step's kernels and held the steps back (396 us per
    # step against 325 us without copies); with four they fit (331 us). The window spans all K
    # steps (no L2 flush: a step's working set, the 1.2 GB of weights, is far larger than L2);
    # the figure is the serving throughput.
    streams = [torch.cuda.Stream(dev) for _ in range(E2E_STREAMS)]
    bufs = []
    for _ in range(E2E_STREAMS):
        bufs.append({"x": torch.empty_like(acts["x"]), "g": torch.empty_like(acts["gating"]),
                     "y": torch.empty_like(y), "tw": torch.empty_like(tw), "ids": torch.empty_like(ids),
                     "ws": torch.zeros_like(ws),
                     "yh": torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16).pin_memory(),
                     "twh": torch.empty((cfg.T, cfg.topk), dtype=torch.float32).pin_memory(),
                     "idh": torch.empty((cfg.T, cfg.topk), dtype=torch.int32).pin_memory()})

    def pipelined_step(i):
        bf = bufs[i % E2E_STREAMS]
        with torch.cuda.stream(streams[i % E2E_STREAMS]):
            bf["x"].copy_(xh, non_blocking=True)
            bf["g"].copy_(gh, non_blocking=True)
            moe.moe_fused_forward(bf["x"], bf["g"], W["w1"], W["w2"], cfg.topk, cfg.renormalize,
                                  cfg.num_expert_group, cfg.topk_group, cfg.scoring, cfg.routed_scaling_factor,
                                  ws=bf["ws"], y=bf["y"], topk_weights=bf["tw"], topk_ids=bf["ids"])
            bf["yh"].copy_(bf["y"], non_blocking=True)
            bf["twh"].copy_(bf["tw"], non_blocking=True)
            bf["idh"].copy_(bf["ids"], non_blocking=True)

    for i in range(E2E_STREAMS * args.warmup):
        pipelined_step(i)
    torch.cuda.synchronize()
    windows = []
    for rep in range(3):
        cur = torch.cuda.current_stream(dev)
        torch.cuda._sleep(4_000_000)  # the host enqueues ahead while the GPU sleeps (outside the window)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(cur)
        for st in streams:
            st.wait_stream(cur)
        for i in range(K):
            pipelined_step(i)
        for st in streams:
            cur.wait_stream(st)
        b.record(cur)
        b.synchronize()
        windows.append(a.elapsed_time(b) / K)
    e2e_ms = max_over_ranks(torch, statistics.median(windows), dev)
    for i in range(E2E_STREAMS):  # every stream's last step returned the layer's outputs
        assert torch.equal(bufs[i]["idh"], ids.cpu()), "pipelined steps returned other routing ids"

    # ---- roofline of the dominant kernel (gate_up grouped GEMM)
    pairs = cfg.T * cfg.topk
    flops_gate_up = 2.0 * pairs * cfg.H * (2 * cfg.I)
    flops_down = 2.0 * pairs * cfg.I * cfg.H
    t_gu = stage_ms["gemm_gate_up"] * 1e-3
    achieved = flops_gate_up / t_gu / 1e12
    peak = float(peaks["bf16_tflops"])
    layer_tflops = (flops_gate_up + flops_down) / (ms * 1e-3) / 1e12

    result = {
        "metric": METRIC,
        "value": round(job_tokens_per_s(cfg.T, world, ms), 1),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded counter-based normal inputs, random-init expert weights)",
        "config": {"workload": cfg.name, "T": cfg.T, "H": cfg.H, "I": cfg.I, "E": cfg.E, "topk": cfg.topk,
                   "routing": "softmax, renormalize, G=1", "l2": "between timed steps: 256 MiB write then 256 MiB read (L2 is 129 MB; the read leaves no dirty lines to write back inside a timed step)",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": {"kernel": "pair::moe_gate_up_kernel", "bound": "tensor", "achieved": round(achieved, 1),
                     "peak": peak, "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                     "peak_source": f"bf16_tflops (burst) of {peaks_kind}",
                     "traffic": kernel_traffic("pair::moe_gate_up_kernel")},
        "layer_tflops": round(layer_tflops, 1),
        "layer_frac_bf16_peak": round(layer_tflops / peak, 4),
        "stage_ms": {k: round(v, 4) for k, v in stage_ms.items()},
        "e2e": {"value": round(job_tokens_per_s(cfg.T, world, e2e_ms), 1), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4),
                "method": f"{K} steps through moe_fused_forward, each copying x and logits from pinned host "
                          "memory and y, weights and ids back, rotating over "
                          f"{E2E_STREAMS} streams with their own device buffers (a step's copies overlap the "
                          "other steps' kernels); one window over all steps, median of 3"},
        "e2e_serial": {"value": round(job_tokens_per_s(cfg.T, world, e2e_serial_ms), 1), "unit": "tokens/s",
                       "ms_per_step": round(e2e_serial_ms, 4),
                       "method": "one step at a time on one stream: copies in, layer, copies out, L2 flushed "
                                 "between steps, mean of the per-step windows"},
        # per step: routing (which also counts each row block's experts), align scan + scatter, gate_up, down, cast
        "gpu_launches": 5 * K,
        "clocks": clk,
    }
    if not args.skip_extra and world == 1:
        result["cublas_context"] = bench_cublas_context(torch, dev, flush, cfg, ids, args)
        result["fp8_layer"] = bench_fp8_layer(moe, torch, dev, flush, peaks, args, cfg, acts, W)
        result["decode"] = bench_decode(moe, synth, torch, dev, flush, peaks, args)
        result["routing"] = bench_routing(moe, synth, torch, dev, flush, peaks, args)
        result["gmm_lowp"] = bench_lowp(moe, synth, torch, dev, flush, peaks, args)
    del W
    return result, cfg


class L2Flush:
    """Untimed work between timed steps: write a 256 MiB buffer (more than the
    129 MB L2), then read another 256 MiB buffer so that the dirty lines of the
    write are written back now and not inside the timed step, then keep the GPU
    busy (~0.1 ms) while the host enqueues the start event and the timed launches,
    so that host-side call overhead (Python, ctypes, tensor-map encoding) never
    shows up inside a device-timed interval."""

    def __init__(self, torch, dev):
        self.torch = torch
        self.w = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        self.r = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        self.sink = torch.empty((), dtype=torch.float32, device=dev)
        self(0)  # the first reduction call sets up state that must not land in a timed step
        torch.cuda.synchronize()

    def __call__(self, k):
        self.w.fill_(float(k))
        self.torch.sum(self.r, dim=0, out=self.sink)
        self.torch.cuda._sleep(200_000)


def bench_decode(moe, synth, torch, dev, flush, peaks, args):
    """Decode layer at T in {1, 8, 32, 128}: weight-stream GB/s = bytes of the active experts / step time."""
    import numpy as np
    out = {}
    cfg0 = synth.decode_config(1)
    W = synth.moe_weights(cfg0, dev)
    for T in (1, 8, 32, 128):
        cfg = synth.decode_config(T)
        acts = synth.moe_activations(cfg, dev)
        ws = torch.zeros(moe.moe_fused_forward_workspace_size(T, cfg.H, cfg.I, cfg.E, cfg.topk),
                         dtype=torch.uint8, device=dev)
        run = lambda: moe.moe_fused_forward(acts["x"], acts["gating"], W["w1"], W["w2"], cfg.topk, cfg.renormalize,
                                            cfg.num_expert_group, cfg.topk_group, cfg.scoring,
                                            cfg.routed_scaling_factor, ws=ws)
        for _ in range(3):
            _, _, ids = run()
        torch.cuda.synchronize()
        n_active = int(np.unique(ids.cpu().numpy()).size)
        times = []
        for k in range(max(5, args.steps)):
            flush(k)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            run()
            b.record()
            b.synchronize()
            times.append(a.elapsed_time(b))
        ms = statistics.median(times)
        wbytes = n_active * 3 * cfg.I * cfg.H * 2
        gbs = wbytes / (ms * 1e-3) / 1e9
        out[f"T{T}"] = {"ms": round(ms, 4), "active_experts": n_active, "weight_bytes": wbytes,
                        "GB/s": round(gbs, 1), "frac_hbm": round(gbs / float(peaks["hbm_gbs"]), 4),
                        "tokens/s": round(T / (ms * 1e-3), 1)}
    # the same layers with FP8-e4m3 weights (per-channel scales, made on the device by torch's e4m3
    # cast) through moe_fused_forward_fp8: one byte per weight streamed
    q1, s1 = device_e4m3_weights(torch, W["w1"])
    q2, s2 = device_e4m3_weights(torch, W["w2"])
    del W
    torch.cuda.empty_cache()
    fp8 = {}
    for T in (1, 8, 32, 128):
        cfg = synth.decode_config(T)
        acts = synth.moe_activations(cfg, dev)
        ws = torch.zeros(moe.moe_fused_forward_fp8_workspace_size(T, cfg.H, cfg.I, cfg.E, cfg.topk),
                         dtype=torch.uint8, device=dev)
        run = lambda: moe.moe_fused_forward_fp8(acts["x"], acts["gating"], q1, s1, q2, s2, cfg.topk,
                                                cfg.renormalize, cfg.num_expert_group, cfg.topk_group, cfg.scoring,
                                                cfg.routed_scaling_factor, ws=ws)
        for _ in range(3):
            _, _, ids = run()
        torch.cuda.synchronize()
        n_active = int(np.unique(ids.cpu().numpy()).size)
        times = []
        for k in range(max(5, args.steps)):
            flush(k)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            run()
            b.record()
            b.synchronize()
            times.append(a.elapsed_time(b))
        ms = statistics.median(times)
        wbytes = n_active * 3 * cfg.I * cfg.H
        gbs = wbytes / (ms * 1e-3) / 1e9
        fp8[f"T{T}"] = {"ms": round(ms, 4), "active_experts": n_active, "weight_bytes": wbytes,
                        "GB/s": round(gbs, 1), "frac_hbm": round(gbs / float(peaks["hbm_gbs"]), 4),
                        "tokens/s": round(T / (ms * 1e-3), 1)}
    out["fp8_e4m3"] = fp8
    del q1, q2, s1, s2
    torch.cuda.empty_cache()
    return out


def fp32_score_collisions(logits, scoring: str, depth: int) -> int:
    """Rows of `logits` [T, E] in which two distinct logits among the row's `depth` largest
    have equal float32 scores: the rows where ranking on rounded scores, instead of on the
    logits as the kernels and the oracle do, could reorder the selection. Information only."""
    import numpy as np
    x = np.asarray(logits, dtype=np.float32)
    order = np.argsort(-x, axis=1, kind="stable")[:, :depth]
    xs = np.take_along_axis(x, order, axis=1)
    one = np.float32(1.0)
    if scoring == "sigmoid":
        sc = (one / (one + np.exp(-xs))).astype(np.float32)
    else:
        m = x.max(axis=1, keepdims=True)
        den = np.exp(x - m).sum(axis=1, keepdims=True, dtype=np.float32)
        sc = (np.exp(xs - m) / den).astype(np.float32)
    tie = (sc[:, 1:] == sc[:, :-1]) & (xs[:, 1:] != xs[:, :-1])
    return int(tie.any(axis=1).sum())


def bench_routing(moe, synth, torch, dev, flush, peaks, args):
    out = {}
    for scoring in ("softmax", "sigmoid"):
        cfg = synth.routing_config(16384, scoring)
        g = synth.gating_logits(cfg, dev).cpu().numpy()
        out[f"fp32_score_ties_T16384_{scoring}"] = {
            "rows": fp32_score_collisions(g, scoring, 2 * cfg.topk), "of": 16384,
            "note": "rows whose 16 largest logits include two distinct ones with equal float32 scores "
                    "(selection ranks on logits; information only)"}
    for T in (16384, 65536):
        cfg = synth.routing_config(T, "sigmoid")
        g0 = synth.gating_logits(cfg, dev)
        nbytes = T * cfg.E * 4 + T * cfg.topk * 8
        # R copies of the logits (and outputs) holding >= 512 MiB together: calls launched back to
        # back in rotation never find their inputs in L2 (129 MB), and the launch and event
        # overheads of one call are spread over many
        R = max(4, -(-(512 << 20) // (T * cfg.E * 4)))
        gs = [g0.clone() for _ in range(R)]
        ws_ = [torch.empty((T, cfg.topk), dtype=torch.float32, device=dev) for _ in range(R)]
        is_ = [torch.empty((T, cfg.topk), dtype=torch.int32, device=dev) for _ in range(R)]
        sink = torch.zeros((), dtype=torch.float32, device=dev)

        def call(j):
            moe.moe_grouped_topk(gs[j % R], cfg.topk, True, cfg.num_expert_group, cfg.topk_group, cfg.scoring,
                                 cfg.routed_scaling_factor, ws_[j % R], is_[j % R])

        def probe(j):
            moe.moe_read_probe(gs[j % R], sink)

        def per_call_us(fn, n):
            times = []
            for rep in range(3):
                flush(rep)
                torch.cuda._sleep(6_000_000)  # the host enqueues all n calls while the GPU sleeps (~3 ms)
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                for j in range(n):
                    fn(j)
                b.record()
                b.synchronize()
                times.append(a.elapsed_time(b) * 1e3 / n)
            return statistics.median(times)

        for j in range(R):
            call(j)
        torch.cuda.synchronize()
        n = 2 * R
        us = per_call_us(call, n)
        floor_us = per_call_us(probe, n)
        gbs = nbytes / (us * 1e-6) / 1e9
        # a single call after an L2 flush, for context (includes the launch and event overheads)
        single = []
        for k in range(max(10, args.steps)):
            flush(k)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            call(0)
            b.record()
            b.synchronize()
            single.append(a.elapsed_time(b))
        out[f"T{T}"] = {"us": round(us, 2), "bytes": nbytes, "GB/s": round(gbs, 1),
                        "frac_hbm": round(gbs / float(peaks["hbm_gbs"]), 4),
                        "timing": f"{n} calls back to back over {R} copies of the inputs ({R * T * cfg.E * 4 >> 20} "
                                  "MiB, > L2), per-call mean of the event window, median of 3",
                        "read_floor_us": round(floor_us, 2),
                        "read_floor_GB/s": round(T * cfg.E * 4 / (floor_us * 1e-6) / 1e9, 1),
                        "read_floor_note": "moe_read_probe: one streaming read of the same logits bytes, timed the "
                                           "same way",
                        "single_call_after_flush_us": round(statistics.median(single) * 1e3, 2)}
        del gs, ws_, is_
        torch.cuda.empty_cache()
    return out


def bench_fp8_layer(moe, torch, dev, flush, peaks, args, cfg, acts, W):
    """The prefill layer with FP8-e4m3 weights (per-channel scales, quantised once by the library)
    and per-token quantised activations: moe_fused_forward_fp8, device-timed like the bf16 layer."""
    E, I, H = cfg.E, cfg.I, cfg.H
    q1, s1 = moe.moe_quant_per_token(W["w1"].view(E * 2 * I, H), torch.float8_e4m3fn)
    q2, s2 = moe.moe_quant_per_token(W["w2"].view(E * H, I), torch.float8_e4m3fn)
    q1, s1, q2, s2 = q1.view(E, 2 * I, H), s1.view(E, 2 * I), q2.view(E, H, I), s2.view(E, H)
    ws = torch.zeros(moe.moe_fused_forward_fp8_workspace_size(cfg.T, H, I, E, cfg.topk), dtype=torch.uint8,
                     device=dev)
    y = torch.empty((cfg.T, H), dtype=torch.bfloat16, device=dev)
    tw = torch.empty((cfg.T, cfg.topk), dtype=torch.float32, device=dev)
    ids = torch.empty((cfg.T, cfg.topk), dtype=torch.int32, device=dev)
    run = lambda: moe.moe_fused_forward_fp8(acts["x"], acts["gating"], q1, s1, q2, s2, cfg.topk, cfg.renormalize,
                                            cfg.num_expert_group, cfg.topk_group, cfg.scoring,
                                            cfg.routed_scaling_factor, ws=ws, y=y, topk_weights=tw, topk_ids=ids)
    for _ in range(args.warmup):
        run()
    K = max(10, args.steps)
    times = []
    for k in range(K):
        flush(k)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        run()
        b.record()
        b.synchronize()
        times.append(a.elapsed_time(b))
    n_ev = 8
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(n_ev)] for _ in range(K)]
    for row in ev:
        for e in row:
            e.record()
    torch.cuda.synchronize()
    for k in range(K):
        flush(k)
        moe.moe_set_stage_events(ev[k])
        run()
        moe.moe_set_stage_events(None)
    torch.cuda.synchronize()
    names = ["routing", "align", "quant_x", "gemm_gate_up", "quant_h", "gemm_down", "cast"]
    stage = {n: statistics.median(ev[k][i].elapsed_time(ev[k][i + 1]) for k in range(K)) for i, n in enumerate(names)}
    if moe.moe_check_device_error(ws):
        raise RuntimeError("moe_fused_forward_fp8 reported a device error")
    ms = statistics.median(times)
    pairs = cfg.T * cfg.topk
    f_gu, f_dn = 2.0 * pairs * H * 2 * I, 2.0 * pairs * I * H
    peak8 = 2.0 * float(peaks["bf16_tflops"])
    gu_tf = f_gu / (stage["gemm_gate_up"] * 1e-3) / 1e12
    dn_tf = f_dn / (stage["gemm_down"] * 1e-3) / 1e12
    return {"workload": cfg.name + "_fp8_e4m3", "ms_per_step": round(ms, 4),
            "tokens/s": round(cfg.T / (ms * 1e-3), 1),
            "layer_TFLOP/s": round((f_gu + f_dn) / (ms * 1e-3) / 1e12, 1),
            "stage_ms": {k: round(v, 4) for k, v in stage.items()},
            "gate_up_TFLOP/s": round(gu_tf, 1), "down_TFLOP/s": round(dn_tf, 1),
            "fp8_peak_TFLOP/s": peak8, "gate_up_frac_fp8_peak": round(gu_tf / peak8, 4),
            "peak_source": "2 x bf16_tflops (burst) of measured: the nominal fp8 / bf16 dense ratio",
            "traffic_bytes_per_launch": {"gemm_gate_up": kernel_traffic("pair::moe_gate_up_kernel<1>"),
                                         "gemm_down": kernel_traffic("moe_down_kernel<1>")},
            "gpu_launches_per_step": 7}  # routing, align, quant x (side stream), gate_up, quant h, down, cast


def bench_cublas_context(torch, dev, flush, cfg, ids, args):
    """Context for the grouped GEMMs: cuBLAS batched GEMMs (torch.bmm) on the same per-expert shapes,
    without the row gather, the SwiGLU and the weighted combine, with every expert holding the same
    number of rows: T*k/E (the routed rows) and the padded row count the grouped kernels execute."""
    import numpy as np
    counts = np.bincount(ids.reshape(-1).cpu().numpy(), minlength=cfg.E)
    padded = int(((counts + 127) // 128 * 128).sum())
    out = {}
    for rows, tag in ((cfg.T * cfg.topk // cfg.E, "routed"), (padded // cfg.E, "padded")):
        for name, (kk, nn) in (("gate_up", (cfg.H, 2 * cfg.I)), ("down", (cfg.I, cfg.H))):
            a = torch.randn(cfg.E, rows, kk, device=dev, dtype=torch.bfloat16)
            b = torch.randn(cfg.E, kk, nn, device=dev, dtype=torch.bfloat16)
            c = torch.empty(cfg.E, rows, nn, device=dev, dtype=torch.bfloat16)
            for _ in range(3):
                torch.bmm(a, b, out=c)
            ts = []
            for k in range(max(10, args.steps)):
                flush(k)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                torch.bmm(a, b, out=c)
                e1.record()
                e1.synchronize()
                ts.append(e0.elapsed_time(e1))
            us = statistics.median(ts) * 1e3
            useful = 2.0 * cfg.T * cfg.topk * kk * nn
            out[f"{name}_{tag}"] = {"shape": f"bmm [{cfg.E}, {rows}, {kk}] x [{cfg.E}, {kk}, {nn}]", "us": round(us, 1),
                                    "routed_TFLOP/s": round(useful / (us * 1e-6) / 1e12, 1)}
            del a, b, c
    torch.cuda.empty_cache()
    return out


def bench_lowp(moe, synth, torch, dev, flush, peaks, args):
    """Low-precision grouped GEMM, M=2048, K=N=4096, E=32 Zipf groups, bf16 out, INT8 and FP8-e4m3;
    and the small-K case K=768, N=3072 under "small_k"."""
    out = bench_lowp_cfg(moe, synth, torch, dev, flush, peaks, args, synth.lowp_config())
    out["small_k"] = bench_lowp_cfg(moe, synth, torch, dev, flush, peaks, args, synth.lowp_small_k_config())
    return out


def bench_lowp_cfg(moe, synth, torch, dev, flush, peaks, args, cfg):
    d = synth.gmm_inputs(cfg, dev)
    out = {"workload": cfg.name}
    sizes = d["expert_sizes"].cpu().tolist()
    n_active = sum(1 for s_ in sizes if s_ > 0)
    flops = 2.0 * cfg.M * cfg.N * cfg.K
    for name, qdt in (("int8", torch.int8), ("e4m3", torch.float8_e4m3fn)):
        qx, sx = moe.moe_quant_per_token(d["x"], qdt)
        qw, sw = moe.moe_quant_per_token(d["w"].view(cfg.E * cfg.N, cfg.K), qdt)
        qw = qw.view(cfg.E, cfg.N, cfg.K)
        sw = sw.view(cfg.E, cfg.N)
        y = torch.empty((cfg.M, cfg.N), dtype=torch.bfloat16, device=dev)
        ws = torch.zeros(moe.gmm_lowp_workspace_size(cfg.M, cfg.K, cfg.N, cfg.E), dtype=torch.uint8, device=dev)
        run = lambda: moe.gmm_lowp(qx, qw, sx, sw, d["expert_offsets"], d["expert_sizes"], torch.bfloat16, y, ws)
        for _ in range(3):
            run()
        times = []
        for k in range(max(10, args.steps)):
            flush(k)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            run()
            b.record()
            b.synchronize()
            times.append(a.elapsed_time(b))
        if moe.moe_check_device_error(ws):
            raise RuntimeError("gmm_lowp reported a device error")
        ms = statistics.median(times)
        nbytes = n_active * cfg.N * cfg.K + cfg.M * cfg.K + cfg.M * cfg.N * 2 + cfg.M * 4 + cfg.E * cfg.N * 4
        gbs = nbytes / (ms * 1e-3) / 1e9
        tf = flops / (ms * 1e-3) / 1e12
        out[name] = {"us": round(ms * 1e3, 2), "TFLOP/s": round(tf, 1),
                     "frac_bf16_peak": round(tf / float(peaks["bf16_tflops"]), 4), "GB/s": round(gbs, 1),
                     "frac_hbm": round(gbs / float(peaks["hbm_gbs"]), 4), "bytes": nbytes}
    del d
    torch.cuda.empty_cache()
    return out


# --------------------------------------------------------------------------- CPU baseline / reference arm
def cpu_baseline(cfg, budget_s: float = 12.0):
    """Times the oracle on the first n tokens of the workload, doubling n until a run takes ~budget_s/4."""
    n, last = 128, None
    x64, g32, w1, w2 = oracle_inputs(cfg, cfg.T)
    while True:
        t0 = time.perf_counter()
        oracle_layer_step(cfg, x64[:n], g32[:n], w1, w2)
        dt = time.perf_counter() - t0
        last = (n, dt)
        if dt > budget_s / 4 or n >= cfg.T:
            break
        n = min(cfg.T, n * 2)
    n, dt = last
    return {"value": round(n / dt, 2), "unit": "tokens/s", "cores": blas_threads(), "kind": "oracle",
            "sample": f"first {n} of {cfg.T} tokens of {cfg.name} (all {cfg.E} experts' weights), float64 numpy, "
                      f"one run of {dt:.2f} s"}


def run_reference(args, rank, world, cfg=None, n: int = 256):
    """The reference arm: the oracle on the first n tokens of the workload per step."""
    import synth
    cfg = cfg or synth.prefill_config()
    n = min(n, cfg.T)
    x64, g32, w1, w2 = oracle_inputs(cfg, n)
    for _ in range(args.warmup):
        oracle_layer_step(cfg, x64, g32, w1, w2)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle_layer_step(cfg, x64, g32, w1, w2)
        times.append(time.perf_counter() - t0)
    ms = statistics.mean(times) * 1e3
    val = round(n / (ms * 1e-3), 2)
    return {
        "impl": "reference", "metric": METRIC, "value": val, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (same seeded inputs as the GPU arm)",
        "config": {"workload": cfg.name, "T": cfg.T, "H": cfg.H, "I": cfg.I, "E": cfg.E, "topk": cfg.topk,
                   "sample_tokens_per_step": n},
        "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": blas_threads(), "kind": "oracle",
                         "sample": f"first {n} of {cfg.T} tokens per step, float64 numpy oracle"},
        "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def device_e4m3_weights(torch, w, chunk=16):
    """Per-output-channel e4m3 codes of bf16 weights [E, R, K] made on the device: torch's float8_e4m3fn
    cast (nearest, ties to even) of w / (absmax / 448) in fp32, a few experts at a time."""
    E_, R_, K_ = w.shape
    q = torch.empty((E_, R_, K_), dtype=torch.uint8, device=w.device)
    sc = torch.empty((E_, R_), dtype=torch.float32, device=w.device)
    for e0 in range(0, E_, chunk):
        w32 = w[e0:e0 + chunk].float()
        amax = w32.abs().amax(dim=2)
        s_ = amax / torch.full_like(amax, 448.0)
        s_ = torch.where(s_ == 0, torch.ones_like(s_), s_)
        q[e0:e0 + chunk] = (w32 / s_[:, :, None]).to(torch.float8_e4m3fn).view(torch.uint8)
        sc[e0:e0 + chunk] = s_
        del w32
    return q, sc


def profile_case(name: str) -> None:
    """Small, fixed workloads for ncu captures (each runs a few calls and exits; the profile
    summaries under profiles/ name the case and the ncu command).

    decode_small  decode-shaped layer with 32 experts (H=7168, I=2048, T=32, top-8 grouped
                  sigmoid; 2.8 GB of bf16 weights, more than L2), bf16 then FP8, twice each
    lowp          gmm_lowp on the C5 and small-K workloads, INT8 then e4m3
    route         grouped top-k at T=65536 (E=256, G=8/4, top-8) and of the prefill layer
    layers        prefill layer (bf16, then FP8) 3 calls each; decode T=32 (E=256) bf16 and FP8
    """
    import torch
    import mixture_experts_routing_grouped_gb300 as moe
    import synth
    from mixture_experts_routing_grouped_gb300 import build as _b
    _b.build()
    dev = "cuda"
    if name == "decode_small":
        cfg = synth.MoEConfig("decode_T32_H7168_I2048_E32_top8", T=32, H=7168, I=2048, E=32, topk=8,
                              num_expert_group=8, topk_group=4, scoring="sigmoid", routed_scaling_factor=2.5,
                              logit_sigma=2.0, seed=41)
        acts, W = synth.moe_activations(cfg, dev), synth.moe_weights(cfg, dev)
        q1, s1 = device_e4m3_weights(torch, W["w1"])
        q2, s2 = device_e4m3_weights(torch, W["w2"])
        for _ in range(2):
            moe.moe_fused_forward(acts["x"], acts["gating"], W["w1"], W["w2"], 8, True, 8, 4, "sigmoid", 2.5)
            moe.moe_fused_forward_fp8(acts["x"], acts["gating"], q1, s1, q2, s2, 8, True, 8, 4, "sigmoid", 2.5)
    elif name == "lowp":
        for cfg in (synth.lowp_config(), synth.lowp_small_k_config()):
            d = synth.gmm_inputs(cfg, dev)
            for qdt in (torch.int8, torch.float8_e4m3fn):
                qx, sx = moe.moe_quant_per_token(d["x"], qdt)
                qw, sw = moe.moe_quant_per_token(d["w"].view(cfg.E * cfg.N, cfg.K), qdt)
                moe.gmm_lowp(qx, qw.view(cfg.E, cfg.N, cfg.K), sx, sw.view(cfg.E, cfg.N), d["expert_offsets"],
                             d["expert_sizes"])
    elif name == "route":
        cfg = synth.routing_config(65536, "sigmoid")
        moe.moe_grouped_topk(synth.gating_logits(cfg, dev), 8, True, 8, 4, "sigmoid", 2.5)
        cfg = synth.prefill_config()
        moe.moe_grouped_topk(synth.gating_logits(cfg, dev), 8, True, 1, 1, "softmax", 1.0)
    elif name == "layers":
        cfg = synth.prefill_config()
        acts, W = synth.moe_activations(cfg, dev), synth.moe_weights(cfg, dev)
        q1, s1 = device_e4m3_weights(torch, W["w1"])
        q2, s2 = device_e4m3_weights(torch, W["w2"])
        for _ in range(3):
            moe.moe_fused_forward(acts["x"], acts["gating"], W["w1"], W["w2"], 8, True)
        for _ in range(3):
            moe.moe_fused_forward_fp8(acts["x"], acts["gating"], q1, s1, q2, s2, 8, True)
        del W, q1, q2
        torch.cuda.empty_cache()
        cfg = synth.decode_config(32)
        acts, W = synth.moe_activations(cfg, dev), synth.moe_weights(cfg, dev)
        for _ in range(2):
            moe.moe_fused_forward(acts["x"], acts["gating"], W["w1"], W["w2"], 8, True, 8, 4, "sigmoid", 2.5)
        q1, s1 = device_e4m3_weights(torch, W["w1"])
        q2, s2 = device_e4m3_weights(torch, W["w2"])
        del W
        torch.cuda.empty_cache()
        for _ in range(2):
            moe.moe_fused_forward_fp8(acts["x"], acts["gating"], q1, s1, q2, s2, 8, True, 8, 4, "sigmoid", 2.5)
    else:
        raise ValueError(f"unknown profile case {name!r}")
    torch.cuda.synchronize()
    print(f"profile case {name}: ok", flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--skip-extra", action="store_true", help="skip the decode and routing sub-benchmarks")
    ap.add_argument("--skip-cpu-baseline", action="store_true")
    ap.add_argument("--only", choices=["routing", "decode", "lowp", "fp8"],
                    help="run just one sub-benchmark on one GPU and print its JSON (profiling cases)")
    ap.add_argument("--profile-case", choices=["decode_small", "lowp", "route", "layers"],
                    help="run one small fixed workload for an ncu capture and exit (no timing)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    rank, world, local_rank = dist_env()
    if args.profile_case:
        profile_case(args.profile_case)
        return

    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(run_reference(args, rank, world)), flush=True)
        return

    if args.only:
        import torch
        import mixture_experts_routing_grouped_gb300 as moe
        import synth
        from mixture_experts_routing_grouped_gb300 import build as _b
        _b.build()
        peaks, _ = load_peaks()
        dev = torch.device("cuda", local_rank)
        flush = L2Flush(torch, dev)
        if args.only == "fp8":
            cfg = synth.prefill_config()
            res = bench_fp8_layer(moe, torch, dev, flush, peaks, args, cfg, synth.moe_activations(cfg, dev),
                                  synth.moe_weights(cfg, dev))
        else:
            fn = {"routing": bench_routing, "decode": bench_decode, "lowp": bench_lowp}[args.only]
            res = fn(moe, synth, torch, dev, flush, peaks, args)
        print(json.dumps({args.only: res}), flush=True)
        return

    if world > 1:
        import torch
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    peaks, kind = load_peaks()
    result, cfg = run_ours(args, peaks, kind, rank, world, local_rank)
    if rank == 0:
        if not args.skip_cpu_baseline:
            result["cpu_baseline"] = cpu_baseline(cfg)
        print(json.dumps(result), flush=True)
    if world > 1:
        import torch
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
