"""Seeded synthetic inputs for the fused MoE layer, shared by tests, bench and smoke.

This module holds no arithmetic of the MoE method (no routing, sorting, GEMM or
combine). It provides:

* a counter-based random generator (two rounds of the MurmurHash3 ``fmix32``
  finalizer, Austin Appleby, public domain) written with torch integer ops that
  give the same bits on CPU and GPU, so any slice of any tensor can be
  regenerated on the host without copying it back from the device;
* a normal variate built from that generator by piecewise-linear interpolation
  of the standard normal inverse CDF tabulated at 65537 points (tails reach
  about +-4.3 sigma); every float op is a separate IEEE-rounded torch op, so
  CPU and GPU produce identical bytes;
* the workload recipes (shapes, distributions, seeds) of the five workloads:
  tiny layer, routing only, prefill layer, decode layer, low-precision GMM.

Random numbers are drawn per (seed, tensor tag, flat element index).
"""
from __future__ import annotations

import functools
import math
import statistics
from dataclasses import dataclass, field

import torch

_M32 = 0xFFFFFFFF
_CHUNK = 1 << 26


def _fmix32_int(h: int) -> int:
    h &= _M32
    h ^= h >> 16
    h = (h * 0x85EBCA6B) & _M32
    h ^= h >> 13
    h = (h * 0xC2B2AE35) & _M32
    h ^= h >> 16
    return h


def _mul32(h: torch.Tensor, c: int) -> torch.Tensor:
    # (h * c) mod 2^32 for 0 <= h < 2^32 without overflowing int64.
    lo, hi = c & 0xFFFF, c >> 16
    return (h * lo + (((h * hi) & 0xFFFF) << 16)) & _M32


def _fmix32(h: torch.Tensor) -> torch.Tensor:
    h = h ^ (h >> 16)
    h = _mul32(h, 0x85EBCA6B)
    h = h ^ (h >> 13)
    h = _mul32(h, 0xC2B2AE35)
    h = h ^ (h >> 16)
    return h


def stream_key(seed: int, tag: int) -> tuple[int, int]:
    """Two 32-bit keys for the stream of tensor ``tag`` under ``seed``."""
    k0 = _fmix32_int((seed * 0x9E3779B1 + tag * 0x7FEB352D + 0x68E31DA4) & _M32)
    k1 = _fmix32_int(((seed >> 32) ^ (tag * 0x846CA68B) ^ 0x1B873593) & _M32)
    return k0, k1


def uniform_u32(key: tuple[int, int], start: int, n: int, device) -> torch.Tensor:
    """int64 tensor of n uniform 32-bit values for flat indices [start, start+n)."""
    i = torch.arange(start, start + n, dtype=torch.int64, device=device)
    h = _fmix32((i & _M32) ^ key[0])
    return _fmix32(h ^ (i >> 32) ^ key[1])


@functools.lru_cache(maxsize=None)
def _normal_table_cpu() -> torch.Tensor:
    nd = statistics.NormalDist()
    n = 65537
    vals = [nd.inv_cdf((j + 0.5) / n) for j in range(n)]
    return torch.tensor(vals, dtype=torch.float64).to(torch.float32)


_table_cache: dict = {}


def _normal_table(device) -> torch.Tensor:
    dev = torch.device(device)
    key = str(dev)
    if key not in _table_cache:
        _table_cache[key] = _normal_table_cpu().to(dev)
    return _table_cache[key]


def normal_f32(key, start: int, n: int, sigma: float, device) -> torch.Tensor:
    """n float32 samples of N(0, sigma^2) for flat indices [start, start+n)."""
    u = uniform_u32(key, start, n, device)
    tab = _normal_table(device)
    idx = u >> 16
    frac = (u & 0xFFFF).to(torch.float32) * (1.0 / 65536.0)
    z0 = tab[idx]
    z1 = tab[idx + 1]
    v = torch.add(z0, torch.mul(frac, torch.sub(z1, z0)))
    return torch.mul(v, torch.tensor(sigma, dtype=torch.float32, device=device))


def fill_normal_(out: torch.Tensor, seed: int, tag: int, sigma: float, start: int = 0) -> torch.Tensor:
    """Fill a contiguous tensor (any float dtype) with N(0, sigma^2), chunked.

    Element j of ``out`` receives the sample at flat index ``start + j`` of the
    (seed, tag) stream, rounded to ``out.dtype`` (round-to-nearest-even).
    """
    flat = out.view(-1)
    key = stream_key(seed, tag)
    n = flat.numel()
    for s in range(0, n, _CHUNK):
        m = min(_CHUNK, n - s)
        flat[s:s + m] = normal_f32(key, start + s, m, sigma, out.device).to(out.dtype)
    return out


def normal(shape, seed: int, tag: int, sigma: float, dtype, device, start: int = 0) -> torch.Tensor:
    out = torch.empty(shape, dtype=dtype, device=device)
    return fill_normal_(out, seed, tag, sigma, start)


# ---------------------------------------------------------------------------
# Workload recipes
# ---------------------------------------------------------------------------
SEED_BASE = 0xC0FFEE

TAG_X, TAG_GATING, TAG_W1, TAG_W2, TAG_WG, TAG_LOWP_X, TAG_LOWP_W, TAG_PERM = 1, 2, 3, 4, 5, 6, 7, 8


@dataclass(frozen=True)
class MoEConfig:
    """One MoE layer workload: shapes, routing parameters and input distributions."""
    name: str
    T: int
    H: int
    I: int
    E: int
    topk: int
    num_expert_group: int = 1
    topk_group: int = 1
    scoring: str = "softmax"          # "softmax" | "sigmoid"
    renormalize: bool = True
    routed_scaling_factor: float = 1.0
    x_sigma: float = 1.0
    w_sigma: float = 0.02
    logit_sigma: float = 1.0          # used when router_sigma is None
    router_sigma: float | None = None # tiny layer: logits = x @ W_g^T, W_g ~ N(0, router_sigma^2)
    seed: int = SEED_BASE

    @property
    def num_pairs(self) -> int:
        return self.T * self.topk


def tiny_config() -> MoEConfig:
    return MoEConfig("tiny_T64_H512_I256_E8_top2", T=64, H=512, I=256, E=8, topk=2,
                     router_sigma=0.05, seed=SEED_BASE + 0)


def routing_config(T: int, scoring: str) -> MoEConfig:
    return MoEConfig(f"routing_T{T}_E256_G8_tg4_top8_{scoring}", T=T, H=7168, I=0, E=256, topk=8,
                     num_expert_group=8, topk_group=4, scoring=scoring, renormalize=True,
                     routed_scaling_factor=2.5, logit_sigma=2.0, seed=SEED_BASE + 1)


def prefill_config(T: int = 4096) -> MoEConfig:
    return MoEConfig(f"prefill_T{T}_H2048_I768_E128_top8", T=T, H=2048, I=768, E=128, topk=8,
                     scoring="softmax", renormalize=True, logit_sigma=1.0, seed=SEED_BASE + 2)


def decode_config(T: int) -> MoEConfig:
    return MoEConfig(f"decode_T{T}_H7168_I2048_E256_top8", T=T, H=7168, I=2048, E=256, topk=8,
                     num_expert_group=8, topk_group=4, scoring="sigmoid", renormalize=True,
                     routed_scaling_factor=2.5, logit_sigma=2.0, seed=SEED_BASE + 3)


def gating_logits(cfg: MoEConfig, device, x: torch.Tensor | None = None) -> torch.Tensor:
    """Router logits [T, E] fp32.

    For the tiny layer the logits are the router projection float(x) @ W_g^T,
    evaluated once on the host in float64 and rounded to fp32 (the router is
    upstream of the routed layer; both sides receive the same logits). The
    other workloads draw the logits directly.
    """
    if cfg.router_sigma is None:
        return normal((cfg.T, cfg.E), cfg.seed, TAG_GATING, cfg.logit_sigma, torch.float32, device)
    if x is None:
        x = normal((cfg.T, cfg.H), cfg.seed, TAG_X, cfg.x_sigma, torch.bfloat16, "cpu")
    wg = normal((cfg.E, cfg.H), cfg.seed, TAG_WG, cfg.router_sigma, torch.float32, "cpu")
    logits = (x.to("cpu", torch.float64) @ wg.to(torch.float64).T).to(torch.float32)
    return logits.to(device)


def moe_activations(cfg: MoEConfig, device) -> dict:
    x = normal((cfg.T, cfg.H), cfg.seed, TAG_X, cfg.x_sigma, torch.bfloat16, device)
    gating = gating_logits(cfg, device, x)
    return {"x": x, "gating": gating}


def moe_weights(cfg: MoEConfig, device) -> dict:
    w1 = normal((cfg.E, 2 * cfg.I, cfg.H), cfg.seed, TAG_W1, cfg.w_sigma, torch.bfloat16, device)
    w2 = normal((cfg.E, cfg.H, cfg.I), cfg.seed, TAG_W2, cfg.w_sigma, torch.bfloat16, device)
    return {"w1": w1, "w2": w2}


def expert_weights(cfg: MoEConfig, e: int, device) -> tuple[torch.Tensor, torch.Tensor]:
    """W1[e] [2I, H] and W2[e] [H, I] alone, identical to the slices of moe_weights."""
    n1 = 2 * cfg.I * cfg.H
    n2 = cfg.H * cfg.I
    w1 = normal((2 * cfg.I, cfg.H), cfg.seed, TAG_W1, cfg.w_sigma, torch.bfloat16, device, start=e * n1)
    w2 = normal((cfg.H, cfg.I), cfg.seed, TAG_W2, cfg.w_sigma, torch.bfloat16, device, start=e * n2)
    return w1, w2


# ---------------------------------------------------------------------------
# Low-precision grouped GEMM workload
# ---------------------------------------------------------------------------
@dataclass(frozen=True)
class GmmConfig:
    name: str
    M: int
    K: int
    N: int
    E: int
    zipf_s: float = 1.2
    x_sigma: float = 1.0
    w_sigma: float = 0.02
    seed: int = SEED_BASE + 4


def lowp_config() -> GmmConfig:
    return GmmConfig("gmm_lowp_M2048_K4096_N4096_E32_zipf1.2", M=2048, K=4096, N=4096, E=32)


def lowp_small_k_config() -> GmmConfig:
    """The low-precision GMM article's small-K case (section 4.2: K=768, N=3072), 32 Zipf groups."""
    return GmmConfig("gmm_lowp_M2048_K768_N3072_E32_zipf1.2", M=2048, K=768, N=3072, E=32)


def _perm(n: int, seed: int, tag: int) -> list[int]:
    """Fisher-Yates permutation of range(n) driven by the counter generator."""
    u = uniform_u32(stream_key(seed, tag), 0, n, "cpu").tolist()
    p = list(range(n))
    for i in range(n - 1, 0, -1):
        j = u[i] % (i + 1)
        p[i], p[j] = p[j], p[i]
    return p


def zipf_group_sizes(M: int, E: int, s: float, seed: int) -> list[int]:
    """Deterministic Zipf(s) group sizes over E experts summing to M.

    Rank r (1-based) gets floor(M * r^-s / sum_q q^-s) rows; the two lowest
    ranks are forced to 1 and 0 rows (a size-1 and an empty group); leftover
    rows go to rank 1; ranks map to experts by a seeded Fisher-Yates shuffle.
    """
    z = sum(r ** -s for r in range(1, E + 1))
    sizes = [int(math.floor(M * (r ** -s) / z)) for r in range(1, E + 1)]
    if E >= 2:
        sizes[-2], sizes[-1] = 1, 0
    sizes[0] += M - sum(sizes)
    perm = _perm(E, seed, TAG_PERM)
    out = [0] * E
    for rank, e in enumerate(perm):
        out[e] = sizes[rank]
    return out


def gmm_inputs(cfg: GmmConfig, device) -> dict:
    """fp32 activations [M, K] (rows pre-sorted by expert), fp32 weights [E, N, K], group metadata."""
    sizes = zipf_group_sizes(cfg.M, cfg.E, cfg.zipf_s, cfg.seed)
    offsets = [0]
    for s_ in sizes:
        offsets.append(offsets[-1] + s_)
    x = normal((cfg.M, cfg.K), cfg.seed, TAG_LOWP_X, cfg.x_sigma, torch.float32, device)
    w = normal((cfg.E, cfg.N, cfg.K), cfg.seed, TAG_LOWP_W, cfg.w_sigma, torch.float32, device)
    return {"x": x, "w": w,
            "expert_sizes": torch.tensor(sizes, dtype=torch.int32, device=device),
            "expert_offsets": torch.tensor(offsets, dtype=torch.int32, device=device)}
