"""ctypes binding of libmoe_gb300.so: argument marshalling only.

Every function takes torch CUDA tensors (PyTorch supplies device memory and the
current stream), checks dtypes/shapes/contiguity, passes raw pointers to the C
ABI declared in include/moe_gb300.h, and raises MoeError on a non-OK status.
No step of the computation runs here.
"""
from __future__ import annotations

import ctypes
import pathlib

import torch

_LIB_PATH = pathlib.Path(__file__).resolve().parent / "libmoe_gb300.so"
_lib = None

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_WORKSPACE, MOE_ERR_CUDA, MOE_ERR_DEVICE_DATA = range(6)
SCORING = {"softmax": 0, "sigmoid": 1}
DTYPES = {torch.bfloat16: 0, torch.float32: 1, torch.int8: 2, torch.float8_e4m3fn: 3}
DEVERR_EXPERT_ID, DEVERR_GROUP_META, DEVERR_TIMEOUT = 0x1, 0x2, 0x4

_c_int, _c_float, _c_size, _vp = ctypes.c_int, ctypes.c_float, ctypes.c_size_t, ctypes.c_void_p

_SIGNATURES = {
    "moe_grouped_topk": (_c_int, [_vp, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_float, _vp, _vp, _vp]),
    "moe_router_topk_workspace_size": (_c_size, [_c_int, _c_int, _c_int]),
    "moe_router_topk": (_c_int, [_vp, _vp, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_float,
                                 _vp, _vp, _vp, _vp, _c_size, _vp]),
    "moe_align_max_padded": (_c_size, [_c_int, _c_int, _c_int]),
    "moe_align_workspace_size": (_c_size, [_c_int, _c_int, _c_int]),
    "moe_align_block_size": (_c_int, [_vp, _c_int, _c_int, _c_int, _vp, _vp, _vp, _vp, _vp, _c_size, _vp]),
    "moe_fused_forward_workspace_size": (_c_size, [_c_int, _c_int, _c_int, _c_int, _c_int]),
    "moe_fused_forward": (_c_int, [_vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int,
                                   _c_int, _c_int, _c_float, _vp, _vp, _vp, _vp, _c_size, _vp]),
    "moe_fused_forward_fp8_workspace_size": (_c_size, [_c_int, _c_int, _c_int, _c_int, _c_int]),
    "moe_fused_forward_fp8": (_c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int,
                                       _c_int, _c_int, _c_int, _c_float, _vp, _vp, _vp, _vp, _c_size, _vp]),
    "moe_fused_forward_noalloc": (_c_int, [_vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int,
                                           _c_int, _c_int, _c_int, _c_float, _vp, _vp, _vp, _vp]),
    "moe_fused_forward_noalloc_check_error": (_c_int, [ctypes.POINTER(_c_int), _vp]),
    "moe_quant_per_token": (_c_int, [_vp, _c_int, _c_int, _c_int, _c_int, _vp, _vp, _vp]),
    "gmm_lowp_workspace_size": (_c_size, [_c_int, _c_int, _c_int, _c_int]),
    "gmm_lowp": (_c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _vp,
                          _c_size, _vp]),
    "moe_read_probe": (_c_int, [_vp, _c_size, _vp, _vp]),
    "moe_wait_timeout_probe": (_c_int, [_vp, ctypes.c_ulonglong, _vp]),
    "moe_check_device_error": (_c_int, [_vp, ctypes.POINTER(_c_int), _vp]),
    "moe_status_string": (ctypes.c_char_p, [_c_int]),
    "moe_set_stage_events": (None, [ctypes.POINTER(_vp), _c_int]),
}


class MoeError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {status_string(status)} ({status})")


def lib():
    """Load libmoe_gb300.so (raises if it was not built: there is no fallback path)."""
    global _lib
    if _lib is None:
        if not _LIB_PATH.exists():
            raise RuntimeError(f"{_LIB_PATH.name} is not built; run mixture_experts_routing_grouped_gb300.build.build() "
                               "(nvcc for sm_103a). There is no CPU or PyTorch fallback.")
        handle = ctypes.CDLL(str(_LIB_PATH))
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def exported_symbols() -> list[str]:
    return list(_SIGNATURES)


def status_string(status: int) -> str:
    return lib().moe_status_string(int(status)).decode()


def _check(fn: str, status: int):
    if status != MOE_OK:
        raise MoeError(fn, status)


def _stream(t: torch.Tensor):
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _ptr(t: torch.Tensor | None):
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _need(t: torch.Tensor, name: str, dtype=None, shape=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


# --------------------------------------------------------------------------- routing
def moe_grouped_topk(gating: torch.Tensor, topk: int, renormalize: bool = True, num_expert_group: int = 1,
                     topk_group: int = 1, scoring_func: str = "softmax", routed_scaling_factor: float = 1.0,
                     topk_weights: torch.Tensor | None = None, topk_ids: torch.Tensor | None = None):
    """Grouped top-k routing of fp32 logits [T, E] -> (weights fp32 [T, topk], ids int32 [T, topk])."""
    _need(gating, "gating", torch.float32)
    T, E = gating.shape
    if topk_weights is None:
        topk_weights = torch.empty((T, topk), dtype=torch.float32, device=gating.device)
    if topk_ids is None:
        topk_ids = torch.empty((T, topk), dtype=torch.int32, device=gating.device)
    _need(topk_weights, "topk_weights", torch.float32, (T, topk))
    _need(topk_ids, "topk_ids", torch.int32, (T, topk))
    st = lib().moe_grouped_topk(_ptr(gating), T, E, num_expert_group, topk_group, topk, SCORING[scoring_func],
                                int(bool(renormalize)), float(routed_scaling_factor), _ptr(topk_weights),
                                _ptr(topk_ids), _stream(gating))
    _check("moe_grouped_topk", st)
    return topk_weights, topk_ids


def moe_router_topk_workspace_size(T: int, H: int, E: int) -> int:
    return int(lib().moe_router_topk_workspace_size(T, H, E))


def moe_router_topk(x: torch.Tensor, w_gate: torch.Tensor, topk: int, renormalize: bool = True,
                    num_expert_group: int = 1, topk_group: int = 1, scoring_func: str = "softmax",
                    routed_scaling_factor: float = 1.0, router_logits: torch.Tensor | None = None,
                    topk_weights: torch.Tensor | None = None, topk_ids: torch.Tensor | None = None,
                    ws: torch.Tensor | None = None):
    """Router projection x [T, H] bf16 @ w_gate [E, H] fp32 ^T, then grouped top-k
    -> (router_logits fp32 [T, E], topk_weights fp32 [T, topk], topk_ids int32 [T, topk])."""
    _need(x, "x", torch.bfloat16)
    T, H = x.shape
    E = w_gate.shape[0]
    _need(w_gate, "w_gate", torch.float32, (E, H))
    dev = x.device
    if router_logits is None:
        router_logits = torch.empty((T, E), dtype=torch.float32, device=dev)
    if topk_weights is None:
        topk_weights = torch.empty((T, topk), dtype=torch.float32, device=dev)
    if topk_ids is None:
        topk_ids = torch.empty((T, topk), dtype=torch.int32, device=dev)
    _need(router_logits, "router_logits", torch.float32, (T, E))
    _need(topk_weights, "topk_weights", torch.float32, (T, topk))
    _need(topk_ids, "topk_ids", torch.int32, (T, topk))
    wsb = moe_router_topk_workspace_size(T, H, E)
    if ws is None and wsb > 0:
        ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
    st = lib().moe_router_topk(_ptr(x), _ptr(w_gate), T, H, E, num_expert_group, topk_group, topk,
                               SCORING[scoring_func], int(bool(renormalize)), float(routed_scaling_factor),
                               _ptr(router_logits), _ptr(topk_weights), _ptr(topk_ids), _ptr(ws),
                               0 if ws is None else ws.numel(), _stream(x))
    _check("moe_router_topk", st)
    return router_logits, topk_weights, topk_ids


# --------------------------------------------------------------------------- align
def moe_align_max_padded(num_pairs: int, num_experts: int, block_m: int) -> int:
    return int(lib().moe_align_max_padded(num_pairs, num_experts, block_m))


def moe_align_block_size(topk_ids: torch.Tensor, block_m: int, num_experts: int, ws: torch.Tensor | None = None):
    """Returns (sorted_token_ids, expert_ids, expert_offsets, num_tokens_post_padded[1]) as int32 CUDA tensors."""
    _need(topk_ids, "topk_ids", torch.int32)
    n = topk_ids.numel()
    cap = moe_align_max_padded(n, num_experts, block_m)
    dev = topk_ids.device
    sorted_ids = torch.empty(cap, dtype=torch.int32, device=dev)
    expert_ids = torch.empty(cap // block_m if block_m > 0 else 0, dtype=torch.int32, device=dev)
    offsets = torch.empty(num_experts + 1, dtype=torch.int32, device=dev)
    ntpp = torch.empty(1, dtype=torch.int32, device=dev)
    wsb = int(lib().moe_align_workspace_size(n, num_experts, block_m))
    if ws is None:
        ws = torch.zeros(max(wsb, 256), dtype=torch.uint8, device=dev)
    st = lib().moe_align_block_size(_ptr(topk_ids), n, num_experts, block_m, _ptr(sorted_ids), _ptr(expert_ids),
                                    _ptr(offsets), _ptr(ntpp), _ptr(ws), ws.numel(), _stream(topk_ids))
    _check("moe_align_block_size", st)
    return sorted_ids, expert_ids, offsets, ntpp


# --------------------------------------------------------------------------- fused layer
def moe_fused_forward_workspace_size(T: int, H: int, I: int, E: int, topk: int) -> int:
    return int(lib().moe_fused_forward_workspace_size(T, H, I, E, topk))


def gmm_lowp_workspace_size(M: int, K: int, N: int, E: int) -> int:
    return int(lib().gmm_lowp_workspace_size(M, K, N, E))


def moe_fused_forward(x: torch.Tensor, gating: torch.Tensor, w_gate_up: torch.Tensor, w_down: torch.Tensor,
                      topk: int, renormalize: bool = True, num_expert_group: int = 1, topk_group: int = 1,
                      scoring_func: str = "softmax", routed_scaling_factor: float = 1.0,
                      ws: torch.Tensor | None = None, y: torch.Tensor | None = None,
                      topk_weights: torch.Tensor | None = None, topk_ids: torch.Tensor | None = None):
    """The routed MoE layer: returns (y bf16 [T, H], topk_weights fp32 [T, k], topk_ids int32 [T, k])."""
    _need(x, "x", torch.bfloat16)
    T, H = x.shape
    E, I2, H2 = w_gate_up.shape
    I = I2 // 2
    _need(gating, "gating", torch.float32, (T, E))
    _need(w_gate_up, "w_gate_up", torch.bfloat16, (E, 2 * I, H))
    _need(w_down, "w_down", torch.bfloat16, (E, H, I))
    dev = x.device
    if y is None:
        y = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    if topk_weights is None:
        topk_weights = torch.empty((T, topk), dtype=torch.float32, device=dev)
    if topk_ids is None:
        topk_ids = torch.empty((T, topk), dtype=torch.int32, device=dev)
    wsb = moe_fused_forward_workspace_size(T, H, I, E, topk)
    if ws is None:
        ws = torch.zeros(max(wsb, 256), dtype=torch.uint8, device=dev)
    st = lib().moe_fused_forward(_ptr(x), _ptr(gating), _ptr(w_gate_up), _ptr(w_down), T, H, I, E,
                                 num_expert_group, topk_group, topk, SCORING[scoring_func], int(bool(renormalize)),
                                 float(routed_scaling_factor), _ptr(y), _ptr(topk_weights), _ptr(topk_ids),
                                 _ptr(ws), ws.numel(), _stream(x))
    _check("moe_fused_forward", st)
    return y, topk_weights, topk_ids


def moe_fused_forward_fp8_workspace_size(T: int, H: int, I: int, E: int, topk: int) -> int:
    return int(lib().moe_fused_forward_fp8_workspace_size(T, H, I, E, topk))


def moe_fused_forward_fp8(x: torch.Tensor, gating: torch.Tensor, w_gate_up: torch.Tensor,
                          scales_gate_up: torch.Tensor, w_down: torch.Tensor, scales_down: torch.Tensor, topk: int,
                          renormalize: bool = True, num_expert_group: int = 1, topk_group: int = 1,
                          scoring_func: str = "softmax", routed_scaling_factor: float = 1.0,
                          ws: torch.Tensor | None = None, y: torch.Tensor | None = None,
                          topk_weights: torch.Tensor | None = None, topk_ids: torch.Tensor | None = None):
    """The routed MoE layer with e4m3 weights (codes as torch.float8_e4m3fn or uint8) and fp32
    per-channel scales: returns (y bf16 [T, H], topk_weights fp32 [T, k], topk_ids int32 [T, k])."""
    _need(x, "x", torch.bfloat16)
    T, H = x.shape
    E, I2, H2 = w_gate_up.shape
    I = I2 // 2
    for t, name, shape in ((w_gate_up, "w_gate_up", (E, 2 * I, H)), (w_down, "w_down", (E, H, I))):
        if t.dtype not in (torch.float8_e4m3fn, torch.uint8):
            raise TypeError(f"{name} must hold e4m3 codes (torch.float8_e4m3fn or uint8), got {t.dtype}")
        _need(t, name, None, shape)
    _need(gating, "gating", torch.float32, (T, E))
    _need(scales_gate_up, "scales_gate_up", torch.float32, (E, 2 * I))
    _need(scales_down, "scales_down", torch.float32, (E, H))
    dev = x.device
    if y is None:
        y = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    if topk_weights is None:
        topk_weights = torch.empty((T, topk), dtype=torch.float32, device=dev)
    if topk_ids is None:
        topk_ids = torch.empty((T, topk), dtype=torch.int32, device=dev)
    wsb = moe_fused_forward_fp8_workspace_size(T, H, I, E, topk)
    if ws is None:
        ws = torch.zeros(max(wsb, 256), dtype=torch.uint8, device=dev)
    st = lib().moe_fused_forward_fp8(_ptr(x), _ptr(gating), _ptr(w_gate_up), _ptr(scales_gate_up), _ptr(w_down),
                                     _ptr(scales_down), T, H, I, E, num_expert_group, topk_group, topk,
                                     SCORING[scoring_func], int(bool(renormalize)), float(routed_scaling_factor),
                                     _ptr(y), _ptr(topk_weights), _ptr(topk_ids), _ptr(ws), ws.numel(), _stream(x))
    _check("moe_fused_forward_fp8", st)
    return y, topk_weights, topk_ids


def moe_fused_forward_noalloc(x: torch.Tensor, gating: torch.Tensor, w_gate_up: torch.Tensor, w_down: torch.Tensor,
                              topk: int, renormalize: bool = True, num_expert_group: int = 1, topk_group: int = 1,
                              scoring_func: str = "softmax", routed_scaling_factor: float = 1.0,
                              y: torch.Tensor | None = None, topk_weights: torch.Tensor | None = None,
                              topk_ids: torch.Tensor | None = None):
    """moe_fused_forward with its scratch taken from the library's fixed device array instead
    of a workspace: for callers that cannot allocate device memory. Outputs may be passed
    in preallocated; problems needing more than MOE_NOALLOC_SCRATCH_BYTES of scratch raise
    MoeError(MOE_ERR_WORKSPACE). Calls that overlap on the GPU race on the shared array."""
    _need(x, "x", torch.bfloat16)
    T, H = x.shape
    E, I2, _ = w_gate_up.shape
    I = I2 // 2
    _need(gating, "gating", torch.float32, (T, E))
    _need(w_gate_up, "w_gate_up", torch.bfloat16, (E, 2 * I, H))
    _need(w_down, "w_down", torch.bfloat16, (E, H, I))
    dev = x.device
    if y is None:
        y = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    if topk_weights is None:
        topk_weights = torch.empty((T, topk), dtype=torch.float32, device=dev)
    if topk_ids is None:
        topk_ids = torch.empty((T, topk), dtype=torch.int32, device=dev)
    st = lib().moe_fused_forward_noalloc(_ptr(x), _ptr(gating), _ptr(w_gate_up), _ptr(w_down), T, H, I, E,
                                         num_expert_group, topk_group, topk, SCORING[scoring_func],
                                         int(bool(renormalize)), float(routed_scaling_factor), _ptr(y),
                                         _ptr(topk_weights), _ptr(topk_ids), _stream(x))
    _check("moe_fused_forward_noalloc", st)
    return y, topk_weights, topk_ids


def moe_fused_forward_noalloc_check_error(device: torch.device | None = None) -> int:
    """Reads and clears the device error word of moe_fused_forward_noalloc's scratch array on
    the current device (synchronises the current stream); returns the MOE_DEVERR_* bits."""
    dev = torch.device("cuda") if device is None else torch.device(device)
    code = _c_int(0)
    with torch.cuda.device(dev):
        st = lib().moe_fused_forward_noalloc_check_error(ctypes.byref(code),
                                                         ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream))
    if st not in (MOE_OK, MOE_ERR_DEVICE_DATA):
        _check("moe_fused_forward_noalloc_check_error", st)
    return int(code.value)


# --------------------------------------------------------------------------- low precision
def moe_quant_per_token(x: torch.Tensor, q_dtype: torch.dtype, q: torch.Tensor | None = None,
                        scales: torch.Tensor | None = None):
    """Symmetric per-row quantisation of [M, K] bf16/fp32 -> (codes int8 or float8_e4m3fn [M, K], scales fp32 [M])."""
    _need(x, "x")
    M, K = x.shape
    if q is None:
        q = torch.empty((M, K), dtype=q_dtype, device=x.device)
    if scales is None:
        scales = torch.empty(M, dtype=torch.float32, device=x.device)
    _need(q, "q", q_dtype, (M, K))
    _need(scales, "scales", torch.float32, (M,))
    st = lib().moe_quant_per_token(_ptr(x), DTYPES[x.dtype], M, K, DTYPES[q_dtype], _ptr(q), _ptr(scales),
                                   _stream(x))
    _check("moe_quant_per_token", st)
    return q, scales


def gmm_lowp(inp: torch.Tensor, weights: torch.Tensor, scales_x: torch.Tensor, scales_w: torch.Tensor,
             expert_offsets: torch.Tensor, expert_sizes: torch.Tensor, out_dtype: torch.dtype = torch.bfloat16,
             out: torch.Tensor | None = None, ws: torch.Tensor | None = None):
    """Low-precision grouped GEMM: out[m, n] = sx[m] sw[e, n] sum_k qx[m, k] qw[e, n, k]."""
    _need(inp, "input")
    M, K = inp.shape
    E, N, K2 = weights.shape
    _need(weights, "weights", inp.dtype, (E, N, K))
    _need(scales_x, "scales_x", torch.float32, (M,))
    _need(scales_w, "scales_w", torch.float32, (E, N))
    _need(expert_offsets, "expert_offsets", torch.int32, (E + 1,))
    _need(expert_sizes, "expert_sizes", torch.int32, (E,))
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype, device=inp.device)
    _need(out, "out", out_dtype, (M, N))
    wsb = int(lib().gmm_lowp_workspace_size(M, K, N, E))
    if ws is None:
        ws = torch.zeros(max(wsb, 256), dtype=torch.uint8, device=inp.device)
    st = lib().gmm_lowp(_ptr(inp), _ptr(weights), _ptr(scales_x), _ptr(scales_w), _ptr(expert_offsets),
                        _ptr(expert_sizes), _ptr(out), M, K, N, E, DTYPES[inp.dtype], DTYPES[out_dtype], _ptr(ws),
                        ws.numel(), _stream(inp))
    _check("gmm_lowp", st)
    return out


def moe_set_stage_events(events) -> None:
    """Record the given torch.cuda.Event objects at the stage boundaries of moe_fused_forward
    (see include/moe_gb300.h); None switches recording off."""
    if not events:
        lib().moe_set_stage_events(None, 0)
        return
    arr = (_vp * len(events))(*[ctypes.c_void_p(e.cuda_event) for e in events])
    lib().moe_set_stage_events(arr, len(events))


def moe_check_device_error(ws: torch.Tensor) -> int:
    """Reads and clears the device error word of a workspace (synchronises the stream)."""
    code = _c_int(0)
    st = lib().moe_check_device_error(_ptr(ws), ctypes.byref(code), _stream(ws))
    if st not in (MOE_OK, MOE_ERR_DEVICE_DATA):
        _check("moe_check_device_error", st)
    return int(code.value)


def moe_read_probe(src: torch.Tensor, sink: torch.Tensor) -> None:
    """Instrumentation: one streaming read of ``src``'s bytes on the current stream (the
    benchmark's read floor)."""
    _need(src, "src")
    _need(sink, "sink", torch.float32)
    st = lib().moe_read_probe(_ptr(src), src.numel() * src.element_size(), _ptr(sink), _stream(src))
    _check("moe_read_probe", st)


def moe_wait_timeout_probe(ws: torch.Tensor, limit_ns: int) -> None:
    """Test of failure detection: one kernel whose bounded wait runs out after limit_ns and
    reports MOE_DEVERR_TIMEOUT into ws's error word (read it with moe_check_device_error)."""
    _need(ws, "ws")
    _check("moe_wait_timeout_probe", lib().moe_wait_timeout_probe(_ptr(ws), int(limit_ns), _stream(ws)))
