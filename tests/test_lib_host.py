"""The C-ABI library builds, loads and exports every declared symbol; host-side
validation and size queries behave as documented. No GPU needed: nothing here
launches a kernel. Every call below is one that the documented checks reject (or
find empty) before any launch, so no fake pointer here ever reaches a kernel."""
import ctypes
import pathlib
import re

import pytest

from conftest import ROOT
from oracle import align as oalign

HEADER = ROOT / "include" / "moe_gb300.h"


@pytest.fixture(scope="module")
def L():
    from mixture_experts_routing_grouped_gb300 import build
    build.build()
    import mixture_experts_routing_grouped_gb300 as moe
    return moe.lib()


def _declared():
    text = HEADER.read_text()
    return sorted(set(re.findall(r"^MOE_API [^(]*?\b(\w+)\(", text, flags=re.M)))


def test_header_declares_the_boundary():
    names = _declared()
    for n in ["moe_grouped_topk", "moe_align_block_size", "moe_align_max_padded", "moe_fused_forward",
              "moe_fused_forward_workspace_size", "gmm_lowp", "moe_quant_per_token", "moe_check_device_error",
              "moe_status_string"]:
        assert n in names


def test_every_declared_symbol_is_exported(L):
    import mixture_experts_routing_grouped_gb300 as moe
    for n in _declared():
        assert hasattr(L, n), n
    assert sorted(moe.exported_symbols()) == _declared()


def test_status_strings(L):
    assert L.moe_status_string(0) == b"MOE_OK"
    assert L.moe_status_string(3) == b"MOE_ERR_WORKSPACE"
    assert L.moe_status_string(99) == b"MOE_ERR_UNKNOWN"


@pytest.mark.parametrize("n,E,bm", [(0, 8, 4), (10, 8, 4), (32768, 128, 128), (1024, 256, 16), (5, 1000, 256)])
def test_align_capacity_matches_oracle(L, n, E, bm):
    assert L.moe_align_max_padded(n, E, bm) == oalign.max_padded(n, E, bm)


FAKE = ctypes.c_void_p(0x10000)  # never dereferenced: validation returns before any launch


def test_routing_validation(L):
    f = L.moe_grouped_topk
    assert f(FAKE, 4, 10, 3, 1, 1, 0, 1, 1.0, FAKE, FAKE, None) == 1      # E % G != 0
    assert f(FAKE, 4, 8, 4, 5, 1, 0, 1, 1.0, FAKE, FAKE, None) == 1       # topk_group > G
    assert f(FAKE, 4, 8, 4, 2, 5, 0, 1, 1.0, FAKE, FAKE, None) == 1       # topk > candidates
    assert f(FAKE, 4, 2048, 8, 4, 8, 0, 1, 1.0, FAKE, FAKE, None) == 1    # E > 1024
    assert f(FAKE, 4, 8, 1, 1, 2, 7, 1, 1.0, FAKE, FAKE, None) == 1       # unknown scoring
    assert f(None, 4, 8, 1, 1, 2, 0, 1, 1.0, FAKE, FAKE, None) == 1       # null input
    assert f(ctypes.c_void_p(0x10004), 4, 8, 1, 1, 2, 0, 1, 1.0, FAKE, FAKE, None) == 2  # misaligned
    assert f(None, 0, 8, 1, 1, 2, 0, 1, 1.0, None, None, None) == 0       # T = 0: nothing to do


def test_align_validation(L):
    f = L.moe_align_block_size
    assert f(FAKE, 10, 8, 3, FAKE, FAKE, FAKE, FAKE, FAKE, 4096, None) == 1  # block_m not a power of 2
    assert f(FAKE, 10, 8, 512, FAKE, FAKE, FAKE, FAKE, FAKE, 4096, None) == 1
    assert f(FAKE, 10, 0, 4, FAKE, FAKE, FAKE, FAKE, FAKE, 4096, None) == 1
    assert f(FAKE, 10, 8, 4, FAKE, FAKE, FAKE, FAKE, None, 4096, None) == 3   # no workspace
    assert f(FAKE, 10, 8, 4, FAKE, FAKE, FAKE, FAKE, FAKE, 8, None) == 3      # workspace too small
    need = L.moe_align_workspace_size(10, 8, 4)
    assert need > 256
    assert f(FAKE, 10, 8, 4, FAKE, FAKE, FAKE, FAKE, FAKE, need - 1, None) == 3


def test_fused_validation_and_sizes(L):
    f = L.moe_fused_forward
    ws = L.moe_fused_forward_workspace_size(4096, 2048, 768, 128, 8)
    cap = oalign.max_padded(4096 * 8, 128, 128)
    assert ws >= cap * 768 * 2 + 4096 * 2048 * 4
    args = lambda H, I, wsb, wsp=FAKE: (FAKE, FAKE, FAKE, FAKE, 64, H, I, 8, 1, 1, 2, 0, 1, 1.0, FAKE, FAKE, FAKE,
                                        wsp, wsb, None)
    assert f(*args(100, 256, 1 << 30)) == 2          # H not a multiple of 256
    assert f(*args(512, 200, 1 << 30)) == 2          # I not a multiple of 128
    need = L.moe_fused_forward_workspace_size(64, 512, 256, 8, 2)
    assert f(*args(512, 256, need - 1)) == 3
    assert f(*args(512, 256, need, ctypes.c_void_p(0x10010))) == 3  # workspace not 256-byte aligned


def test_gmm_lowp_workspace_holds_the_widened_activations(L):
    # INT8 inputs are widened to fp16 once, into the workspace: M*K*2 bytes beyond the metadata
    for M, K, N, E in ((2048, 4096, 4096, 32), (1, 128, 128, 1), (0, 256, 128, 4)):
        assert L.gmm_lowp_workspace_size(M, K, N, E) >= M * K * 2 + 256
    assert L.gmm_lowp_workspace_size(16, 128, 128, 0) == 0


def test_fused_fp8_validation_and_sizes(L):
    f = L.moe_fused_forward_fp8
    ws = L.moe_fused_forward_fp8_workspace_size(4096, 2048, 768, 128, 8)
    cap = oalign.max_padded(4096 * 8, 128, 128)
    # the bf16 layout, plus e4m3 codes of x and of h with their scales
    assert ws >= cap * 768 * 2 + 4096 * 2048 * 4 + 4096 * 2048 + cap * 768
    assert L.moe_fused_forward_fp8_workspace_size(16, 512, 256, 0, 2) == 0
    args = lambda H, I, wsb, wsp=FAKE, s1=FAKE, s2=FAKE: (FAKE, FAKE, FAKE, s1, FAKE, s2, 64, H, I, 8, 1, 1, 2, 0, 1,
                                                         1.0, FAKE, FAKE, FAKE, wsp, wsb, None)
    assert f(*args(100, 256, 1 << 30)) == 2          # H not a multiple of 256
    assert f(*args(512, 200, 1 << 30)) == 2          # I not a multiple of 128
    assert f(*args(512, 256, 1 << 30, s1=None)) == 1  # missing gate_up scales
    assert f(*args(512, 256, 1 << 30, s2=None)) == 1  # missing down scales
    assert f(*args(512, 256, 1 << 30, s1=ctypes.c_void_p(0x10004))) == 2  # scales not 16-byte aligned
    need = L.moe_fused_forward_fp8_workspace_size(64, 512, 256, 8, 2)
    assert need > L.moe_fused_forward_workspace_size(64, 512, 256, 8, 2)
    assert f(*args(512, 256, need - 1)) == 3
    assert f(*args(512, 256, need, ctypes.c_void_p(0x10010))) == 3  # workspace not 256-byte aligned


def test_gmm_lowp_validation(L):
    f = L.gmm_lowp
    I8, E4, BF, F32 = 2, 3, 0, 1
    ws = 1 << 30

    def call(M=256, K=256, N=256, E=4, in_dt=E4, out_dt=BF, inp=FAKE, w=FAKE, sx=FAKE, sw=FAKE, off=FAKE,
             sz=FAKE, out=FAKE, wsp=FAKE, wsb=ws):
        return f(inp, w, sx, sw, off, sz, out, M, K, N, E, in_dt, out_dt, wsp, wsb, None)

    assert call(in_dt=BF) == 1                          # inputs must be int8 or e4m3
    assert call(out_dt=I8) == 1                         # output must be bf16 or fp32
    assert call(E=0) == 1 and call(E=2048) == 1         # 1 <= E <= 1024
    assert call(M=-1) == 1 and call(K=0) == 1 and call(N=0) == 1
    assert call(w=None) == 1 and call(sw=None) == 1 and call(off=None) == 1 and call(sz=None) == 1
    assert call(inp=None) == 1 and call(sx=None) == 1 and call(out=None) == 1
    assert call(K=200) == 2 and call(N=200) == 2       # K and N in whole 128-wide tiles
    assert call(inp=ctypes.c_void_p(0x10008)) == 2      # operands 16-byte aligned
    assert call(wsp=None) == 3
    assert call(wsp=ctypes.c_void_p(0x10010)) == 3      # workspace 256-byte aligned
    need8 = L.gmm_lowp_workspace_size(256, 256, 256, 4)
    assert call(in_dt=I8, wsb=need8 - 1) == 3           # INT8 needs room for the widened codes
    assert call(M=0, inp=None, sx=None, out=None) == 0  # no rows: nothing to do


def test_quant_validation(L):
    f = L.moe_quant_per_token
    BF, F32, I8, E4 = 0, 1, 2, 3
    assert f(FAKE, I8, 4, 64, E4, FAKE, FAKE, None) == 1    # x must be bf16 or fp32
    assert f(FAKE, BF, 4, 64, BF, FAKE, FAKE, None) == 1    # codes must be int8 or e4m3
    assert f(FAKE, BF, -1, 64, I8, FAKE, FAKE, None) == 1
    assert f(FAKE, BF, 4, 0, I8, FAKE, FAKE, None) == 1
    assert f(None, BF, 4, 64, I8, FAKE, FAKE, None) == 1
    assert f(FAKE, BF, 4, 64, I8, FAKE, None, None) == 1
    assert f(FAKE, BF, 4, 60, I8, FAKE, FAKE, None) == 2     # K a multiple of 8
    assert f(ctypes.c_void_p(0x10008), BF, 4, 64, I8, FAKE, FAKE, None) == 2  # x 16-byte aligned
    assert f(FAKE, F32, 4, 64, I8, ctypes.c_void_p(0x10004), FAKE, None) == 2  # codes 8-byte aligned
    assert f(None, BF, 0, 64, I8, None, None, None) == 0     # no rows: nothing to do


def test_check_device_error_needs_its_arguments(L):
    code = ctypes.c_int(0)
    assert L.moe_check_device_error(None, ctypes.byref(code), None) == 1
    assert L.moe_check_device_error(FAKE, None, None) == 1


def test_noalloc_rejects_on_the_host(L):
    """The allocation-free forward refuses, before touching any device, a problem whose
    workspace exceeds its fixed scratch array, and arguments that size no workspace."""
    f = L.moe_fused_forward_noalloc
    T, H, I, E, k = 4096, 2048, 768, 128, 8
    assert L.moe_fused_forward_workspace_size(T, H, I, E, k) > 64 * 1024 * 1024
    assert f(FAKE, FAKE, FAKE, FAKE, T, H, I, E, 1, 1, k, 0, 1, 1.0, FAKE, FAKE, FAKE, None) == 3
    assert f(FAKE, FAKE, FAKE, FAKE, 64, 0, 256, 8, 1, 1, 2, 0, 1, 1.0, FAKE, FAKE, FAKE, None) == 1
