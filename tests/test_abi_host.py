"""Host-side checks of the C ABI: the library builds/loads, exports every
function include/tokengate.h declares, and rejects bad arguments before any
CUDA call (so these run without a GPU)."""
import ctypes
import os
import re

import pytest

import learned_token_pruning_residual_b300 as tg
from learned_token_pruning_residual_b300 import build as tgbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tokengate.h")


@pytest.fixture(scope="module")
def L():
    tgbuild.build()
    return tg.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(tg_[a-z_]+)\s*\(", src)))


def test_header_and_binding_agree():
    assert declared_functions() == sorted(tg.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), name


def test_status_strings_and_version(L):
    assert L.tg_abi_version() == 3
    names = [L.tg_status_string(i).decode() for i in range(7)]
    assert names == ["TG_OK", "TG_ERR_INVALID_ARG", "TG_ERR_UNSUPPORTED", "TG_ERR_CUDA",
                     "TG_ERR_NAN_SCORE", "TG_ERR_BAD_INDEX", "TG_ERR_TIMEOUT"]
    assert L.tg_status_string(99).decode() == "TG_ERR_UNKNOWN"


def _m():
    return ctypes.c_int64(-1)


def test_select_argument_errors_and_host_M(L):
    m = _m()
    ws = ctypes.c_void_p(0x20000)
    wsb = L.tg_select_workspace_bytes(0)
    assert wsb == L.tg_select_workspace_bytes(1 << 30) == 106496  # independent of N
    # doc_end > N
    assert L.tg_select_topk(None, 10, 2, 20, 1, None, ctypes.byref(m), ws, wsb, None) == 1
    assert b"doc_end" in L.tg_last_error_message()
    # K > D
    assert L.tg_select_topk(None, 10, 2, 5, 4, None, ctypes.byref(m), ws, wsb, None) == 1
    # negative K
    assert L.tg_select_topk(None, 10, 2, 5, -1, None, ctypes.byref(m), ws, wsb, None) == 1
    # N == 0 is valid and launches nothing; M is computed on the host
    assert L.tg_select_topk(None, 0, 0, 0, 0, None, ctypes.byref(m), None, 0, None) == 0
    assert m.value == 0
    # nothing kept (M == 0) is valid and launches nothing
    assert L.tg_select_topk(None, 3, 0, 3, 0, None, ctypes.byref(m), None, 0, None) == 0
    assert m.value == 0
    # NULL pointers with work to do
    assert L.tg_select_topk(None, 10, 2, 5, 1, None, ctypes.byref(m), ws, wsb, None) == 1
    assert m.value == 8                                   # 10 - 3 + 1, reported before the check
    # misaligned pointer
    assert L.tg_select_topk(ctypes.c_void_p(0x1004), 10, 2, 5, 1, ctypes.c_void_p(0x2000),
                            ctypes.byref(m), ws, wsb, None) == 1
    # the workspace: missing, too small, misaligned
    p = ctypes.c_void_p(0x10000)
    assert L.tg_select_topk(p, 10, 2, 5, 1, p, ctypes.byref(m), None, wsb, None) == 1
    assert b"workspace" in L.tg_last_error_message()
    assert L.tg_select_topk(p, 10, 2, 5, 1, p, ctypes.byref(m), ws, wsb - 1, None) == 1
    assert L.tg_select_topk(p, 10, 2, 5, 1, p, ctypes.byref(m), ctypes.c_void_p(0x20010), wsb,
                            None) == 1


def test_gate_argument_errors(L):
    p = ctypes.c_void_p(0x10000)
    g = lambda *a, ws=None, b=0, e=0: L.tg_gate_score(*a, ws, b, e, None)
    assert g(p, 7, 10, 64, p, None, 16, p, 0.0, p) == 1          # dtype
    assert g(p, 1, -1, 64, p, None, 16, p, 0.0, p) == 1          # N
    assert g(p, 1, 10, 64, None, None, 16, p, 0.0, p) == 1       # NULL W1
    assert g(p, 1, 10, 96, p, None, 16, p, 0.0, p) == 2          # d % 64
    assert g(p, 1, 10, 64, p, None, 300, p, 0.0, p) == 2         # Hg > 256
    assert g(p, 1, 10, 64, p, None, 24, p, 0.0, p) == 2          # Hg % 16
    assert g(None, 1, 0, 64, None, None, 16, None, 0.0, None) == 0  # N == 0
    # with a select workspace: the span must lie in [0, N], the workspace be aligned
    ws = ctypes.c_void_p(0x20000)
    assert g(p, 1, 10, 64, p, None, 16, p, 0.0, p, ws=ws, b=3, e=11) == 1
    assert g(p, 1, 10, 64, p, None, 16, p, 0.0, p, ws=ws, b=5, e=4) == 1
    assert g(p, 1, 10, 64, p, None, 16, p, 0.0, p, ws=ctypes.c_void_p(0x20040), b=0, e=8) == 1
    # without a workspace the span is ignored
    assert g(p, 1, 10, 96, p, None, 16, p, 0.0, p, b=5, e=4) == 2


def test_gather_rmsnorm_qkv_attn_argument_errors(L):
    p = ctypes.c_void_p(0x10000)
    # f32 -> bf16 gather is not a supported pair
    assert L.tg_gather_rows(p, 0, 10, 64, p, 5, p, 1, None, None, None) == 2
    # idx NULL needs M == N
    assert L.tg_gather_rows(p, 1, 10, 64, None, 5, p, 1, None, None, None) == 1
    # scores without logsig output
    assert L.tg_gather_rows(p, 1, 10, 64, p, 5, p, 1, p, None, None) == 1
    # row bytes not a multiple of 16
    assert L.tg_gather_rows(p, 1, 10, 4, p, 5, p, 1, None, None, None) == 1
    assert L.tg_rmsnorm(p, 0, 10, 12, p, 1e-6, p, 1, None) == 1                     # d % 8
    assert L.tg_rmsnorm(p, 0, 10, 16, p, -1.0, p, 1, None) == 1                     # eps < 0
    assert L.tg_qkv_proj(p, 1, 10, 100, p, 16, 8, 128, p, None) == 2                # d % 64
    assert L.tg_keybias_attn(p, 1, 10, 16, 5, 128, None, None, 1.0, p, None, None) == 1  # Hq % Hkv
    assert L.tg_keybias_attn(p, 1, 10, 16, 8, 64, None, None, 1.0, p, None, None) == 2   # dh != 128
    assert L.tg_keybias_attn(p, 1, 10, 16, 16, 128, None, None, 1.0, p, None, None) == 2  # G odd
    assert L.tg_keybias_attn(p, 1, 10, 16, 8, 128, p, None, 1.0, p, None, None) == 1     # bias, no gain
    assert L.tg_keybias_attn(p, 1, 10, 16, 8, 128, None, None, float("nan"), p, None, None) == 1
    # bf16: the temperature must be finite and > 0
    for t in (0.0, -1.1, float("inf")):
        assert L.tg_keybias_attn(p, 1, 10, 16, 8, 128, None, None, t, p, None, None) == 2
        assert b"temperature" in L.tg_last_error_message()
    assert L.tg_keybias_attn(p, 0, 10, 4, 2, 48, None, None, 1.0, p, None, None) == 2    # f32 dh
    assert L.tg_keybias_attn(None, 1, 0, 16, 8, 128, None, None, 1.0, None, None, None) == 0


def test_python_binding_raises_without_device():
    import torch
    if torch.cuda.is_available():
        pytest.skip("has a device")
    x = torch.zeros(4, 64)
    with pytest.raises(ValueError):
        tg.tg_gate_score(x, x, None, x[0], 0.0)


def test_backward_argument_errors(L):
    p = ctypes.c_void_p(0x10000)
    odd = ctypes.c_void_p(0x10004)
    # forward with lse: a NULL lse is an error, M == 0 launches nothing
    assert L.tg_keybias_attn_lse(p, 1, 10, 16, 8, 128, None, None, 1.0, p, None, None, None) == 1
    assert L.tg_keybias_attn_lse(None, 1, 0, 16, 8, 128, None, None, 1.0, None, None, None,
                                 None) == 0
    assert L.tg_keybias_attn_lse(p, 1, 10, 16, 8, 128, None, None, 1.0, p, None, odd, None) == 1
    # delta: dtype, sizes, unsupported dh, NULL and misaligned pointers
    assert L.tg_attn_bwd_delta(p, p, 7, 10, 16, 128, p, None) == 1
    assert L.tg_attn_bwd_delta(p, p, 1, -1, 16, 128, p, None) == 1
    assert L.tg_attn_bwd_delta(p, p, 1, 10, 16, 96, p, None) == 2
    assert L.tg_attn_bwd_delta(p, p, 0, 10, 16, 256, p, None) == 2
    assert L.tg_attn_bwd_delta(p, None, 1, 10, 16, 128, p, None) == 1
    assert L.tg_attn_bwd_delta(p, odd, 1, 10, 16, 128, p, None) == 1
    assert L.tg_attn_bwd_delta(None, None, 1, 0, 16, 128, None, None) == 0
    assert L.tg_attn_bwd_delta(p, p, 1, 2**31 - 1, 4096, 256, p, None) == 2   # grid too large
    # bias gradient
    args = lambda **kw: [kw.get("qkv", p), kw.get("do", p), kw.get("dt", 1), kw.get("M", 10),
                         kw.get("Hq", 16), kw.get("Hkv", 8), kw.get("dh", 128), kw.get("ls", p),
                         kw.get("g", p), kw.get("t", 1.0), kw.get("lse", p), kw.get("delta", p),
                         kw.get("db", p), None]
    assert L.tg_keybias_attn_bias_grad(*args(dt=5)) == 1
    assert L.tg_keybias_attn_bias_grad(*args(Hq=12)) == 1                 # Hq % Hkv
    assert L.tg_keybias_attn_bias_grad(*args(t=float("nan"))) == 1
    assert L.tg_keybias_attn_bias_grad(*args(t=float("inf"))) == 1
    assert L.tg_keybias_attn_bias_grad(*args(lse=None)) == 1
    assert L.tg_keybias_attn_bias_grad(*args(g=None)) == 1                # bias without gain
    assert L.tg_keybias_attn_bias_grad(*args(db=odd)) == 1
    assert L.tg_keybias_attn_bias_grad(*args(dh=64)) == 2                 # bf16 needs dh 128
    assert L.tg_keybias_attn_bias_grad(*args(dt=0, dh=96)) == 2
    assert L.tg_keybias_attn_bias_grad(*args(M=0, qkv=None, do=None)) == 0
    assert L.tg_keybias_attn_bias_grad(*args(M=2**31 - 1, Hq=2**16, Hkv=2**15)) == 2
    # reduction
    assert L.tg_bias_grad_reduce(p, 10, 0, p, p, p, p, None, None) == 1     # Hq
    assert L.tg_bias_grad_reduce(p, 10, 4, None, p, p, p, None, None) == 1  # logsig
    assert L.tg_bias_grad_reduce(p, 10, 4, p, p, p, None, None, None) == 1  # dgain
    assert L.tg_bias_grad_reduce(p, 10, 4, p, p, p, p, odd, None) == 1      # dscore alignment


def test_selftest_bounded_wait_argument_errors(L):
    assert L.tg_selftest_bounded_wait(0, None, None) == 1            # timeout 0
    assert L.tg_selftest_bounded_wait(1000001, None, None) == 1      # longer than 1 s
    assert b"timeout_us" in L.tg_last_error_message()
    assert L.tg_selftest_bounded_wait(100, ctypes.c_void_p(0x1004), None) == 1  # misaligned report


def test_plan_argument_errors(L):
    assert L.tg_gated_layer_plan_create(None, None) == 1
    assert L.tg_plan_launch(None, None) == 1
    assert L.tg_plan_destroy(None) == 0
