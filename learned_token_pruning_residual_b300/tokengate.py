"""Thin Python binding of libtokengate.so (ctypes).

Argument marshalling only: every step of the gated prefill runs in the
library's CUDA kernels.  torch supplies device memory and the stream (the
caller's current CUDA stream).  If the library has not been built, or no
CUDA device is present, the calls raise; there is no fallback path.

Functions carry the C names:

    tg_gate_score     scores = w2 . GELU(W1 x + b1) + b2 per token
    tg_select_topk    kept indices: non-document tokens + top-K document tokens
    tg_gather_rows    kept rows and log(sigmoid(score)) of each kept token
    tg_rmsnorm        RMSNorm of a pruned layer's input
    tg_qkv_proj       packed q|k|v projection of the kept rows
    tg_keybias_attn   causal GQA attention with the per-key bias g_h * logsig
    tg_keybias_attn_lse        the same, also writing each row's log-sum-exp
    tg_attn_bwd_delta          D = dO . O per head and row
    tg_keybias_attn_bias_grad  dL/db for the per-head key bias b = g_h * logsig
    tg_bias_grad_reduce        dL/dlogsig, dL/dgain and dL/dscore from dL/db
    tg_get_device_status
    tg_selftest_bounded_wait   a wait that must give up (the failure path)
    tg_select_topk_noalloc     the select without a workspace (scratch compiled in)
    tg_rope_table              rotary (cos, sin) of the kept rows at their prompt positions
    tg_qkv_proj_qknorm_rope    QKV projection + per-head q/k RMSNorm + rotary embedding
    tg_linear_residual         residual += X W^T (o-projection, MLP down-projection)
    tg_swiglu                  silu(X W_gate^T) * (X W_up^T)
    tg_gated_delta_rule        the gated delta rule of a Gated-DeltaNet layer, chunked
    tg_gated_layer_plan_create / tg_plan_launch / tg_plan_destroy
                               the five calls of a gated layer as one CUDA graph

plus compositions of them: ``gated_layer``, ``pruned_stack``, ``qwen3_layer``,
``qwen3_pruned_stack`` and ``bias_backward``.
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "TokenGateError", "lib", "library_path", "TG_F32", "TG_BF16",
    "tg_gate_score", "tg_select_workspace_bytes", "new_select_workspace", "tg_select_topk", "tg_gather_rows", "tg_rmsnorm", "tg_qkv_proj",
    "tg_keybias_attn", "tg_keybias_attn_lse", "tg_attn_bwd_delta", "tg_keybias_attn_bias_grad",
    "tg_bias_grad_reduce", "tg_get_device_status", "tg_selftest_bounded_wait",
    "tg_select_topk_noalloc", "tg_rope_table", "tg_qkv_proj_qknorm_rope", "tg_linear_residual",
    "tg_swiglu", "tg_gated_delta_rule", "GatedLayerPlan", "qwen3_layer", "qwen3_pruned_stack", "gated_layer",
    "pruned_stack",
    "bias_backward", "EXPORTED_SYMBOLS",
]

TG_F32, TG_BF16 = 0, 1
_STATUS = {0: "TG_OK", 1: "TG_ERR_INVALID_ARG", 2: "TG_ERR_UNSUPPORTED", 3: "TG_ERR_CUDA",
           4: "TG_ERR_NAN_SCORE", 5: "TG_ERR_BAD_INDEX", 6: "TG_ERR_TIMEOUT"}

_HERE = os.path.dirname(os.path.abspath(__file__))
library_path = os.path.join(_HERE, "libtokengate.so")

_p, _i32, _i64, _f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
# name -> argtypes, in the order of include/tokengate.h
_SIGNATURES = {
    "tg_status_string": [ctypes.c_int],
    "tg_abi_version": [],
    "tg_last_error_message": [],
    "tg_gate_score": [_p, ctypes.c_int, _i64, _i32, _p, _p, _i32, _p, _f32, _p, _p, _i64, _i64,
                      _p],
    "tg_select_workspace_bytes": [_i64],
    "tg_select_topk": [_p, _i64, _i64, _i64, _i64, _p, ctypes.POINTER(_i64), _p, ctypes.c_size_t,
                       _p],
    "tg_gather_rows": [_p, ctypes.c_int, _i64, _i32, _p, _i64, _p, ctypes.c_int, _p, _p, _p],
    "tg_rmsnorm": [_p, ctypes.c_int, _i64, _i32, _p, _f32, _p, ctypes.c_int, _p],
    "tg_qkv_proj": [_p, ctypes.c_int, _i64, _i32, _p, _i32, _i32, _i32, _p, _p],
    "tg_keybias_attn": [_p, ctypes.c_int, _i64, _i32, _i32, _i32, _p, _p, _f32, _p, _p, _p],
    "tg_keybias_attn_lse": [_p, ctypes.c_int, _i64, _i32, _i32, _i32, _p, _p, _f32, _p, _p, _p,
                            _p],
    "tg_attn_bwd_delta": [_p, _p, ctypes.c_int, _i64, _i32, _i32, _p, _p],
    "tg_keybias_attn_bias_grad": [_p, _p, ctypes.c_int, _i64, _i32, _i32, _i32, _p, _p, _f32, _p,
                                  _p, _p, _p],
    "tg_bias_grad_reduce": [_p, _i64, _i32, _p, _p, _p, _p, _p, _p],
    "tg_get_device_status": [_p],
    "tg_selftest_bounded_wait": [ctypes.c_uint32, _p, _p],
    "tg_select_topk_noalloc": [_p, _i64, _i64, _i64, _i64, _p, ctypes.POINTER(_i64), _p],
    "tg_rope_table": [_p, _i64, _i32, ctypes.c_double, _p, _p],
    "tg_qkv_proj_qknorm_rope": [_p, _i64, _i32, _p, _i32, _i32, _i32, _p, _p, _f32, _p, _p, _p],
    "tg_linear_residual": [_p, _i64, _i32, _p, _i32, _p, _p],
    "tg_swiglu": [_p, _i64, _i32, _p, _p, _i32, _p, _p],
    "tg_gated_delta_rule_workspace_bytes": [_i64, _i32],
    "tg_gated_delta_rule": [_p, _p, _p, ctypes.c_int, _p, _p, _i64, _i32, _i32, _i32, _p, _p, _p,
                            _p, ctypes.c_size_t, _p],
    "tg_gated_layer_plan_create": [_p, ctypes.POINTER(_p)],
    "tg_plan_launch": [_p, _p],
    "tg_plan_destroy": [_p],
}
EXPORTED_SYMBOLS = tuple(_SIGNATURES)

_lib = None


class TokenGateError(RuntimeError):
    def __init__(self, status: int, message: str = ""):
        self.status = status
        name = _STATUS.get(status, f"status {status}")
        super().__init__(f"{name}: {message}" if message else name)


def lib() -> ctypes.CDLL:
    """Load the shared library (once).  Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(library_path):
            raise RuntimeError(
                f"{library_path} is missing; build it with "
                "`python -m learned_token_pruning_residual_b300.build`")
        L = ctypes.CDLL(library_path)
        for name, args in _SIGNATURES.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = ctypes.c_char_p if name in ("tg_status_string", "tg_last_error_message") \
                else (ctypes.c_size_t if name.endswith("_workspace_bytes") else ctypes.c_int)
        _lib = L
    return _lib


def _check(status: int) -> None:
    if status != 0:
        msg = lib().tg_last_error_message().decode(errors="replace")
        raise TokenGateError(status, msg)


def _stream() -> int:
    return torch.cuda.current_stream().cuda_stream


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return TG_F32
    if t.dtype == torch.bfloat16:
        return TG_BF16
    raise TypeError(f"unsupported dtype {t.dtype}")


def _ptr(t: torch.Tensor | None) -> int | None:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensor must live on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return t.data_ptr()


def tg_gate_score(X, W1, b1, w2, b2: float, out=None, select_ws=None, doc_begin: int = 0,
                  doc_end: int = 0):
    """Gate scores [N] fp32 of the residual rows X [N][d] (bf16 or fp32).
    With ``select_ws`` (a select workspace) the bf16 path also counts the
    first radix pass of the selection over [doc_begin, doc_end) into it, for
    the tg_select_topk that follows on the same workspace."""
    N, d = X.shape
    Hg = W1.shape[0]
    if out is None:
        out = torch.empty(N, dtype=torch.float32, device=X.device)
    _check(lib().tg_gate_score(_ptr(X), _dt(X), N, d, _ptr(W1), _ptr(b1), Hg, _ptr(w2),
                               float(b2), _ptr(out), _ptr(select_ws), int(doc_begin),
                               int(doc_end), _stream()))
    return out


def tg_select_workspace_bytes(N: int = 0) -> int:
    return int(lib().tg_select_workspace_bytes(int(N)))


def new_select_workspace(device=None) -> torch.Tensor:
    """A zeroed select workspace (uint8, tg_select_workspace_bytes() bytes)
    on ``device``.  Every successful select leaves it zeroed again; use one
    per stream."""
    return torch.zeros(tg_select_workspace_bytes(), dtype=torch.uint8,
                       device=device if device is not None else torch.cuda.current_device())


_WORKSPACES: dict = {}


def _default_workspace(device: torch.device) -> torch.Tensor:
    key = (device.index, torch.cuda.current_stream(device).cuda_stream)
    ws = _WORKSPACES.get(key)
    if ws is None:
        ws = _WORKSPACES[key] = new_select_workspace(device)
    return ws


def tg_select_topk(scores, doc_begin: int, doc_end: int, K: int, out=None, workspace=None):
    """Ascending int32 indices of the kept tokens: all tokens outside
    [doc_begin, doc_end) plus the K best-scoring document tokens.
    ``workspace``: a select workspace (default: one kept per device and
    stream by this module)."""
    N = scores.shape[0]
    M = N - (doc_end - doc_begin) + K
    if out is None:
        out = torch.empty(max(M, 0), dtype=torch.int32, device=scores.device)
    if workspace is None:
        workspace = _default_workspace(scores.device)
    m_out = _i64(0)
    _check(lib().tg_select_topk(_ptr(scores), N, doc_begin, doc_end, K, _ptr(out),
                                ctypes.byref(m_out), _ptr(workspace),
                                workspace.numel() * workspace.element_size(), _stream()))
    assert m_out.value == M
    return out


def tg_select_topk_noalloc(scores, doc_begin: int, doc_end: int, K: int, out=None):
    """tg_select_topk for callers that cannot provide a workspace: the
    library uses a scratch array compiled into it (one per device, shared by
    all calls; calls must not overlap on the GPU)."""
    N = scores.shape[0]
    M = N - (doc_end - doc_begin) + K
    if out is None:
        out = torch.empty(max(M, 0), dtype=torch.int32, device=scores.device)
    m_out = _i64(0)
    _check(lib().tg_select_topk_noalloc(_ptr(scores), N, doc_begin, doc_end, K, _ptr(out),
                                        ctypes.byref(m_out), _stream()))
    assert m_out.value == M
    return out


def tg_gather_rows(X, idx, scores=None, out=None, out_dtype=None, logsig_out=None):
    """(Y, logsig): Y[m] = X[idx[m]] (idx None: identity) in out_dtype, and
    log(sigmoid(scores[idx[m]])) when scores are given."""
    N, d = X.shape
    M = N if idx is None else idx.shape[0]
    out_dtype = out_dtype or X.dtype
    if out is None:
        out = torch.empty(M, d, dtype=out_dtype, device=X.device)
    if scores is not None and logsig_out is None:
        logsig_out = torch.empty(M, dtype=torch.float32, device=X.device)
    _check(lib().tg_gather_rows(_ptr(X), _dt(X), N, d, _ptr(idx), M, _ptr(out), _dt(out),
                                _ptr(scores), _ptr(logsig_out) if scores is not None else None,
                                _stream()))
    return out, (logsig_out if scores is not None else None)


def tg_rmsnorm(X, gamma, eps: float, out=None, out_dtype=torch.bfloat16):
    M, d = X.shape
    if out is None:
        out = torch.empty(M, d, dtype=out_dtype, device=X.device)
    _check(lib().tg_rmsnorm(_ptr(X), _dt(X), M, d, _ptr(gamma), float(eps), _ptr(out), _dt(out),
                            _stream()))
    return out


def tg_qkv_proj(X, Wqkv, Hq: int, Hkv: int, dh: int, out=None):
    M, d = X.shape
    if out is None:
        out = torch.empty(M, (Hq + 2 * Hkv) * dh, dtype=X.dtype, device=X.device)
    _check(lib().tg_qkv_proj(_ptr(X), _dt(X), M, d, _ptr(Wqkv), Hq, Hkv, dh, _ptr(out), _stream()))
    return out


def tg_keybias_attn(QKV, Hq: int, Hkv: int, dh: int, logsig, gain, temperature: float,
                    out=None, residual=None):
    """O [M][Hq dh] (or residual += O in fp32 when residual is given)."""
    M = QKV.shape[0]
    if out is None and residual is None:
        out = torch.empty(M, Hq * dh, dtype=QKV.dtype, device=QKV.device)
    _check(lib().tg_keybias_attn(_ptr(QKV), _dt(QKV), M, Hq, Hkv, dh, _ptr(logsig), _ptr(gain),
                                 float(temperature), _ptr(out), _ptr(residual), _stream()))
    return out if residual is None else residual


def tg_keybias_attn_lse(QKV, Hq: int, Hkv: int, dh: int, logsig, gain, temperature: float,
                        out=None, residual=None, lse=None):
    """(O, lse): tg_keybias_attn plus lse [Hq][M] fp32, the natural-log
    normaliser log sum_{j <= i} exp(l_ij) of every head and row."""
    M = QKV.shape[0]
    if out is None and residual is None:
        out = torch.empty(M, Hq * dh, dtype=QKV.dtype, device=QKV.device)
    if lse is None:
        lse = torch.empty(Hq, M, dtype=torch.float32, device=QKV.device)
    _check(lib().tg_keybias_attn_lse(_ptr(QKV), _dt(QKV), M, Hq, Hkv, dh, _ptr(logsig),
                                     _ptr(gain), float(temperature), _ptr(out), _ptr(residual),
                                     _ptr(lse), _stream()))
    return (out if residual is None else residual), lse


def tg_attn_bwd_delta(dO, O, Hq: int, dh: int, out=None):
    """D [Hq][M] fp32: dO_i . o_i over the dh columns of each head."""
    M = dO.shape[0]
    if out is None:
        out = torch.empty(Hq, M, dtype=torch.float32, device=dO.device)
    _check(lib().tg_attn_bwd_delta(_ptr(dO), _ptr(O), _dt(dO), M, Hq, dh, _ptr(out), _stream()))
    return out


def tg_keybias_attn_bias_grad(QKV, dO, Hq: int, Hkv: int, dh: int, logsig, gain,
                              temperature: float, lse, delta, out=None):
    """dL/db [Hq][M] fp32 for the key bias b_hj = g_h logsig_j."""
    M = QKV.shape[0]
    if out is None:
        out = torch.empty(Hq, M, dtype=torch.float32, device=QKV.device)
    _check(lib().tg_keybias_attn_bias_grad(_ptr(QKV), _ptr(dO), _dt(QKV), M, Hq, Hkv, dh,
                                           _ptr(logsig), _ptr(gain), float(temperature),
                                           _ptr(lse), _ptr(delta), _ptr(out), _stream()))
    return out


def tg_bias_grad_reduce(dbias, logsig, gain, dlogsig=None, dgain=None, dscore=None,
                        want_dscore: bool = True):
    """(dL/dlogsig [M], dL/dgain [Hq], dL/dscore [M] or None) from dL/db."""
    Hq, M = dbias.shape
    dev = dbias.device
    if dlogsig is None:
        dlogsig = torch.empty(M, dtype=torch.float32, device=dev)
    if dgain is None:
        dgain = torch.empty(Hq, dtype=torch.float32, device=dev)
    if dscore is None and want_dscore:
        dscore = torch.empty(M, dtype=torch.float32, device=dev)
    _check(lib().tg_bias_grad_reduce(_ptr(dbias), M, Hq, _ptr(logsig), _ptr(gain), _ptr(dlogsig),
                                     _ptr(dgain), _ptr(dscore), _stream()))
    return dlogsig, dgain, dscore


def tg_get_device_status(raise_on_error: bool = True) -> int:
    st = lib().tg_get_device_status(_stream())
    if raise_on_error:
        _check(st)
    return st


def tg_selftest_bounded_wait(timeout_us: int, report=None) -> None:
    """Launch the failure-path self-check (one CTA waits on an mbarrier that
    nothing completes and gives up after timeout_us).  ``report`` (uint64
    [4] on the device, optional) receives (ok, ns) of the short-bound waiter
    and of the abort-driven waiter.  Read the result with
    tg_get_device_status(raise_on_error=False): it returns TG_ERR_TIMEOUT."""
    _check(lib().tg_selftest_bounded_wait(int(timeout_us), _ptr(report), _stream()))


def tg_rope_table(positions, dh: int, base: float, out=None):
    """[M][dh/2][2] fp32 (cos, sin) of positions[m] * base^(-2c/dh)."""
    M = positions.shape[0]
    if out is None:
        out = torch.empty(M, dh // 2, 2, dtype=torch.float32, device=positions.device)
    _check(lib().tg_rope_table(_ptr(positions), M, dh, float(base), _ptr(out), _stream()))
    return out


def tg_qkv_proj_qknorm_rope(X, Wqkv, Hq: int, Hkv: int, dh: int, gamma_q, gamma_k, eps: float,
                            rope_table, out=None):
    M, d = X.shape
    if out is None:
        out = torch.empty(M, (Hq + 2 * Hkv) * dh, dtype=X.dtype, device=X.device)
    _check(lib().tg_qkv_proj_qknorm_rope(_ptr(X), M, d, _ptr(Wqkv), Hq, Hkv, dh, _ptr(gamma_q),
                                         _ptr(gamma_k), float(eps), _ptr(rope_table), _ptr(out),
                                         _stream()))
    return out


def tg_linear_residual(X, W, residual):
    """residual (fp32 [M][N], in place) += X W^T."""
    M, K = X.shape
    N = W.shape[0]
    _check(lib().tg_linear_residual(_ptr(X), M, K, _ptr(W), N, _ptr(residual), _stream()))
    return residual


def tg_swiglu(X, W_gate, W_up, out=None):
    M, d = X.shape
    F = W_gate.shape[0]
    if out is None:
        out = torch.empty(M, F, dtype=X.dtype, device=X.device)
    _check(lib().tg_swiglu(_ptr(X), M, d, _ptr(W_gate), _ptr(W_up), F, _ptr(out), _stream()))
    return out


def tg_gated_delta_rule(q, k, v, alpha, beta, S0=None, out=None, S_out=None, workspace=None):
    """o [T][H][dv] (q's dtype) of the gated delta rule over T tokens;
    q, k [T][H][dk], v [T][H][dv], alpha, beta [T][H] fp32, S0 / S_out
    [H][dv][dk] fp32 (optional).  Returns (o, S_out)."""
    T, H, dk = k.shape
    dv = v.shape[2]
    if out is None:
        out = torch.empty(T, H, dv, dtype=q.dtype, device=q.device)
    nb = int(lib().tg_gated_delta_rule_workspace_bytes(T, H))
    if workspace is None:
        workspace = torch.empty(max(nb, 16), dtype=torch.uint8, device=q.device)
    _check(lib().tg_gated_delta_rule(_ptr(q), _ptr(k), _ptr(v), _dt(q), _ptr(alpha), _ptr(beta), T,
                                     H, dk, dv, _ptr(S0), _ptr(out), _ptr(S_out), _ptr(workspace),
                                     workspace.numel(), _stream()))
    return out, S_out


class _GatedLayerDesc(ctypes.Structure):
    _fields_ = [("X", _p), ("N", _i64), ("d", _i32), ("W1", _p), ("b1", _p), ("Hg", _i32),
                ("w2", _p), ("b2", _f32), ("doc_begin", _i64), ("doc_end", _i64), ("K", _i64),
                ("Wqkv", _p), ("Hq", _i32), ("Hkv", _i32), ("dh", _i32), ("gain", _p),
                ("temperature", _f32), ("scores", _p), ("select_ws", _p),
                ("select_ws_bytes", ctypes.c_size_t), ("kept_idx", _p), ("Xk", _p),
                ("logsig_kept", _p), ("QKV", _p), ("O", _p)]


class GatedLayerPlan:
    """The five calls of one gated layer on fixed device buffers, captured
    once into a CUDA graph by the library (tg_gated_layer_plan_create);
    launch() replays it on the current stream.  Write a new prompt into
    ``X`` between launches.  ``bufs`` holds the outputs (scores, idx, Xk,
    logsig, qkv, out) and the select workspace (select_ws); missing ones are
    allocated here.  The tensors are kept alive with the plan."""

    def __init__(self, X, W1, b1, w2, b2, doc_begin, doc_end, K, Wqkv, Hq, Hkv, dh, gain,
                 temperature, bufs: dict | None = None):
        N, d = X.shape
        M = N - (doc_end - doc_begin) + K
        dev = X.device
        b = dict(bufs or {})
        f32, bf = torch.float32, torch.bfloat16
        b.setdefault("scores", torch.empty(N, dtype=f32, device=dev))
        b.setdefault("select_ws", new_select_workspace(dev))
        b.setdefault("idx", torch.empty(M, dtype=torch.int32, device=dev))
        b.setdefault("Xk", torch.empty(M, d, dtype=bf, device=dev))
        b.setdefault("logsig", torch.empty(M, dtype=f32, device=dev))
        b.setdefault("qkv", torch.empty(M, (Hq + 2 * Hkv) * dh, dtype=bf, device=dev))
        b.setdefault("out", torch.empty(M, Hq * dh, dtype=bf, device=dev))
        self.bufs = b
        self._keep = (X, W1, b1, w2, Wqkv, gain)
        ws = b["select_ws"]
        desc = _GatedLayerDesc(
            _ptr(X), N, d, _ptr(W1), _ptr(b1), W1.shape[0], _ptr(w2), float(b2), doc_begin,
            doc_end, K, _ptr(Wqkv), Hq, Hkv, dh, _ptr(gain), float(temperature), _ptr(b["scores"]),
            _ptr(ws), ws.numel() * ws.element_size(), _ptr(b["idx"]), _ptr(b["Xk"]),
            _ptr(b["logsig"]), _ptr(b["qkv"]), _ptr(b["out"]))
        handle = _p()
        _check(lib().tg_gated_layer_plan_create(ctypes.byref(desc), ctypes.byref(handle)))
        self._handle = handle

    def launch(self, stream: int | None = None):
        _check(lib().tg_plan_launch(self._handle, _stream() if stream is None else stream))
        return self.bufs

    def close(self):
        if self._handle is not None and self._handle.value:
            lib().tg_plan_destroy(self._handle)
        self._handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def qwen3_layer(x, rope_table, L: dict, Hq: int, Hkv: int, dh: int, logsig, eps: float = 1e-6,
                bufs: dict | None = None):
    """One Qwen3 decoder layer on the kept rows, x (fp32 [M][d]) updated in
    place: RMSNorm -> QKV + q/k RMSNorm + rotary embedding (rope_table of the
    rows' prompt positions) -> token-gated attention -> x += o Wo^T ->
    RMSNorm -> SwiGLU -> x += u Wd^T.  Seven library calls.  ``L`` holds
    gamma_attn, Wqkv, gamma_q, gamma_k, gain, temperature, Wo, gamma_mlp, Wg,
    Wu, Wd (bf16 weights, fp32 vectors); ``bufs`` may hold xn, qkv, o, hn, u."""
    M, d = x.shape
    b = bufs or {}
    dev = x.device
    bf = torch.bfloat16
    F = L["Wg"].shape[0]
    xn = b.get("xn") if b.get("xn") is not None else torch.empty(M, d, dtype=bf, device=dev)
    qkv = b.get("qkv") if b.get("qkv") is not None else \
        torch.empty(M, (Hq + 2 * Hkv) * dh, dtype=bf, device=dev)
    o = b.get("o") if b.get("o") is not None else torch.empty(M, Hq * dh, dtype=bf, device=dev)
    u = b.get("u") if b.get("u") is not None else torch.empty(M, F, dtype=bf, device=dev)
    tg_rmsnorm(x, L["gamma_attn"], eps, out=xn)
    tg_qkv_proj_qknorm_rope(xn, L["Wqkv"], Hq, Hkv, dh, L["gamma_q"], L["gamma_k"], eps,
                            rope_table, out=qkv)
    tg_keybias_attn(qkv, Hq, Hkv, dh, logsig, L["gain"], L["temperature"], out=o)
    tg_linear_residual(o, L["Wo"], x)
    tg_rmsnorm(x, L["gamma_mlp"], eps, out=xn)
    tg_swiglu(xn, L["Wg"], L["Wu"], out=u)
    tg_linear_residual(u, L["Wd"], x)
    return x


def qwen3_pruned_stack(x, positions, layers, Hq: int, Hkv: int, dh: int, logsig,
                       rope_base: float = 1e6, eps: float = 1e-6, bufs: dict | None = None):
    """The Qwen3 layers above the gate on the kept rows: the rotary table of
    the rows' prompt positions is built once, then qwen3_layer per layer."""
    table = tg_rope_table(positions, dh, rope_base)
    b = dict(bufs or {})
    M, d = x.shape
    bf = torch.bfloat16
    for key, shape in (("xn", (M, d)), ("qkv", (M, (Hq + 2 * Hkv) * dh)), ("o", (M, Hq * dh))):
        if b.get(key) is None:
            b[key] = torch.empty(*shape, dtype=bf, device=x.device)
    if layers and b.get("u") is None:
        b["u"] = torch.empty(M, layers[0]["Wg"].shape[0], dtype=bf, device=x.device)
    for L in layers:
        qwen3_layer(x, table, L, Hq, Hkv, dh, logsig, eps, bufs=b)
    return x


def gated_layer(X, W1, b1, w2, b2, doc_begin, doc_end, K, Wqkv, Hq, Hkv, dh, gain, temperature,
                bufs: dict | None = None):
    """One gated layer: score -> select -> gather -> QKV -> key-bias
    attention, five library calls on the current stream.  The gate counts
    the select's first radix pass into the select workspace.  ``bufs`` may
    hold preallocated outputs (scores, idx, Xk, logsig, qkv, out) and the
    workspace (select_ws)."""
    b = bufs or {}
    ws = b.get("select_ws")
    if ws is None:
        ws = _default_workspace(X.device)
    s = tg_gate_score(X, W1, b1, w2, b2, out=b.get("scores"), select_ws=ws, doc_begin=doc_begin,
                      doc_end=doc_end)
    idx = tg_select_topk(s, doc_begin, doc_end, K, out=b.get("idx"), workspace=ws)
    Xk, ls = tg_gather_rows(X, idx, s, out=b.get("Xk"), logsig_out=b.get("logsig"))
    qkv = tg_qkv_proj(Xk, Wqkv, Hq, Hkv, dh, out=b.get("qkv"))
    O = tg_keybias_attn(qkv, Hq, Hkv, dh, ls, gain, temperature, out=b.get("out"))
    return {"scores": s, "idx": idx, "Xk": Xk, "logsig": ls, "qkv": qkv, "O": O}


def pruned_stack(x, layers, Hq, Hkv, dh, logsig, eps: float = 1e-6, bufs: dict | None = None):
    """x (fp32 [M][d], updated in place) <- x + attn(qkv(RMSNorm(x))) per
    layer; ``layers`` holds dicts with Wqkv (bf16), gamma, gain, temperature.
    logsig None runs the layers without the bias (full prefill)."""
    M, d = x.shape
    b = bufs or {}
    xn = b.get("xn") if b.get("xn") is not None else torch.empty(M, d, dtype=torch.bfloat16, device=x.device)
    qkv = b.get("qkv") if b.get("qkv") is not None else \
        torch.empty(M, (Hq + 2 * Hkv) * dh, dtype=torch.bfloat16, device=x.device)
    for L in layers:
        tg_rmsnorm(x, L["gamma"], eps, out=xn)
        tg_qkv_proj(xn, L["Wqkv"], Hq, Hkv, dh, out=qkv)
        tg_keybias_attn(qkv, Hq, Hkv, dh, logsig, L["gain"], L["temperature"], residual=x)
    return x


def bias_backward(qkv, O, lse, dO, Hq, Hkv, dh, logsig, gain, temperature,
                  bufs: dict | None = None):
    """The gradient path from the attention output back to the scorer, three
    library calls on the current stream: D = dO . O, dL/db, then dL/dlogsig,
    dL/dgain and dL/dscore.  ``O`` and ``lse`` come from tg_keybias_attn_lse.
    ``bufs`` may hold preallocated outputs (delta, dbias, dlogsig, dgain, dscore)."""
    b = bufs or {}
    delta = tg_attn_bwd_delta(dO, O, Hq, dh, out=b.get("delta"))
    dbias = tg_keybias_attn_bias_grad(qkv, dO, Hq, Hkv, dh, logsig, gain, temperature, lse, delta,
                                      out=b.get("dbias"))
    dls, dg, ds = tg_bias_grad_reduce(dbias, logsig, gain, dlogsig=b.get("dlogsig"),
                                      dgain=b.get("dgain"), dscore=b.get("dscore"))
    return {"delta": delta, "dbias": dbias, "dlogsig": dls, "dgain": dg, "dscore": ds}
