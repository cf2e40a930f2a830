"""Plain, slow fp64 definitions of every step of TokenGate's gated prefill.

TEST INFRASTRUCTURE ONLY -- used by the tests, the smoke check and the
CPU-baseline timing; never by the product path.

Sources (five web pages about one paper, "TokenGate: Adapting LLMs for Fast
and Memory-Efficient Prefill with Learned Token Pruning"):

[RU] telohudelo.online, "TokenGate ускоряет prefill в LLM до 11,3 раза за
     счёт обучаемого отсева", section "Механизм token-gated attention".
[TH] ai4bro.com, "Stanford เปิดตัว TokenGate เร่งความเร็ว Prefill ใน LLM
     สูงสุด 11.3 เท่า", section "กลไกการทำงานของ Learned Token Pruning"
     (three phases; token-gated attention; per-head gain and temperature).
[DE] spke.com, "TokenGate – Token-Gated Attention macht das Vollfüllen von
     langen Kontexten bis zu 11,3-mal schneller", sections "Wie hat TokenGate
     das Pruning von Tokens verstanden?" and "Was ist token-gated Attention?".
[IT] ai.info, "TokenGate riporta un prefill fino a 11,3 volte più veloce sui
     contesti lunghi", section "TokenGate impara quali token mantenere".

What the pages state: below gate layer L every token is processed; at L a
small MLP scores each token from its post-attention residual and a top-K
selector keeps the best-scoring document tokens ([DE], [TH] phase 2); the
question part of the prompt is never pruned ([DE], [TH] phase 3); only the
kept rows go up ([IT]); the layers above build no KV for pruned tokens
([DE]); each kept token's score becomes a bias on the attention logits above
the gate, MoE-router style, with a learnable per-head gain and a learnable
temperature ([TH], [DE] "Was ist token-gated Attention?", [RU]).

What they leave open, and the reading taken here (one line each):

* logit form: l_ij = t * (q_i . k_j) / sqrt(dh) + g_h * log(sigmoid(s_j)),
  causal on original positions, GQA with kv head = h // (Hq / Hkv).
* gate MLP: s = w2 . GELU(W1 x + b1) + b2, GELU the exact erf form.
* selection order: fp32 score bits mapped to a total order (-0 < +0, ties go
  to the lower index); K counts document tokens only; output ascending.
* every kept key gets the bias, query tokens included (the MLP scores every
  token).
* a pruned layer of the stack: x <- x + attn(qkv(RMSNorm(x))) (no RoPE, no
  o-proj, no MLP).
* a full decoder layer above the gate (the pages say only that the layers
  above L process the kept tokens; their internals are the base model's):
  Qwen3 order -- RMSNorm, q|k|v, per-head RMSNorm of q and k, rotary
  embedding at the kept tokens' ORIGINAL prompt positions (rotate-half
  pairing, theta_c = base^(-2c/dh)), key-bias attention, o-projection,
  residual add, RMSNorm, SwiGLU MLP, residual add.
* the gradient the bias carries back to the scorer ([DE] "Was ist
  token-gated Attention?": the bias gives the gradient a way back to the
  scorer; [TH] the same, MoE-router style): the plain chain rule through
  the logit form above, with the scorer's output s_j entering only through
  ls_j = log(sigmoid(s_j)) of the kept keys.

Everything runs in float64 on values widened exactly from their stored
formats.  numpy's matmul, sort and erf are used as library primitives; there
is no blocking or fusion beyond processing independent query rows in chunks.
"""
from __future__ import annotations

import math

import numpy as np
from scipy.special import erf as _erf
from scipy.special import expit as _expit

__all__ = [
    "bf16_bits_to_f64", "f32_to_f64", "gelu_erf", "gate_score",
    "score_key", "select_topk", "select_topk_by_rank", "SelectNaNError",
    "logsigmoid", "gather_rows", "rmsnorm", "linear", "qkv_proj", "split_qkv",
    "keybias_attn", "gated_layer", "pruned_stack",
    "keybias_attn_lse", "attn_delta", "keybias_attn_bias_grad", "bias_grad_reduce",
    "qk_rmsnorm", "rope_angles", "rope", "swiglu_hidden", "swiglu_mlp", "qwen3_pruned_layer",
    "gated_delta_rule", "gated_delta_rule_chunked",
]


# --------------------------------------------------------------------------
# storage formats -> float64 (exact widening)
# --------------------------------------------------------------------------
def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 is the top half of an fp32 pattern; widening is exact."""
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def f32_to_f64(a: np.ndarray) -> np.ndarray:
    return np.asarray(a, dtype=np.float32).astype(np.float64)


def _widen(a: np.ndarray) -> np.ndarray:
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return bf16_bits_to_f64(a)
    return a.astype(np.float64)


# --------------------------------------------------------------------------
# phase 2a: the gate MLP  ([DE] "Wie hat TokenGate ...", Gate-Modul; [TH] phase 2)
# --------------------------------------------------------------------------
def gelu_erf(z: np.ndarray) -> np.ndarray:
    """GELU(z) = z * Phi(z) = 0.5 z (1 + erf(z / sqrt 2))."""
    return 0.5 * z * (1.0 + _erf(z / math.sqrt(2.0)))


def gate_score(X, W1, b1, w2, b2) -> np.ndarray:
    """Score of every token from its residual row at the gate layer:
    z = W1 x_i + b1 ; h = GELU(z) ; s_i = w2 . h + b2.

    X [N][d], W1 [Hg][d] (bf16 bits or fp32), b1 [Hg] or None, w2 [Hg], b2.
    Returns s [N] in float64."""
    x = _widen(X)
    W = _widen(W1)
    z = x @ W.T
    if b1 is not None:
        z = z + _widen(b1)[None, :]
    h = gelu_erf(z)
    return h @ _widen(w2) + float(b2)


# --------------------------------------------------------------------------
# phase 2b: top-K over the document span, question never pruned
#   ([DE] "Wie hat TokenGate ..."; [TH] phase 2 and 3; [IT])
# --------------------------------------------------------------------------
class SelectNaNError(ValueError):
    """A NaN score inside the document span has no place in the order."""


def score_key(scores_f32: np.ndarray) -> np.ndarray:
    """Map fp32 score bits to uint32 keys whose unsigned order is the total
    order used for selection: negative patterns are bit-inverted, the rest
    get the sign bit set.  So -inf < ... < -0.0 < +0.0 < ... < +inf."""
    u = np.ascontiguousarray(scores_f32, dtype=np.float32).view(np.uint32)
    neg = (u & np.uint32(0x80000000)) != 0
    return np.where(neg, ~u, u | np.uint32(0x80000000)).astype(np.uint32)


def select_topk(scores_f32, doc_begin: int, doc_end: int, K: int) -> np.ndarray:
    """Indices kept at the gate: every token outside [doc_begin, doc_end)
    plus the K document tokens ranked first by (key descending, index
    ascending); returned ascending as int64.  Raises SelectNaNError when a
    document score is NaN."""
    s = np.asarray(scores_f32, dtype=np.float32)
    N = s.shape[0]
    if not (0 <= doc_begin <= doc_end <= N) or not (0 <= K <= doc_end - doc_begin):
        raise ValueError("bad span or K")
    doc = s[doc_begin:doc_end]
    if np.isnan(doc).any():
        raise SelectNaNError("NaN score in the document span")
    keys = score_key(doc).astype(np.int64)
    pos = np.arange(doc_begin, doc_end, dtype=np.int64)
    # lexsort: last key is primary -> sort by key descending, then index ascending
    order = np.lexsort((pos, -keys))
    kept_doc = np.sort(pos[order[:K]])
    outside = np.concatenate([np.arange(0, doc_begin), np.arange(doc_end, N)]).astype(np.int64)
    return np.sort(np.concatenate([outside, kept_doc]))


def select_topk_by_rank(scores_f32, doc_begin: int, doc_end: int, K: int) -> np.ndarray:
    """Second, independent definition for small inputs (pure Python): a
    document token j is kept iff fewer than K document tokens beat it, where
    i beats j when key_i > key_j, or key_i == key_j and i < j."""
    s = [float(v) for v in np.asarray(scores_f32, dtype=np.float32)]
    keys = [int(k) for k in score_key(np.asarray(scores_f32, dtype=np.float32))]
    N = len(s)
    out = []
    for j in range(N):
        if j < doc_begin or j >= doc_end:
            out.append(j)
            continue
        if math.isnan(s[j]):
            raise SelectNaNError("NaN score in the document span")
        beats = 0
        for i in range(doc_begin, doc_end):
            if keys[i] > keys[j] or (keys[i] == keys[j] and i < j):
                beats += 1
        if beats < K:
            out.append(j)
    return np.asarray(out, dtype=np.int64)


# --------------------------------------------------------------------------
# phase 3 entry: gather the kept rows and their bias input
#   ([IT] only the kept representations go up; [DE] "Was ist token-gated
#   Attention?": the kept token's score becomes the bias)
# --------------------------------------------------------------------------
def logsigmoid(s) -> np.ndarray:
    """log(sigmoid(s)) = min(s, 0) - log1p(exp(-|s|)), in float64."""
    s = np.asarray(s, dtype=np.float64)
    return np.minimum(s, 0.0) - np.log1p(np.exp(-np.abs(s)))


def gather_rows(X, idx, scores_f32=None):
    """Y[m] = X[idx[m]] (an exact copy, same storage format) and, when scores
    are given, ls[m] = log(sigmoid(s[idx[m]])) in float64."""
    X = np.asarray(X)
    idx = np.asarray(idx, dtype=np.int64)
    Y = X[idx].copy()
    ls = None
    if scores_f32 is not None:
        ls = logsigmoid(np.asarray(scores_f32, dtype=np.float32).astype(np.float64)[idx])
    return Y, ls


# --------------------------------------------------------------------------
# phase 3: the pruned layers ([DE] "Prune-Front-Behandlung"; [TH] phase 3)
# --------------------------------------------------------------------------
def rmsnorm(x, gamma, eps: float) -> np.ndarray:
    """RMSNorm(x) = x * gamma / sqrt(mean(x^2) + eps), row-wise."""
    x = _widen(x)
    ms = np.mean(x * x, axis=1, keepdims=True)
    return x * _widen(gamma)[None, :] / np.sqrt(ms + float(eps))


def linear(X, W) -> np.ndarray:
    """X W^T with W [out][in] (nn.Linear layout, no bias)."""
    return _widen(X) @ _widen(W).T


def qkv_proj(X, Wqkv) -> np.ndarray:
    """QKV = X Wqkv^T with Wqkv [(Hq + 2 Hkv) dh][d] (nn.Linear layout)."""
    return linear(X, Wqkv)


def split_qkv(QKV, Hq: int, Hkv: int, dh: int):
    """Column blocks of the packed rows: q heads, then k heads, then v heads."""
    q = QKV[:, : Hq * dh]
    k = QKV[:, Hq * dh: (Hq + Hkv) * dh]
    v = QKV[:, (Hq + Hkv) * dh: (Hq + 2 * Hkv) * dh]
    return q, k, v


def keybias_attn(QKV, Hq: int, Hkv: int, dh: int, logsig_kept, gain, temperature: float,
                 rows=None, return_rowsum: bool = False, chunk: int = 512):
    """Token-gated causal attention over the kept rows.

    For query head h (kv head h // (Hq / Hkv)) and kept row i:
        l_ij = t * (q_i . k_j) / sqrt(dh) + g_h * ls_j   for j <= i
        o_i  = sum_j softmax_j(l_ij) v_j
    ``logsig_kept`` None drops the bias term (full prefill).  The causal
    mask on compacted rows equals the mask on original positions because the
    kept indices ascend.  ``rows`` (optional) restricts the output to those
    query rows; the result is then [len(rows)][Hq dh].
    Returns O (float64), and the largest |row sum of p - 1| if asked."""
    Q = _widen(QKV)
    M = Q.shape[0]
    assert Hq % Hkv == 0, "GQA needs Hq divisible by Hkv"
    G = Hq // Hkv
    q_all, k_all, v_all = split_qkv(Q, Hq, Hkv, dh)
    ls = None if logsig_kept is None else np.asarray(logsig_kept, dtype=np.float64)
    g = np.asarray(gain, dtype=np.float64)
    t = float(temperature)
    rows = np.arange(M, dtype=np.int64) if rows is None else np.asarray(rows, dtype=np.int64)
    O = np.zeros((rows.shape[0], Hq * dh), dtype=np.float64)
    worst_rowsum = 0.0
    for h in range(Hq):
        hk = h // G
        q = q_all[:, h * dh:(h + 1) * dh]
        k = k_all[:, hk * dh:(hk + 1) * dh]
        v = v_all[:, hk * dh:(hk + 1) * dh]
        for c0 in range(0, rows.shape[0], chunk):
            r = rows[c0:c0 + chunk]
            jmax = int(r.max()) + 1
            logits = t * (q[r] @ k[:jmax].T) / math.sqrt(dh)
            if ls is not None:
                logits = logits + g[h] * ls[None, :jmax]
            causal = np.arange(jmax)[None, :] <= r[:, None]
            logits = np.where(causal, logits, -np.inf)
            mx = logits.max(axis=1, keepdims=True)
            p = np.exp(logits - mx)
            p = p / p.sum(axis=1, keepdims=True)
            if return_rowsum:
                worst_rowsum = max(worst_rowsum, float(np.abs(p.sum(axis=1) - 1.0).max()))
            O[c0:c0 + chunk, h * dh:(h + 1) * dh] = p @ v[:jmax]
    if return_rowsum:
        return O, worst_rowsum
    return O


def gated_layer(X, W1, b1, w2, b2, doc_begin, doc_end, K, Wqkv, Hq, Hkv, dh, gain,
                temperature, scores_f32=None):
    """One gated layer end to end: score, select, gather, project, attend.

    Selection is decided on fp32 scores (the format the selector reads); by
    default the oracle's own scores rounded to fp32."""
    s = gate_score(X, W1, b1, w2, b2)
    s32 = s.astype(np.float32) if scores_f32 is None else np.asarray(scores_f32, np.float32)
    idx = select_topk(s32, doc_begin, doc_end, K)
    Xk, ls = gather_rows(X, idx, s32)
    QKV = qkv_proj(Xk, Wqkv)
    O = keybias_attn(QKV, Hq, Hkv, dh, ls, gain, temperature)
    return {"scores": s, "idx": idx, "Xk": Xk, "logsig": ls, "QKV": QKV, "O": O}


def pruned_stack(x0, layers, Hq, Hkv, dh, logsig_kept, eps: float = 1e-6):
    """The layers above the gate on the kept rows:
    x <- x + keybias_attn(qkv_proj(RMSNorm(x))) for each layer.
    ``layers`` is a list of dicts with Wqkv, gamma, gain, temperature.
    ``logsig_kept`` None runs the same layers as full prefill (no bias)."""
    x = _widen(x0)
    assert x.shape[1] == Hq * dh, "the residual add needs Hq * dh == d_model"
    for L in layers:
        xn = rmsnorm(x, L["gamma"], eps)
        qkv = qkv_proj(xn, L["Wqkv"])
        x = x + keybias_attn(qkv, Hq, Hkv, dh, logsig_kept, L["gain"], L["temperature"])
    return x


# --------------------------------------------------------------------------
# the gradient path to the scorer ([DE] "Was ist token-gated Attention?":
# the kept tokens' scores become a bias on the attention logits, which gives
# the gradient a way back to the scorer; [TH] token-gated attention, the
# MoE-router device; [RU] "Механизм token-gated attention")
#
# With b_hj = g_h ls_j the bias of key j in head h, l_ij = t q_i.k_j/sqrt(dh)
# + b_hj, P = softmax_j(l), o_i = sum_j P_ij v_j and an upstream gradient
# dO, the chain rule gives
#   dP_ij = dO_i . v_j,   D_i = sum_j P_ij dP_ij,   dl_ij = P_ij (dP_ij - D_i)
#   dL/db_hj = sum_{i >= j} dl_ij      (b_hj enters every row i >= j)
#   dL/dls_j = sum_h g_h dL/db_hj,     dL/dg_h = sum_j ls_j dL/db_hj
#   dL/ds_j  = dL/dls_j * sigmoid(-s_j)  (d log sigmoid(s) / ds)
# --------------------------------------------------------------------------
def _head_logits(q, k, r, ls, g_h: float, t: float, dh: int) -> np.ndarray:
    """l_ij for query rows r against keys [0, max(r)], -inf where j > i."""
    jmax = int(r.max()) + 1
    logits = t * (q[r] @ k[:jmax].T) / math.sqrt(dh)
    if ls is not None:
        logits = logits + g_h * ls[None, :jmax]
    causal = np.arange(jmax)[None, :] <= r[:, None]
    return np.where(causal, logits, -np.inf)


def keybias_attn_lse(QKV, Hq: int, Hkv: int, dh: int, logsig_kept, gain, temperature: float,
                     chunk: int = 512, rows_from: int = 0) -> np.ndarray:
    """lse[h][i] = log sum_{j <= i} exp(l_ij), natural log, float64 [Hq][M]:
    the per-row normaliser of the softmax that the backward re-uses.  Rows
    below ``rows_from`` are left at 0 (not computed)."""
    Q = _widen(QKV)
    M = Q.shape[0]
    G = Hq // Hkv
    q_all, k_all, _ = split_qkv(Q, Hq, Hkv, dh)
    ls = None if logsig_kept is None else np.asarray(logsig_kept, dtype=np.float64)
    g = np.asarray(gain, dtype=np.float64)
    lse = np.zeros((Hq, M), dtype=np.float64)
    for h in range(Hq):
        hk = h // G
        q = q_all[:, h * dh:(h + 1) * dh]
        k = k_all[:, hk * dh:(hk + 1) * dh]
        for c0 in range(rows_from, M, chunk):
            r = np.arange(c0, min(M, c0 + chunk))
            logits = _head_logits(q, k, r, ls, g[h], float(temperature), dh)
            mx = logits.max(axis=1, keepdims=True)
            lse[h, r] = mx[:, 0] + np.log(np.exp(logits - mx).sum(axis=1))
    return lse


def attn_delta(dO, O_out, Hq: int, dh: int) -> np.ndarray:
    """D[h][i] = dO_i^h . o_i^h over the dh columns of head h, float64 [Hq][M]
    (equal to sum_j P_ij dP_ij when o is the exact attention output)."""
    a = _widen(dO)
    b = _widen(O_out)
    M = a.shape[0]
    return (a * b).reshape(M, Hq, dh).sum(axis=2).T.copy()


def keybias_attn_bias_grad(QKV, Hq: int, Hkv: int, dh: int, logsig_kept, gain,
                           temperature: float, dO, chunk: int = 256,
                           return_terms: bool = False, keys_from: int = 0):
    """dL/db_hj = sum_{i >= j} P_ij (dP_ij - D_i) for every head h and kept
    key j, float64 [Hq][M], with P recomputed from the logits, dP_ij =
    dO_i . v_j and D_i = sum_j P_ij dP_ij (its definition, not dO_i . o_i).
    ``logsig_kept`` None means b = 0 (the gradient is still defined).

    With ``return_terms`` it also returns two magnitudes per (h, j) that size
    the rounding of a finite-precision evaluation (they are not part of the
    gradient): cond = sum_i P_ij (|dP_ij| + |D_i|), the sum of the absolute
    terms, and oerr = sum_i P_ij sum_c |dO_ic| (|o_ic| + (P |V|)_ic), what a
    relative error in every p and o element feeds into D and on into dL/db.

    ``keys_from`` > 0 evaluates only the keys j >= keys_from: rows i <
    keys_from (which reach no such key) are skipped, and the returned
    columns below keys_from are 0."""
    Q = _widen(QKV)
    dOw = _widen(dO)
    M = Q.shape[0]
    G = Hq // Hkv
    q_all, k_all, v_all = split_qkv(Q, Hq, Hkv, dh)
    ls = None if logsig_kept is None else np.asarray(logsig_kept, dtype=np.float64)
    g = np.asarray(gain, dtype=np.float64)
    dB = np.zeros((Hq, M), dtype=np.float64)
    cond = np.zeros((Hq, M), dtype=np.float64)
    oerr = np.zeros((Hq, M), dtype=np.float64)
    for h in range(Hq):
        hk = h // G
        q = q_all[:, h * dh:(h + 1) * dh]
        k = k_all[:, hk * dh:(hk + 1) * dh]
        v = v_all[:, hk * dh:(hk + 1) * dh]
        do = dOw[:, h * dh:(h + 1) * dh]
        for c0 in range(keys_from, M, chunk):
            r = np.arange(c0, min(M, c0 + chunk))
            logits = _head_logits(q, k, r, ls, g[h], float(temperature), dh)
            jmax = logits.shape[1]
            mx = logits.max(axis=1, keepdims=True)
            p = np.exp(logits - mx)
            p = p / p.sum(axis=1, keepdims=True)
            dp = do[r] @ v[:jmax].T
            D = (p * dp).sum(axis=1, keepdims=True)
            dB[h, :jmax] += (p * (dp - D)).sum(axis=0)
            if return_terms:
                cond[h, :jmax] += (p * (np.abs(dp) + np.abs(D))).sum(axis=0)
                o = p @ v[:jmax]
                w = (np.abs(do[r]) * (np.abs(o) + p @ np.abs(v[:jmax]))).sum(axis=1)
                oerr[h, :jmax] += (p * w[:, None]).sum(axis=0)
    if keys_from > 0:
        dB[:, :keys_from] = 0.0
        cond[:, :keys_from] = 0.0
        oerr[:, :keys_from] = 0.0
    if return_terms:
        return dB, cond, oerr
    return dB


def bias_grad_reduce(dbias, logsig_kept, gain):
    """From dL/db [Hq][M]: dL/dls_j = sum_h g_h dL/db_hj, dL/dg_h = sum_j ls_j
    dL/db_hj, and dL/ds_j = dL/dls_j * sigmoid(-s_j) where ls_j = log
    sigmoid(s_j), so sigmoid(-s_j) = 1 - exp(ls_j) = -expm1(ls_j).  Returns
    (dls [M], dgain [Hq], ds [M]), float64."""
    dB = np.asarray(dbias, dtype=np.float64)
    ls = np.asarray(logsig_kept, dtype=np.float64)
    g = np.asarray(gain, dtype=np.float64)
    dls = g @ dB
    dgain = dB @ ls
    ds = dls * -np.expm1(ls)
    return dls, dgain, ds


# --------------------------------------------------------------------------
# a full decoder layer on the kept rows ([DE] "Prune-Front-Behandlung": the
# layers above L process only the K kept tokens; [IT] only the kept
# representations go up).  The layer's internals are the base model's
# (Qwen3); the one pruning-specific choice is that every kept row keeps its
# original prompt position for the rotary embedding.
# --------------------------------------------------------------------------
def qk_rmsnorm(QKV, Hq: int, Hkv: int, dh: int, gamma_q, gamma_k, eps: float) -> np.ndarray:
    """RMSNorm of every q head and every k head over its own dh columns, with
    weights gamma_q [dh] and gamma_k [dh] shared by all heads of a kind; the
    v columns are returned unchanged.  float64 [M][(Hq + 2 Hkv) dh]."""
    Y = _widen(QKV).copy()
    M = Y.shape[0]
    for first, heads, gamma in ((0, Hq, gamma_q), (Hq, Hkv, gamma_k)):
        blk = Y[:, first * dh:(first + heads) * dh].reshape(M, heads, dh)
        ms = np.mean(blk * blk, axis=2, keepdims=True)
        blk = blk / np.sqrt(ms + float(eps)) * _widen(gamma)[None, None, :]
        Y[:, first * dh:(first + heads) * dh] = blk.reshape(M, heads * dh)
    return Y


def rope_angles(positions, dh: int, base: float):
    """(cos, sin) of positions[m] * theta_c, theta_c = base^(-2c / dh),
    c < dh / 2: float64 [M][dh / 2] each."""
    h2 = dh // 2
    theta = float(base) ** (-2.0 * np.arange(h2, dtype=np.float64) / dh)
    ang = np.asarray(positions, dtype=np.float64)[:, None] * theta[None, :]
    return np.cos(ang), np.sin(ang)


def rope(QKV, Hq: int, Hkv: int, dh: int, positions, base: float) -> np.ndarray:
    """Rotary embedding of the q and k heads: with h2 = dh / 2 and
    theta_c = base^(-2c / dh) for c < h2, row m's pair (x_c, x_{c + h2}) of
    every q and k head is rotated by the angle positions[m] * theta_c:
        x_c'      = x_c cos - x_{c+h2} sin
        x_{c+h2}' = x_{c+h2} cos + x_c sin.
    ``positions`` are the rows' token positions in the original prompt (for
    kept rows: the kept indices).  v unchanged.  float64."""
    Y = _widen(QKV).copy()
    M = Y.shape[0]
    h2 = dh // 2
    cos, sin = rope_angles(positions, dh, base)
    cos, sin = cos[:, None, :], sin[:, None, :]
    heads = Hq + Hkv
    blk = Y[:, :heads * dh].reshape(M, heads, dh)
    lo, hi = blk[:, :, :h2].copy(), blk[:, :, h2:].copy()
    blk[:, :, :h2] = lo * cos - hi * sin
    blk[:, :, h2:] = hi * cos + lo * sin
    Y[:, :heads * dh] = blk.reshape(M, heads * dh)
    return Y


def swiglu_hidden(x, Wg, Wu) -> np.ndarray:
    """silu(x Wg^T) * (x Wu^T) with silu(z) = z * sigmoid(z); Wg, Wu
    [ffn][d] (nn.Linear layout).  float64 [M][ffn]."""
    x = _widen(x)
    g = x @ _widen(Wg).T
    return g * _expit(g) * (x @ _widen(Wu).T)


def swiglu_mlp(x, Wg, Wu, Wd) -> np.ndarray:
    """The SwiGLU MLP: swiglu_hidden(x, Wg, Wu) Wd^T, Wd [d][ffn]."""
    return swiglu_hidden(x, Wg, Wu) @ _widen(Wd).T


def qwen3_pruned_layer(x, positions, L: dict, Hq: int, Hkv: int, dh: int, logsig_kept,
                       eps: float = 1e-6, rows=None) -> np.ndarray:
    """One decoder layer on the kept rows, in Qwen3's order:
        a = RMSNorm(x; gamma_attn);  qkv = a Wqkv^T
        qkv = rope(qk_rmsnorm(qkv; gamma_q, gamma_k), positions; rope_base)
        x = x + keybias_attn(qkv; logsig_kept, gain, temperature) Wo^T
        x = x + swiglu_mlp(RMSNorm(x; gamma_mlp); Wg, Wu, Wd)
    ``L`` holds those weights.  gamma_q None skips the q/k norm, rope_base
    None skips the rotary embedding, Wd None skips the MLP (the reductions
    the pins use).  ``rows`` (optional) restricts the output to those rows
    (every row's keys still enter the attention).  float64 [M or len(rows)][d]."""
    x = _widen(x)
    qkv = qkv_proj(rmsnorm(x, L["gamma_attn"], eps), L["Wqkv"])
    if L.get("gamma_q") is not None:
        qkv = qk_rmsnorm(qkv, Hq, Hkv, dh, L["gamma_q"], L["gamma_k"], eps)
    if L.get("rope_base") is not None:
        qkv = rope(qkv, Hq, Hkv, dh, positions, L["rope_base"])
    o = keybias_attn(qkv, Hq, Hkv, dh, logsig_kept, L["gain"], L["temperature"], rows=rows)
    x = (x if rows is None else x[np.asarray(rows)]) + linear(o, L["Wo"])
    if L.get("Wd") is not None:
        x = x + swiglu_mlp(rmsnorm(x, L["gamma_mlp"], eps), L["Wg"], L["Wu"], L["Wd"])
    return x


# --------------------------------------------------------------------------
# Gated-DeltaNet layers of a hybrid model ([TH] "การใช้งานกับโมเดล
# hybrid-attention"; [DE] "Wird es auf Hybrid-Attention-Modellen
# funktionieren?"; [IT] "I modelli ibridi ampliano le possibilità di
# selezione dei token": the gate can sit in a Gated-DeltaNet layer of a
# hybrid model whose other layers are full attention, and the DeltaNet layers
# above it are pruned too).  The pages give no formula; the layer's
# recurrence is the published gated delta rule, per head, with a state
# S in R^{dv x dk}:
#     S_t = alpha_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T
#     o_t = S_t q_t
# alpha_t in (0, 1] a decay gate, beta_t in [0, 1] the write strength.  A
# pruned DeltaNet layer runs this recurrence over the kept tokens only, in
# their prompt order (a pruned token neither decays nor writes the state).
# --------------------------------------------------------------------------
def gated_delta_rule(q, k, v, alpha, beta, S0=None):
    """The recurrence, token by token (the definition).
    q, k [T][H][dk], v [T][H][dv], alpha, beta [T][H]; S0 [H][dv][dk] or
    None (zeros).  Returns (o [T][H][dv], S_T [H][dv][dk]), float64."""
    q, k, v = _widen(q), _widen(k), _widen(v)
    a, b = np.asarray(alpha, np.float64), np.asarray(beta, np.float64)
    T, H, dk = k.shape
    dv = v.shape[2]
    S = np.zeros((H, dv, dk)) if S0 is None else np.array(S0, dtype=np.float64)
    o = np.zeros((T, H, dv))
    for t in range(T):
        for h in range(H):
            kt = k[t, h]
            # S (I - beta k k^T) = S - beta (S k) k^T
            S[h] = a[t, h] * (S[h] - b[t, h] * np.outer(S[h] @ kt, kt)) + b[t, h] * np.outer(v[t, h], kt)
            o[t, h] = S[h] @ q[t, h]
    return o, S


def gated_delta_rule_chunked(q, k, v, alpha, beta, S0=None, chunk: int = 64):
    """The same recurrence evaluated chunk by chunk.  Within a chunk that
    starts from state S (before its first token), with g_i the cumulative
    product of alpha up to token i of the chunk, the delta-rule errors
    u_i = v_i - alpha_i S_{i-1} k_i satisfy the unit lower-triangular system
        u_i + sum_{j<i} (g_i / g_j) beta_j (k_i . k_j) u_j = v_i - g_i S k_i,
    and then
        o_i = g_i S q_i + sum_{j<=i} (g_i / g_j) beta_j (k_j . q_i) u_j
        S  <- g_C S + sum_j (g_C / g_j) beta_j u_j k_j^T.
    Same arguments and results as gated_delta_rule (float64)."""
    q, k, v = _widen(q), _widen(k), _widen(v)
    a, b = np.asarray(alpha, np.float64), np.asarray(beta, np.float64)
    T, H, dk = k.shape
    dv = v.shape[2]
    S = np.zeros((H, dv, dk)) if S0 is None else np.array(S0, dtype=np.float64)
    o = np.zeros((T, H, dv))
    for c0 in range(0, T, chunk):
        c1 = min(T, c0 + chunk)
        for h in range(H):
            K, Q, V = k[c0:c1, h], q[c0:c1, h], v[c0:c1, h]
            bet = b[c0:c1, h]
            lg = np.cumsum(np.log(a[c0:c1, h]))          # log g_i
            G = np.exp(lg[:, None] - lg[None, :])          # g_i / g_j
            n = c1 - c0
            A = np.tril(G * (K @ K.T) * bet[None, :], -1)  # j < i
            rhs = V - np.exp(lg)[:, None] * (K @ S[h].T)
            U = np.linalg.solve(np.eye(n) + A, rhs)
            P = np.tril(G * (Q @ K.T)) * bet[None, :]      # j <= i
            o[c0:c1, h] = np.exp(lg)[:, None] * (Q @ S[h].T) + P @ U
            wC = np.exp(lg[-1] - lg) * bet                 # (g_C / g_j) beta_j
            S[h] = np.exp(lg[-1]) * S[h] + (U * wC[:, None]).T @ K
    return o, S
