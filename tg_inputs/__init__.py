"""Seeded synthetic inputs for the gated-prefill path.

This module only draws random numbers and stores them in the formats the
kernels and the fp64 oracle both read (fp32 arrays, and bf16 as uint16 bit
patterns rounded to nearest-even).  It holds none of the method's
arithmetic: no scoring, selection, projection or attention happens here.

Workload shapes follow the pages' Qwen3-1.7B setting (TokenGate on one GPU,
batch 1, a long document followed by a short question; the gate sits at a
layer L and the layers above see only the kept tokens).  The pages publish
no tensors, so every value is drawn here:

* residual rows x_i ~ N(0, 1)
* weights ~ N(0, 1/fan_in) (W1 of the gate MLP, w2, the packed QKV weight)
* per-head gains g_h ~ U(0.5, 1.5), temperature t = 1.1
* RMSNorm weight gamma ~ U(0.9, 1.1)
* gate biases b1, b2 are zero unless ``gate_biases=True``

Each tensor has its own stream ``(seed, stream id)`` so adding a tensor never
changes another one.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass
from fractions import Fraction

import numpy as np

__all__ = [
    "Workload", "WORKLOADS", "kept_count", "f32_to_bf16_bits",
    "residual", "gate_params", "qkv_weight", "attn_params", "rms_gamma", "qwen3_layer_params",
    "random_scores", "random_qkv", "random_logsig", "random_dout", "adversarial_scores",
    "deltanet_inputs",
    "DELTANET_SHAPE",
]

# stream ids: one per tensor kind, so that draws never overlap
_S_RESIDUAL, _S_W1, _S_B1, _S_W2, _S_B2, _S_WQKV, _S_GAIN, _S_GAMMA = range(8)
_S_SCORES, _S_QKV, _S_LOGSIG, _S_ADV, _S_DOUT = 20, 21, 22, 23, 24
# the other weights of a full (Qwen3-shaped) decoder layer
_S_QK_GAMMA, _S_WO, _S_MLP_GAMMA, _S_WG, _S_WU, _S_WD = 30, 31, 32, 33, 34, 35
_S_DN = 40  # Gated-DeltaNet layer inputs


@dataclass(frozen=True)
class Workload:
    """One synthetic prompt: a document span [doc_begin, doc_end) followed
    by a question that is never pruned, plus the model shapes around the
    gate layer."""

    name: str
    N: int                      # tokens in the prompt
    doc_begin: int
    doc_end: int
    d: int                      # d_model
    Hg: int                     # gate MLP hidden width
    Hq: int                     # query heads
    Hkv: int                    # key/value heads (GQA groups)
    dh: int                     # head dim
    dtype: str                  # "f32" or "bf16"
    seed: int
    budgets: tuple = (Fraction(1, 10),)   # fraction of the document kept
    layers: int = 1             # layers above the gate that run pruned
    gate_layer: int = 0         # index L of the gate layer (context only)
    temperature: float = 1.1
    K_fixed: int | None = None  # overrides the budget with an exact count

    @property
    def D(self) -> int:
        return self.doc_end - self.doc_begin

    def Ks(self) -> list[int]:
        if self.K_fixed is not None:
            return [self.K_fixed]
        return [kept_count(self.D, b) for b in self.budgets]

    def M(self, K: int) -> int:
        return self.N - self.D + K

    @property
    def qkv_cols(self) -> int:
        return (self.Hq + 2 * self.Hkv) * self.dh


def kept_count(D: int, budget) -> int:
    """Kept document tokens for a budget fraction: floor(D * budget) in exact
    rational arithmetic (no float rounding of the fraction)."""
    b = Fraction(budget)
    return (D * b.numerator) // b.denominator


WORKLOADS: dict[str, Workload] = {w.name: w for w in [
    # the small case: every op on fp32, oracle finishes in well under a second
    Workload("tiny_f32_n512", N=512, doc_begin=0, doc_end=448, d=256, Hg=64,
             Hq=4, Hkv=2, dh=64, dtype="f32", seed=0, K_fixed=128),
    # one gated layer at 16k tokens, 10% of the document kept
    Workload("qwen3_1p7b_n16k_keep10", N=16384, doc_begin=0, doc_end=16128,
             d=2048, Hg=256, Hq=16, Hkv=8, dh=128, dtype="bf16", seed=1,
             budgets=(Fraction(10, 100),)),
    # one input at 32k, four budgets swept over the same scores
    Workload("qwen3_1p7b_n32k_sweep", N=32768, doc_begin=0, doc_end=32512,
             d=2048, Hg=256, Hq=16, Hkv=8, dh=128, dtype="bf16", seed=2,
             budgets=(Fraction(5, 100), Fraction(10, 100), Fraction(25, 100),
                      Fraction(50, 100))),
    # long context, 6.25% kept
    Workload("qwen3_1p7b_n128k_keep6p25", N=131072, doc_begin=0,
             doc_end=130816, d=2048, Hg=256, Hq=16, Hkv=8, dh=128,
             dtype="bf16", seed=3, budgets=(Fraction(625, 10000),)),
    # 20 pruned layers above gate layer 8 at 64k, 10% kept
    Workload("qwen3_1p7b_n64k_stack20_keep10", N=65536, doc_begin=0,
             doc_end=65280, d=2048, Hg=256, Hq=16, Hkv=8, dh=128,
             dtype="bf16", seed=4, budgets=(Fraction(10, 100),), layers=20,
             gate_layer=8),
]}


def _rng(seed: int, stream: int, sub: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64([seed, stream, sub]))


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (round to nearest, ties to even) and return
    the 16-bit patterns.  Inputs are finite by construction."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32)
    # finite inputs: the largest finite pattern plus 0x8000 still fits 32 bits
    r = (u >> 16) & np.uint32(1)
    r += np.uint32(0x7FFF)
    r += u
    r >>= np.uint32(16)
    return r.astype(np.uint16)


def _normal(seed: int, stream: int, sub: int, shape, std: float, dtype: str,
            chunk_rows: int = 4096) -> np.ndarray:
    """N(0, std^2) as fp32, or as bf16 bits.  Row chunk c is drawn from its
    own stream (seed, stream, sub, c), so chunks fill in parallel and the
    result does not depend on the thread count."""
    shape = tuple(shape)
    rows = shape[0]
    rest = int(np.prod(shape[1:])) if len(shape) > 1 else 1
    out = np.empty((rows, rest), dtype=np.uint16 if dtype == "bf16" else np.float32)

    def fill(c: int) -> None:
        r0, r1 = c * chunk_rows, min(rows, (c + 1) * chunk_rows)
        g = np.random.Generator(np.random.PCG64([seed, stream, sub, c]))
        v = g.standard_normal((r1 - r0, rest), dtype=np.float32)
        if std != 1.0:
            v *= np.float32(std)
        out[r0:r1] = f32_to_bf16_bits(v) if dtype == "bf16" else v

    n_chunks = (rows + chunk_rows - 1) // chunk_rows
    if n_chunks == 1:
        fill(0)
    else:
        with ThreadPoolExecutor(max_workers=min(n_chunks, os.cpu_count() or 1)) as ex:
            list(ex.map(fill, range(n_chunks)))
    return out.reshape(shape)


def residual(w: Workload) -> np.ndarray:
    """Post-attention residual at the gate layer, [N][d]."""
    return _normal(w.seed, _S_RESIDUAL, 0, (w.N, w.d), 1.0, w.dtype)


def gate_params(w: Workload, gate_biases: bool = False) -> dict:
    """Gate MLP d -> Hg -> 1: W1 [Hg][d] (dtype of the residual), b1 [Hg]
    fp32, w2 [Hg] fp32, b2 scalar."""
    W1 = _normal(w.seed, _S_W1, 0, (w.Hg, w.d), 1.0 / np.sqrt(w.d), w.dtype)
    if gate_biases:
        b1 = _rng(w.seed, _S_B1).standard_normal(w.Hg, dtype=np.float32) * np.float32(1 / np.sqrt(w.d))
        b2 = float(_rng(w.seed, _S_B2).standard_normal(dtype=np.float32) * np.float32(1 / np.sqrt(w.Hg)))
    else:
        b1 = np.zeros(w.Hg, dtype=np.float32)
        b2 = 0.0
    w2 = _rng(w.seed, _S_W2).standard_normal(w.Hg, dtype=np.float32) * np.float32(1 / np.sqrt(w.Hg))
    return {"W1": W1, "b1": b1.astype(np.float32), "w2": w2.astype(np.float32), "b2": np.float32(b2).item()}


def qkv_weight(w: Workload, layer: int = 0) -> np.ndarray:
    """Packed projection weight [(Hq + 2 Hkv) dh][d] (nn.Linear out x in):
    rows [0, Hq dh) give q, the next Hkv dh give k, the last Hkv dh give v."""
    return _normal(w.seed, _S_WQKV, layer, (w.qkv_cols, w.d), 1.0 / np.sqrt(w.d), w.dtype)


def attn_params(w: Workload, layer: int = 0) -> dict:
    """Per query head gain g [Hq] ~ U(0.5, 1.5) and the temperature t."""
    g = _rng(w.seed, _S_GAIN, layer).uniform(0.5, 1.5, size=w.Hq).astype(np.float32)
    return {"gain": g, "temperature": float(np.float32(w.temperature))}


def rms_gamma(w: Workload, layer: int = 0) -> np.ndarray:
    return _rng(w.seed, _S_GAMMA, layer).uniform(0.9, 1.1, size=w.d).astype(np.float32)


def qwen3_layer_params(w: Workload, layer: int = 0, ffn: int = 6144) -> dict:
    """All weights of one Qwen3-shaped decoder layer above the gate (the
    pages' layers above L are the base model's layers; Qwen3-1.7B has an
    MLP width of 6144 and a rotary base of 1e6):
      gamma_attn, gamma_mlp [d] ~ U(0.9, 1.1); Wqkv as qkv_weight;
      gamma_q, gamma_k [dh] ~ U(0.9, 1.1); gain, temperature as attn_params;
      Wo [d][Hq dh] ~ N(0, 1/(Hq dh)); Wg, Wu [ffn][d] ~ N(0, 1/d);
      Wd [d][ffn] ~ N(0, 1/ffn); matrices in the workload's dtype."""
    qg = _rng(w.seed, _S_QK_GAMMA, layer)
    return {
        "gamma_attn": rms_gamma(w, layer), "Wqkv": qkv_weight(w, layer),
        "gamma_q": qg.uniform(0.9, 1.1, size=w.dh).astype(np.float32),
        "gamma_k": qg.uniform(0.9, 1.1, size=w.dh).astype(np.float32),
        "rope_base": 1e6, **attn_params(w, layer),
        "Wo": _normal(w.seed, _S_WO, layer, (w.d, w.Hq * w.dh), 1.0 / np.sqrt(w.Hq * w.dh),
                      w.dtype),
        "gamma_mlp": _rng(w.seed, _S_MLP_GAMMA, layer).uniform(0.9, 1.1, size=w.d)
                       .astype(np.float32),
        "Wg": _normal(w.seed, _S_WG, layer, (ffn, w.d), 1.0 / np.sqrt(w.d), w.dtype),
        "Wu": _normal(w.seed, _S_WU, layer, (ffn, w.d), 1.0 / np.sqrt(w.d), w.dtype),
        "Wd": _normal(w.seed, _S_WD, layer, (w.d, ffn), 1.0 / np.sqrt(ffn), w.dtype),
    }


def random_scores(n: int, seed: int, scale: float = 1.0) -> np.ndarray:
    """Continuous fp32 gate scores, for testing selection on its own."""
    return (_rng(seed, _S_SCORES).standard_normal(n, dtype=np.float32) * np.float32(scale))


def random_qkv(M: int, Hq: int, Hkv: int, dh: int, seed: int, dtype: str = "bf16",
               std: float = 1.0) -> np.ndarray:
    """Packed [M][(Hq + 2 Hkv) dh] q|k|v rows, for testing attention on its own."""
    return _normal(seed, _S_QKV, 0, (M, (Hq + 2 * Hkv) * dh), std, dtype)


def random_dout(M: int, Hq: int, dh: int, seed: int, dtype: str = "bf16",
                std: float = 1.0) -> np.ndarray:
    """An upstream gradient dL/dO [M][Hq dh] for the attention output."""
    return _normal(seed, _S_DOUT, 0, (M, Hq * dh), std, dtype)


def random_logsig(M: int, seed: int) -> np.ndarray:
    """Non-positive per-key bias inputs (the range of a log-sigmoid), drawn as
    minus an exponential variate with mean 0.7."""
    return (-_rng(seed, _S_LOGSIG).exponential(0.7, size=M)).astype(np.float32)


def adversarial_scores(kind: str, n: int, seed: int = 0) -> np.ndarray:
    """Score vectors that stress a selector: ties, signed zeros, infinities,
    denormals and few distinct values."""
    rng = _rng(seed, _S_ADV, ADVERSARIAL_KINDS.index(kind) if kind in ADVERSARIAL_KINDS else 99)
    f32 = np.float32
    if kind == "all_equal":
        return np.full(n, f32(0.25), dtype=np.float32)
    if kind == "quantised":          # 5 distinct values, many ties
        return (rng.integers(-2, 3, size=n).astype(np.float32) * f32(0.5))
    if kind == "signed_zero":        # only +0.0 and -0.0
        z = np.zeros(n, dtype=np.float32)
        z[rng.random(n) < 0.5] = f32(-0.0)
        return z
    if kind == "infinities":         # finite values mixed with +-inf
        v = rng.standard_normal(n, dtype=np.float32)
        m = rng.random(n)
        v[m < 0.05] = np.inf
        v[(m >= 0.05) & (m < 0.10)] = -np.inf
        return v
    if kind == "denormal":           # subnormals of both signs and zeros
        bits = rng.integers(0, 1 << 23, size=n, dtype=np.uint32)
        bits[rng.random(n) < 0.5] |= np.uint32(0x80000000)
        return bits.view(np.float32)
    if kind == "same_top_bits":      # all keys share their top 21 bits
        base = np.uint32(0x3F800000)
        bits = base + rng.integers(0, 1 << 10, size=n, dtype=np.uint32)
        return bits.view(np.float32)
    if kind == "descending":
        return np.linspace(1.0, -1.0, n, dtype=np.float32)
    if kind == "ascending":
        return np.linspace(-1.0, 1.0, n, dtype=np.float32)
    raise ValueError(kind)


ADVERSARIAL_KINDS = ("all_equal", "quantised", "signed_zero", "infinities", "denormal",
                     "same_top_bits", "descending", "ascending")


# Head shape of a Gated-DeltaNet layer: the pages name the hybrid model but
# give none of its sizes; 16 heads with dk = dv = 128 are taken.
DELTANET_SHAPE = {"H": 16, "dk": 128, "dv": 128}


def deltanet_inputs(T: int, H: int, dk: int, dv: int, seed: int, dtype: str = "f32") -> dict:
    """Inputs of a Gated-DeltaNet layer's recurrence over T tokens: q ~
    N(0, 1/dk), k uniform on the unit sphere (a normal draw scaled to unit
    length), v ~ N(0, 1), decay alpha ~ U(0.9, 1), write strength beta ~
    U(0, 1); q, k, v as fp32 or bf16 bits ([T][H][d]), alpha and beta fp32
    [T][H].  For bf16 the unit keys are rounded after scaling."""
    g = _rng(seed, _S_DN)
    q = g.standard_normal((T, H, dk), dtype=np.float32) * np.float32(1 / np.sqrt(dk))
    k = g.standard_normal((T, H, dk), dtype=np.float32)
    k /= np.linalg.norm(k, axis=2, keepdims=True)
    v = g.standard_normal((T, H, dv), dtype=np.float32)
    alpha = g.uniform(0.9, 1.0, (T, H)).astype(np.float32)
    beta = g.uniform(0.0, 1.0, (T, H)).astype(np.float32)
    if dtype == "bf16":
        q, k, v = f32_to_bf16_bits(q), f32_to_bf16_bits(k), f32_to_bf16_bits(v)
    return {"q": q, "k": k, "v": v, "alpha": alpha, "beta": beta}
