"""The delta rule's bf16 tolerance against a model of where the tensor-core
kernels round (CPU).  The model evaluates the chunked form (chunks of 64) in
fp32 and rounds to bf16 exactly where the kernels hand an operand to the
tensor cores: P, T, -T diag(g) and the product W- built from it, diag(g) Q,
diag(beta g_C / g) K, the state S before each chunk, U, and the output.
Correct bf16 arithmetic of that shape must sit inside the tolerance the GPU
tests use; a planted mistake in the model (a dropped term, a wrong sign, a
missing decay) must not."""
import numpy as np
import pytest

import oracle as O
import tg_inputs as TI
from gpu_helpers import DELTA_MAX_REL, DELTA_MEAN_REL

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _bf(x):
    return O.bf16_bits_to_f64(TI.f32_to_bf16_bits(np.asarray(x, np.float32))).astype(np.float32)


def _model(q, k, v, alpha, beta, plant=None, C=64):
    T, H, d = q.shape
    f32 = np.float32
    o = np.zeros((T, H, d), f32)
    for h in range(H):
        S = np.zeros((d, d), f32)
        for c0 in range(0, T, C):
            n = min(C, T - c0)
            Q, K, V = (np.zeros((C, d), f32) for _ in range(3))
            Q[:n], K[:n], V[:n] = q[c0:c0 + n, h], k[c0:c0 + n, h], v[c0:c0 + n, h]
            la, b = np.zeros(C, f32), np.zeros(C, f32)
            la[:n], b[:n] = np.log(alpha[c0:c0 + n, h]), beta[c0:c0 + n, h]
            lg = np.cumsum(la).astype(f32)
            g = np.exp(lg).astype(f32)
            R = np.exp(lg[:, None] - lg[None, :]).astype(f32)
            A = np.tril(R * b[None, :] * (K @ K.T), -1).astype(f32)
            P = _bf(np.tril(R * b[None, :] * (Q @ K.T), 0 if plant != "strict_P" else -1))
            Tm = np.linalg.inv(np.eye(C, dtype=f32) + A).astype(f32)
            Wn = _bf(_bf(-Tm * g[None, :]) @ K)
            if plant == "sign_W":
                Wn = -Wn
            Qg = _bf(g[:, None] * Q)
            Kp = _bf((b * np.exp(lg[-1] - lg))[:, None] * K)
            Sb = _bf(S)
            U = _bf(_bf(Tm) @ V + Wn @ Sb.T)
            Oc = Qg @ Sb.T + (P @ U if plant != "drop_PU" else 0)
            o[c0:c0 + n, h] = _bf(Oc[:n])
            S = ((g[-1] if plant != "no_decay" else 1.0) * S + U.T @ Kp).astype(f32)
    return o


def _errors(got, ref):
    rms = float(np.sqrt(np.mean(ref * ref)))
    err = np.abs(got - ref)
    return float((err / (np.abs(ref) + rms)).max()), float(err.mean()) / rms


@pytest.fixture(scope="module")
def case():
    T, H = 320, 2
    x = TI.deltanet_inputs(T, H, 128, 128, seed=21, dtype="bf16")
    q, k, v = (O.bf16_bits_to_f64(x[n]) for n in ("q", "k", "v"))
    ref, _ = O.gated_delta_rule(q, k, v, x["alpha"], x["beta"])
    return [a.astype(np.float32) for a in (q, k, v)] + [x["alpha"], x["beta"], ref]


def test_bf16_rounding_model_is_inside_the_tolerance(case):
    q, k, v, a, b, ref = case
    mx, mean = _errors(_model(q, k, v, a, b), ref)
    assert mx <= DELTA_MAX_REL / 1.5, mx
    assert mean <= DELTA_MEAN_REL / 2, mean


@pytest.mark.parametrize("plant", ["sign_W", "drop_PU", "no_decay", "strict_P"])
def test_planted_mistakes_exceed_the_tolerance(case, plant):
    q, k, v, a, b, ref = case
    mx, mean = _errors(_model(q, k, v, a, b, plant=plant), ref)
    assert mx > DELTA_MAX_REL or mean > DELTA_MEAN_REL, (plant, mx, mean)
