"""GPU parity of the gradient path from the attention bias back to the
scorer (the forward's log-sum-exp, D = dO . O, dL/db, and the reduction to
dL/dlogsig, dL/dgain, dL/dscore) against the fp64 oracle, through the C ABI.

Tolerances are derived from the arithmetic, per element, from magnitudes the
oracle returns (``return_terms``):

* dL/db_hj = sum_i P_ij (dP_ij - D_i) on the GPU carries relative errors of
  about 1e-5 in each p (fp32 logits, the forward's fp32 lse, ex2.approx),
  about 1e-6 in each dP (fp32 accumulation of exact bf16 products) and the
  fp32 rounding of the running sums; each is bounded by
  EPS_ARITH * cond_hj, cond = sum_i P_ij (|dP_ij| + |D_i|).
* When D comes from the forward's bf16 output O, each o element is off by
  at most 2^-9 of |o| (the store) plus 2^-9 of (P |V|) (P is rounded to bf16
  before the P V product); the bound uses 2^-8 for both, times oerr =
  sum_i P_ij sum_c |dO_ic| (|o_ic| + (P |V|)_ic).
"""
import numpy as np
import pytest
import torch

import oracle as O
import tg_inputs as TI
from learned_token_pruning_residual_b300 import build as tgbuild
import learned_token_pruning_residual_b300 as tg
from gpu_helpers import f64, to_dev

pytestmark = pytest.mark.gpu

EPS_ARITH = 2e-4          # relative error of p, dP and the sums (fp32 arithmetic)
EPS_O = 2.0 ** -8         # relative error of a bf16 attention output element


@pytest.fixture(scope="module", autouse=True)
def _lib():
    tgbuild.build()
    tg.lib()
    assert tg.tg_get_device_status(raise_on_error=False) == 0


def _status():
    return tg.tg_get_device_status(raise_on_error=False)


def _case(M, Hq=16, Hkv=8, dh=128, bias=True, seed=0, dtype="bf16"):
    QKV = TI.random_qkv(M, Hq, Hkv, dh, seed=seed, dtype=dtype)
    ls = TI.random_logsig(M, seed=seed) if bias else None
    g = TI._rng(seed, 30).uniform(0.5, 1.5, Hq).astype(np.float32)
    dO = TI.random_dout(M, Hq, dh, seed=seed, dtype=dtype)
    return QKV, ls, g, dO


def _widen(a):
    return O.bf16_bits_to_f64(a) if a.dtype == np.uint16 else a.astype(np.float64)


def assert_dbias_close(got, ref, cond, oerr=None, eps_o=0.0):
    tol = EPS_ARITH * cond + 1e-6 * max(float(np.abs(ref).max()), 1e-30)
    if oerr is not None:
        tol = tol + eps_o * oerr
    err = np.abs(got - ref)
    bad = err > tol
    assert not bad.any(), (f"{int(bad.sum())} of {bad.size} off; worst excess "
                           f"{float((err - tol).max()):.3e}, worst err {float(err.max()):.3e}")
    return float(err.max())


def _lse_close(got, ref):
    err = np.abs(got - ref)
    assert (err <= 2e-4 * np.maximum(1.0, np.abs(ref))).all(), f"lse off by {float(err.max()):.3e}"


def _unit(M, Hq=16, Hkv=8, t=1.1, bias=True, seed=0, scale_ls=1.0, scale_g=1.0):
    """dL/db on the GPU from the oracle's lse and D (rounded to fp32)."""
    QKV, ls, g, dO = _case(M, Hq, Hkv, bias=bias, seed=seed)
    if ls is not None:
        ls = (ls * scale_ls).astype(np.float32)
    g = (g * scale_g).astype(np.float32)
    q64, do64 = _widen(QKV), _widen(dO)
    lse = O.keybias_attn_lse(q64, Hq, Hkv, 128, ls, g, t)
    o = O.keybias_attn(q64, Hq, Hkv, 128, ls, g, t)
    D = O.attn_delta(do64, o, Hq, 128)
    ref, cond, _ = O.keybias_attn_bias_grad(q64, Hq, Hkv, 128, ls, g, t, do64, return_terms=True)
    got = tg.tg_keybias_attn_bias_grad(to_dev(QKV), to_dev(dO), Hq, Hkv, 128,
                                       to_dev(ls) if ls is not None else None, to_dev(g), t,
                                       to_dev(lse.astype(np.float32)), to_dev(D.astype(np.float32)))
    assert_dbias_close(f64(got), ref, cond)
    assert _status() == 0
    return got


# ------------------------------------------------- dL/db from given lse, D --
@pytest.mark.parametrize("M", [1, 2, 127, 128, 129, 300, 1000])
def test_bias_grad_bf16_ragged_sizes(M):
    _unit(M, seed=M)


@pytest.mark.parametrize("Hq,Hkv", [(2, 1), (4, 1), (6, 6), (8, 2)])
def test_bias_grad_bf16_group_sizes(Hq, Hkv):
    _unit(450, Hq=Hq, Hkv=Hkv, seed=Hq + Hkv)


def test_bias_grad_bf16_no_bias_and_strong_bias():
    _unit(400, bias=False, seed=3)
    _unit(700, t=2.5, seed=4, scale_ls=8.0, scale_g=3.0)


def test_bias_grad_bf16_zero_upstream_gradient_is_zero_and_deterministic():
    M = 600
    QKV, ls, g, _ = _case(M, seed=5)
    zero = torch.zeros(M, 16 * 128, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(16, M, dtype=torch.float32, device="cuda")
    D = torch.zeros(16, M, dtype=torch.float32, device="cuda")
    q, l, gg = to_dev(QKV), to_dev(ls), to_dev(g)
    got = tg.tg_keybias_attn_bias_grad(q, zero, 16, 8, 128, l, gg, 1.1, lse, D)
    assert torch.count_nonzero(got).item() == 0
    _, _, _, dO = _case(M, seed=5)
    out, lse = tg.tg_keybias_attn_lse(q, 16, 8, 128, l, gg, 1.1)
    D = tg.tg_attn_bwd_delta(to_dev(dO), out, 16, 128)
    a = tg.tg_keybias_attn_bias_grad(q, to_dev(dO), 16, 8, 128, l, gg, 1.1, lse, D)
    b = tg.tg_keybias_attn_bias_grad(q, to_dev(dO), 16, 8, 128, l, gg, 1.1, lse, D)
    assert torch.equal(a, b)
    assert _status() == 0


# ------------------------------------------------------------- forward lse --
@pytest.mark.parametrize("M", [1, 129, 1000])
def test_forward_lse_bf16(M):
    QKV, ls, g, _ = _case(M, seed=10 + M)
    out, lse = tg.tg_keybias_attn_lse(to_dev(QKV), 16, 8, 128, to_dev(ls), to_dev(g), 1.1)
    q64 = _widen(QKV)
    _lse_close(f64(lse), O.keybias_attn_lse(q64, 16, 8, 128, ls, g, 1.1))
    # the output is the same as without lse
    plain = tg.tg_keybias_attn(to_dev(QKV), 16, 8, 128, to_dev(ls), to_dev(g), 1.1)
    assert torch.equal(out, plain)


def test_forward_lse_f32_and_residual_mode():
    w = TI.WORKLOADS["tiny_f32_n512"]
    QKV, ls, g, _ = _case(192, w.Hq, w.Hkv, w.dh, seed=2, dtype="f32")
    _, lse = tg.tg_keybias_attn_lse(to_dev(QKV), w.Hq, w.Hkv, w.dh, to_dev(ls), to_dev(g), 1.1)
    ref = O.keybias_attn_lse(QKV, w.Hq, w.Hkv, w.dh, ls, g, 1.1)
    np.testing.assert_allclose(f64(lse), ref, rtol=1e-5, atol=1e-5)
    QKV, ls, g, _ = _case(300, seed=3)
    x = torch.zeros(300, 16 * 128, dtype=torch.float32, device="cuda")
    _, lse = tg.tg_keybias_attn_lse(to_dev(QKV), 16, 8, 128, to_dev(ls), to_dev(g), 1.1,
                                    residual=x)
    _lse_close(f64(lse), O.keybias_attn_lse(_widen(QKV), 16, 8, 128, ls, g, 1.1))


# ------------------------------------------------------------------- delta --
@pytest.mark.parametrize("dtype,dh", [("bf16", 128), ("bf16", 64), ("f32", 64), ("f32", 32)])
def test_delta(dtype, dh):
    M, Hq = 333, 4
    dO = TI.random_dout(M, Hq, dh, seed=7, dtype=dtype)
    Oa = TI.random_dout(M, Hq, dh, seed=8, dtype=dtype)
    got = f64(tg.tg_attn_bwd_delta(to_dev(dO), to_dev(Oa), Hq, dh))
    a, b = _widen(dO), _widen(Oa)
    ref = O.attn_delta(a, b, Hq, dh)
    absum = O.attn_delta(np.abs(a), np.abs(b), Hq, dh)
    assert (np.abs(got - ref) <= dh * 2.0 ** -24 * absum + 1e-30).all()


# --------------------------------------------------------------- reduction --
@pytest.mark.parametrize("M,Hq", [(0, 4), (1, 16), (1868, 16), (8432, 16)])
def test_bias_grad_reduce(M, Hq):
    rng = np.random.default_rng(M + Hq)
    dB = rng.standard_normal((Hq, M)).astype(np.float32)
    s = (rng.standard_normal(M) * 4).astype(np.float32)
    if M > 1:
        s[0], s[1] = 40.0, -40.0
    ls = O.logsigmoid(s.astype(np.float64)).astype(np.float32)
    g = rng.uniform(0.5, 1.5, Hq).astype(np.float32)
    dls, dg, ds = tg.tg_bias_grad_reduce(to_dev(dB) if M else torch.empty(Hq, 0, device="cuda"),
                                         to_dev(ls), to_dev(g))
    r_dls, r_dg, r_ds = O.bias_grad_reduce(dB, ls, g)
    np.testing.assert_allclose(f64(dg), r_dg, rtol=0,
                               atol=1e-5 * (np.abs(dB).astype(np.float64) @ np.abs(ls)).max() + 1e-30)
    if M:
        tol = 1e-6 * (np.abs(g).astype(np.float64) @ np.abs(dB))
        assert (np.abs(f64(dls) - r_dls) <= tol).all()
        # sigmoid(-s) from -expm1(ls): a few ulp relative, on top of dls
        assert (np.abs(f64(ds) - r_ds) <= 1e-6 * np.abs(r_ds) + tol * -np.expm1(ls)).all()
        assert f64(ds)[0] != 0.0 or r_dls[0] == 0.0   # sigmoid(-40) survives
    # fixed summation order: bitwise reproducible
    dls2, dg2, _ = tg.tg_bias_grad_reduce(to_dev(dB) if M else torch.empty(Hq, 0, device="cuda"),
                                          to_dev(ls), to_dev(g))
    assert torch.equal(dg, dg2) and torch.equal(dls, dls2)
    assert _status() == 0


# ------------------------------------------------------- the whole backward --
def _chain(M, Hq, Hkv, dh, ls, g, t, QKV, dO):
    q = to_dev(QKV)
    out, lse = tg.tg_keybias_attn_lse(q, Hq, Hkv, dh, to_dev(ls), to_dev(g), t)
    res = tg.bias_backward(q, out, lse, to_dev(dO), Hq, Hkv, dh, to_dev(ls), to_dev(g), t)
    return lse, res


def test_backward_chain_tiny_f32():
    w = TI.WORKLOADS["tiny_f32_n512"]
    QKV, ls, g, dO = _case(192, w.Hq, w.Hkv, w.dh, seed=1, dtype="f32")
    _, res = _chain(192, w.Hq, w.Hkv, w.dh, ls, g, 1.1, QKV, dO)
    ref, cond, oerr = O.keybias_attn_bias_grad(QKV, w.Hq, w.Hkv, w.dh, ls, g, 1.1, dO,
                                               return_terms=True)
    # fp32 throughout: D from the fp32 output, whose elements are off by ~1e-6
    assert_dbias_close(f64(res["dbias"]), ref, cond, oerr, 1e-5)
    r_dls, r_dg, r_ds = O.bias_grad_reduce(ref, ls, g)
    np.testing.assert_allclose(f64(res["dlogsig"]), r_dls, rtol=1e-3, atol=1e-3 * np.abs(r_dls).max())
    np.testing.assert_allclose(f64(res["dgain"]), r_dg, rtol=1e-3, atol=1e-3 * np.abs(r_dg).max())
    np.testing.assert_allclose(f64(res["dscore"]), r_ds, rtol=1e-3, atol=1e-3 * np.abs(r_ds).max())
    assert _status() == 0


@pytest.mark.parametrize("M", [300, 1868])
def test_backward_chain_bf16(M):
    # M = 1868: the kept rows of the 16k workload (10% of the document kept)
    QKV, ls, g, dO = _case(M, seed=20 + M)
    lse, res = _chain(M, 16, 8, 128, ls, g, 1.1, QKV, dO)
    q64, do64 = _widen(QKV), _widen(dO)
    _lse_close(f64(lse), O.keybias_attn_lse(q64, 16, 8, 128, ls, g, 1.1))
    ref, cond, oerr = O.keybias_attn_bias_grad(q64, 16, 8, 128, ls, g, 1.1, do64,
                                               return_terms=True)
    assert_dbias_close(f64(res["dbias"]), ref, cond, oerr, EPS_O)
    # the reduction of the GPU's dL/db, against the oracle's reduction of the
    # same values (the reduction's own parity is tested above)
    dB = f64(res["dbias"])
    r_dls, r_dg, r_ds = O.bias_grad_reduce(dB, ls, g)
    abs_dls = np.abs(np.asarray(g, np.float64)) @ np.abs(dB)      # sums of |terms|
    abs_dg = np.abs(dB) @ np.abs(np.asarray(ls, np.float64))
    assert (np.abs(f64(res["dlogsig"]) - r_dls) <= 1e-6 * abs_dls).all()
    assert (np.abs(f64(res["dgain"]) - r_dg) <= 1e-5 * abs_dg).all()
    assert (np.abs(f64(res["dscore"]) - r_ds) <= 1e-6 * np.abs(r_ds) + 1e-6 * abs_dls).all()
    # and the end result against the exact gradient: each dL/dls_j is a sum
    # over heads of dL/db_hj, so its error is bounded by the same sum of bounds
    e_dls = np.asarray(g, np.float64) @ (EPS_ARITH * cond + EPS_O * oerr)
    exact_dls = O.bias_grad_reduce(ref, ls, g)[0]
    assert (np.abs(f64(res["dlogsig"]) - exact_dls) <= e_dls + 1e-5 * np.abs(exact_dls).max()).all()
    assert _status() == 0


def test_backward_chain_bf16_128k_last_keys():
    # M = 8432: the kept rows of the 128k workload (6.25% of the document);
    # the oracle evaluates the last 384 keys, which need only the last 384 rows
    M, j0 = 8432, 8432 - 384
    QKV, ls, g, dO = _case(M, seed=128)
    lse, res = _chain(M, 16, 8, 128, ls, g, 1.1, QKV, dO)
    q64, do64 = _widen(QKV), _widen(dO)
    _lse_close(f64(lse)[:, j0:], O.keybias_attn_lse(q64, 16, 8, 128, ls, g, 1.1,
                                                    rows_from=j0)[:, j0:])
    ref, cond, oerr = O.keybias_attn_bias_grad(q64, 16, 8, 128, ls, g, 1.1, do64,
                                               return_terms=True, keys_from=j0)
    assert_dbias_close(f64(res["dbias"])[:, j0:], ref[:, j0:], cond[:, j0:], oerr[:, j0:], EPS_O)
    # every key: finite, and each head's gradient sums to (almost) zero --
    # shifting all biases of a head changes nothing -- up to what the bf16
    # output feeds into D (sum_i |dD_i| <= 2^-8 sum_i sum_c |dO_ic| |o_ic| ... )
    dB = f64(res["dbias"])
    assert np.isfinite(dB).all()
    assert (np.abs(dB.sum(axis=1)) <= 1e-2 * np.abs(dB).sum(axis=1)).all()
    assert _status() == 0
