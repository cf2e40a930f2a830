"""GPU parity of each kernel against the fp64 oracle, on seeded inputs that
span several tiles and a ragged tail, plus the edge cases of each op.
Everything goes through the C ABI (via the ctypes binding)."""
import math

import numpy as np
import pytest
import torch

import oracle as O
import tg_inputs as TI
from learned_token_pruning_residual_b300 import build as tgbuild
import learned_token_pruning_residual_b300 as tg
from gpu_helpers import (assert_attn_close, assert_gate_close, assert_qkv_close, bits, f64,
                         to_dev)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    tgbuild.build()
    tg.lib()
    assert tg.tg_get_device_status(raise_on_error=False) == 0


def _status():
    return tg.tg_get_device_status(raise_on_error=False)


# ------------------------------------------------------------------ select --
SELECT_SHAPES = [
    # N, doc_begin, doc_end, K
    (1, 0, 1, 0), (1, 0, 1, 1), (7, 0, 7, 3), (100, 10, 90, 40), (512, 0, 448, 128),
    (5000, 123, 4871, 1), (5000, 123, 4871, 4747), (5000, 0, 5000, 2500), (5000, 2500, 2500, 0),
    (16384, 0, 16128, 1612), (16384, 0, 16128, 0), (16384, 0, 16128, 16128),
    (65536, 0, 65280, 6528), (131072, 0, 130816, 8176), (200003, 77, 199990, 12345),
    # more than 8 x 24576 keys: the kernel streams keys from global memory
    (300000, 1000, 299000, 29800),
]


@pytest.mark.parametrize("N,b,e,K", SELECT_SHAPES)
def test_select_random_bit_exact(N, b, e, K):
    s = TI.random_scores(N, seed=N + K)
    got = tg.tg_select_topk(to_dev(s), b, e, K).cpu().numpy()
    ref = O.select_topk(s, b, e, K)
    assert got.shape == ref.shape
    assert np.array_equal(got, ref)
    assert _status() == 0


@pytest.mark.parametrize("kind", TI.ADVERSARIAL_KINDS)
@pytest.mark.parametrize("N,b,e", [(3000, 100, 2800), (70001, 5, 70000)])
def test_select_adversarial_bit_exact(kind, N, b, e):
    s = TI.adversarial_scores(kind, N, seed=3)
    D = e - b
    for K in (0, 1, 17, D // 3, D - 1, D):
        got = tg.tg_select_topk(to_dev(s), b, e, K).cpu().numpy()
        assert np.array_equal(got, O.select_topk(s, b, e, K)), (kind, K)
    assert _status() == 0


def test_select_hand_worked_fixture_on_gpu():
    from test_oracle_pins import _read_golden_select
    g = _read_golden_select()
    s = np.array([float(v) for v in g["scores"]], dtype=np.float32)
    b, e = int(g["doc_begin"][0]), int(g["doc_end"][0])
    for K, expect in g["cases"]:
        assert tg.tg_select_topk(to_dev(s), b, e, K).cpu().tolist() == expect


def test_select_32k_budget_sweep_bit_exact():
    w = TI.WORKLOADS["qwen3_1p7b_n32k_sweep"]
    s = TI.random_scores(w.N, seed=w.seed)
    sd = to_dev(s)
    for K in w.Ks():
        got = tg.tg_select_topk(sd, w.doc_begin, w.doc_end, K).cpu().numpy()
        assert np.array_equal(got, O.select_topk(s, w.doc_begin, w.doc_end, K)), K


def test_select_is_deterministic():
    s = to_dev(TI.adversarial_scores("quantised", 131072, seed=9))
    a = tg.tg_select_topk(s, 0, 130816, 8176)
    for _ in range(3):
        assert torch.equal(a, tg.tg_select_topk(s, 0, 130816, 8176))


def test_select_nan_in_span_sets_status():
    s = TI.random_scores(4000, seed=1)
    s[1234] = np.nan
    tg.tg_select_topk(to_dev(s), 0, 3000, 100)
    assert tg.tg_get_device_status(raise_on_error=False) == 4       # TG_ERR_NAN_SCORE
    assert _status() == 0                                             # cleared after reading
    # a NaN outside the span is not an error
    s3 = TI.random_scores(4000, seed=1)
    s3[3500] = np.nan
    got = tg.tg_select_topk(to_dev(s3), 0, 3000, 100).cpu().numpy()
    assert _status() == 0
    assert np.array_equal(got, O.select_topk(s3, 0, 3000, 100))


def _ws_reset_words(ws):
    """The workspace words that must be zero before a select call: the four
    2048-word histograms, then (after 2 x 256 per-CTA count words) the
    4-word header, the barrier's arrival counter and (after the barrier's
    generation word) the candidate reservation counter."""
    w = ws.view(torch.int32)
    base = 4 * 2048 + 512
    return torch.cat([w[:4 * 2048], w[base:base + 5], w[base + 6:base + 7]])


def test_select_leaves_workspace_zeroed():
    ws = tg.new_select_workspace()
    for N, b, e, K in [(131072, 0, 130816, 8176), (5000, 123, 4871, 4747), (5000, 0, 5000, 0),
                       (300000, 1000, 299000, 29800)]:
        s = TI.random_scores(N, seed=K + 1)
        got = tg.tg_select_topk(to_dev(s), b, e, K, workspace=ws).cpu().numpy()
        assert np.array_equal(got, O.select_topk(s, b, e, K))
        assert int(_ws_reset_words(ws).count_nonzero()) == 0, (N, K)
    assert _status() == 0


@pytest.mark.parametrize("N,b,e,K", [(16384, 0, 16128, 1612), (131072, 0, 130816, 8176),
                                     (20000, 300, 19000, 0), (20000, 300, 19000, 18700),
                                     (4097, 1, 4096, 2000)])
def test_gate_fills_first_select_pass(N, b, e, K):
    """The gate epilogue counts the first radix pass into the select
    workspace; the select on the same span uses it.  Bit-exact against the
    oracle on the GPU's own scores, twice in a row on one workspace, and the
    workspace is zero afterwards."""
    d, Hg = 256, 64
    rng = np.random.default_rng(N + K)
    X = TI.f32_to_bf16_bits(rng.standard_normal((N, d)).astype(np.float32))
    W1 = TI.f32_to_bf16_bits((rng.standard_normal((Hg, d)) / np.sqrt(d)).astype(np.float32))
    w2 = (rng.standard_normal(Hg) / np.sqrt(Hg)).astype(np.float32)
    Xd, W1d, w2d = to_dev(X), to_dev(W1), to_dev(w2)
    ws = tg.new_select_workspace()
    for _ in range(2):
        sc = tg.tg_gate_score(Xd, W1d, None, w2d, 0.0, select_ws=ws, doc_begin=b, doc_end=e)
        assert int(_ws_reset_words(ws).count_nonzero()) > 0 or e == b
        idx = tg.tg_select_topk(sc, b, e, K, workspace=ws).cpu().numpy()
        assert np.array_equal(idx, O.select_topk(sc.cpu().numpy(), b, e, K))
        assert int(_ws_reset_words(ws).count_nonzero()) == 0
    assert _status() == 0


def test_gate_histogram_of_another_span_is_ignored():
    N, d, Hg = 9000, 128, 32
    rng = np.random.default_rng(4)
    X = TI.f32_to_bf16_bits(rng.standard_normal((N, d)).astype(np.float32))
    W1 = TI.f32_to_bf16_bits((rng.standard_normal((Hg, d)) / np.sqrt(d)).astype(np.float32))
    w2 = (rng.standard_normal(Hg) / np.sqrt(Hg)).astype(np.float32)
    ws = tg.new_select_workspace()
    sc = tg.tg_gate_score(to_dev(X), to_dev(W1), None, to_dev(w2), 0.0, select_ws=ws,
                          doc_begin=0, doc_end=8000)
    idx = tg.tg_select_topk(sc, 100, 8500, 1234, workspace=ws).cpu().numpy()
    assert np.array_equal(idx, O.select_topk(sc.cpu().numpy(), 100, 8500, 1234))
    assert int(_ws_reset_words(ws).count_nonzero()) == 0
    assert _status() == 0


# ------------------------------------------------------------------ gather --
@pytest.mark.parametrize("mode", ["bf16", "f32", "bf16_to_f32"])
def test_gather_exact_and_logsig(mode):
    N, d = 3001, 256 if mode != "f32" else 260
    rng = np.random.default_rng(5)
    Xf = rng.standard_normal((N, d)).astype(np.float32)
    X = TI.f32_to_bf16_bits(Xf) if mode != "f32" else Xf
    s = (rng.standard_normal(N) * 20).astype(np.float32)
    s[:4] = [0.0, -100.0, 100.0, -0.0]
    idx = np.sort(rng.choice(N, 1777, replace=False)).astype(np.int32)
    idx[0] = 0
    Y, ls = tg.tg_gather_rows(to_dev(X), to_dev(idx), to_dev(s),
                              out_dtype=torch.float32 if mode == "bf16_to_f32" else None)
    Yr, lsr = O.gather_rows(X, idx, s)
    if mode == "bf16":
        assert np.array_equal(bits(Y), Yr)
    elif mode == "f32":
        assert np.array_equal(Y.cpu().numpy(), Yr)
    else:
        assert np.array_equal(Y.cpu().numpy().astype(np.float64), O.bf16_bits_to_f64(Yr))
    np.testing.assert_allclose(f64(ls), lsr, rtol=2e-6, atol=1e-7)
    assert _status() == 0


@pytest.mark.parametrize("dtype,d,N,M", [
    ("bf16", 2048, 20000, 8432),   # the 128k workload's row size and kept count
    ("bf16", 2048, 5000, 4999),    # nearly every row kept
    ("f32", 2048, 3000, 1000),     # 8 KB rows
    ("bf16", 8192, 1500, 700),     # 16 KB rows: several vector rounds per lane
    ("bf16", 8, 300000, 140000),   # 16-byte rows (one lane), rows past one grid stride
])
def test_gather_large_rows_exact(dtype, d, N, M):
    rng = np.random.default_rng(d + M)
    Xf = rng.standard_normal((N, d)).astype(np.float32)
    X = TI.f32_to_bf16_bits(Xf) if dtype == "bf16" else Xf
    s = (rng.standard_normal(N) * 5).astype(np.float32)
    idx = np.sort(rng.choice(N, M, replace=False)).astype(np.int32)
    Y, ls = tg.tg_gather_rows(to_dev(X), to_dev(idx), to_dev(s))
    Yr, lsr = O.gather_rows(X, idx, s)
    got = bits(Y) if dtype == "bf16" else Y.cpu().numpy()
    assert np.array_equal(got, Yr)
    np.testing.assert_allclose(f64(ls), lsr, rtol=2e-6, atol=1e-7)
    assert _status() == 0


def test_gather_bad_indices_among_many_rows():
    """Out-of-range indices at both ends, next to each other and in the
    middle of a 3000-row gather of 4 KB rows: those rows are zero, every
    other row exact."""
    N, d, M = 4000, 2048, 3000
    rng = np.random.default_rng(9)
    X = TI.f32_to_bf16_bits(rng.standard_normal((N, d)).astype(np.float32) + 3.0)
    idx = rng.integers(0, N, M).astype(np.int32)
    bad = np.array([0, 17, 18, 40, 1500, 2999])
    idx[bad] = np.array([-1, N, N + 5, -7, 1 << 30, N], dtype=np.int32)
    Y, _ = tg.tg_gather_rows(to_dev(X), to_dev(idx))
    assert tg.tg_get_device_status(raise_on_error=False) == 5   # TG_ERR_BAD_INDEX
    got = bits(Y)
    assert not got[bad].any()
    good = np.setdiff1d(np.arange(M), bad)
    assert np.array_equal(got[good], X[idx[good]])
    assert _status() == 0


def test_gather_identity_and_empty():
    X = TI.f32_to_bf16_bits(np.random.default_rng(1).standard_normal((130, 64)).astype(np.float32))
    Y, _ = tg.tg_gather_rows(to_dev(X), None)
    assert np.array_equal(bits(Y), X)
    Y0, _ = tg.tg_gather_rows(to_dev(X), torch.empty(0, dtype=torch.int32, device="cuda"))
    assert Y0.shape == (0, 64)


def test_gather_bad_index_sets_status():
    X = to_dev(TI.f32_to_bf16_bits(np.ones((10, 64), np.float32)))
    idx = to_dev(np.array([0, 3, 10, 2], dtype=np.int32))           # 10 is out of range
    Y, _ = tg.tg_gather_rows(X, idx)
    assert tg.tg_get_device_status(raise_on_error=False) == 5        # TG_ERR_BAD_INDEX
    assert not f64(Y)[2].any()                                       # that row is zeroed
    assert (f64(Y)[[0, 1, 3]] == 1.0).all()


# ----------------------------------------------------------------- rmsnorm --
@pytest.mark.parametrize("xin,yout", [("f32", "bf16"), ("bf16", "bf16"), ("f32", "f32")])
def test_rmsnorm(xin, yout):
    rng = np.random.default_rng(2)
    M, d = 777, 2048
    xf = (rng.standard_normal((M, d)) * 1.7).astype(np.float32)
    x = TI.f32_to_bf16_bits(xf) if xin == "bf16" else xf
    gm = rng.uniform(0.9, 1.1, d).astype(np.float32)
    y = tg.tg_rmsnorm(to_dev(x), to_dev(gm), 1e-6,
                      out_dtype=torch.bfloat16 if yout == "bf16" else torch.float32)
    ref = O.rmsnorm(x, gm, 1e-6)
    err = np.abs(f64(y) - ref)
    bound = (2.0 ** -8 if yout == "bf16" else 1e-6) * np.abs(ref) + 1e-6
    assert (err <= bound).all(), float((err - bound).max())


# -------------------------------------------------------------------- gate --
def test_gate_tiny_f32():
    w = TI.WORKLOADS["tiny_f32_n512"]
    X = TI.residual(w)
    gp = TI.gate_params(w, gate_biases=True)
    s = tg.tg_gate_score(to_dev(X), to_dev(gp["W1"]), to_dev(gp["b1"]), to_dev(gp["w2"]), gp["b2"])
    assert_gate_close(f64(s), O.gate_score(X, gp["W1"], gp["b1"], gp["w2"], gp["b2"]))


@pytest.mark.parametrize("N,Hg,biases", [(1, 256, False), (1000, 256, True), (4097, 128, True),
                                         (16384, 256, False), (300, 64, True), (200, 16, False)])
def test_gate_bf16(N, Hg, biases):
    w = TI.Workload("g", N=N, doc_begin=0, doc_end=N, d=2048, Hg=Hg, Hq=16, Hkv=8, dh=128,
                    dtype="bf16", seed=N + Hg)
    X = TI.residual(w)
    gp = TI.gate_params(w, gate_biases=biases)
    b1 = to_dev(gp["b1"]) if biases else None
    s = tg.tg_gate_score(to_dev(X), to_dev(gp["W1"]), b1, to_dev(gp["w2"]), gp["b2"])
    ref = O.gate_score(X, gp["W1"], gp["b1"] if biases else None, gp["w2"], gp["b2"])
    assert_gate_close(f64(s), ref)
    assert _status() == 0


@pytest.mark.parametrize("N,d", [(5000, 128), (70001, 128), (20000, 320)])
def test_gate_bf16_short_k_loop(N, d):
    """Hg = 256 with 2 or 5 K blocks per tile: the W1 fills, which trail the
    residual's by a few K steps, cross tile boundaries (and with one tile per
    CTA pair the whole K loop is shorter than that lag)."""
    Hg = 256
    rng = np.random.default_rng(N + d)
    X = TI.f32_to_bf16_bits(rng.standard_normal((N, d)).astype(np.float32))
    W1 = TI.f32_to_bf16_bits((rng.standard_normal((Hg, d)) / np.sqrt(d)).astype(np.float32))
    b1 = (rng.standard_normal(Hg) * 0.1).astype(np.float32)
    w2 = (rng.standard_normal(Hg) / np.sqrt(Hg)).astype(np.float32)
    s = tg.tg_gate_score(to_dev(X), to_dev(W1), to_dev(b1), to_dev(w2), 0.25)
    assert_gate_close(f64(s), O.gate_score(X, W1, b1, w2, 0.25))
    assert _status() == 0


def test_gate_bf16_zero_weight_closed_form():
    N, d, Hg = 333, 256, 32
    X = TI.f32_to_bf16_bits(np.random.default_rng(3).standard_normal((N, d)).astype(np.float32))
    W1 = np.zeros((Hg, d), dtype=np.uint16)
    b1 = np.linspace(-2, 2, Hg).astype(np.float32)
    w2 = np.linspace(1, -1, Hg).astype(np.float32)
    s = f64(tg.tg_gate_score(to_dev(X), to_dev(W1), to_dev(b1), to_dev(w2), 0.5))
    const = O.gate_score(X[:1], W1, b1, w2, 0.5)[0]
    assert_gate_close(s, np.full(N, const))


# --------------------------------------------------------------------- qkv --
@pytest.mark.parametrize("M", [1, 127, 129, 1868])
def test_qkv_bf16(M):
    w = TI.WORKLOADS["qwen3_1p7b_n16k_keep10"]
    X = TI.residual(TI.Workload("x", N=M, doc_begin=0, doc_end=M, d=2048, Hg=256, Hq=16, Hkv=8,
                                dh=128, dtype="bf16", seed=40 + M))
    W = TI.qkv_weight(w)
    got = tg.tg_qkv_proj(to_dev(X), to_dev(W), 16, 8, 128)
    assert_qkv_close(f64(got), O.qkv_proj(X, W), K=2048)


def test_qkv_bf16_identity_weight_reproduces_input():
    M, d = 300, 128
    X = TI.f32_to_bf16_bits(np.random.default_rng(4).standard_normal((M, d)).astype(np.float32))
    W = np.zeros((3 * 128, d), dtype=np.float32)                # [(Hq + 2 Hkv) dh][d]
    W[:d, :d] = np.eye(d)
    got = tg.tg_qkv_proj(to_dev(X), to_dev(TI.f32_to_bf16_bits(W)), 1, 1, 128)   # cols = 3*128
    g = bits(got)
    assert np.array_equal(g[:, :d], X)
    assert not g[:, d:].any()


def test_qkv_tiny_f32():
    w = TI.WORKLOADS["tiny_f32_n512"]
    X = TI.residual(w)[:192]
    W = TI.qkv_weight(w)
    got = f64(tg.tg_qkv_proj(to_dev(X), to_dev(W), w.Hq, w.Hkv, w.dh))
    np.testing.assert_allclose(got, O.qkv_proj(X, W), rtol=1e-4, atol=1e-5)


# -------------------------------------------------------------------- attn --
def _attn_case(M, Hq=16, Hkv=8, dh=128, bias=True, seed=0, dtype="bf16"):
    QKV = TI.random_qkv(M, Hq, Hkv, dh, seed=seed, dtype=dtype)
    ls = TI.random_logsig(M, seed=seed) if bias else None
    g = TI._rng(seed, 30).uniform(0.5, 1.5, Hq).astype(np.float32)
    return QKV, ls, g


@pytest.mark.parametrize("M", [1, 2, 100, 128, 129, 256, 1000, 1868])
def test_attn_bf16_all_rows(M):
    QKV, ls, g = _attn_case(M, seed=M)
    got = tg.tg_keybias_attn(to_dev(QKV), 16, 8, 128, to_dev(ls), to_dev(g), 1.1)
    ref = O.keybias_attn(QKV, 16, 8, 128, ls, g, 1.1)
    assert_attn_close(f64(got), ref)
    assert _status() == 0


@pytest.mark.parametrize("Hq,Hkv", [(2, 1), (4, 1), (8, 2)])
def test_attn_bf16_other_group_sizes(Hq, Hkv):
    QKV, ls, g = _attn_case(700, Hq=Hq, Hkv=Hkv, seed=Hq)
    got = tg.tg_keybias_attn(to_dev(QKV), Hq, Hkv, 128, to_dev(ls), to_dev(g), 0.9)
    assert_attn_close(f64(got), O.keybias_attn(QKV, Hq, Hkv, 128, ls, g, 0.9))


def test_attn_bf16_no_bias_is_causal_softmax():
    QKV, _, g = _attn_case(600, bias=False, seed=7)
    got = tg.tg_keybias_attn(to_dev(QKV), 16, 8, 128, None, None, 1.0)
    assert_attn_close(f64(got), O.keybias_attn(QKV, 16, 8, 128, None, g, 1.0))


def test_attn_bf16_strong_bias_and_large_logits():
    # large logits exercise the delayed rescale; a dominant bias concentrates rows
    M = 900
    QKV, ls, g = _attn_case(M, seed=11)
    ls = ls * 8.0
    got = tg.tg_keybias_attn(to_dev(QKV), 16, 8, 128, to_dev(ls), to_dev(g * 3), 2.5)
    assert_attn_close(f64(got), O.keybias_attn(QKV, 16, 8, 128, ls, g * 3, 2.5))


def test_attn_bf16_residual_mode():
    M = 513
    QKV, ls, g = _attn_case(M, seed=12)
    x = np.random.default_rng(0).standard_normal((M, 16 * 128)).astype(np.float32)
    xd = to_dev(x)
    tg.tg_keybias_attn(to_dev(QKV), 16, 8, 128, to_dev(ls), to_dev(g), 1.1, residual=xd)
    ref = x.astype(np.float64) + O.keybias_attn(QKV, 16, 8, 128, ls, g, 1.1)
    assert_attn_close(f64(xd), ref)


def test_attn_bf16_deterministic():
    QKV, ls, g = _attn_case(1000, seed=13)
    a = tg.tg_keybias_attn(to_dev(QKV), 16, 8, 128, to_dev(ls), to_dev(g), 1.1)
    b = tg.tg_keybias_attn(to_dev(QKV), 16, 8, 128, to_dev(ls), to_dev(g), 1.1)
    assert torch.equal(a, b)


@pytest.mark.parametrize("bias", [True, False])
def test_attn_tiny_f32(bias):
    w = TI.WORKLOADS["tiny_f32_n512"]
    QKV, ls, g = _attn_case(192, Hq=w.Hq, Hkv=w.Hkv, dh=w.dh, bias=bias, seed=1, dtype="f32")
    got = tg.tg_keybias_attn(to_dev(QKV), w.Hq, w.Hkv, w.dh, to_dev(ls) if bias else None,
                             to_dev(g), 1.1)
    ref = O.keybias_attn(QKV, w.Hq, w.Hkv, w.dh, ls, g, 1.1)
    np.testing.assert_allclose(f64(got), ref, rtol=1e-4, atol=1e-5)


# ------------------------------------------------------------- the plan --
def test_gated_layer_plan_matches_the_calls():
    """The library's CUDA graph of the five calls gives exactly the outputs
    of the calls made one by one (the same kernels), launch after launch,
    also after a new prompt is written into its input buffer."""
    w = TI.Workload("plan_bf16_n4096", N=4096, doc_begin=64, doc_end=3900, d=2048, Hg=256, Hq=16,
                    Hkv=8, dh=128, dtype="bf16", seed=21, K_fixed=700)
    gp, Wqkv, ap = TI.gate_params(w, gate_biases=True), TI.qkv_weight(w), TI.attn_params(w)
    X = to_dev(TI.residual(w))
    args = (to_dev(gp["W1"]), to_dev(gp["b1"]), to_dev(gp["w2"]), gp["b2"], w.doc_begin,
            w.doc_end, w.Ks()[0], to_dev(Wqkv), w.Hq, w.Hkv, w.dh, to_dev(ap["gain"]),
            ap["temperature"])
    plan = tg.GatedLayerPlan(X, *args)
    for k in range(3):
        if k == 2:  # a new prompt in the same buffer
            X.copy_(to_dev(TI.f32_to_bf16_bits(np.random.default_rng(3).standard_normal(
                (w.N, w.d)).astype(np.float32))))
        got = plan.launch()
        ref = tg.gated_layer(X, *args)
        torch.cuda.synchronize()
        for a, b in (("scores", "scores"), ("idx", "idx"), ("logsig", "logsig")):
            assert torch.equal(got[a], ref[b]), a
        assert torch.equal(got["out"].view(torch.int16), ref["O"].view(torch.int16))
    plan.close()
    assert _status() == 0
