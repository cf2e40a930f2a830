"""GPU parity of the full Qwen3 decoder layer on the kept rows against the
fp64 oracle: the rotary table at the kept rows' prompt positions, the QKV
projection with per-head q/k RMSNorm and rotary embedding fused into its
epilogue, the residual-add projections, the SwiGLU hidden layer, and one
whole layer at the pruned-stack workload's size (M = 6784 kept rows of a
65536-token prompt) on sampled rows plus the question rows."""
import numpy as np
import pytest

import oracle as O
import tg_inputs as TI
from learned_token_pruning_residual_b300 import build as tgbuild
import learned_token_pruning_residual_b300 as tg
from gpu_helpers import assert_attn_close, assert_qkv_close, f64, to_dev

pytestmark = pytest.mark.gpu

W64 = TI.WORKLOADS["qwen3_1p7b_n64k_stack20_keep10"]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    tgbuild.build()
    tg.lib()
    assert tg.tg_get_device_status(raise_on_error=False) == 0


def _kept_positions(N, M, seed):
    rng = np.random.default_rng(seed)
    return np.sort(rng.choice(N, M, replace=False)).astype(np.int32)


def _bf16(a, seed_scale=1.0):
    return TI.f32_to_bf16_bits(np.asarray(a, dtype=np.float32) * np.float32(seed_scale))


def _dev_layer(P):
    out = {}
    for k, v in P.items():
        out[k] = to_dev(v) if isinstance(v, np.ndarray) else v
    return out


def test_rope_table_matches_the_angles():
    for pos in (np.arange(1000, dtype=np.int32), _kept_positions(131072, 8432, 1)):
        tab = tg.tg_rope_table(to_dev(pos), 128, 1e6).cpu().numpy().astype(np.float64)
        cos, sin = O.rope_angles(pos, 128, 1e6)
        err = max(np.abs(tab[..., 0] - cos).max(), np.abs(tab[..., 1] - sin).max())
        assert err <= 2e-6, err
    assert tg.tg_get_device_status(raise_on_error=False) == 0


@pytest.mark.parametrize("M", [1, 129, 1868])
def test_qkv_qknorm_rope(M):
    w = W64
    P = TI.qwen3_layer_params(w, layer=1)
    rng = np.random.default_rng(M)
    X = _bf16(rng.standard_normal((M, w.d)))
    pos = _kept_positions(w.N, M, M)
    table = tg.tg_rope_table(to_dev(pos), w.dh, P["rope_base"])
    got = tg.tg_qkv_proj_qknorm_rope(to_dev(X), to_dev(P["Wqkv"]), w.Hq, w.Hkv, w.dh,
                                     to_dev(P["gamma_q"]), to_dev(P["gamma_k"]), 1e-6, table)
    ref = O.rope(O.qk_rmsnorm(O.qkv_proj(X, P["Wqkv"]), w.Hq, w.Hkv, w.dh, P["gamma_q"],
                              P["gamma_k"], 1e-6), w.Hq, w.Hkv, w.dh, pos, P["rope_base"])
    assert_qkv_close(f64(got), ref, w.d)
    assert tg.tg_get_device_status(raise_on_error=False) == 0


@pytest.mark.parametrize("M,K,N", [(1868, 2048, 2048), (300, 6144, 2048), (5, 128, 96)])
def test_linear_residual(M, K, N):
    rng = np.random.default_rng(K + N)
    X = _bf16(rng.standard_normal((M, K)))
    W = _bf16(rng.standard_normal((N, K)) / np.sqrt(K))
    r0 = rng.standard_normal((M, N)).astype(np.float32)
    r = to_dev(r0)
    tg.tg_linear_residual(to_dev(X), to_dev(W), r)
    ref = r0.astype(np.float64) + O.linear(X, W)
    lin = O.linear(X, W)
    rms = float(np.sqrt(np.mean(lin * lin)))
    err = np.abs(f64(r) - ref)
    # fp32 accumulation of K bf16 products, and the fp32 add into the residual
    assert (err <= 1e-3 * rms + 2.0 ** -22 * np.abs(ref)).all(), float(err.max())
    assert tg.tg_get_device_status(raise_on_error=False) == 0


@pytest.mark.parametrize("M,F", [(1868, 6144), (77, 256), (130, 96)])
def test_swiglu(M, F):
    d = 2048
    rng = np.random.default_rng(M + F)
    X = _bf16(rng.standard_normal((M, d)))
    Wg = _bf16(rng.standard_normal((F, d)) / np.sqrt(d))
    Wu = _bf16(rng.standard_normal((F, d)) / np.sqrt(d))
    got = tg.tg_swiglu(to_dev(X), to_dev(Wg), to_dev(Wu))
    assert_qkv_close(f64(got), O.swiglu_hidden(X, Wg, Wu), d)
    assert tg.tg_get_device_status(raise_on_error=False) == 0


def _sample_rows(M, n, seed):
    rng = np.random.default_rng(seed)
    tail = np.arange(max(0, M - 256), M)
    head = rng.choice(max(1, M - 256), size=min(n, max(1, M - 256)), replace=False)
    return np.unique(np.concatenate([head, tail, [0]])).astype(np.int64)


def test_qwen3_layer_full_size_one_layer():
    """One whole Qwen3 layer on the stack workload's M = 6784 kept rows at
    their prompt positions (a 65536-token prompt), compared on 1024 sampled
    rows plus the 256 question rows at the attention tolerance."""
    w = W64
    M = w.M(w.Ks()[0])
    P = TI.qwen3_layer_params(w, layer=0)
    rng = np.random.default_rng(12)
    x0 = rng.standard_normal((M, w.d)).astype(np.float32)
    pos = _kept_positions(w.N, M, 12)
    pos[-256:] = np.arange(w.N - 256, w.N)  # the question is always kept
    pos = np.sort(pos)
    ls = TI.random_logsig(M, seed=12)
    x = to_dev(x0)
    table = tg.tg_rope_table(to_dev(pos), w.dh, P["rope_base"])
    tg.qwen3_layer(x, table, _dev_layer(P), w.Hq, w.Hkv, w.dh, to_dev(ls))
    rows = _sample_rows(M, 1024, seed=12)
    ref = O.qwen3_pruned_layer(x0, pos, P, w.Hq, w.Hkv, w.dh, ls, rows=rows)
    mx, mean = assert_attn_close(f64(x)[rows], ref)
    print(f"Qwen3 layer, M={M}: max-abs {mx:.2e} mean-abs {mean:.2e}")
    assert tg.tg_get_device_status(raise_on_error=False) == 0


def test_qwen3_stack_teacher_forced_small():
    """Four layers through qwen3_pruned_stack's per-layer call, each layer
    teacher-forced (the oracle takes the GPU's input of that layer), at
    M = 640 kept rows of a 16384-token prompt, all rows compared."""
    w = TI.WORKLOADS["qwen3_1p7b_n16k_keep10"]
    M = 640
    rng = np.random.default_rng(13)
    x = to_dev(rng.standard_normal((M, w.d)).astype(np.float32))
    pos = _kept_positions(w.N, M, 13)
    ls = TI.random_logsig(M, seed=13)
    table = tg.tg_rope_table(to_dev(pos), w.dh, 1e6)
    for layer in range(4):
        P = TI.qwen3_layer_params(w, layer=layer, ffn=1024)
        x_in = x.cpu().numpy()
        tg.qwen3_layer(x, table, _dev_layer(P), w.Hq, w.Hkv, w.dh, to_dev(ls))
        ref = O.qwen3_pruned_layer(x_in, pos, P, w.Hq, w.Hkv, w.dh, ls)
        assert_attn_close(f64(x), ref)
    assert tg.tg_get_device_status(raise_on_error=False) == 0


def test_kept_rows_at_prompt_positions_equal_the_masked_full_layer():
    """The pin of the oracle's layer, on the GPU: the kept rows at their
    original positions give the full prompt's layer output at those rows with
    every pruned key masked (logsig = -inf for pruned rows, a finite bias for
    kept ones), here with the full prompt's layer run on the GPU too."""
    w = TI.WORKLOADS["qwen3_1p7b_n16k_keep10"]
    N, M = 512, 200
    P = TI.qwen3_layer_params(w, layer=2, ffn=512)
    rng = np.random.default_rng(14)
    xf = rng.standard_normal((N, w.d)).astype(np.float32)
    idx = _kept_positions(N, M, 14)
    ls_full = np.full(N, -np.inf, dtype=np.float32)
    ls_full[idx] = TI.random_logsig(M, seed=14)
    Pd = _dev_layer(P)
    x_full = to_dev(xf)
    tg.qwen3_layer(x_full, tg.tg_rope_table(to_dev(np.arange(N, dtype=np.int32)), w.dh, 1e6), Pd,
                   w.Hq, w.Hkv, w.dh, to_dev(ls_full))
    x_kept = to_dev(xf[idx])
    tg.qwen3_layer(x_kept, tg.tg_rope_table(to_dev(idx), w.dh, 1e6), Pd, w.Hq, w.Hkv, w.dh,
                   to_dev(ls_full[idx]))
    # both equal the oracle's layer on the kept rows at their positions (which
    # the oracle's pins show equals its full layer with the pruned keys masked)
    ref = O.qwen3_pruned_layer(xf[idx], idx, P, w.Hq, w.Hkv, w.dh, ls_full[idx])
    assert_attn_close(f64(x_kept), ref)
    assert_attn_close(f64(x_full)[idx], ref)
    assert tg.tg_get_device_status(raise_on_error=False) == 0
