"""GPU parity of the gated delta rule (the recurrence of the Gated-DeltaNet
layers of a hybrid model, run over the kept tokens) against the fp64
oracle: ragged chunks, an initial state and the final state, fp32 inputs
(CUDA-core kernels, tight tolerance) and bf16 inputs (tensor-core kernels,
the bf16 tolerance), pruning as no-op tokens, the hybrid workload's size
(6784 kept tokens, 16 heads of 128) and the 32k prompt the bench times in
full (sampled heads)."""
import numpy as np
import pytest
import torch

import oracle as O
import tg_inputs as TI
from learned_token_pruning_residual_b300 import build as tgbuild
import learned_token_pruning_residual_b300 as tg
from gpu_helpers import assert_delta_close, f64, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    tgbuild.build()
    tg.lib()
    assert tg.tg_get_device_status(raise_on_error=False) == 0


def _widen(a):
    return O.bf16_bits_to_f64(a) if a.dtype == np.uint16 else a.astype(np.float64)


def _close(got, ref, what):
    # fp32 arithmetic over chunks of 64: a few units of 2^-24 per operation,
    # grown by the unit-triangular solve; bounded at 1e-4 of the output scale
    rms = float(np.sqrt(np.mean(ref * ref)))
    err = np.abs(got - ref)
    bad = err > 1e-4 * (np.abs(ref) + rms)
    assert not bad.any(), f"{what}: {bad.sum()} off, worst {float(err.max()):.3e} (rms {rms:.3e})"
    return float(err.max())


@pytest.mark.parametrize("T,H", [(1, 2), (64, 3), (65, 3), (300, 4)])
def test_delta_rule_f32_matches_recurrence(T, H):
    d = 128
    x = TI.deltanet_inputs(T, H, d, d, seed=T + H, dtype="f32")
    S0 = (np.random.default_rng(T).standard_normal((H, d, d)) * 0.05).astype(np.float32)
    S_out = torch.empty(H, d, d, dtype=torch.float32, device="cuda")
    o, _ = tg.tg_gated_delta_rule(to_dev(x["q"]), to_dev(x["k"]), to_dev(x["v"]),
                                  to_dev(x["alpha"]), to_dev(x["beta"]), S0=to_dev(S0),
                                  S_out=S_out)
    ref_o, ref_S = O.gated_delta_rule(x["q"], x["k"], x["v"], x["alpha"], x["beta"], S0)
    _close(f64(o), ref_o, "o")
    _close(f64(S_out), ref_S, "state")
    assert tg.tg_get_device_status(raise_on_error=False) == 0


@pytest.mark.parametrize("T,H,with_S0", [(1, 2, True), (63, 1, False), (64, 3, True),
                                         (65, 2, True), (128, 1, False), (129, 3, True),
                                         (257, 2, True), (1000, 2, False), (1999, 5, True)])
def test_delta_rule_bf16_tensor_cores(T, H, with_S0):
    """Chunk counts odd and even (the prep kernel pairs chunks), ragged last
    chunks, one token, with and without an initial state."""
    d = 128
    x = TI.deltanet_inputs(T, H, d, d, seed=T + 7 * H, dtype="bf16")
    S0 = (np.random.default_rng(T).standard_normal((H, d, d)) * 0.05).astype(np.float32) \
        if with_S0 else None
    S_out = torch.empty(H, d, d, dtype=torch.float32, device="cuda")
    o, _ = tg.tg_gated_delta_rule(to_dev(x["q"]), to_dev(x["k"]), to_dev(x["v"]),
                                  to_dev(x["alpha"]), to_dev(x["beta"]),
                                  S0=to_dev(S0) if with_S0 else None, S_out=S_out)
    ref_o, ref_S = O.gated_delta_rule(_widen(x["q"]), _widen(x["k"]), _widen(x["v"]),
                                      x["alpha"], x["beta"], S0)
    mo = assert_delta_close(f64(o), ref_o, "o")
    ms = assert_delta_close(f64(S_out), ref_S, "state")
    print(f"T={T} H={H}: o max/rms {mo[0]:.2e} mean/rms {mo[1]:.2e}; "
          f"S max/rms {ms[0]:.2e} mean/rms {ms[1]:.2e}")
    assert tg.tg_get_device_status(raise_on_error=False) == 0


def test_delta_rule_bf16_is_deterministic():
    T, H, d = 700, 3, 128
    x = TI.deltanet_inputs(T, H, d, d, seed=3, dtype="bf16")
    args = [to_dev(x[n]) for n in ("q", "k", "v", "alpha", "beta")]
    a, _ = tg.tg_gated_delta_rule(*args)
    b, _ = tg.tg_gated_delta_rule(*args)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_pruned_layer_equals_noop_tokens(dtype):
    """On either path, the recurrence over the kept tokens equals the
    recurrence over every token with the pruned ones made no-ops (alpha = 1,
    beta = 0): both are compared with the oracle on the kept tokens."""
    T, H, d = 400, 2, 128
    x = TI.deltanet_inputs(T, H, d, d, seed=6, dtype=dtype)
    idx = np.sort(np.random.default_rng(6).choice(T, 150, replace=False))
    a2, b2 = np.ones((T, H), np.float32), np.zeros((T, H), np.float32)
    a2[idx], b2[idx] = x["alpha"][idx], x["beta"][idx]
    full, _ = tg.tg_gated_delta_rule(to_dev(x["q"]), to_dev(x["k"]), to_dev(x["v"]), to_dev(a2),
                                     to_dev(b2))
    kept, _ = tg.tg_gated_delta_rule(to_dev(x["q"][idx]), to_dev(x["k"][idx]),
                                     to_dev(x["v"][idx]), to_dev(x["alpha"][idx]),
                                     to_dev(x["beta"][idx]))
    ref, _ = O.gated_delta_rule(_widen(x["q"][idx]), _widen(x["k"][idx]), _widen(x["v"][idx]),
                                x["alpha"][idx], x["beta"][idx])
    check = _close if dtype == "f32" else assert_delta_close
    check(f64(kept), ref, "kept")
    check(f64(full)[idx], ref, "full with no-op tokens")


def test_hybrid_workload_size():
    """6784 kept tokens (the 64k prompt at 10% of its document plus the
    question), 16 heads of 128, bf16 inputs, against the oracle's chunked
    form (equal to its recurrence, pinned) on every token, and the final
    state."""
    T, H, d = 6784, 16, 128
    x = TI.deltanet_inputs(T, H, d, d, seed=9, dtype="bf16")
    S_out = torch.empty(H, d, d, dtype=torch.float32, device="cuda")
    o, _ = tg.tg_gated_delta_rule(to_dev(x["q"]), to_dev(x["k"]), to_dev(x["v"]),
                                  to_dev(x["alpha"]), to_dev(x["beta"]), S_out=S_out)
    ref, ref_S = O.gated_delta_rule_chunked(_widen(x["q"]), _widen(x["k"]), _widen(x["v"]),
                                            x["alpha"], x["beta"])
    print("o", assert_delta_close(f64(o), ref, "o"))
    print("S", assert_delta_close(f64(S_out), ref_S, "state"))
    assert tg.tg_get_device_status(raise_on_error=False) == 0


def test_full_32k_prompt_sampled_heads():
    """The 32k prompt that --mode deltanet times in full (32768 tokens, 16
    heads): all heads on the GPU in one call, as the bench launches it; heads
    0 and 11 (independent of the others) against the oracle."""
    T, H, d = 32768, 16, 128
    x = TI.deltanet_inputs(T, H, d, d, seed=2, dtype="bf16")
    S_out = torch.empty(H, d, d, dtype=torch.float32, device="cuda")
    o, _ = tg.tg_gated_delta_rule(to_dev(x["q"]), to_dev(x["k"]), to_dev(x["v"]),
                                  to_dev(x["alpha"]), to_dev(x["beta"]), S_out=S_out)
    o, S_out = f64(o), f64(S_out)
    for h in (0, 11):
        sl = slice(h, h + 1)
        ref, ref_S = O.gated_delta_rule_chunked(_widen(x["q"][:, sl]), _widen(x["k"][:, sl]),
                                                _widen(x["v"][:, sl]), x["alpha"][:, sl],
                                                x["beta"][:, sl])
        assert_delta_close(o[:, sl], ref, f"o head {h}")
        assert_delta_close(S_out[sl], ref_S, f"state head {h}")
    assert tg.tg_get_device_status(raise_on_error=False) == 0
