"""GPU parity of the gated delta rule (the recurrence of the Gated-DeltaNet
layers of a hybrid model, run over the kept tokens) against the fp64
oracle's recurrence: ragged chunks, an initial state and the final state,
bf16 and fp32 inputs, pruning as no-op tokens, and the hybrid workload's
size (6784 kept tokens, 16 heads of 128)."""
import numpy as np
import pytest
import torch

import oracle as O
import tg_inputs as TI
from learned_token_pruning_residual_b300 import build as tgbuild
import learned_token_pruning_residual_b300 as tg
from gpu_helpers import f64, to_dev

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


@pytest.mark.parametrize("T,H,dtype", [(1, 2, "f32"), (64, 3, "f32"), (65, 3, "f32"),
                                       (300, 4, "f32"), (257, 2, "bf16")])
def test_delta_rule_matches_recurrence(T, H, dtype):
    d = 128
    x = TI.deltanet_inputs(T, H, d, d, seed=T + H, dtype=dtype)
    S0 = (np.random.default_rng(T).standard_normal((H, d, d)) * 0.05).astype(np.float32)
    S_out = torch.empty(H, d, d, dtype=torch.float32, device="cuda")
    o, _ = tg.tg_gated_delta_rule(to_dev(x["q"]), to_dev(x["k"]), to_dev(x["v"]),
                                  to_dev(x["alpha"]), to_dev(x["beta"]), S0=to_dev(S0),
                                  S_out=S_out)
    ref_o, ref_S = O.gated_delta_rule(_widen(x["q"]), _widen(x["k"]), _widen(x["v"]), x["alpha"],
                                      x["beta"], S0)
    if dtype == "f32":
        _close(f64(o), ref_o, "o")
    else:
        _close_bf16(f64(o), ref_o)
    _close(f64(S_out), ref_S, "state")
    assert tg.tg_get_device_status(raise_on_error=False) == 0


def _close_bf16(got, ref):
    # the bf16 output adds its store rounding (2^-9 relative)
    rms = float(np.sqrt(np.mean(ref * ref)))
    err = np.abs(got - ref)
    assert (err <= 2.0 ** -8 * np.abs(ref) + 1e-4 * rms).all(), float(err.max())


def test_pruned_layer_equals_noop_tokens_on_the_gpu():
    T, H, d = 400, 2, 128
    x = TI.deltanet_inputs(T, H, d, d, seed=5)
    idx = np.sort(np.random.default_rng(5).choice(T, 150, replace=False))
    a2, b2 = np.ones((T, H), np.float32), np.zeros((T, H), np.float32)
    a2[idx], b2[idx] = x["alpha"][idx], x["beta"][idx]
    full, _ = tg.tg_gated_delta_rule(to_dev(x["q"]), to_dev(x["k"]), to_dev(x["v"]), to_dev(a2),
                                     to_dev(b2))
    kept, _ = tg.tg_gated_delta_rule(to_dev(x["q"][idx]), to_dev(x["k"][idx]),
                                     to_dev(x["v"][idx]), to_dev(x["alpha"][idx]),
                                     to_dev(x["beta"][idx]))
    ref, _ = O.gated_delta_rule(x["q"][idx], x["k"][idx], x["v"][idx], x["alpha"][idx],
                                x["beta"][idx])
    _close(f64(kept), ref, "kept")
    _close(f64(full)[idx], ref, "full with no-op tokens")


def test_hybrid_workload_size():
    """6784 kept tokens (the 64k prompt at 10% of its document plus the
    question), 16 heads of 128, bf16 inputs, against the oracle's chunked
    form (equal to its recurrence, pinned) on every token."""
    T, H, d = 6784, 16, 128
    x = TI.deltanet_inputs(T, H, d, d, seed=9, dtype="bf16")
    o, _ = tg.tg_gated_delta_rule(to_dev(x["q"]), to_dev(x["k"]), to_dev(x["v"]),
                                  to_dev(x["alpha"]), to_dev(x["beta"]))
    ref, _ = O.gated_delta_rule_chunked(_widen(x["q"]), _widen(x["k"]), _widen(x["v"]),
                                        x["alpha"], x["beta"])
    _close_bf16(f64(o), ref)
    assert tg.tg_get_device_status(raise_on_error=False) == 0
