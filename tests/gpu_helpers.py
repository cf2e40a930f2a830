"""Helpers for the GPU parity tests: move generator outputs to the device,
bring results back widened exactly, and the tolerances used."""
import numpy as np
import torch


def to_dev(a: np.ndarray) -> torch.Tensor:
    """numpy -> CUDA tensor; uint16 arrays are bf16 bit patterns."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(a).cuda()


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> uint16 bit patterns on the host."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def f64(t: torch.Tensor) -> np.ndarray:
    """Any float tensor -> float64 on the host (bf16 and fp32 widen exactly)."""
    return t.detach().cpu().float().numpy().astype(np.float64)


# ---- tolerances -----------------------------------------------------------
GATE_REL = 1e-4          # scores: |gpu - orc| <= 1e-4 * max(|orc|, rms(orc))
ATTN_MAX_ABS = 2e-2      # attention: max |gpu - orc| over compared outputs
ATTN_MEAN_ABS = 1e-2     #            mean |gpu - orc|
# gated delta rule on the tensor cores (bf16 operands, fp32 state and sums):
# per element |gpu - orc| <= 2^-5 (|orc| + rms(orc)), mean |gpu - orc| <= 2^-7
# rms(orc); about twice / three times what a model of the kernels' bf16
# rounding points reaches (tests/test_deltanet_rounding_model.py)
DELTA_MAX_REL = 2.0 ** -5
DELTA_MEAN_REL = 2.0 ** -7


def assert_gate_close(got, ref):
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 1.0
    tol = GATE_REL * np.maximum(np.abs(ref), rms)
    err = np.abs(got - ref)
    bad = err > tol
    assert not bad.any(), f"{bad.sum()} scores off; worst rel {float((err / np.maximum(np.abs(ref), rms)).max()):.3e}"
    return float((err / np.maximum(np.abs(ref), rms)).max()) if ref.size else 0.0


def assert_qkv_close(got, ref, K: int):
    """bf16 output of an fp32-accumulated dot product of length K: the store
    rounds to nearest (|err| <= 2^-8 |orc|), and fp32 accumulation adds at
    most a few units of 2^-24 * sqrt(K) * rms(orc) in practice; 1e-3 * rms
    is a generous allowance for it."""
    rms = float(np.sqrt(np.mean(ref * ref)))
    tol = 2.0 ** -8 * np.abs(ref) + 1e-3 * rms
    err = np.abs(got - ref)
    bad = err > tol
    assert not bad.any(), f"{bad.sum()} of {bad.size} off; worst {float((err - tol).max()):.3e} over"
    return float(err.max())


def assert_stack_drift_sane(got, ref, layers: int):
    """Sanity bound for the untethered drift of a `layers`-deep stack (not a
    parity tolerance: parity of the stack is checked per layer, teacher-
    forced, at the attention tolerance).  Each layer's bf16 roundings (of
    the RMSNorm output, of q, k, v and of P) are independent, so their
    effects on the residual add roughly in quadrature: sqrt(layers) times
    the attention tolerance."""
    err = np.abs(got - ref)
    mx, mean = float(err.max()), float(err.mean())
    f = float(np.sqrt(layers))
    assert mx <= f * ATTN_MAX_ABS and mean <= f * ATTN_MEAN_ABS, f"max {mx:.3e} mean {mean:.3e}"
    return mx, mean


def assert_attn_close(got, ref):
    err = np.abs(got - ref)
    mx, mean = float(err.max()), float(err.mean())
    assert mx <= ATTN_MAX_ABS and mean <= ATTN_MEAN_ABS, f"max {mx:.3e} mean {mean:.3e}"
    return mx, mean


def assert_delta_close(got, ref, what=""):
    """The delta rule's bf16 tolerance; returns (max, mean) error over rms."""
    rms = float(np.sqrt(np.mean(ref * ref)))
    err = np.abs(got - ref)
    bad = err > DELTA_MAX_REL * (np.abs(ref) + rms)
    assert not bad.any(), (f"{what}: {int(bad.sum())} off, worst {float(err.max()):.3e} "
                           f"(rms {rms:.3e})")
    assert float(err.mean()) <= DELTA_MEAN_REL * rms, (what, float(err.mean()), rms)
    return float(err.max()) / rms, float(err.mean()) / rms
