"""tg_select_topk_noalloc: the select for callers that cannot allocate
device memory or pass the library a workspace (a host that owns all device
memory and allows no allocation after start-up, a plug-in inside another
framework's allocator, a latency-critical path where cudaMalloc/cudaFree
would synchronise).  It uses a scratch array compiled into the library
instead of a workspace.

Called through the C ABI (ctypes), its indices must equal those of the
regular tg_select_topk on the same scores, bit for bit, on two calls in a
row: the second call finds the array as the first left it.  The first case
runs the multi-CTA select, whose grid barriers and histograms live in the
scratch; the second a span short enough for the single-CTA select.  This
file is named to be collected last, so that a run stopping at its first
failure has already run every other test; it also passes alone."""
import ctypes

import numpy as np
import pytest
import torch

import tg_inputs as TI
from learned_token_pruning_residual_b300 import build as tgbuild
import learned_token_pruning_residual_b300 as tg
from gpu_helpers import to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    tgbuild.build()
    tg.lib()
    assert tg.tg_get_device_status(raise_on_error=False) == 0


def _noalloc(L, s, b, e, K):
    N = s.shape[0]
    M = N - (e - b) + K
    out = torch.full((M,), -1, dtype=torch.int32, device=s.device)
    m = ctypes.c_int64(-1)
    st = L.tg_select_topk_noalloc(ctypes.c_void_p(s.data_ptr()), N, b, e, K,
                                  ctypes.c_void_p(out.data_ptr()), ctypes.byref(m),
                                  ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, L.tg_last_error_message()
    assert m.value == M
    return out


def test_noalloc_select_matches_select_on_two_calls_in_a_row():
    L = tg.lib()
    cases = [(131072, 0, 130816, 8176, 21), (16384, 0, 16128, 1612, 22)]
    for N, b, e, K, seed in cases:
        s = to_dev(TI.random_scores(N, seed=seed))
        ref = tg.tg_select_topk(s, b, e, K, workspace=tg.new_select_workspace())
        got = _noalloc(L, s, b, e, K)
        torch.cuda.synchronize()
        assert torch.equal(got, ref), (N, K)
    assert tg.tg_get_device_status(raise_on_error=False) == 0


def test_noalloc_select_argument_errors():
    L = tg.lib()
    m = ctypes.c_int64(-1)
    assert L.tg_select_topk_noalloc(None, 10, 2, 20, 1, None, ctypes.byref(m), None) == 1
    assert L.tg_select_topk_noalloc(None, 10, 2, 5, 4, None, ctypes.byref(m), None) == 1
    assert L.tg_select_topk_noalloc(None, 3, 0, 3, 0, None, ctypes.byref(m), None) == 0
    assert m.value == 0
