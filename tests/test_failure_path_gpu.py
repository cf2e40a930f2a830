"""The failure path on the GPU: a bounded wait that runs out.

Every pipeline wait of the library gives up after a bound, sets
TG_ERR_TIMEOUT in the device status word and an abort flag that makes the
CTA's other waiters leave.  tg_selftest_bounded_wait builds that situation
with an mbarrier that nothing completes.  The test checks the status, that
reading it clears it, that the abort flag ended the second waiter long
before its own 2 s bound, and that the next real call still matches the
oracle.  No trap, no fault, no unbounded wait."""
import time

import numpy as np
import pytest
import torch

import oracle as O
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


@pytest.mark.parametrize("timeout_us", [200, 5000])
def test_wait_runs_out_and_sets_timeout(timeout_us):
    report = torch.zeros(4, dtype=torch.int64, device="cuda")
    t0 = time.perf_counter()
    tg.tg_selftest_bounded_wait(timeout_us, report)
    st = tg.tg_get_device_status(raise_on_error=False)
    host_s = time.perf_counter() - t0
    assert st == 6  # TG_ERR_TIMEOUT
    # reading the status cleared it
    assert tg.tg_get_device_status(raise_on_error=False) == 0
    ok0, ns0, ok1, ns1 = report.cpu().tolist()
    assert ok0 == 0 and ok1 == 0  # both waits gave up
    assert ns0 >= timeout_us * 1000  # the short bound ran out ...
    assert ns0 < timeout_us * 1000 + 5_000_000  # ... and not much later
    assert ns1 < 1_000_000_000  # the 2 s waiter left on the abort flag, well before its bound
    assert host_s < 1.9


def test_device_usable_after_timeout():
    tg.tg_selftest_bounded_wait(100)
    assert tg.tg_get_device_status(raise_on_error=False) == 6
    s = TI.adversarial_scores("quantised", 40000, seed=3)
    idx = tg.tg_select_topk(to_dev(s), 100, 39000, 4321).cpu().numpy()
    assert np.array_equal(idx, O.select_topk(s, 100, 39000, 4321))
    assert tg.tg_get_device_status(raise_on_error=False) == 0
