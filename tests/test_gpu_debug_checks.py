"""Debug runs (MOE_CHECK_PLANS=1): every call's plan and slot table are checked
on the host after the call; the real plans of every schedule must pass, and
the outputs stay those of the oracle (GPU)."""
import os

import numpy as np
import pytest

import synth
from tests.gpu_util import DECODE_TOL, Pair, assert_plan_equal, pinned_store, row_rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture
def checks_on():
    os.environ["MOE_CHECK_PLANS"] = "1"
    yield
    del os.environ["MOE_CHECK_PLANS"]


@pytest.mark.parametrize("fill_mode,policy,T,S", [(1, 0, 1, 32), (0, 0, 1, 32), (1, 1, 1, 32), (0, 0, 64, 8),
                                                (1, 2, 64, 8), (1, 0, 64, 128)])
def test_checked_calls_pass(checks_on, fill_mode, policy, T, S):
    sh = synth.SWEEP
    store = pinned_store(1, sh.E, sh.H, sh.F, seed=0)
    p = Pair(1, sh.E, sh.k, sh.H, sh.F, S, store, max_tokens=T, fill_mode=fill_mode, policy=policy)
    assert p.gpu.cfg.max_tokens == T
    _, logits, x = synth.batch_inputs(sh, 6, T, seed=2, zipf=1.2, sticky=0.3, act="f32")
    for b in range(6):
        check = b in (0, 5)
        g, plan, r = p.step(0, logits[b, 0], x[b, 0], compute_oracle=check)
        assert_plan_equal(plan, r, f"batch {b}")
        if check:
            assert row_rel_err(g, r["out"]).max() <= DECODE_TOL
    st = p.gpu.stats(-1)
    assert st["poisoned"] == 0 and st["calls"] == 6
    p.close()


def test_checks_are_off_by_default():
    sh = synth.TINY
    store = pinned_store(1, sh.E, sh.H, sh.F, seed=0)
    assert "MOE_CHECK_PLANS" not in os.environ
    p = Pair(1, sh.E, sh.k, sh.H, sh.F, sh.S, store, max_tokens=4)
    lg, x = synth.tiny_inputs(0)
    g, plan, r = p.step(0, lg, x)
    assert np.array_equal(plan["gpu_slot"], r["gpu_slot"])
    p.close()
