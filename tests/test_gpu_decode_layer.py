"""The decode layer kernel (pull fill, single-stage calls of at most 8 tokens)
against the oracle and against the GEMV kernels of the other schedules (GPU).

Every kernel of the decode path reduces in one canonical order, so the decode
layer kernel must give bitwise the outputs of the staged GEMV path (any slot
budget) and of the copy-engine schedule, besides the oracle's slot maps and
outputs within 1e-3 max relative error."""
import numpy as np
import pytest

import synth
from tests.gpu_util import (DECODE_TOL, Pair, assert_plan_equal, assert_stats_equal,
                            pinned_store, row_rel_err)

pytestmark = pytest.mark.gpu

TINY = synth.TINY


@pytest.fixture(scope="module")
def tiny_store():
    return pinned_store(TINY.L, TINY.E, TINY.H, TINY.F, seed=0)


def test_budget_invariance_pull(tiny_store):
    # S = 8 = E: every call single-stage -> decode layer kernel (4-token and
    # 1-token variants); smaller budgets run the staged GEMV path
    logits, x = synth.tiny_inputs(0)
    outs = {}
    for S in range(1, TINY.E + 1):
        p = Pair(TINY.L, TINY.E, TINY.k, TINY.H, TINY.F, S, tiny_store, max_tokens=4, fill_mode=1)
        got = []
        g, plan, r = p.step(0, logits, x)
        assert_plan_equal(plan, r, f"S={S}")
        assert row_rel_err(g, r["out"]).max() <= DECODE_TOL
        got.append(g)
        for t in range(4):
            g, plan, r = p.step(0, logits[t:t + 1], x[t:t + 1])
            assert_plan_equal(plan, r, f"S={S} t={t}")
            got.append(g)
        outs[S] = got
        assert_stats_equal(p.gpu.stats(0), p.orc.stats(0))
        p.close()
    for S in outs:
        for a, b in zip(outs[S], outs[TINY.E]):
            assert np.array_equal(a, b), S


def test_decode_kernel_matches_copy_engine_schedule():
    # decode model shapes, 2 layers: pull (decode layer kernel) and memcpy
    # (copy engine + GEMV kernels + combine) give the same plans and bitwise
    # the same outputs
    sh = synth.DECODE
    layers = [0, 1]
    store = pinned_store(len(layers), sh.E, sh.H, sh.F, seed=1)
    steps = 24
    picks, logits, x = synth.decode_inputs(sh, steps, batch=1, seed=1, layers=layers)
    pull = Pair(len(layers), sh.E, sh.k, sh.H, sh.F, sh.S, store, max_tokens=1, fill_mode=1)
    copy = Pair(len(layers), sh.E, sh.k, sh.H, sh.F, sh.S, store, max_tokens=1, fill_mode=0)
    worst = 0.0
    for s in range(steps):
        for li in range(len(layers)):
            check = s in (0, 7, steps - 1)
            ga, pa, ra = pull.step(li, logits[s, li], x[s, li], compute_oracle=check)
            gb, pb, _ = copy.step(li, logits[s, li], x[s, li], compute_oracle=False)
            assert_plan_equal(pa, ra, f"step {s} layer {li}")
            assert np.array_equal(pa["gpu_slot"], pb["gpu_slot"])
            assert np.array_equal(ga, gb), (s, li)
            if check:
                worst = max(worst, row_rel_err(ga, ra["out"]).max())
    assert worst <= DECODE_TOL, worst
    st = pull.gpu.stats(-1)
    assert st["unique_misses"] > 0 and st["unique_hits"] > 0
    pull.close()
    copy.close()


@pytest.mark.parametrize("T", [1, 3, 4])
def test_bf16_inputs_decode_kernel(T):
    # bf16 activations through the decode layer kernel (T * k <= 32 slots: single stage)
    sh = synth.PREFILL
    store = pinned_store(1, sh.E, sh.H, sh.F, seed=2)
    _, logits, x = synth.batch_inputs(sh, 3, T, seed=2, layers=[0], act="bf16")
    p = Pair(1, sh.E, sh.k, sh.H, sh.F, sh.S, store, max_tokens=T, act="bf16", fill_mode=1)
    for b in range(3):
        g, plan, r = p.step(0, logits[b, 0], x[b, 0])
        assert_plan_equal(plan, r, f"batch {b}")
        assert row_rel_err(g, r["out"]).max() <= DECODE_TOL
    assert_stats_equal(p.gpu.stats(0), p.orc.stats(0))
    p.close()


def test_weight_mode_renormalised_pull(tiny_store):
    logits, x = synth.tiny_inputs(1)
    p = Pair(TINY.L, TINY.E, TINY.k, TINY.H, TINY.F, 8, tiny_store, max_tokens=4, weight_mode=1, fill_mode=1)
    for _ in range(2):
        g, plan, r = p.step(0, logits, x)
        assert_plan_equal(plan, r)
        np.testing.assert_allclose(plan["w"].sum(axis=1), 1.0, rtol=1e-6)
        assert row_rel_err(g, r["out"]).max() <= DECODE_TOL
    p.close()


def test_repeated_calls_reuse_slots_written_on_the_way():
    # a miss is written into its slot by the decode layer kernel while it is
    # computed; the next call's hits read those slots (checked against the oracle)
    sh = synth.DECODE
    store = pinned_store(1, sh.E, sh.H, sh.F, seed=3)
    rng = np.random.default_rng(3)
    p = Pair(1, sh.E, sh.k, sh.H, sh.F, sh.S, store, max_tokens=1, fill_mode=1)
    x = rng.standard_normal((1, sh.H)).astype(np.float32)
    lg = rng.standard_normal((1, sh.E)).astype(np.float32)
    g0, plan0, r0 = p.step(0, lg, x)           # all 8 picks miss (empty cache)
    assert_plan_equal(plan0, r0)
    g1, plan1, r1 = p.step(0, lg, x)           # same picks: all hits now
    assert_plan_equal(plan1, r1)
    assert np.array_equal(g0, g1)              # slot contents equal the host blocks
    assert row_rel_err(g1, r1["out"]).max() <= DECODE_TOL
    st = p.gpu.stats(0)
    assert st["unique_misses"] == 8 and st["unique_hits"] == 8
    p.close()
