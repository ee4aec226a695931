"""CUDA path vs the CPU oracle, through the C ABI (GPU).

Slot maps, miss lists (expert, slot, evicted, stage), stage assignment and
counters must match bit for bit; outputs within 1e-3 max relative error per
token row (fp32-accumulate paths)."""
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


@pytest.mark.parametrize("fill_mode", [0, 1])
def test_tiny_parity(tiny_store, fill_mode):
    logits, x = synth.tiny_inputs(0)
    p = Pair(TINY.L, TINY.E, TINY.k, TINY.H, TINY.F, TINY.S, tiny_store, max_tokens=4,
             fill_mode=fill_mode)
    # one call of 4 tokens (usually staged: more distinct experts than 4 slots) ...
    g, plan, r = p.step(0, logits, x)
    assert_plan_equal(plan, r, "T=4")
    assert row_rel_err(g, r["out"]).max() <= DECODE_TOL
    # ... then the same tokens as 4 sequential single-token calls (evictions)
    for t in range(4):
        g, plan, r = p.step(0, logits[t:t + 1], x[t:t + 1])
        assert_plan_equal(plan, r, f"t={t}")
        assert row_rel_err(g, r["out"]).max() <= DECODE_TOL
    assert_stats_equal(p.gpu.stats(0), p.orc.stats(0))
    p.close()


def test_tiny_budget_invariance(tiny_store):
    logits, x = synth.tiny_inputs(0)
    outs = {}
    for S in range(1, TINY.E + 1):
        p = Pair(TINY.L, TINY.E, TINY.k, TINY.H, TINY.F, S, tiny_store, max_tokens=4)
        got = []
        g, plan, r = p.step(0, logits, x)
        assert_plan_equal(plan, r, f"S={S}")
        got.append(g)
        for t in range(4):
            g, plan, r = p.step(0, logits[t:t + 1], x[t:t + 1])
            assert_plan_equal(plan, r, f"S={S} t={t}")
            got.append(g)
        outs[S] = got
        p.close()
    for S in outs:
        for a, b in zip(outs[S], outs[TINY.E]):
            assert np.array_equal(a, b), S      # bitwise: any budget, same result


@pytest.mark.parametrize("fill_mode", [0, 1])
def test_decode_shape_parity(fill_mode):
    # the decode model's shapes (E=128, H=2816, F=704, 32 slots) on 2 of its layers
    sh = synth.DECODE
    layers = [0, 1]
    store = pinned_store(len(layers), sh.E, sh.H, sh.F, seed=0)
    steps = 40
    picks, logits, x = synth.decode_inputs(sh, steps, batch=1, seed=0, layers=layers)
    p = Pair(len(layers), sh.E, sh.k, sh.H, sh.F, sh.S, store, max_tokens=1, fill_mode=fill_mode)
    worst = 0.0
    for s in range(steps):
        for li in range(len(layers)):
            check = (s % 8 == 0) or s == steps - 1
            g, plan, r = p.step(li, logits[s, li], x[s, li], compute_oracle=check)
            assert_plan_equal(plan, r, f"step {s} layer {li}")
            assert set(plan["ids"][0].tolist()) == set(picks[s, li, 0].tolist())
            if check:
                worst = max(worst, row_rel_err(g, r["out"]).max())
    assert worst <= DECODE_TOL, worst
    for li in range(len(layers)):
        assert_stats_equal(p.gpu.stats(li), p.orc.stats(li))
    st = p.gpu.stats(-1)
    assert st["pick_hits"] > 0 and st["unique_misses"] > 0
    p.close()


@pytest.mark.parametrize("routing", ["uniform", "zipf"])
def test_sweep_budgets(routing):
    # over-budget sweep: 64 tokens/batch, budgets 8..128 (staged below |U|)
    sh = synth.SWEEP
    store = pinned_store(1, sh.E, sh.H, sh.F, seed=0)
    n_batches = 4
    zipf = 0.0 if routing == "uniform" else 1.2
    _, logits, x = synth.batch_inputs(sh, n_batches, 64, seed=0, zipf=zipf, sticky=0.0, act="f32")
    outs = {}
    for S in (8, 16, 32, 64, 128):
        p = Pair(1, sh.E, sh.k, sh.H, sh.F, S, store, max_tokens=64)
        got = []
        for b in range(n_batches):
            check = S in (8, 128) and b in (0, n_batches - 1)
            g, plan, r = p.step(0, logits[b, 0], x[b, 0], compute_oracle=check)
            assert_plan_equal(plan, r, f"S={S} batch {b}")
            if check:
                assert row_rel_err(g, r["out"]).max() <= DECODE_TOL
            got.append(g)
        assert_stats_equal(p.gpu.stats(0), p.orc.stats(0))
        if S == 8:
            assert p.gpu.stats(0)["staged_calls"] == n_batches
        outs[S] = got
        p.close()
    for S in outs:
        for a, b in zip(outs[S], outs[128]):
            assert np.array_equal(a, b), S


def test_bf16_activations_gemv_path():
    sh = synth.PREFILL
    store = pinned_store(1, sh.E, sh.H, sh.F, seed=0)
    _, logits, x = synth.batch_inputs(sh, 2, 32, seed=0, layers=[0], act="bf16")
    p = Pair(1, sh.E, sh.k, sh.H, sh.F, sh.S, store, max_tokens=32, act="bf16")
    for b in range(2):
        g, plan, r = p.step(0, logits[b, 0], x[b, 0])
        assert_plan_equal(plan, r, f"batch {b}")
        assert row_rel_err(g, r["out"]).max() <= DECODE_TOL
    p.close()


def test_weight_mode_renormalised(tiny_store):
    logits, x = synth.tiny_inputs(0)
    p = Pair(TINY.L, TINY.E, TINY.k, TINY.H, TINY.F, 8, tiny_store, max_tokens=4, weight_mode=1)
    g, plan, r = p.step(0, logits, x)
    assert_plan_equal(plan, r)
    np.testing.assert_allclose(plan["w"].sum(axis=1), 1.0, rtol=1e-6)
    assert row_rel_err(g, r["out"]).max() <= DECODE_TOL
    p.close()


@pytest.mark.parametrize("batch", [1, 8])
def test_large_shape_subset(batch):
    # the large model's shapes (E=256, H=4096, F=1536, 64 slots) on one layer
    sh = synth.LARGE
    store = pinned_store(1, sh.E, sh.H, sh.F, seed=0)
    steps = 24
    _, logits, x = synth.decode_inputs(sh, steps, batch=batch, seed=0, layers=[0])
    p = Pair(1, sh.E, sh.k, sh.H, sh.F, sh.S, store, max_tokens=batch, fill_mode=1)
    for s in range(steps):
        check = s in (0, steps // 2, steps - 1)
        g, plan, r = p.step(0, logits[s, 0], x[s, 0], compute_oracle=check)
        assert_plan_equal(plan, r, f"step {s}")
        if check:
            assert row_rel_err(g, r["out"]).max() <= DECODE_TOL
    assert_stats_equal(p.gpu.stats(0), p.orc.stats(0))
    p.close()


def test_single_expert_dense_case():
    # E = k = 1: one dense Q4_0 SwiGLU FFN, router weight exactly 1
    H, F = 256, 512
    store = pinned_store(1, 1, H, F, seed=5)
    rng = np.random.default_rng(5)
    p = Pair(1, 1, 1, H, F, 1, store, max_tokens=3)
    x = rng.standard_normal((3, H)).astype(np.float32)
    lg = rng.standard_normal((3, 1)).astype(np.float32)
    g, plan, r = p.step(0, lg, x)
    assert np.all(plan["w"] == 1.0)
    assert row_rel_err(g, r["out"]).max() <= DECODE_TOL
    p.close()
