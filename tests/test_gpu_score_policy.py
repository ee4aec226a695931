"""The decayed-score admission policy (MOE_POLICY_SCORE) on the GPU against the
oracle: every call's plan (slots, bypassed misses, evictions) bit-exact, outputs
within 1e-3, counters equal; outputs bitwise those of an LRU handle (every pair
is computed from the same bytes in the same order, cached or not)."""
import numpy as np
import pytest

import synth
from tests.gpu_util import DECODE_TOL, Pair, assert_plan_equal, assert_stats_equal, pinned_store, row_rel_err

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("fill_mode", [1, 0])
@pytest.mark.parametrize("budget", [0, 1])
def test_score_policy_decode_shape(fill_mode, budget):
    sh = synth.DECODE
    L = 2
    store = pinned_store(L, sh.E, sh.H, sh.F, seed=7)
    steps = 40
    _, logits, x = synth.decode_inputs(sh, steps, batch=1, seed=7, layers=list(range(L)))
    p = Pair(L, sh.E, sh.k, sh.H, sh.F, sh.S, store, max_tokens=1, fill_mode=fill_mode, policy=1,
             admit_budget=budget)
    worst = 0.0
    for s in range(steps):
        for li in range(L):
            check = s in (0, 10, steps - 1) or s % 7 == 3
            g, plan, r = p.step(li, logits[s, li], x[s, li], compute_oracle=check)
            assert_plan_equal(plan, r, f"step {s} layer {li}")
            if check:
                worst = max(worst, row_rel_err(g, r["out"]).max())
    assert worst <= DECODE_TOL, worst
    for li in range(L):
        assert_stats_equal(p.gpu.stats(li), p.orc.stats(li))
    st = p.gpu.stats(-1)
    assert st["evictions"] > 0 and st["poisoned"] == 0
    if budget == 1:                                # calls with two or more misses bypass all but one
        assert st["bypassed"] > 0
    p.close()


@pytest.mark.parametrize("fill_mode,sticky", [(1, 300), (0, 300), (1, 1000)])
def test_sticky_share(fill_mode, sticky):
    # the highest-scoring share of occupied slots is never evicted: plans
    # bit-exact against the oracle; a share of 1000 evicts nothing at all
    sh = synth.DECODE
    store = pinned_store(1, sh.E, sh.H, sh.F, seed=9)
    steps = 60
    _, logits, x = synth.decode_inputs(sh, steps, batch=1, seed=9, layers=[0])
    p = Pair(1, sh.E, sh.k, sh.H, sh.F, sh.S, store, max_tokens=1, fill_mode=fill_mode, policy=1,
             sticky=sticky)
    for s in range(steps):
        check = s in (0, 30, steps - 1)
        g, plan, r = p.step(0, logits[s, 0], x[s, 0], compute_oracle=check)
        assert_plan_equal(plan, r, f"step {s}")
        if check:
            assert row_rel_err(g, r["out"]).max() <= DECODE_TOL
    assert_stats_equal(p.gpu.stats(0), p.orc.stats(0))
    st = p.gpu.stats(0)
    assert (st["evictions"] == 0) == (sticky == 1000)
    if sticky == 1000:                             # full slots: every later miss is bypassed
        assert st["bypassed"] > 0
    p.close()


def test_score_policy_four_token_calls():
    # 4 tokens x top-8 = 32 picks <= 32 slots: still one stage
    sh = synth.DECODE
    store = pinned_store(1, sh.E, sh.H, sh.F, seed=8)
    _, logits, x = synth.batch_inputs(sh, 12, 4, seed=8, layers=[0], act="f32")
    p = Pair(1, sh.E, sh.k, sh.H, sh.F, sh.S, store, max_tokens=4, fill_mode=1, policy=1)
    for b in range(12):
        g, plan, r = p.step(0, logits[b, 0], x[b, 0], compute_oracle=b % 4 == 3)
        assert_plan_equal(plan, r, f"batch {b}")
        if b % 4 == 3:
            assert row_rel_err(g, r["out"]).max() <= DECODE_TOL
    assert_stats_equal(p.gpu.stats(0), p.orc.stats(0))
    p.close()


def test_score_policy_outputs_equal_lru_outputs():
    import torch
    import router_softmax_top_gb300 as moe
    sh = synth.DECODE
    store = pinned_store(1, sh.E, sh.H, sh.F, seed=9)
    _, logits, x = synth.decode_inputs(sh, 30, batch=1, seed=9, layers=[0])
    kw = dict(n_layers=1, n_experts=sh.E, top_k=sh.k, hidden=sh.H, ffn=sh.F, slots_per_layer=sh.S,
              max_tokens=1, store=store, fill_mode=moe.MOE_FILL_PULL)
    a = moe.MoECache(**kw)
    b = moe.MoECache(**kw, policy=moe.MOE_POLICY_SCORE, admit_budget=1)
    for s in range(30):
        lg = torch.from_numpy(logits[s, 0]).cuda()
        xd = torch.from_numpy(x[s, 0]).cuda()
        assert torch.equal(a.forward(0, lg, xd), b.forward(0, lg, xd)), s
    assert b.stats(0)["bypassed"] > 0
    assert a.stats(0)["unique_hits"] != b.stats(0)["unique_hits"] or a.stats(0)["evictions"] != b.stats(0)["evictions"]
    a.close()
    b.close()


def test_score_policy_rejects_multi_stage_configs():
    import router_softmax_top_gb300 as moe
    sh = synth.TINY
    store = pinned_store(1, sh.E, sh.H, sh.F, seed=0)
    with pytest.raises(moe.MoeError) as ei:       # 4 tokens x top-2 > 4 slots: calls could stage
        moe.MoECache(n_layers=1, n_experts=sh.E, top_k=sh.k, hidden=sh.H, ffn=sh.F, slots_per_layer=sh.S,
                     max_tokens=4, store=store, fill_mode=moe.MOE_FILL_PULL, policy=moe.MOE_POLICY_SCORE)
    assert ei.value.code == moe.MOE_ERR_UNSUPPORTED
    c = moe.MoECache(n_layers=1, n_experts=sh.E, top_k=sh.k, hidden=sh.H, ffn=sh.F, slots_per_layer=sh.S,
                     max_tokens=2, store=store, fill_mode=moe.MOE_FILL_PULL, policy=moe.MOE_POLICY_SCORE)
    c.close()
