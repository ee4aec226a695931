"""Warm start from a usage profile on the GPU against the oracle: the slot maps
after the preload and through the following calls bit-exact, outputs within
1e-3, the slots holding the right bytes (bitwise the outputs of a cold handle)."""
import numpy as np
import pytest

import synth
from tests.gpu_util import DECODE_TOL, Pair, assert_plan_equal, assert_stats_equal, pinned_store, row_rel_err

pytestmark = pytest.mark.gpu


def _profile(picks, L, E):
    # usage counts [L, E] from a trace's picks [steps, L, T, k]
    counts = np.zeros((L, E), np.uint32)
    for li in range(L):
        np.add.at(counts[li], picks[:, li].reshape(-1), 1)
    return counts


@pytest.mark.parametrize("fill_mode", [1, 0])
def test_preload_then_decode_parity(fill_mode):
    sh = synth.DECODE
    L = 2
    store = pinned_store(L, sh.E, sh.H, sh.F, seed=11)
    picks, logits, x = synth.decode_inputs(sh, 200, batch=1, seed=11, layers=list(range(L)))
    counts = _profile(picks[40:], L, sh.E)        # the same routing, other tokens
    p = Pair(L, sh.E, sh.k, sh.H, sh.F, sh.S, store, max_tokens=1, fill_mode=fill_mode)
    p.gpu.preload(counts)
    p.orc.preload(counts)
    worst = 0.0
    for s in range(30):
        for li in range(L):
            check = s in (0, 1, 29) or s % 9 == 4
            g, plan, r = p.step(li, logits[s, li], x[s, li], compute_oracle=check)
            assert_plan_equal(plan, r, f"step {s} layer {li}")
            if check:
                worst = max(worst, row_rel_err(g, r["out"]).max())
    assert worst <= DECODE_TOL, worst
    for li in range(L):
        assert_stats_equal(p.gpu.stats(li), p.orc.stats(li))
    p.close()


def test_preloaded_slots_hold_the_store_blocks():
    # a call whose picks were all preloaded: all hits, and bitwise the outputs of
    # a cold handle (which reads the same blocks from the host store)
    import torch
    import router_softmax_top_gb300 as moe
    sh = synth.DECODE
    store = pinned_store(1, sh.E, sh.H, sh.F, seed=12)
    picks, logits, x = synth.decode_inputs(sh, 12, batch=1, seed=12, layers=[0])
    n = max(s for s in range(1, 13) if len(np.unique(picks[:s, 0])) <= sh.S)
    assert n >= 3
    counts = np.zeros((1, sh.E), np.uint32)
    counts[0, np.unique(picks[:n, 0])] = 1
    kw = dict(n_layers=1, n_experts=sh.E, top_k=sh.k, hidden=sh.H, ffn=sh.F, slots_per_layer=sh.S,
              max_tokens=1, store=store, fill_mode=moe.MOE_FILL_PULL)
    warm, cold = moe.MoECache(**kw), moe.MoECache(**kw)
    warm.preload(counts)
    for s in range(n):
        lg = torch.from_numpy(logits[s, 0]).cuda()
        xd = torch.from_numpy(x[s, 0]).cuda()
        assert torch.equal(warm.forward(0, lg, xd), cold.forward(0, lg, xd)), s
    st = warm.stats(0)
    assert st["unique_misses"] == 0 and st["unique_hits"] == n * sh.k and st["calls"] == n
    warm.close()
    cold.close()
