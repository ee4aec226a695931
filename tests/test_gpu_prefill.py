"""Prefill path: token-sorted grouped GEMM on tcgen05 tensor cores (bf16 operands,
fp32 accumulate), against the CPU oracle (GPU).

Tolerance 2e-2 max relative error per token row (weights and h rounded to bf16
on the tensor-core path; the oracle is exact in double).  Slot maps bit-exact."""
import numpy as np
import pytest

import oracle
import synth
from tests.gpu_util import (PREFILL_TOL, Pair, assert_plan_equal, assert_stats_equal,
                            pinned_store, row_rel_err)

pytestmark = pytest.mark.gpu


def _pair(sh, store, S, T, gemm=True, fill_mode=0):
    return Pair(1, sh.E, sh.k, sh.H, sh.F, S, store, max_tokens=T, act="bf16", fill_mode=fill_mode,
                gemm_min_tokens=16 if gemm else 0)


@pytest.mark.parametrize("fill_mode", [0, 1])
def test_prefill_shape_gemm_parity(fill_mode):
    sh = synth.PREFILL
    store = pinned_store(1, sh.E, sh.H, sh.F, seed=0)
    T = 96
    _, logits, x = synth.batch_inputs(sh, 2, T, seed=0, layers=[0], act="bf16")
    p = _pair(sh, store, sh.S, T, fill_mode=fill_mode)
    for b in range(2):
        g, plan, r = p.step(0, logits[b, 0], x[b, 0])
        assert_plan_equal(plan, r, f"batch {b}")
        err = row_rel_err(g, r["out"])
        assert err.max() <= PREFILL_TOL, err.max()
    assert p.gpu.stats(0)["staged_calls"] >= 1      # more distinct experts than 32 slots
    assert_stats_equal(p.gpu.stats(0), p.orc.stats(0))
    p.close()


def test_tiny_shape_gemm_parity():
    # H = 256, F = 512: several M tiles, 4 K chunks, 4 slots (staged)
    sh = synth.TINY
    store = pinned_store(1, sh.E, sh.H, sh.F, seed=0)
    rng = np.random.default_rng(3)
    T = 40
    lg = rng.standard_normal((T, sh.E)).astype(np.float32)
    x = synth.normal_bf16_bits(T * sh.H, 0, synth.PURPOSE_X, 99, 0).reshape(T, sh.H)
    p = Pair(1, sh.E, sh.k, sh.H, sh.F, sh.S, store, max_tokens=T, act="bf16", gemm_min_tokens=16)
    g, plan, r = p.step(0, lg, x)
    assert_plan_equal(plan, r)
    assert row_rel_err(g, r["out"]).max() <= PREFILL_TOL
    p.close()


def test_gemm_budget_invariance_and_gemv_agreement():
    sh = synth.PREFILL
    store = pinned_store(1, sh.E, sh.H, sh.F, seed=0)
    T = 64
    _, logits, x = synth.batch_inputs(sh, 1, T, seed=1, layers=[0], act="bf16")
    outs = {}
    for S in (8, 32, 128):
        p = _pair(sh, store, S, T)
        g, plan, r = p.step(0, logits[0, 0], x[0, 0], compute_oracle=(S == 128))
        assert_plan_equal(plan, r, f"S={S}")
        if S == 128:
            assert row_rel_err(g, r["out"]).max() <= PREFILL_TOL
        outs[S] = g
        p.close()
    assert np.array_equal(outs[8], outs[128])
    assert np.array_equal(outs[32], outs[128])
    # the fp32 GEMV path on the same inputs agrees within the bf16 tolerance
    p = _pair(sh, store, 128, T, gemm=False)
    g, _, _ = p.step(0, logits[0, 0], x[0, 0], compute_oracle=False)
    assert row_rel_err(outs[128], g).max() <= PREFILL_TOL
    p.close()


@pytest.mark.parametrize("fill_mode", [0, 1])
def test_full_prefill_batch_all_rows(fill_mode):
    # two 512-token batches of the prefill model through the GEMM path, every
    # output row compared with the oracle.  Their hottest experts get 428 and
    # 439 routed pairs, so the GEMM's units of 128 pairs reach a fourth N tile
    # of one expert; slot maps and counters bit-exact
    sh = synth.PREFILL
    store = pinned_store(1, sh.E, sh.H, sh.F, seed=0)
    T = 512
    picks, logits, x = synth.batch_inputs(sh, 2, T, seed=0, layers=[0], act="bf16")
    assert max(np.bincount(picks[b, 0].ravel()).max() for b in range(2)) > 3 * 128
    p = _pair(sh, store, sh.S, T, fill_mode=fill_mode)
    for b in range(2):
        g, plan, r = p.step(0, logits[b, 0], x[b, 0])
        assert_plan_equal(plan, r, f"batch {b}")
        err = row_rel_err(g, r["out"])
        assert err.max() <= PREFILL_TOL, (b, int(err.argmax()), err.max())
    assert_stats_equal(p.gpu.stats(0), p.orc.stats(0))
    p.close()


def test_prefill_all_resident_and_hot_experts():
    # every expert resident (128 slots), then a batch whose 512 tokens all pick
    # among 16 experts (each expert ~256 pairs: two full N tiles): all rows
    sh = synth.PREFILL
    store = pinned_store(1, sh.E, sh.H, sh.F, seed=0)
    T = 512
    _, logits, x = synth.batch_inputs(sh, 2, T, seed=3, layers=[0], act="bf16")
    hot = synth.trace(T, 16, sh.k, 0.0, 0.0, 5, 0, 0)
    hot_logits = synth.logits_from_picks(hot, sh.E, 5, 0, 0, 1)
    p = _pair(sh, store, sh.E, T)
    for b, lg in enumerate([logits[0, 0], logits[1, 0], hot_logits]):
        g, plan, r = p.step(0, lg, x[b % 2, 0])
        assert_plan_equal(plan, r, f"batch {b}")
        assert row_rel_err(g, r["out"]).max() <= PREFILL_TOL, b
    assert_stats_equal(p.gpu.stats(0), p.orc.stats(0))
    p.close()
