"""Whole-layer oracle pins: exactly-once, budget invariance, stats, and an
independent numpy restatement of the layer on the tiny workload (CPU only)."""
import numpy as np
import pytest

import oracle
import synth
from tests.test_oracle_ffn import _dequant_numpy

TINY = synth.TINY


def _tiny_store():
    return synth.store(TINY.L, TINY.E, TINY.H, TINY.F, seed=0)


def _numpy_layer(store, L_idx, E, k, H, F, logits, x, weight_mode=0):
    """Independent restatement: argsort top-k, numpy softmax, numpy decode, float64 matmuls."""
    eb = 3 * F * H // 32 * 18
    mat = F * H // 32 * 18
    T = logits.shape[0]
    out = np.zeros((T, H))
    for t in range(T):
        row = logits[t].astype(np.float64)
        order = np.lexsort((np.arange(E), -row))[:k]
        p = np.exp(row - row.max())
        p /= p.sum()
        w = p[order]
        if weight_mode == 1:
            w = w / w.sum()
        for q, e in enumerate(order):
            base = (L_idx * E + e) * eb
            blk = store[base:base + eb]
            Wg = _dequant_numpy(blk[:mat].tobytes(), F, H)
            Wu = _dequant_numpy(blk[mat:2 * mat].tobytes(), F, H)
            Wd = _dequant_numpy(blk[2 * mat:].tobytes(), H, F)
            g, u = Wg @ x[t], Wu @ x[t]
            out[t] += w[q] * (Wd @ (g / (1 + np.exp(-g)) * u))
    return out


def test_tiny_layer_matches_numpy_restatement():
    store = _tiny_store()
    logits, x = synth.tiny_inputs(0)
    c = oracle.Cache(TINY.L, TINY.E, TINY.k, TINY.H, TINY.F, TINY.S, store)
    r = c.forward(0, logits, x)
    ref = _numpy_layer(store, 0, TINY.E, TINY.k, TINY.H, TINY.F, logits, x.astype(np.float64))
    np.testing.assert_allclose(r["out"], ref, rtol=1e-6, atol=1e-6 * np.abs(ref).max())
    assert np.all(r["visits"] == 1)


@pytest.mark.parametrize("mode", [0, 1])
def test_weight_modes_numpy(mode):
    store = _tiny_store()
    logits, x = synth.tiny_inputs(0)
    c = oracle.Cache(TINY.L, TINY.E, TINY.k, TINY.H, TINY.F, 8, store, weight_mode=mode)
    r = c.forward(0, logits, x)
    ref = _numpy_layer(store, 0, TINY.E, TINY.k, TINY.H, TINY.F, logits, x.astype(np.float64), mode)
    np.testing.assert_allclose(r["out"], ref, rtol=1e-6, atol=1e-6 * np.abs(ref).max())


def test_budget_invariance_and_exactly_once():
    store = _tiny_store()
    logits, x = synth.tiny_inputs(0)
    outs = {}
    for S in range(1, TINY.E + 1):
        c = oracle.Cache(TINY.L, TINY.E, TINY.k, TINY.H, TINY.F, S, store)
        # one T=4 call, then the same 4 tokens as 4 sequential T=1 calls
        r = c.forward(0, logits, x)
        assert np.all(r["visits"] == 1)
        seq = []
        for t in range(4):
            rt = c.forward(0, logits[t:t + 1], x[t:t + 1])
            assert np.all(rt["visits"] == 1)
            seq.append(rt["out"])
        outs[S] = (r["out"], np.concatenate(seq))
        st = c.stats(0)
        assert st["calls"] == 5
        assert st["pick_hits"] + st["pick_misses"] == (4 + 4) * TINY.k
    for S in outs:
        assert np.array_equal(outs[S][0], outs[TINY.E][0]), S
        assert np.array_equal(outs[S][1], outs[TINY.E][1]), S
        # a T=1 call sees the same arithmetic as its row of the T=4 call
        assert np.array_equal(outs[S][1], outs[S][0])


def test_tiny_one_call_stages_with_four_slots():
    store = _tiny_store()
    logits, x = synth.tiny_inputs(0)
    c = oracle.Cache(TINY.L, TINY.E, TINY.k, TINY.H, TINY.F, TINY.S, store)
    r = c.forward(0, logits, x)
    info = r["info"]
    n_unique = len(set(r["ids"].ravel().tolist()))
    assert info["n_unique"] == n_unique
    assert info["n_stages"] == (1 if n_unique <= 4 else 1 + -(-(n_unique - 4) // 4))
    st = c.stats(0)
    assert st["unique_misses"] == n_unique and st["unique_hits"] == 0   # cold start
    assert st["bytes_uploaded"] == n_unique * TINY.expert_bytes


def test_single_expert_reduces_to_dense_ffn():
    # E = k = 1: the router weight is 1 and the layer is one dense Q4_0 SwiGLU FFN
    H, F = 256, 512
    store = synth.store(1, 1, H, F, seed=5)
    x = np.random.default_rng(5).standard_normal((3, H)).astype(np.float32)
    logits = np.random.default_rng(6).standard_normal((3, 1)).astype(np.float32)
    c = oracle.Cache(1, 1, 1, H, F, 1, store)
    r = c.forward(0, logits, x)
    assert np.all(r["w"] == 1.0)
    for t in range(3):
        y = oracle.expert_ffn(store, H, F, x[t].astype(np.float64))
        assert np.array_equal(r["out"][t], y.astype(np.float32))


def test_identical_experts_add_weights():
    H, F = 64, 64
    one = synth.store(1, 1, H, F, seed=9)
    store = np.concatenate([one, one])
    x = np.random.default_rng(10).standard_normal((1, H)).astype(np.float32)
    logits = np.array([[0.25, -0.5]], np.float32)
    c = oracle.Cache(1, 2, 2, H, F, 2, store)
    r = c.forward(0, logits, x)
    y = oracle.expert_ffn(one, H, F, x[0].astype(np.float64))
    np.testing.assert_allclose(r["out"][0], (r["w"][0].sum() * y), rtol=1e-6, atol=1e-7)
    np.testing.assert_allclose(r["w"][0].sum(), 1.0, atol=1e-15)   # k = E: whole softmax


def test_non_finite_logit_leaves_state():
    store = _tiny_store()
    logits, x = synth.tiny_inputs(0)
    c = oracle.Cache(TINY.L, TINY.E, TINY.k, TINY.H, TINY.F, TINY.S, store)
    bad = logits.copy()
    bad[2, 1] = np.nan
    with pytest.raises(ValueError):
        c.forward(0, bad, x)
    assert c.lru(0).state()["clock"] == 0
    assert c.stats(0)["calls"] == 0


def test_plan_only_mode_matches_full():
    store = _tiny_store()
    logits, x = synth.tiny_inputs(0)
    a = oracle.Cache(TINY.L, TINY.E, TINY.k, TINY.H, TINY.F, 3, store)
    b = oracle.Cache(TINY.L, TINY.E, TINY.k, TINY.H, TINY.F, 3, store)
    for t in range(4):
        ra = a.forward(0, logits[t:t + 1], x[t:t + 1], compute=True)
        rb = b.forward(0, logits[t:t + 1], None, compute=False)
        for key in ("ids", "gpu_slot", "stage", "miss_expert", "miss_slot", "miss_evicted"):
            assert np.array_equal(ra[key], rb[key])
