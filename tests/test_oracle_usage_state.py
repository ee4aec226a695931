"""Lifetime usage counts and resumable slot-table state (the oracle, CPU only).

"Persistent hot experts" ("llama.cpp: fork with multi gpu acceleration ...")
keeps how often each expert was used, per layer, and preloads the most-used
ones at the next start.  The counts are pinned here against a numpy top-k of
the logits (not the oracle's router) and hand-worked cases; the resumable
state against hand-worked eviction traces and against an uninterrupted run."""
import numpy as np
import pytest

import oracle
import synth


def _topk(lg: np.ndarray, k: int) -> np.ndarray:
    # highest logit first, ties to the lower id (stable sort of the negated row)
    return np.argsort(-lg, axis=1, kind="stable")[:, :k]


def _tiny(L=1, S=4, E=8, **kw):
    sh = synth.TINY
    store = synth.store(L, E, sh.H, sh.F, seed=4)
    return oracle.Cache(L, E, sh.k, sh.H, sh.F, S, store, **kw)


def _picks(E, *tokens):
    lg = np.full((len(tokens), E), -3.0, np.float32)
    for t, tok in enumerate(tokens):
        for j, e in enumerate(tok):
            lg[t, e] = 2.0 - j
    return lg


def test_usage_hand_worked():
    c = _tiny()
    assert c.k == 2
    c.forward(0, _picks(8, (1, 7), (1, 3)), None, compute=False)
    c.forward(0, _picks(8, (3, 1)), None, compute=False)
    assert c.usage()[0].tolist() == [0, 3, 0, 2, 0, 0, 0, 1]


@pytest.mark.parametrize("policy,budget,S", [(oracle.POLICY_LRU, 0, 8), (oracle.POLICY_SCORE, 1, 16),
                                             (oracle.POLICY_ADOPT, 0, 8)])
def test_usage_counts_every_routed_pick(policy, budget, S):
    # hits, misses, bypassed misses (score policy, budget 1) and staged calls
    # all count once per (token, pick); each layer counts its own calls
    sh = synth.SWEEP
    L = 2
    c = oracle.Cache(L, sh.E, sh.k, sh.H, sh.F, S, np.zeros(1, np.uint8), policy=policy, admit_budget=budget)
    rng = np.random.default_rng(11)
    want = np.zeros((L, sh.E), np.int64)
    for i in range(12):
        layer = i % L
        T = 1 if policy == oracle.POLICY_SCORE else int(rng.integers(1, 24))
        lg = (rng.standard_normal((T, sh.E)) * 2).astype(np.float32)
        c.forward(layer, lg, None, compute=False)
        np.add.at(want[layer], _topk(lg, sh.k).ravel(), 1)
    assert np.array_equal(c.usage().astype(np.int64), want)
    assert int(c.usage().sum()) == sum(c.stats(l)["pick_hits"] + c.stats(l)["pick_misses"] for l in range(L))
    if policy == oracle.POLICY_SCORE:
        assert sum(c.stats(l)["bypassed"] for l in range(L)) > 0
    if policy == oracle.POLICY_ADOPT:
        assert sum(c.stats(l)["staged_calls"] for l in range(L)) > 0


def test_rejected_calls_and_preload_count_nothing():
    c = _tiny(policy=oracle.POLICY_SCORE)
    c.forward(0, _picks(8, (2, 5)), None, compute=False)
    before = c.usage().copy()
    bad = _picks(8, (1, 3))
    bad[0, 6] = np.nan
    with pytest.raises(ValueError):
        c.forward(0, bad, None, compute=False)
    with pytest.raises(ValueError):                                # 6 distinct experts > 4 slots
        c.forward(0, _picks(8, (0, 1), (2, 3), (4, 6)), None, compute=False)
    c.preload(np.ones((1, 8), np.uint32))
    assert np.array_equal(c.usage(), before)


def test_usage_feeds_the_next_preload():
    # the page's loop: counts kept by one session warm the next one's slots
    a = _tiny(S=3)
    a.forward(0, _picks(8, (4, 6), (4, 1)), None, compute=False)
    a.forward(0, _picks(8, (6, 4), (2, 0)), None, compute=False)
    assert a.usage()[0].tolist() == [1, 1, 1, 0, 3, 0, 2, 0]
    b = _tiny(S=3)
    b.preload(a.usage())
    assert b.lru(0).state()["slot_expert"].tolist() == [4, 6, 0]   # 3, 2, then the 1s by id


def test_set_state_hand_worked_evictions():
    c = _tiny(S=4)
    assert c.set_state(0, [3, -1, 5, 0], np.array([7, 0, 2, 9], np.uint64), 9,
                       np.zeros(8, np.float32), np.zeros(8, np.uint32))
    st = c.lru(0).state()
    assert st["expert_slot"].tolist() == [3, -1, -1, 0, -1, 2, -1, -1] and st["clock"] == 9
    r = c.forward(0, _picks(8, (6, 5)), None, compute=False)       # 5 hits slot 2; 6 takes empty slot 1
    assert r["gpu_slot"].tolist() == [[1, 2]]
    assert r["miss_slot"].tolist() == [1] and r["miss_evicted"].tolist() == [-1]
    r = c.forward(0, _picks(8, (1, 2)), None, compute=False)       # victims: slot 0 (stamp 7), slot 3 (9)
    assert r["miss_expert"].tolist() == [1, 2]
    assert r["miss_slot"].tolist() == [0, 3] and r["miss_evicted"].tolist() == [3, 0]
    st = c.lru(0).state()
    assert st["slot_stamp"].tolist() == [11, 10, 10, 11] and st["clock"] == 11


def test_set_state_restores_scores_and_usage():
    c = _tiny(S=2, policy=oracle.POLICY_SCORE)
    score = np.array([0, 0, 0, 3.0, 0, 0.5, 0, 0], np.float32)
    usage = np.arange(8, dtype=np.uint32) * 10
    assert c.set_state(0, [3, 5], np.array([1, 1], np.uint64), 1, score, usage)
    # expert 6 missed: score 1.0 after this token; the weakest unpicked slot
    # holds 5 (0.5 x 0.9 = 0.45), so 6 is admitted over it
    r = c.forward(0, _picks(8, (3, 6)), None, compute=False)
    assert r["miss_expert"].tolist() == [6] and r["miss_slot"].tolist() == [1]
    assert r["miss_evicted"].tolist() == [5]
    assert c.usage()[0].tolist() == (usage + np.array([0, 0, 0, 1, 0, 0, 1, 0], np.uint32)).tolist()
    assert c.lru(0).scores()[3] == np.float32(np.float32(3.0) * np.float32(0.9)) + np.float32(1.0)


@pytest.mark.parametrize("edit", ["range", "dup", "stamp", "nan", "neg"])
def test_set_state_rejects_invalid_tables(edit):
    c = _tiny(S=4)
    c.forward(0, _picks(8, (2, 5)), None, compute=False)
    before = c.state(0)
    se, ss = np.array([1, 4, -1, 6], np.int32), np.array([3, 2, 0, 1], np.uint64)
    sc, us = np.zeros(8, np.float32), np.zeros(8, np.uint32)
    if edit == "range":
        se[2] = 8
    elif edit == "dup":
        se[3] = 1
    elif edit == "stamp":
        ss[0] = 4
    elif edit == "nan":
        sc[2] = np.nan
    else:
        sc[2] = -1.0
    assert not c.set_state(0, se, ss, 3, sc, us)
    after = c.state(0)
    for key in before:
        assert np.array_equal(np.asarray(before[key]), np.asarray(after[key])), key


@pytest.mark.parametrize("policy,S", [(oracle.POLICY_LRU, 4), (oracle.POLICY_SCORE, 6), (oracle.POLICY_ADOPT, 3)])
def test_resumed_cache_equals_uninterrupted(policy, S):
    sh = synth.TINY
    L = 2
    store = synth.store(L, sh.E, sh.H, sh.F, seed=9)
    a = oracle.Cache(L, sh.E, sh.k, sh.H, sh.F, S, store, policy=policy, admit_budget=1)
    rng, rng_x = np.random.default_rng(5), np.random.default_rng(6)
    batches = []
    for i in range(24):
        # short calls leave slots untouched, so recency decides evictions;
        # adopt needs the odd staged call (more distinct experts than slots)
        T = 1 if policy == oracle.POLICY_SCORE else (3 if policy == oracle.POLICY_ADOPT and i % 4 == 3 else
                                                     int(rng.integers(1, 3)))
        batches.append((i % L, rng.standard_normal((T, sh.E)).astype(np.float32) * 2,
                        rng_x.standard_normal((T, sh.H)).astype(np.float32)))
    for layer, lg, x in batches[:12]:
        a.forward(layer, lg, x)
    b = oracle.Cache(L, sh.E, sh.k, sh.H, sh.F, S, store, policy=policy, admit_budget=1)
    stale = oracle.Cache(L, sh.E, sh.k, sh.H, sh.F, S, store, policy=policy, admit_budget=1)
    for layer in range(L):
        st = a.state(layer)
        assert b.set_state(layer, st["slot_expert"], st["slot_stamp"], st["clock"], st["score"], st["usage"])
        # the same slot contents with every recency stamp and score dropped
        assert stale.set_state(layer, st["slot_expert"], np.zeros(S, np.uint64), st["clock"],
                               np.zeros(sh.E, np.float32), st["usage"])
    diverged = False
    for layer, lg, x in batches[12:]:
        ra, rb, rs = a.forward(layer, lg, x), b.forward(layer, lg, x), stale.forward(layer, lg, x)
        for key in ("gpu_slot", "stage", "miss_expert", "miss_slot", "miss_evicted"):
            assert np.array_equal(ra[key], rb[key]), key
            diverged |= not np.array_equal(ra[key], rs[key])
        assert np.array_equal(ra["out"], rb["out"])
        assert np.array_equal(ra["out"], rs["out"])                # outputs never depend on the slots
    assert np.array_equal(a.usage(), b.usage())
    assert diverged, "the trace must be one on which the dropped stamps and scores change a plan"
