"""The adopt policy of the oracle (CPU only): a staged call ends holding its
most-used experts ("Prefill preheat"), with the uploads and stages of LRU.

Pinned against an independent brute-force simulator (exhaustive small traces,
long random ones), hand-worked calls, and its relations to LRU."""
import itertools
import random

import numpy as np
import pytest

import oracle
import synth
from tests.adopt_bruteforce import BruteAdopt
from tests.lru_bruteforce import BruteLRU


def _compare(S, E, trace):
    o = oracle.LRU(S, E, policy=oracle.POLICY_ADOPT)
    b = BruteAdopt(S, E)
    for call in trace:
        po = o.plan(np.array(call, dtype=np.int32))
        pb = b.call([list(t) for t in call])
        where = (S, trace)
        assert po["gpu_slot"].tolist() == pb["gpu_slot"], where
        assert po["stage"].tolist() == pb["stage"], where
        recs = list(zip(po["miss_expert"].tolist(), po["miss_slot"].tolist(),
                        po["miss_evicted"].tolist(), po["miss_stage"].tolist()))
        assert recs == pb["misses"], where
        for key in ("n_unique", "n_hits", "n_miss", "n_stages", "n_evict", "pick_hits", "pick_misses"):
            assert po["info"][key] == pb[key], (key, where)
        so, sb = o.state(), b.state()
        assert so["slot_expert"].tolist() == sb["slot_expert"], where
        assert so["expert_slot"].tolist() == sb["expert_slot"], where
        assert so["slot_stamp"].tolist() == sb["slot_stamp"], where
        assert so["clock"] == sb["clock"]


@pytest.mark.parametrize("S", [1, 2, 3])
@pytest.mark.parametrize("k,T,length", [(1, 2, 3), (2, 2, 2), (2, 3, 1), (1, 3, 2)])
def test_exhaustive_small(S, k, T, length):
    E = 4
    toks = [list(p) for p in itertools.permutations(range(E), k)]
    calls = list(itertools.product(toks, repeat=T))
    for trace in itertools.product(calls, repeat=length):
        _compare(S, E, [list(c) for c in trace])


@pytest.mark.parametrize("S,E,k,T", [(2, 6, 2, 3), (3, 8, 2, 5), (4, 16, 4, 6), (5, 16, 4, 3),
                                     (8, 32, 8, 8), (32, 128, 8, 64), (32, 128, 8, 512), (7, 64, 6, 40)])
def test_random_long(S, E, k, T):
    # Zipf-like picks within a call, so that pick counts differ and tie
    rng = random.Random(S * 977 + E * 13 + k * 7 + T)
    w = [1.0 / (i + 1) ** 1.1 for i in range(E)]
    perm = list(range(E))
    rng.shuffle(perm)
    trace = []
    for _ in range(12 if T >= 64 else 30):
        call = []
        for _t in range(T):
            tok = []
            while len(tok) < k:
                e = perm[rng.choices(range(E), weights=w)[0]]
                if e not in tok:
                    tok.append(e)
            call.append(tok)
        trace.append(call)
    _compare(S, E, trace)


def test_hand_worked_cold_call():
    # E = 6, S = 2, picks 0 three times, 1, 2, 3 once: rank 0 > 1 > 2 > 3.
    # Misses lowest rank first: 3, 2 | 1, 0.  Stage 0: 3 -> slot 0, 2 -> slot 1.
    # m = 2 later misses, G = 1, C = 2: no slot kept; 1 -> slot 0, 0 -> slot 1.
    o = oracle.LRU(2, 6, policy=oracle.POLICY_ADOPT)
    p = o.plan(np.array([[0, 1], [0, 2], [0, 3]], dtype=np.int32))
    assert p["miss_expert"].tolist() == [3, 2, 1, 0]
    assert p["miss_slot"].tolist() == [0, 1, 0, 1]
    assert p["miss_evicted"].tolist() == [-1, -1, 3, 2]
    assert p["miss_stage"].tolist() == [0, 0, 1, 1]
    assert o.state()["slot_expert"].tolist() == [1, 0]           # the call's top 2
    lru = oracle.LRU(2, 6)
    lru.plan(np.array([[0, 1], [0, 2], [0, 3]], dtype=np.int32))
    assert lru.state()["slot_expert"].tolist() == [2, 3]         # LRU: the last two by id


def test_hand_worked_kept_slot():
    # S = 3 holding 5, 6, 7.  Picks: 5 x3, 6 x2, 0, 1, 2 once each (E = 8).
    # rank: 5 > 6 > 0 > 1 > 2; hits 5, 6; misses lowest rank first 2, 1, 0.
    # Stage 0: 2 -> slot 2 (expert 7, not picked).  m = 2 later misses: G = 1,
    # C = 2, keep S - C = 1 slot: slot 0 (expert 5, the top rank).  Streaming
    # slots 1, 2: 1 -> slot 1 (evicts 6), 0 -> slot 2 (evicts 2).
    o = oracle.LRU(3, 8, policy=oracle.POLICY_ADOPT)
    o.plan(np.array([[5], [6], [7]], dtype=np.int32))           # slots 0, 1, 2 <- 5, 6, 7
    p = o.plan(np.array([[5, 6], [5, 6], [5, 0], [1, 2]], dtype=np.int32))
    assert p["miss_expert"].tolist() == [2, 1, 0]
    assert p["miss_slot"].tolist() == [2, 1, 2]
    assert p["miss_evicted"].tolist() == [7, 6, 2]
    assert p["miss_stage"].tolist() == [0, 1, 1]
    assert p["info"]["n_stages"] == 2
    assert o.state()["slot_expert"].tolist() == [5, 1, 0]


def test_single_stage_calls_are_lru():
    rng = np.random.default_rng(4)
    a, b = oracle.LRU(8, 32, policy=oracle.POLICY_ADOPT), oracle.LRU(8, 32)
    for _ in range(200):
        ids = np.stack([rng.choice(32, 2, replace=False) for _ in range(3)]).astype(np.int32)  # <= 6 distinct
        pa, pb = a.plan(ids), b.plan(ids)
        for key in ("gpu_slot", "stage", "miss_expert", "miss_slot", "miss_evicted", "miss_stage"):
            assert np.array_equal(pa[key], pb[key]), key
    assert np.array_equal(a.state()["slot_expert"], b.state()["slot_expert"])


def test_uploads_and_stages_as_lru_from_the_same_state():
    # warm both policies identically with single-stage calls, then one staged call
    for seed in range(20):
        rng = np.random.default_rng(seed)
        S, E, k = 6, 40, 4
        a, b = BruteAdopt(S, E), BruteLRU(S, E)
        for _ in range(10):
            call = [list(rng.choice(E, k, replace=False)) for _ in range(1)]
            a.call(call), b.call(call)
        call = [list(rng.choice(E, k, replace=False)) for _ in range(6)]
        pa, pb = a.call(call), b.call(call)
        for key in ("n_miss", "n_stages", "n_evict", "pick_hits"):
            assert pa[key] == pb[key], (seed, key)


def test_final_state_ranks():
    # after a staged call: kept slots hold the top-ranked stage-0 experts, and
    # every later miss still resident ranks above every later miss evicted
    rng = random.Random(7)
    S, E = 8, 64
    o = oracle.LRU(S, E, policy=oracle.POLICY_ADOPT)
    for trial in range(40):
        call = [[rng.choice(range(E // 2)) if rng.random() < 0.5 else rng.randrange(E) for _ in range(1)]
                for _ in range(rng.randrange(10, 30))]
        ids = np.array(call, dtype=np.int32)
        cnt = np.bincount(ids.ravel(), minlength=E)
        p = o.plan(ids)
        final = set(o.state()["slot_expert"].tolist())
        later = [e for e, st in zip(p["miss_expert"].tolist(), p["miss_stage"].tolist()) if st >= 1]
        if not later:
            continue
        key = lambda e: (-cnt[e], e)
        kept_in = [e for e in later if e in final]
        gone = [e for e in later if e not in final]
        if kept_in and gone:
            assert max(key(e) for e in kept_in) < min(key(e) for e in gone), trial


def test_outputs_equal_lru():
    sh = synth.TINY
    store = synth.store(1, sh.E, sh.H, sh.F, seed=8)
    a = oracle.Cache(1, sh.E, sh.k, sh.H, sh.F, sh.S, store, policy=oracle.POLICY_ADOPT)
    b = oracle.Cache(1, sh.E, sh.k, sh.H, sh.F, sh.S, store)
    rng = np.random.default_rng(8)
    staged = 0
    for _ in range(6):
        lg = rng.standard_normal((5, sh.E)).astype(np.float32)
        x = rng.standard_normal((5, sh.H)).astype(np.float32)
        ra, rb = a.forward(0, lg, x), b.forward(0, lg, x)
        assert np.array_equal(ra["out"], rb["out"])
        staged += ra["info"]["n_stages"] > 1
    assert staged >= 3
