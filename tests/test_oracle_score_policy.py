"""The oracle's decayed-score admission policy against an independent
brute-force simulator (CPU only), exhaustive on tiny traces and on long random
traces, plus closed forms, invariants and the policy's independence of outputs."""
import itertools
import random

import numpy as np
import pytest

import oracle
import synth
from tests.score_bruteforce import BruteScore


def _compare(S, E, trace, budget=0, sticky=0):
    o = oracle.LRU(S, E, policy=oracle.POLICY_SCORE, budget=budget, sticky=sticky)
    b = BruteScore(S, E, budget, sticky)
    for call in trace:
        po = o.plan(np.array(call, dtype=np.int32))
        pb = b.call([list(t) for t in call])
        assert po["gpu_slot"].tolist() == pb["gpu_slot"], (S, budget, trace)
        assert (po["stage"] == 0).all()
        recs = list(zip(po["miss_expert"].tolist(), po["miss_slot"].tolist(),
                        po["miss_evicted"].tolist(), po["miss_stage"].tolist()))
        assert recs == pb["misses"], (S, budget, trace)
        for key in ("n_unique", "n_hits", "n_miss", "n_stages", "n_evict", "n_bypass", "pick_hits",
                    "pick_misses"):
            assert po["info"][key] == pb[key], (key, S, budget, trace)
        so, sb = o.state(), b.state()
        assert so["slot_expert"].tolist() == sb["slot_expert"]
        assert so["expert_slot"].tolist() == sb["expert_slot"]
        assert so["slot_stamp"].tolist() == sb["slot_stamp"]
        assert so["clock"] == sb["clock"]
        assert o.scores().tolist() == [float(v) for v in b.score]   # bit for bit: same fp32 operations
        # a bypass happens only with no empty slot left or the budget used up
        assert po["info"]["n_hits"] + po["info"]["n_miss"] == po["info"]["n_unique"]


def _token_choices(E, k):
    return [list(p) for p in itertools.permutations(range(E), k)]


@pytest.mark.parametrize("budget", [0, 1])
@pytest.mark.parametrize("S,k,T,length", [(1, 1, 1, 6), (2, 1, 1, 6), (3, 1, 1, 5), (2, 2, 1, 4),
                                          (3, 1, 2, 3), (2, 1, 2, 3), (3, 3, 1, 3)])
def test_exhaustive_small(S, k, T, length, budget):
    E = 4
    calls = [c for c in itertools.product(_token_choices(E, k), repeat=T)
             if len({e for tok in c for e in tok}) <= S]
    for trace in itertools.product(calls, repeat=length):
        _compare(S, E, [list(c) for c in trace], budget)


@pytest.mark.parametrize("S,E,k,T,budget", [(4, 8, 2, 2, 0), (8, 16, 4, 2, 0), (8, 16, 4, 2, 2),
                                            (32, 128, 8, 1, 0), (32, 128, 8, 4, 0), (32, 128, 8, 1, 3)])
def test_random_long(S, E, k, T, budget):
    rng = random.Random(S * 7 + E * 3 + k + T + budget)
    zipf = np.array([1.0 / (r + 1) ** 1.1 for r in range(E)])
    zipf /= zipf.sum()
    trace = []
    for _ in range(60):
        call = []
        for _t in range(T):
            tok = []
            while len(tok) < k:
                e = int(np.searchsorted(np.cumsum(zipf), rng.random()))
                if e < E and e not in tok:
                    tok.append(e)
            call.append(tok)
        if len({e for tok in call for e in tok}) <= S:
            trace.append(call)
    _compare(S, E, trace, budget)


def test_score_closed_form():
    # one expert picked n times in a row: 1 + 0.9 + ... + 0.9^(n-1) = 10 (1 - 0.9^n),
    # within fp32 rounding of n steps
    o = oracle.LRU(4, 8, policy=oracle.POLICY_SCORE)
    for n in range(1, 60):
        o.plan(np.array([[3]], dtype=np.int32))
        assert abs(float(o.scores()[3]) - 10.0 * (1.0 - 0.9 ** n)) < 1e-5
        assert o.scores()[0] == 0.0
    # then unused for m tokens: decays by 0.9^m
    s0 = float(o.scores()[3])
    for m in range(1, 20):
        o.plan(np.array([[5]], dtype=np.int32))
        assert abs(float(o.scores()[3]) - s0 * 0.9 ** m) < 1e-5


def test_hot_expert_survives_one_off_misses():
    # LRU evicts the hot expert for a stream of one-off experts; the score
    # policy keeps it (the one-offs are bypassed once the slot is full)
    S, E = 1, 16
    lru = oracle.LRU(S, E)
    sc = oracle.LRU(S, E, policy=oracle.POLICY_SCORE)
    for _ in range(5):
        lru.plan(np.array([[0]], dtype=np.int32))
        sc.plan(np.array([[0]], dtype=np.int32))
    for e in range(1, 6):
        lru.plan(np.array([[e]], dtype=np.int32))
        p = sc.plan(np.array([[e]], dtype=np.int32))
        assert p["miss_slot"].tolist() == [-1] and p["info"]["n_bypass"] == 1
    assert sc.state()["slot_expert"].tolist() == [0]
    assert lru.state()["slot_expert"].tolist() == [5]


def test_multi_stage_call_rejected():
    o = oracle.LRU(2, 8, policy=oracle.POLICY_SCORE)
    with pytest.raises(ValueError):
        o.plan(np.array([[0, 1, 2]], dtype=np.int32))
    assert o.state()["clock"] == 0                   # state untouched


def test_outputs_do_not_depend_on_the_policy():
    # every pair is computed from its expert's store bytes either way
    sh = synth.TINY
    store = synth.store(1, sh.E, sh.H, sh.F, seed=3)
    a = oracle.Cache(1, sh.E, sh.k, sh.H, sh.F, sh.S, store)
    b = oracle.Cache(1, sh.E, sh.k, sh.H, sh.F, sh.S, store, policy=oracle.POLICY_SCORE)
    rng = np.random.default_rng(3)
    bypassed = 0
    for _ in range(12):
        lg = rng.standard_normal((1, sh.E)).astype(np.float32)
        x = rng.standard_normal((1, sh.H)).astype(np.float32)
        ra, rb = a.forward(0, lg, x), b.forward(0, lg, x)
        assert np.array_equal(ra["out"], rb["out"])
        bypassed += rb["info"]["n_bypass"]
    assert b.stats(0)["bypassed"] == bypassed > 0
    assert a.stats(0)["bypassed"] == 0


@pytest.mark.parametrize("sticky", [500, 1000])
@pytest.mark.parametrize("S,k,T,length", [(2, 1, 1, 6), (3, 1, 1, 5), (3, 1, 2, 3), (2, 2, 1, 4)])
def test_exhaustive_small_sticky(S, k, T, length, sticky):
    E = 4
    calls = [c for c in itertools.product(_token_choices(E, k), repeat=T)
             if len({e for tok in c for e in tok}) <= S]
    for trace in itertools.product(calls, repeat=length):
        _compare(S, E, [list(c) for c in trace], 0, sticky)


@pytest.mark.parametrize("S,E,k,T,budget,sticky", [(8, 16, 4, 2, 0, 500), (32, 128, 8, 1, 0, 300),
                                                   (32, 128, 8, 4, 2, 300), (7, 32, 2, 3, 0, 999)])
def test_random_long_sticky(S, E, k, T, budget, sticky):
    rng = random.Random(S * 11 + E + k + T + sticky)
    zipf = np.array([1.0 / (r + 1) ** 1.1 for r in range(E)])
    cdf = np.cumsum(zipf / zipf.sum())
    trace = []
    for _ in range(60):
        call = []
        for _t in range(T):
            tok = []
            while len(tok) < k:
                e = int(np.searchsorted(cdf, rng.random()))
                if e < E and e not in tok:
                    tok.append(e)
            call.append(tok)
        if len({e for tok in call for e in tok}) <= S:
            trace.append(call)
    _compare(S, E, trace, budget, sticky)


def test_full_sticky_share_never_evicts():
    # every occupied slot protected: once the slots are full, misses are bypassed
    o = oracle.LRU(4, 16, policy=oracle.POLICY_SCORE, sticky=1000)
    rng = np.random.default_rng(2)
    for i in range(50):
        p = o.plan(rng.choice(16, (1, 2), replace=False).astype(np.int32))
        assert p["info"]["n_evict"] == 0
    assert (o.state()["slot_expert"] >= 0).all()


def test_sticky_hand_worked():
    # S = 2, E = 4.  Calls [0] x3, then [1]: slot 0 holds expert 0 (score
    # 2.439), slot 1 expert 1 (1.0).  Then one call of four tokens 1, 2, 2, 2:
    # after it expert 0 scores 1.6002, expert 1 1.3851, expert 2 2.71.  Expert
    # 1 is picked (pinned), so the only evictable slot is 0, whose 1.6002 is
    # below 2.71: without a sticky share, expert 2 replaces expert 0.  With a share
    # of 500 (one slot) the highest-scoring occupied slot, slot 0, is kept, and
    # expert 2 is computed without a slot (bypassed).
    for sticky, slot, state in ((0, 0, [2, 1]), (500, -1, [0, 1])):
        o = oracle.LRU(2, 4, policy=oracle.POLICY_SCORE, sticky=sticky)
        for ids in ([[0]], [[0]], [[0]], [[1]]):
            o.plan(np.array(ids, dtype=np.int32))
        p = o.plan(np.array([[1], [2], [2], [2]], dtype=np.int32))
        assert p["miss_expert"].tolist() == [2] and p["miss_slot"].tolist() == [slot], sticky
        assert p["info"]["n_bypass"] == (1 if slot < 0 else 0)
        assert o.state()["slot_expert"].tolist() == state, sticky
        np.testing.assert_allclose(o.scores(), [1.6002, 1.3851, 2.71, 0.0], rtol=1e-4)


def test_single_precision_reading_decides_an_admission():
    """Hand-worked trace on which the precision of the score decides who is admitted.

    "Keeping the cache fresh" gives the decay (x0.9 per token) but no arithmetic
    precision; the reading taken is single precision, each operation rounded.
    Two slots, experts A=0, B=1, C=2, D=3, one token per call, no budget limit:
      * A and D fill the slots (calls [A], [D]) and are then picked alternately,
        which keeps both scores near 4.3-5.3;
      * B is picked once, 200 tokens before the last call, and C once, 190
        tokens before it: both are bypassed (score 1 against slots above 4);
      * the 189 calls before the last pick A only, so D's score decays to ~1e-8;
      * the last call picks B and C together (k = 2).
    In the last call B's score is 1 + 0.9^200 and C's is 1 + 0.9^190 in exact
    arithmetic.  Both powers are below 2^-24, half a unit in the last place of
    1.0 in single precision, so both scores round to exactly 1.0: a tie, which
    goes to the lower id.  B is considered first, is stronger than the weakest
    slot (D, ~1e-8), and takes D's slot 1; C then faces A (~9) and is bypassed.
    A double-precision reading keeps 1 + 0.9^190 > 1 + 0.9^200 and would admit
    C instead of B."""
    from fractions import Fraction
    # the two facts the expectation rests on, in exact rational arithmetic
    assert Fraction(9, 10) ** 190 < Fraction(1, 2 ** 24)
    assert Fraction(1) + Fraction(9, 10) ** 190 > Fraction(1) + Fraction(9, 10) ** 200
    A, B, C, D = 0, 1, 2, 3
    N = 600                                   # the last call is token N
    o = oracle.LRU(2, 4, policy=oracle.POLICY_SCORE)
    calls = [[[A]], [[D]]]
    t = 3
    while t < N - 200:
        calls.append([[A]] if t % 2 else [[D]]); t += 1
    calls.append([[B]]); t += 1               # token N - 200
    while t < N - 190:
        calls.append([[A]] if t % 2 else [[D]]); t += 1
    calls.append([[C]]); t += 1               # token N - 190
    while t < N:
        calls.append([[A]]); t += 1
    for c in calls:
        p = o.plan(np.array(c, dtype=np.int32))
        if c in ([[B]], [[C]]):
            assert p["gpu_slot"].tolist() == [[-1]] and p["info"]["n_bypass"] == 1
    assert o.state()["slot_expert"].tolist() == [A, D]
    p = o.plan(np.array([[B, C]], dtype=np.int32))
    assert p["gpu_slot"].tolist() == [[1, -1]]
    assert list(zip(p["miss_expert"].tolist(), p["miss_slot"].tolist(), p["miss_evicted"].tolist())) == \
        [(B, 1, D), (C, -1, -1)]
    assert p["info"]["n_bypass"] == 1 and p["info"]["n_evict"] == 1
    sc = o.scores()
    assert sc[B] == np.float32(1.0) and sc[C] == np.float32(1.0)
    assert o.state()["slot_expert"].tolist() == [A, B]
