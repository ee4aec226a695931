"""The oracle's slot map against an independent brute-force simulator (CPU only).

Exhaustive over every trace of a few calls for E = 4 experts, S in {1, 2, 3}
slots, k in {1, 2} picks and T in {1, 2} tokens, plus long random traces.
"""
import itertools
import random

import numpy as np
import pytest

import oracle
from tests.lru_bruteforce import BruteLRU


def _compare(S, E, trace):
    o = oracle.LRU(S, E)
    b = BruteLRU(S, E)
    for call in trace:
        ids = np.array(call, dtype=np.int32)
        po = o.plan(ids)
        pb = b.call([list(t) for t in call])
        assert po["gpu_slot"].tolist() == pb["gpu_slot"], (S, trace)
        assert po["stage"].tolist() == pb["stage"], (S, trace)
        recs = list(zip(po["miss_expert"].tolist(), po["miss_slot"].tolist(),
                        po["miss_evicted"].tolist(), po["miss_stage"].tolist()))
        assert recs == pb["misses"], (S, trace)
        for key in ("n_unique", "n_hits", "n_miss", "n_stages", "n_evict", "pick_hits", "pick_misses"):
            assert po["info"][key] == pb[key], (key, S, trace)
        so, sb = o.state(), b.state()
        assert so["slot_expert"].tolist() == sb["slot_expert"]
        assert so["expert_slot"].tolist() == sb["expert_slot"]
        assert so["slot_stamp"].tolist() == sb["slot_stamp"]
        assert so["clock"] == sb["clock"]
        # invariants: resident count <= S, hits + misses = |U|
        assert (so["slot_expert"] >= 0).sum() <= S
        assert po["info"]["n_hits"] + po["info"]["n_miss"] == po["info"]["n_unique"]


def _token_choices(E, k):
    # router output order is rank order; both orders of a pair matter for gpu_slot
    return [list(p) for p in itertools.permutations(range(E), k)]


@pytest.mark.parametrize("S", [1, 2, 3])
@pytest.mark.parametrize("k,T,length", [(1, 1, 5), (2, 1, 4), (1, 2, 3), (2, 2, 2)])
def test_exhaustive_small(S, k, T, length):
    E = 4
    toks = _token_choices(E, k)
    calls = list(itertools.product(toks, repeat=T))
    n = 0
    for trace in itertools.product(calls, repeat=length):
        _compare(S, E, [list(c) for c in trace])
        n += 1
    assert n == len(calls) ** length


@pytest.mark.parametrize("S,E,k,T", [(1, 4, 2, 2), (2, 6, 2, 3), (3, 8, 2, 4), (4, 8, 2, 4),
                                     (5, 16, 4, 3), (8, 32, 8, 2), (32, 128, 8, 1), (8, 128, 8, 64)])
def test_random_long(S, E, k, T):
    rng = random.Random(S * 1000 + E * 10 + k + T)
    trace = []
    prev = None
    for _ in range(40):
        call = []
        for _t in range(T):
            if prev is not None and rng.random() < 0.4:
                tok = list(prev)
                rng.shuffle(tok)
                tok = tok[: k // 2] + [e for e in rng.sample(range(E), E) if e not in tok[: k // 2]][: k - k // 2]
            else:
                tok = rng.sample(range(E), k)
            call.append(tok)
            prev = tok
        trace.append(call)
    _compare(S, E, trace)


def test_cold_start_fills_empty_slots_in_order():
    o = oracle.LRU(4, 8)
    p = o.plan(np.array([[5, 2]], np.int32))
    # misses in ascending expert order onto slots 0, 1
    assert p["miss_expert"].tolist() == [2, 5]
    assert p["miss_slot"].tolist() == [0, 1]
    assert p["miss_evicted"].tolist() == [-1, -1]
    assert p["gpu_slot"].tolist() == [[1, 0]]


def test_pinned_experts_never_evicted_within_call():
    # S = 2, call 1 loads {0,1}; call 2 wants {1,2}: 1 is a hit, 2 must evict 0 (not 1)
    o = oracle.LRU(2, 4)
    o.plan(np.array([[0, 1]], np.int32))
    p = o.plan(np.array([[2, 1]], np.int32))
    assert p["miss_expert"].tolist() == [2]
    assert p["miss_evicted"].tolist() == [0]
    assert p["gpu_slot"].tolist() == [[0, 1]]


def test_staged_call_partitions_pairs():
    # 4 distinct experts, 1 slot -> 4 stages; every pair in exactly one stage
    o = oracle.LRU(1, 8)
    p = o.plan(np.array([[3, 1], [7, 5]], np.int32))
    assert p["info"]["n_stages"] == 4
    assert sorted(p["stage"].ravel().tolist()) == [0, 1, 2, 3]
    assert p["miss_expert"].tolist() == [1, 3, 5, 7]
    assert p["miss_stage"].tolist() == [0, 1, 2, 3]
    assert p["miss_evicted"].tolist() == [-1, 1, 3, 5]
