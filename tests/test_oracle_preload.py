"""Warm start from a usage profile (the oracle, CPU only): which experts land in
which slots, how the next calls see them, and that outputs do not change."""
import numpy as np

import oracle
import synth


def _cache(S=4, E=8, **kw):
    sh = synth.TINY
    store = synth.store(1, E, sh.H, sh.F, seed=4)
    return oracle.Cache(1, E, sh.k, sh.H, sh.F, S, store, **kw), store


def test_top_s_by_count_then_id():
    c, _ = _cache(S=4)
    c.preload(np.array([[0, 5, 5, 1, 0, 9, 2, 0]], dtype=np.uint32))
    st = c.lru(0).state()
    assert st["slot_expert"].tolist() == [5, 1, 2, 6]          # 9, then the 5s by id, then 2
    assert st["expert_slot"].tolist() == [-1, 1, 2, -1, -1, 0, 3, -1]
    assert st["slot_stamp"].tolist() == [0, 0, 0, 0] and st["clock"] == 0


def test_fewer_used_experts_than_slots_leave_slots_empty():
    c, _ = _cache(S=8)
    c.preload(np.array([[0, 5, 5, 1, 0, 9, 2, 0]], dtype=np.uint32))
    assert c.lru(0).state()["slot_expert"].tolist() == [5, 1, 2, 6, 3, -1, -1, -1]


def test_preloaded_experts_hit_and_empty_slots_fill_first():
    c, _ = _cache(S=8)
    c.preload(np.array([[0, 5, 5, 1, 0, 9, 2, 0]], dtype=np.uint32))
    lg = np.full((1, 8), -3.0, np.float32)
    lg[0, 1], lg[0, 7] = 2.0, 1.0                                 # picks 1 (cached) and 7
    r = c.forward(0, lg, None, compute=False)
    assert r["info"]["n_hits"] == 1 and r["miss_expert"].tolist() == [7]
    assert r["miss_slot"].tolist() == [5] and r["miss_evicted"].tolist() == [-1]
    assert c.stats(0)["calls"] == 1                               # the preload is not a call


def test_preload_replaces_the_cached_set():
    c, _ = _cache(S=4)
    lg = np.full((1, 8), -3.0, np.float32)
    lg[0, 0], lg[0, 4] = 2.0, 1.0
    c.forward(0, lg, None, compute=False)                         # 0 and 4 cached
    c.preload(np.array([[0, 0, 3, 0, 0, 0, 0, 1]], dtype=np.uint32))
    st = c.lru(0).state()
    assert st["slot_expert"].tolist() == [2, 7, -1, -1]
    assert st["expert_slot"][0] == -1 and st["expert_slot"][4] == -1


def test_outputs_do_not_depend_on_the_preload():
    sh = synth.TINY
    store = synth.store(1, sh.E, sh.H, sh.F, seed=6)
    a = oracle.Cache(1, sh.E, sh.k, sh.H, sh.F, sh.S, store)
    b = oracle.Cache(1, sh.E, sh.k, sh.H, sh.F, sh.S, store)
    b.preload(np.arange(sh.E, dtype=np.uint32)[None, :])
    rng = np.random.default_rng(6)
    for _ in range(6):
        lg = rng.standard_normal((2, sh.E)).astype(np.float32)
        x = rng.standard_normal((2, sh.H)).astype(np.float32)
        assert np.array_equal(a.forward(0, lg, x)["out"], b.forward(0, lg, x)["out"])
    assert b.stats(0)["unique_hits"] > a.stats(0)["unique_hits"]


def test_preloaded_slots_are_evicted_in_slot_order():
    # all preloaded slots carry stamp 0: the least recently used is the lowest
    # slot index, and a slot used since is younger than every untouched one
    c, _ = _cache(S=4)
    c.preload(np.array([[0, 5, 5, 1, 0, 9, 2, 0]], dtype=np.uint32))   # slots: 5 1 2 6
    lg = np.full((1, 8), -3.0, np.float32)
    lg[0, 5], lg[0, 7] = 2.0, 1.0                                 # 5 hits (slot 0), 7 misses
    r = c.forward(0, lg, None, compute=False)
    assert r["miss_expert"].tolist() == [7]
    assert r["miss_slot"].tolist() == [1] and r["miss_evicted"].tolist() == [1]
    lg = np.full((1, 8), -3.0, np.float32)
    lg[0, 0], lg[0, 4] = 2.0, 1.0                                 # two misses
    r = c.forward(0, lg, None, compute=False)
    assert sorted(r["miss_slot"].tolist()) == [2, 3]
    assert sorted(r["miss_evicted"].tolist()) == [2, 6]
