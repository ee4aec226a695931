"""Lifetime usage counts and saved / resumed cache state on the GPU, against the
oracle (GPU).

* moe_cache_usage equals the oracle's counts bit for bit after decode calls
  (single-warp plan), staged batch calls (block plan, grid router) and the
  score and adopt policies.
* moe_cache_save_state holds the oracle's slot tables, stamps, clocks, scores
  and counts bit for bit.
* A fresh handle that loads the state plans (bit-exact) and computes (within
  tolerance) exactly as the oracle that never stopped: the slots it refilled
  hold the right blocks.
* A planted random state, loaded into both sides, gives the same plans.
* Malformed states are rejected with MOE_ERR_INVALID_ARG and leave the handle
  as it was; a poisoned handle refuses to save but still reports its counts.
"""
import numpy as np
import pytest

import synth
from tests.gpu_util import DECODE_TOL, Pair, assert_plan_equal, pinned_store, row_rel_err

pytestmark = pytest.mark.gpu

HDR = 48


def unpack_state(blob: bytes, L: int, E: int, S: int):
    """The arrays of a saved state, by the layout moe_cache.h documents."""
    import router_softmax_top_gb300 as moe
    hdr = moe.MoeStateHeader.from_buffer_copy(blob[:HDR])
    off = HDR
    out = {}
    for name, dt, n in (("clock", np.uint64, L), ("slot_stamp", np.uint64, L * S),
                        ("slot_expert", np.int32, L * S), ("score", np.float32, L * E),
                        ("usage", np.uint32, L * E)):
        a = np.frombuffer(blob, dtype=dt, count=n, offset=off).copy()
        off += a.nbytes
        out[name] = a if name == "clock" else a.reshape(L, -1)
    assert off == len(blob) == hdr.total_bytes
    return hdr, out


def pack_state(hdr, st) -> bytes:
    return bytes(hdr) + b"".join(np.ascontiguousarray(st[n], dtype=dt).tobytes() for n, dt in
                                 (("clock", np.uint64), ("slot_stamp", np.uint64), ("slot_expert", np.int32),
                                  ("score", np.float32), ("usage", np.uint32)))


def assert_state_equals_oracle(blob, orc, L, E, S):
    hdr, st = unpack_state(blob, L, E, S)
    assert (hdr.n_layers, hdr.n_experts, hdr.slots_per_layer) == (L, E, S)
    for l in range(L):
        o = orc.state(l)
        assert st["clock"][l] == o["clock"], l
        assert np.array_equal(st["slot_expert"][l], o["slot_expert"]), l
        assert np.array_equal(st["slot_stamp"][l], o["slot_stamp"]), l
        assert np.array_equal(st["score"][l].view(np.uint32), o["score"].view(np.uint32)), l
        assert np.array_equal(st["usage"][l], o["usage"]), l


# (T, S, fill_mode, policy, admit_budget): single-warp plan at T = 1, the
# block plan with the grid router and stages at T = 64
CASES = [(1, 32, 1, 0, 0), (1, 32, 0, 0, 0), (1, 32, 1, 1, 2), (64, 8, 1, 0, 0), (64, 8, 1, 2, 0),
         (64, 32, 0, 0, 0)]


def _inputs(T, n, seed):
    sh = synth.SWEEP
    if T == 1:
        _, lg, x = synth.decode_inputs(sh, n, batch=1, seed=seed, layers=[0, 1])
        return [(s % 2, lg[s, s % 2], x[s, s % 2]) for s in range(n)]
    _, lg, x = synth.batch_inputs(sh, n, T, seed=seed, layers=[0, 1], zipf=1.2, sticky=0.3, act="f32")
    return [(b % 2, lg[b, b % 2], x[b, b % 2]) for b in range(n)]


def _pair(T, S, fill_mode, policy, budget, store):
    sh = synth.SWEEP
    return Pair(2, sh.E, sh.k, sh.H, sh.F, S, store, max_tokens=T, fill_mode=fill_mode, policy=policy,
                admit_budget=budget)


@pytest.mark.parametrize("T,S,fill_mode,policy,budget", CASES)
def test_usage_and_saved_state_match_oracle(T, S, fill_mode, policy, budget):
    sh = synth.SWEEP
    store = pinned_store(2, sh.E, sh.H, sh.F, seed=21)
    p = _pair(T, S, fill_mode, policy, budget, store)
    for i, (layer, lg, x) in enumerate(_inputs(T, 8, seed=21)):
        _, plan, r = p.step(layer, lg, x, compute_oracle=False)
        assert_plan_equal(plan, r, f"call {i}")
    assert np.array_equal(p.gpu.usage(), p.orc.usage())
    assert int(p.gpu.usage().sum()) == 8 * T * sh.k
    assert_state_equals_oracle(p.gpu.save_state(), p.orc, 2, sh.E, S)
    p.close()


@pytest.mark.parametrize("T,S,fill_mode,policy,budget", CASES)
def test_resumed_handle_continues_as_uninterrupted(T, S, fill_mode, policy, budget):
    sh = synth.SWEEP
    store = pinned_store(2, sh.E, sh.H, sh.F, seed=22)
    calls = _inputs(T, 14, seed=22)
    a = _pair(T, S, fill_mode, policy, budget, store)
    for layer, lg, x in calls[:7]:
        a.step(layer, lg, x, compute_oracle=False)
    blob = a.gpu.save_state()
    orc_stats = [a.orc.stats(l) for l in range(2)]
    a.gpu.close()
    b = _pair(T, S, fill_mode, policy, budget, store)
    b.orc = a.orc                                   # the oracle that never stopped
    b.gpu.load_state(blob)
    assert_state_equals_oracle(b.gpu.save_state(), b.orc, 2, sh.E, S)
    worst = 0.0
    for i, (layer, lg, x) in enumerate(calls[7:]):
        check = i in (0, 1, 6)
        g, plan, r = b.step(layer, lg, x, compute_oracle=check)
        assert_plan_equal(plan, r, f"resumed call {i}")
        if check:
            worst = max(worst, row_rel_err(g, r["out"]).max())
    assert worst <= DECODE_TOL, worst
    assert np.array_equal(b.gpu.usage(), b.orc.usage())
    for l in range(2):                              # the resumed handle counts from zero
        got, o = b.gpu.stats(l), b.orc.stats(l)
        for key in ("calls", "pick_hits", "unique_misses", "evictions", "stages", "bypassed"):
            assert got[key] == o[key] - orc_stats[l][key], key
    b.close()


@pytest.mark.parametrize("T,S,policy", [(1, 32, 0), (1, 16, 1), (64, 16, 0)])
def test_planted_state_plans_as_oracle(T, S, policy):
    import router_softmax_top_gb300 as moe
    sh = synth.SWEEP
    store = pinned_store(2, sh.E, sh.H, sh.F, seed=23)
    p = _pair(T, S, 1, policy, 3 if policy == 1 else 0, store)
    rng = np.random.default_rng(23)
    hdr = moe.MoeStateHeader(moe.MOE_STATE_MAGIC, moe.MOE_STATE_VERSION, 2, sh.E, S, policy,
                             moe.moe_expert_bytes(sh.H, sh.F), 0, 0)
    st = {"clock": np.array([1000, 57], np.uint64), "slot_stamp": np.zeros((2, S), np.uint64),
          "slot_expert": np.full((2, S), -1, np.int32), "score": np.zeros((2, sh.E), np.float32),
          "usage": rng.integers(0, 2**32, (2, sh.E), dtype=np.uint64).astype(np.uint32)}
    for l in range(2):
        held = rng.choice(sh.E, S - 3, replace=False)
        where = rng.choice(S, S - 3, replace=False)          # three slots stay empty
        st["slot_expert"][l, where] = held
        # few distinct stamps: ties broken by slot index on both sides
        st["slot_stamp"][l, where] = (rng.integers(0, 4, S - 3) * int(st["clock"][l] // 4)).astype(np.uint64)
        st["score"][l] = (rng.random(sh.E) * 4).astype(np.float32)
    hdr.total_bytes = HDR + len(pack_state(hdr, st)) - len(bytes(hdr))
    blob = pack_state(hdr, st)
    p.gpu.load_state(blob)
    for l in range(2):
        assert p.orc.set_state(l, st["slot_expert"][l], st["slot_stamp"][l], int(st["clock"][l]),
                               st["score"][l], st["usage"][l])
    assert unpack_state(p.gpu.save_state(), 2, sh.E, S)[1]["usage"].tobytes() == st["usage"].tobytes()
    for i, (layer, lg, x) in enumerate(_inputs(T, 8, seed=24)):
        check = i in (0, 5)
        g, plan, r = p.step(layer, lg, x, compute_oracle=check)
        assert_plan_equal(plan, r, f"call {i}")
        if check:
            assert row_rel_err(g, r["out"]).max() <= DECODE_TOL
    assert np.array_equal(p.gpu.usage(), p.orc.usage())
    p.close()


def test_malformed_states_are_rejected():
    import router_softmax_top_gb300 as moe
    sh = synth.SWEEP
    S = 16
    store = pinned_store(2, sh.E, sh.H, sh.F, seed=25)
    p = _pair(1, S, 1, 0, 0, store)
    calls = _inputs(1, 10, seed=25)
    for layer, lg, x in calls[:4]:
        p.step(layer, lg, x, compute_oracle=False)
    good = p.gpu.save_state()
    hdr, st = unpack_state(good, 2, sh.E, S)

    def variant(edit):
        h2 = moe.MoeStateHeader.from_buffer_copy(bytes(hdr))
        s2 = {k: v.copy() for k, v in st.items()}
        edit(h2, s2)
        return pack_state(h2, s2)

    held = int(np.nonzero(st["slot_expert"][0] >= 0)[0][0])
    bad = {
        "magic": variant(lambda h, s: setattr(h, "magic", 0)),
        "version": variant(lambda h, s: setattr(h, "version", 2)),
        "slots": variant(lambda h, s: setattr(h, "slots_per_layer", S + 1)),
        "expert_bytes": variant(lambda h, s: setattr(h, "expert_bytes", h.expert_bytes + 18)),
        "id": variant(lambda h, s: s["slot_expert"].__setitem__((1, 0), sh.E)),
        "dup": variant(lambda h, s: s["slot_expert"].__setitem__((0, (held + 1) % S), s["slot_expert"][0, held])),
        "stamp": variant(lambda h, s: s["slot_stamp"].__setitem__((0, held), s["clock"][0] + 1)),
        "clock": variant(lambda h, s: s["clock"].__setitem__(1, 1 << 48)),
        "nan": variant(lambda h, s: s["score"].__setitem__((1, 3), np.nan)),
        "neg": variant(lambda h, s: s["score"].__setitem__((0, 3), -0.5)),
        "short": good[:-4],
        "long": good + b"\0" * 4,
    }
    for name, blob in bad.items():
        assert p.gpu.load_state_rc(blob) == moe.MOE_ERR_INVALID_ARG, name
    assert p.gpu.save_state() == good               # unchanged, not poisoned
    assert p.gpu.stats(-1)["poisoned"] == 0
    for i, (layer, lg, x) in enumerate(calls[4:]):
        _, plan, r = p.step(layer, lg, x, compute_oracle=False)
        assert_plan_equal(plan, r, f"call {i} after the rejected loads")
    p.close()


def test_poisoned_handle_refuses_to_save():
    import router_softmax_top_gb300 as moe
    sh = synth.TINY
    store = pinned_store(1, sh.E, sh.H, sh.F, seed=26)
    c = moe.MoECache(n_layers=1, n_experts=sh.E, top_k=sh.k, hidden=sh.H, ffn=sh.F, slots_per_layer=sh.S,
                     max_tokens=1, store=store, fill_mode=moe.MOE_FILL_MEMCPY, timeout_us=200_000)
    lg, x = synth.tiny_inputs(26)
    import torch
    lgd, xd = torch.from_numpy(lg).cuda(), torch.from_numpy(x).cuda()
    out = torch.empty((1, sh.H), device="cuda")
    assert c.forward_rc(0, lgd[:1], xd[:1], out) == moe.MOE_OK
    counts = c.usage()
    assert int(counts.sum()) == sh.k
    c.inject(moe.MOE_INJECT_MEMCPY_FAIL)
    rc = moe.MOE_OK
    for t in range(1, 4):                            # the next call with a miss meets the failed copy
        rc = c.forward_rc(0, lgd[t:t + 1], xd[t:t + 1], out)
        if rc != moe.MOE_OK:
            break
    assert rc == moe.MOE_ERR_CUDA
    with pytest.raises(moe.MoeError) as e:
        c.save_state()
    assert e.value.code == moe.MOE_ERR_POISONED
    assert c.load_state_rc(b"\0" * 64) == moe.MOE_ERR_POISONED
    assert int(c.usage().sum()) >= sh.k               # still readable
    c.close()
