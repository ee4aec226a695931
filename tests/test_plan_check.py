"""The library's host-side plan check (debug runs, MOE_CHECK_PLANS=1), on the CPU.

The check is a self-contained header; this test compiles it with g++ behind a
small C wrapper and feeds it plans from the CPU oracle (which it must accept)
and the same plans with one planted mistake each (which it must reject with
the number of the broken rule)."""
import ctypes
import os
import subprocess

import numpy as np
import pytest

import oracle
import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER_DIR = os.path.join(ROOT, "router_softmax_top_gb300", "csrc")

WRAPPER = r'''
#include "plan_check.h"
extern "C" int check(int T, int k, int E, int S, int n_stages, int n_miss, const int32_t *ids,
                     const int32_t *gs, const int32_t *stage, const int32_t *miss,
                     const int32_t *slot_expert, const int32_t *expert_slot) {
  return moe::plan_check(T, k, E, S, n_stages, n_miss, ids, gs, stage, miss, slot_expert, expert_slot);
}
'''


@pytest.fixture(scope="module")
def check(tmp_path_factory):
    d = tmp_path_factory.mktemp("plan_check")
    src, so = d / "w.cpp", d / "libw.so"
    src.write_text(WRAPPER)
    subprocess.run(["g++", "-O1", "-std=c++17", "-shared", "-fPIC", "-I", HEADER_DIR, "-o", str(so), str(src)],
                   check=True)
    lib = ctypes.CDLL(str(so))
    lib.check.restype = ctypes.c_int
    return lib.check


def _run(check, T, k, E, S, plan, state):
    miss = np.stack([plan["miss_expert"], plan["miss_slot"], plan["miss_evicted"], plan["miss_stage"]], axis=1) \
        if len(plan["miss_expert"]) else np.zeros((1, 4), np.int32)
    keep = [np.ascontiguousarray(a, dtype=np.int32) for a in
            (plan["ids"], plan["gpu_slot"], plan["stage"], miss, state["slot_expert"], state["expert_slot"])]
    return check(T, k, E, S, plan["info"]["n_stages"], len(plan["miss_expert"]),
                 *[k2.ctypes.data_as(ctypes.c_void_p) for k2 in keep])


def _oracle_plans(S, T, n, policy=oracle.POLICY_LRU, seed=0):
    sh = synth.SWEEP
    c = oracle.Cache(1, sh.E, sh.k, sh.H, sh.F, S, np.zeros(1, np.uint8), policy=policy)
    _, logits, _ = synth.batch_inputs(sh, n, T, seed=seed, zipf=1.2, sticky=0.0, act="f32")
    out = []
    for b in range(n):
        r = c.forward(0, logits[b, 0], None, compute=False)
        st = c.lru(0).state()
        out.append((r, {"slot_expert": st["slot_expert"].copy(), "expert_slot": st["expert_slot"].copy()}))
    return sh, out


@pytest.mark.parametrize("S,T,policy", [(32, 1, 0), (8, 64, 0), (32, 64, 0), (128, 64, 0), (8, 64, 2)])
def test_oracle_plans_pass(check, S, T, policy):
    sh, plans = _oracle_plans(S, T, 4, policy)
    for r, st in plans:
        assert _run(check, T, sh.k, sh.E, S, r, st) == 0


def test_planted_mistakes_are_caught(check):
    S, T = 8, 64
    sh, plans = _oracle_plans(S, T, 2)
    r, st = plans[-1]
    assert r["info"]["n_stages"] > 1

    def broken(edit):
        r2 = {k2: (v.copy() if isinstance(v, np.ndarray) else dict(v) if isinstance(v, dict) else v)
              for k2, v in r.items()}
        st2 = {k2: v.copy() for k2, v in st.items()}
        edit(r2, st2)
        return _run(check, T, sh.k, sh.E, S, r2, st2)

    def dup_id(r2, _):
        r2["ids"][3, 1] = r2["ids"][3, 0]
    assert broken(dup_id) == 1

    def bad_id(r2, _):
        r2["ids"][0, 0] = sh.E
    assert broken(bad_id) == 1

    def bad_slot(r2, _):
        r2["gpu_slot"][5, 2] = S
    assert broken(bad_slot) == 2

    def bad_stage(r2, _):
        r2["stage"][1, 1] = r2["info"]["n_stages"]
    assert broken(bad_stage) == 3

    def bad_miss(r2, _):
        r2["miss_evicted"][0] = sh.E
    assert broken(bad_miss) == 4

    def two_slots(_, st2):
        st2["slot_expert"][1] = st2["slot_expert"][0]
    assert broken(two_slots) == 5

    def wrong_last_stage(r2, _):
        last = r2["info"]["n_stages"] - 1
        t, q = np.argwhere(r2["stage"] == last)[0]
        r2["gpu_slot"][t, q] = (r2["gpu_slot"][t, q] + 1) % S
    assert broken(wrong_last_stage) == 6

    def wrong_early_stage(r2, _):
        t, q = np.argwhere(r2["stage"] == 1)[0] if r2["info"]["n_stages"] > 2 else np.argwhere(r2["stage"] == 0)[0]
        e = r2["ids"][t, q]
        # a stage whose miss record of this expert names another slot
        i = int(np.nonzero(r2["miss_expert"] == e)[0][0]) if e in r2["miss_expert"] else None
        if i is None:
            pytest.skip("picked pair is a hit")
        r2["miss_slot"][i] = (r2["miss_slot"][i] + 1) % S
    assert broken(wrong_early_stage) in (6, 7)
