"""Adopt policy on the GPU against the oracle: staged calls (more distinct
experts than slots) plan bit-exact, through the tensor-core GEMM and the GEMV
kernels, both fill modes; the blocks the final state maps are the right ones
(later single-token calls that hit them give bitwise the outputs of an LRU
handle, which holds or fetches the same blocks)."""
import numpy as np
import pytest

import synth
from tests.gpu_util import (DECODE_TOL, PREFILL_TOL, Pair, assert_plan_equal, assert_stats_equal,
                            pinned_store, row_rel_err)

pytestmark = pytest.mark.gpu

SH = synth.PREFILL
ADOPT = 2


@pytest.fixture(scope="module")
def store():
    return pinned_store(1, SH.E, SH.H, SH.F, seed=31)


@pytest.mark.parametrize("gemm", [True, False])
@pytest.mark.parametrize("fill_mode", [1, 0])
def test_staged_calls_then_decode(store, gemm, fill_mode):
    T = 96
    act = "bf16" if gemm else "f32"
    _, logits, x = synth.batch_inputs(SH, 3, T, seed=31, layers=[0], act=act)
    p = Pair(1, SH.E, SH.k, SH.H, SH.F, SH.S, store, max_tokens=T, act=act, fill_mode=fill_mode,
             gemm_min_tokens=16 if gemm else 0, policy=ADOPT)
    tol = PREFILL_TOL if gemm else DECODE_TOL
    for b in range(3):
        g, plan, r = p.step(0, logits[b, 0], x[b, 0], compute_oracle=(b != 1))
        assert_plan_equal(plan, r, f"batch {b}")
        assert plan["n_stages"] >= 2
        if b != 1:
            assert row_rel_err(g, r["out"]).max() <= tol
    # single tokens afterwards: plans still bit-exact, hits read the adopted slots
    picks, lg1, x1 = synth.decode_inputs(SH, 12, batch=1, seed=32, layers=[0])
    for s in range(12):
        xs = x1[s, 0, :1] if act == "f32" else _bf16(x1[s, 0, :1])
        g, plan, r = p.step(0, lg1[s, 0, :1], xs)
        assert_plan_equal(plan, r, f"decode {s}")
        assert row_rel_err(g, r["out"]).max() <= tol
    assert_stats_equal(p.gpu.stats(0), p.orc.stats(0))
    p.close()


def _bf16(a):
    # round-to-nearest-even fp32 -> bf16 raw bits
    u = np.ascontiguousarray(a, np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def test_outputs_bitwise_lru_and_slots_hold_the_right_blocks(store):
    # the same staged calls and following single tokens on an adopt handle and
    # an LRU handle: bitwise equal outputs (the policy moves blocks, not sums)
    T = 128
    _, logits, x = synth.batch_inputs(SH, 2, T, seed=33, layers=[0], act="f32")
    _, lg1, x1 = synth.decode_inputs(SH, 16, batch=1, seed=34, layers=[0])
    outs = {}
    for pol in (0, ADOPT):
        p = Pair(1, SH.E, SH.k, SH.H, SH.F, SH.S, store, max_tokens=T, act="f32", fill_mode=1, policy=pol)
        o = [p.step(0, logits[b, 0], x[b, 0], compute_oracle=False)[0] for b in range(2)]
        o += [p.step(0, lg1[s, 0, :1], x1[s, 0, :1], compute_oracle=False)[0] for s in range(16)]
        outs[pol] = o
        p.close()
    for i, (a, b) in enumerate(zip(outs[0], outs[ADOPT])):
        assert np.array_equal(a, b), i
