"""Small batches (2 to 31 tokens: speculative verification, short prompts) on the
decode model against the oracle, through each compute path:

* the GEMV path: the decode layer kernel while a call fits one stage for sure
  (up to 4 tokens at 8 picks and 32 slots, two compute groups), the staged GEMV
  kernels beyond; fp32 and bf16 inputs; 1e-3 per token row;
* the tensor-core grouped GEMM (switch point at 1 token); 2e-2 per token row.

Slot maps bit-exact on every call; the statistics equal at the end."""
import numpy as np
import pytest

import synth
from tests.gpu_util import (DECODE_TOL, PREFILL_TOL, Pair, assert_plan_equal, assert_stats_equal,
                            pinned_store, row_rel_err)

pytestmark = pytest.mark.gpu

SH = synth.DECODE
CALLS = 3


@pytest.fixture(scope="module")
def store():
    return pinned_store(1, SH.E, SH.H, SH.F, seed=21)


@pytest.mark.parametrize("path", ["gemv-f32", "gemv-bf16", "gemm"])
@pytest.mark.parametrize("T", [2, 3, 4, 5, 8, 9, 16, 31])
def test_small_batch_parity(store, T, path):
    act = "f32" if path == "gemv-f32" else "bf16"
    gemm = path == "gemm"
    _, logits, x = synth.batch_inputs(SH, CALLS, T, seed=21 + T, layers=[0], act=act)
    p = Pair(1, SH.E, SH.k, SH.H, SH.F, SH.S, store, max_tokens=T, act=act, fill_mode=1,
             gemm_min_tokens=1 if gemm else 0)
    tol = PREFILL_TOL if gemm else DECODE_TOL
    for b in range(CALLS):
        check = b != 1
        g, plan, r = p.step(0, logits[b, 0], x[b, 0], compute_oracle=check)
        assert_plan_equal(plan, r, f"T={T} call {b}")
        if check:
            err = row_rel_err(g, r["out"]).max()
            assert err <= tol, (T, path, b, err)
    assert_stats_equal(p.gpu.stats(0), p.orc.stats(0))
    p.close()


@pytest.mark.parametrize("T", [2, 4])
def test_two_group_decode_kernel_matches_staged_gemv(store, T):
    # the same calls with 8 slots (more possible experts than slots: the GEMV
    # kernels, staged where needed) and with 32 (one stage for sure: the decode
    # layer kernel, two compute groups): bitwise equal outputs
    _, logits, x = synth.batch_inputs(SH, 4, T, seed=40 + T, layers=[0], act="f32")
    outs = {}
    for S in (8, 32):
        p = Pair(1, SH.E, SH.k, SH.H, SH.F, S, store, max_tokens=T, act="f32", fill_mode=1)
        outs[S] = [p.step(0, logits[b, 0], x[b, 0], compute_oracle=False)[0] for b in range(4)]
        p.close()
    for b in range(4):
        assert np.array_equal(outs[8][b], outs[32][b]), b
