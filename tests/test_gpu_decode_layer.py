"""The decode layer kernel (pull fill, single-stage calls of at most 8 tokens)
against the oracle and against the GEMV kernels of the other schedules (GPU).

Every kernel of the decode path reduces in one canonical order, so the decode
layer kernel must give bitwise the outputs of the staged GEMV path (any slot
budget) and of the copy-engine schedule, besides the oracle's slot maps and
outputs within 1e-3 max relative error."""
import numpy as np
import pytest

import synth
from tests.gpu_util import (DECODE_TOL, Pair, assert_plan_equal, assert_stats_equal,
                            pinned_store, row_rel_err)

pytestmark = pytest.mark.gpu

TINY = synth.TINY


@pytest.fixture(scope="module")
def tiny_store():
    return pinned_store(TINY.L, TINY.E, TINY.H, TINY.F, seed=0)


def test_budget_invariance_pull(tiny_store):
    # S = 8 = E: every call single-stage -> decode layer kernel (4-token and
    # 1-token variants); smaller budgets run the staged GEMV path
    logits, x = synth.tiny_inputs(0)
    outs = {}
    for S in range(1, TINY.E + 1):
        p = Pair(TINY.L, TINY.E, TINY.k, TINY.H, TINY.F, S, tiny_store, max_tokens=4, fill_mode=1)
        got = []
        g, plan, r = p.step(0, logits, x)
        assert_plan_equal(plan, r, f"S={S}")
        assert row_rel_err(g, r["out"]).max() <= DECODE_TOL
        got.append(g)
        for t in range(4):
            g, plan, r = p.step(0, logits[t:t + 1], x[t:t + 1])
            assert_plan_equal(plan, r, f"S={S} t={t}")
            got.append(g)
        outs[S] = got
        assert_stats_equal(p.gpu.stats(0), p.orc.stats(0))
        p.close()
    for S in outs:
        for a, b in zip(outs[S], outs[TINY.E]):
            assert np.array_equal(a, b), S


def test_decode_kernel_matches_copy_engine_schedule():
    # decode model shapes, 2 layers: pull (decode layer kernel) and memcpy
    # (copy engine + GEMV kernels + combine) give the same plans and bitwise
    # the same outputs
    sh = synth.DECODE
    layers = [0, 1]
    store = pinned_store(len(layers), sh.E, sh.H, sh.F, seed=1)
    steps = 24
    picks, logits, x = synth.decode_inputs(sh, steps, batch=1, seed=1, layers=layers)
    pull = Pair(len(layers), sh.E, sh.k, sh.H, sh.F, sh.S, store, max_tokens=1, fill_mode=1)
    copy = Pair(len(layers), sh.E, sh.k, sh.H, sh.F, sh.S, store, max_tokens=1, fill_mode=0)
    worst = 0.0
    for s in range(steps):
        for li in range(len(layers)):
            check = s in (0, 7, steps - 1)
            ga, pa, ra = pull.step(li, logits[s, li], x[s, li], compute_oracle=check)
            gb, pb, _ = copy.step(li, logits[s, li], x[s, li], compute_oracle=False)
            assert_plan_equal(pa, ra, f"step {s} layer {li}")
            assert np.array_equal(pa["gpu_slot"], pb["gpu_slot"])
            assert np.array_equal(ga, gb), (s, li)
            if check:
                worst = max(worst, row_rel_err(ga, ra["out"]).max())
    assert worst <= DECODE_TOL, worst
    st = pull.gpu.stats(-1)
    assert st["unique_misses"] > 0 and st["unique_hits"] > 0
    pull.close()
    copy.close()


@pytest.mark.parametrize("T", [1, 3, 4])
def test_bf16_inputs_decode_kernel(T):
    # bf16 activations through the decode layer kernel (T * k <= 32 slots: single stage)
    sh = synth.PREFILL
    store = pinned_store(1, sh.E, sh.H, sh.F, seed=2)
    _, logits, x = synth.batch_inputs(sh, 3, T, seed=2, layers=[0], act="bf16")
    p = Pair(1, sh.E, sh.k, sh.H, sh.F, sh.S, store, max_tokens=T, act="bf16", fill_mode=1)
    for b in range(3):
        g, plan, r = p.step(0, logits[b, 0], x[b, 0])
        assert_plan_equal(plan, r, f"batch {b}")
        assert row_rel_err(g, r["out"]).max() <= DECODE_TOL
    assert_stats_equal(p.gpu.stats(0), p.orc.stats(0))
    p.close()


def test_weight_mode_renormalised_pull(tiny_store):
    logits, x = synth.tiny_inputs(1)
    p = Pair(TINY.L, TINY.E, TINY.k, TINY.H, TINY.F, 8, tiny_store, max_tokens=4, weight_mode=1, fill_mode=1)
    for _ in range(2):
        g, plan, r = p.step(0, logits, x)
        assert_plan_equal(plan, r)
        np.testing.assert_allclose(plan["w"].sum(axis=1), 1.0, rtol=1e-6)
        assert row_rel_err(g, r["out"]).max() <= DECODE_TOL
    p.close()


def test_repeated_calls_reuse_slots_written_on_the_way():
    # a miss is written into its slot by the decode layer kernel while it is
    # computed; the next call's hits read those slots (checked against the oracle)
    sh = synth.DECODE
    store = pinned_store(1, sh.E, sh.H, sh.F, seed=3)
    rng = np.random.default_rng(3)
    p = Pair(1, sh.E, sh.k, sh.H, sh.F, sh.S, store, max_tokens=1, fill_mode=1)
    x = rng.standard_normal((1, sh.H)).astype(np.float32)
    lg = rng.standard_normal((1, sh.E)).astype(np.float32)
    g0, plan0, r0 = p.step(0, lg, x)           # all 8 picks miss (empty cache)
    assert_plan_equal(plan0, r0)
    g1, plan1, r1 = p.step(0, lg, x)           # same picks: all hits now
    assert_plan_equal(plan1, r1)
    assert np.array_equal(g0, g1)              # slot contents equal the host blocks
    assert row_rel_err(g1, r1["out"]).max() <= DECODE_TOL
    st = p.gpu.stats(0)
    assert st["unique_misses"] == 8 and st["unique_hits"] == 8
    p.close()


def test_step_graph_replay_matches_eager_calls():
    # pull fill, single-token calls: a step of layer calls captured as a CUDA
    # graph and replayed gives bitwise the outputs and statistics of the same
    # calls issued one by one
    import ctypes
    import torch
    import router_softmax_top_gb300 as moe
    sh = synth.DECODE
    layers = [0, 1]
    L = len(layers)
    store = pinned_store(L, sh.E, sh.H, sh.F, seed=4)
    steps = 12
    _, logits, x = synth.decode_inputs(sh, steps, batch=1, seed=4, layers=layers)
    lg_d = torch.from_numpy(logits).cuda()
    x_d = torch.from_numpy(x).cuda()

    def make():
        return moe.MoECache(n_layers=L, n_experts=sh.E, top_k=sh.k, hidden=sh.H, ffn=sh.F,
                            slots_per_layer=sh.S, max_tokens=1, store=store, fill_mode=moe.MOE_FILL_PULL)

    fwd = moe.lib().moe_layer_forward
    # eager
    a = make()
    out_a = torch.empty((steps, L, 1, sh.H), device="cuda")
    sa = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for s in range(steps):
        for l in range(L):
            assert fwd(a.handle, l, ctypes.c_void_p(lg_d[s, l].data_ptr()), ctypes.c_void_p(x_d[s, l].data_ptr()),
                       1, ctypes.c_void_p(out_a[s, l].data_ptr()), sa) == 0
    torch.cuda.synchronize()
    # graph: first step eager (warms the library up), then capture one step and replay
    b = make()
    out_b = torch.empty((steps, L, 1, sh.H), device="cuda")
    lg_cur = torch.empty((L, 1, sh.E), device="cuda")
    x_cur = torch.empty((L, 1, sh.H), device="cuda")
    out_cur = torch.empty((L, 1, sh.H), device="cuda")
    for l in range(L):
        assert fwd(b.handle, l, ctypes.c_void_p(lg_d[0, l].data_ptr()), ctypes.c_void_p(x_d[0, l].data_ptr()),
                   1, ctypes.c_void_p(out_b[0, l].data_ptr()), sa) == 0
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream()
    with torch.cuda.graph(g, stream=cap):
        cs = ctypes.c_void_p(cap.cuda_stream)
        for l in range(L):
            assert fwd(b.handle, l, ctypes.c_void_p(lg_cur[l].data_ptr()), ctypes.c_void_p(x_cur[l].data_ptr()),
                       1, ctypes.c_void_p(out_cur[l].data_ptr()), cs) == 0
    for s in range(1, steps):
        lg_cur.copy_(lg_d[s])
        x_cur.copy_(x_d[s])
        g.replay()
        out_b[s].copy_(out_cur)
    torch.cuda.synchronize()
    assert torch.equal(out_a, out_b)
    sa_, sb_ = a.stats(-1), b.stats(-1)
    for key in ("calls", "pick_hits", "pick_misses", "unique_hits", "unique_misses", "evictions"):
        assert sa_[key] == sb_[key], key
    assert sb_["unique_misses"] > 0 and sb_["poisoned"] == 0
    a.close()
    b.close()


def test_full_decode_config_graph_sampled():
    # the decode workload at full size (30 layers, 12.8 GB host store) in the
    # launch configuration the bench times: one step of 30 layer calls
    # captured as a CUDA graph and replayed.  The oracle follows every call
    # (its cache state) and computes the outputs of sampled steps, one eager
    # and two replayed; statistics must agree exactly at the end.
    import ctypes
    import torch
    import oracle
    import router_softmax_top_gb300 as moe
    sh = synth.DECODE
    L = sh.L
    store = pinned_store(L, sh.E, sh.H, sh.F, seed=0)
    W, K = 6, 18
    steps = W + K
    _, logits, x = synth.decode_inputs(sh, steps, batch=1, seed=0)
    lg_d = torch.from_numpy(logits).cuda()
    x_d = torch.from_numpy(x).cuda()
    c = moe.MoECache(n_layers=L, n_experts=sh.E, top_k=sh.k, hidden=sh.H, ffn=sh.F,
                     slots_per_layer=sh.S, max_tokens=1, store=store, fill_mode=moe.MOE_FILL_PULL)
    orc = oracle.Cache(L, sh.E, sh.k, sh.H, sh.F, sh.S, store.numpy())
    fwd = moe.lib().moe_layer_forward
    out = torch.empty((L, 1, sh.H), device="cuda")
    check = {W - 1, W + K // 2, steps - 1}
    worst = 0.0

    def follow(s):
        # the oracle's calls of step s; the outputs of sampled steps compared
        nonlocal worst
        res = [orc.forward(l, logits[s, l], x[s, l] if s in check else None, compute=s in check)
               for l in range(L)]
        if s in check:
            torch.cuda.synchronize()
            got = out.cpu().numpy()
            for l in range(L):
                worst = max(worst, row_rel_err(got[l], res[l]["out"]).max())

    sa = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for s in range(W):
        for l in range(L):
            assert fwd(c.handle, l, ctypes.c_void_p(lg_d[s, l].data_ptr()), ctypes.c_void_p(x_d[s, l].data_ptr()),
                       1, ctypes.c_void_p(out[l].data_ptr()), sa) == 0
        follow(s)
    lg_cur = torch.empty((L, 1, sh.E), device="cuda")
    x_cur = torch.empty((L, 1, sh.H), device="cuda")
    g = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=cap):
        cs = ctypes.c_void_p(cap.cuda_stream)
        for l in range(L):
            assert fwd(c.handle, l, ctypes.c_void_p(lg_cur[l].data_ptr()), ctypes.c_void_p(x_cur[l].data_ptr()),
                       1, ctypes.c_void_p(out[l].data_ptr()), cs) == 0
    for s in range(W, steps):
        lg_cur.copy_(lg_d[s])
        x_cur.copy_(x_d[s])
        g.replay()
        follow(s)
    torch.cuda.synchronize()
    assert worst <= DECODE_TOL, worst
    per_layer = [orc.stats(l) for l in range(L)]
    assert_stats_equal(c.stats(-1), {key: sum(d[key] for d in per_layer) for key in per_layer[0]})
    st = c.stats(-1)
    assert st["poisoned"] == 0 and st["calls"] == L * steps and st["unique_misses"] > 0
    c.close()
