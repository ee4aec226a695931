"""Error paths of the C ABI on the GPU: edge sizes, rejected inputs, poisoning,
failure injection (a host wait whose limit is too short; a device wait for a
value that is never written, ended by its limit).  Nothing here faults or
hangs the device: every failure is made on the host, is a value check the
kernels perform, or is a bounded device wait that runs out."""
import numpy as np
import pytest

import router_softmax_top_gb300 as moe
import synth
from tests.gpu_util import pinned_store

pytestmark = pytest.mark.gpu

TINY = synth.TINY


def _cache(store, **kw):
    args = dict(n_layers=1, n_experts=TINY.E, top_k=TINY.k, hidden=TINY.H, ffn=TINY.F,
                slots_per_layer=TINY.S, max_tokens=4, store=store)
    args.update(kw)
    return moe.MoECache(**args)


@pytest.fixture(scope="module")
def store():
    return pinned_store(1, TINY.E, TINY.H, TINY.F, seed=0)


def _inputs(T=4):
    import torch
    lg, x = synth.tiny_inputs(0)
    return torch.from_numpy(lg[:T].copy()).cuda(), torch.from_numpy(x[:T].copy()).cuda()


def test_zero_tokens_is_noop(store):
    import torch
    c = _cache(store)
    lg, x = _inputs()
    out = torch.full((4, TINY.H), 7.0, device="cuda")
    assert c.forward_rc(0, lg[:0], x[:0], out) == moe.MOE_OK
    torch.cuda.synchronize()
    assert torch.all(out == 7.0)
    assert c.stats(0)["calls"] == 0
    c.close()


def test_too_many_tokens_and_bad_layer(store):
    import torch
    c = _cache(store, max_tokens=2)
    lg, x = _inputs(4)
    out = torch.empty((4, TINY.H), device="cuda")
    assert c.forward_rc(0, lg, x, out) == moe.MOE_ERR_INVALID_ARG
    assert moe.moe_layer_forward(c.handle, 3, lg.data_ptr(), x.data_ptr(), 1, out.data_ptr()) \
        == moe.MOE_ERR_INVALID_ARG
    assert c.stats(-1)["poisoned"] == 0     # argument errors do not poison
    c.forward(0, lg[:2], x[:2])
    c.close()


@pytest.mark.parametrize("fill_mode", [0, 1])
@pytest.mark.parametrize("bad", [float("nan"), float("inf")])
def test_non_finite_logit_poisons(store, fill_mode, bad):
    import torch
    c = _cache(store, fill_mode=fill_mode, slots_per_layer=8)
    lg, x = _inputs(2)
    out = torch.empty((2, TINY.H), device="cuda")
    c.forward(0, lg, x, out)                       # a good call first
    before = c.stats(0)
    lg2 = lg.clone()
    lg2[1, 3] = bad
    rc = c.forward_rc(0, lg2, x, out)
    if rc == moe.MOE_OK:                           # pull mode reports after the fact
        rc = c.sync()
    assert rc == moe.MOE_ERR_INVALID_ARG
    st = c.stats(0)
    assert st["poisoned"] == 1 and st["last_error"] == moe.MOE_ERR_INVALID_ARG
    assert st["calls"] == before["calls"]          # the layer's state did not move
    assert c.forward_rc(0, lg, x, out) == moe.MOE_ERR_POISONED
    c.close()


@pytest.mark.parametrize("fill_mode", [0, 1])
def test_non_finite_logit_large_call_poisons(store, fill_mode):
    # more than 64 tokens: routing runs in its own grid and reports through a
    # device flag that the plan kernel reads
    import numpy as np
    import torch
    T = 100
    c = _cache(store, fill_mode=fill_mode, max_tokens=T)
    rng = np.random.default_rng(7)
    lg = torch.from_numpy(rng.standard_normal((T, TINY.E)).astype(np.float32)).cuda()
    x = torch.from_numpy(rng.standard_normal((T, TINY.H)).astype(np.float32)).cuda()
    out = torch.empty((T, TINY.H), device="cuda")
    c.forward(0, lg, x, out)
    before = c.stats(0)
    lg2 = lg.clone()
    lg2[77, 5] = float("nan")
    rc = c.forward_rc(0, lg2, x, out)
    if rc == moe.MOE_OK:
        rc = c.sync()
    assert rc == moe.MOE_ERR_INVALID_ARG
    st = c.stats(0)
    assert st["poisoned"] == 1 and st["calls"] == before["calls"]
    c.close()
    # a fresh handle on the same device routes large calls normally again
    c = _cache(store, fill_mode=fill_mode, max_tokens=T)
    c.forward(0, lg, x, out)
    assert c.stats(0)["calls"] == 1 and c.stats(0)["poisoned"] == 0
    c.close()


def test_timeout_on_host_wait_poisons(store):
    # the stream is kept busy (~25 ms of device sleep) ahead of the call, so its
    # plan cannot have written the mailbox when the host's wait (limit 1 ms)
    # gives up: the call returns MOE_ERR_TIMEOUT every time
    import torch
    c = _cache(store, timeout_us=1000)           # memcpy fill, 4 tokens: the host reads the mailbox
    lg, x = _inputs(4)
    out = torch.empty((4, TINY.H), device="cuda")
    torch.cuda.synchronize()
    torch.cuda._sleep(50_000_000)                  # ~25 ms at 2 GHz on the current stream
    assert c.forward_rc(0, lg, x, out) == moe.MOE_ERR_TIMEOUT
    st = c.stats(-1)
    assert st["poisoned"] == 1 and st["last_error"] == moe.MOE_ERR_TIMEOUT
    assert c.forward_rc(0, lg, x, out) == moe.MOE_ERR_POISONED
    c.close()                                      # waits for the work in flight, frees all
    torch.cuda.synchronize()


@pytest.mark.parametrize("T,S,n", [(1, 8, 1), (1, 8, 2), (4, 4, 2)])
def test_failed_fill_copy_poisons(store, T, S, n):
    # the n-th host-to-device copy of a missed block fails before it is issued
    # (host-side injection): the call returns MOE_ERR_CUDA, the handle is
    # poisoned, the statistics stay readable, and kernels of the call that wait
    # for the missing block end by their bounded wait (timeout_us / 4 = 50 ms)
    import torch
    c = _cache(store, fill_mode=moe.MOE_FILL_MEMCPY, slots_per_layer=S, max_tokens=T, timeout_us=200_000)
    lg, x = _inputs(4)
    out = torch.empty((T, TINY.H), device="cuda")
    c.inject(moe.MOE_INJECT_MEMCPY_FAIL | (n << 8))
    rc = moe.MOE_OK
    for t in range(4):                             # calls with misses until the n-th copy
        s0 = t if T == 1 else 0
        rc = c.forward_rc(0, lg[s0:s0 + T], x[s0:s0 + T], out)
        if rc != moe.MOE_OK:
            break
    assert rc == moe.MOE_ERR_CUDA
    st = c.stats(-1)
    assert st["poisoned"] == 1 and st["last_error"] == moe.MOE_ERR_CUDA and st["cuda_error"] == 999
    assert st["calls"] >= 1
    assert c.forward_rc(0, lg[:T], x[:T], out) == moe.MOE_ERR_POISONED
    c.close()
    torch.cuda.synchronize()
    c2 = _cache(store, fill_mode=moe.MOE_FILL_MEMCPY, slots_per_layer=S, max_tokens=T)
    c2.forward(0, lg[:T], x[:T], out)
    assert c2.sync() == moe.MOE_OK and torch.isfinite(out).all()
    c2.close()


def test_device_wait_limit_poisons(store):
    # injected fault, no GPU fault: the decode layer kernel waits for a gate
    # value carrying a call number that is never written.  Its bounded wait
    # (timeout_us / 4 = 50 ms) gives up, ends the other CTAs' waits, the kernel
    # finishes, and the handle reports MOE_ERR_TIMEOUT at the next sync; the
    # device stays usable.
    import torch
    c = _cache(store, fill_mode=moe.MOE_FILL_PULL, timeout_us=200_000)
    lg, x = _inputs(1)
    out = torch.empty((1, TINY.H), device="cuda")
    c.forward(0, lg, x, out)                       # a normal call first
    assert c.sync() == moe.MOE_OK
    c.inject(moe.MOE_INJECT_DECODE_WAIT)
    assert c.forward_rc(0, lg, x, out) == moe.MOE_OK   # launched: the failure shows at the sync
    assert c.sync() == moe.MOE_ERR_TIMEOUT
    st = c.stats(-1)
    assert st["poisoned"] == 1 and st["last_error"] == moe.MOE_ERR_TIMEOUT
    assert c.forward_rc(0, lg, x, out) == moe.MOE_ERR_POISONED
    c.close()
    torch.cuda.synchronize()
    # a fresh handle on the same device computes normally
    c2 = _cache(store, fill_mode=moe.MOE_FILL_PULL)
    c2.forward(0, lg, x, out)
    assert c2.sync() == moe.MOE_OK and c2.stats(-1)["poisoned"] == 0
    assert torch.isfinite(out).all()
    c2.close()


def test_inject_rejects_unknown_code(store):
    c = _cache(store)
    with pytest.raises(moe.MoeError):
        c.inject(7)
    with pytest.raises(moe.MoeError):
        c.inject(moe.MOE_INJECT_MEMCPY_FAIL | (-1 << 8))
    c.inject(moe.MOE_INJECT_MEMCPY_FAIL | (3 << 8))
    c.inject(0)                                    # clears both kinds
    c.close()


def test_unaligned_store_rejected(store):
    import ctypes
    cfg = moe.MoeCacheConfig(1, TINY.E, TINY.k, TINY.H, TINY.F, TINY.S, 4, 0, 0, 0, 0, 0, 0, 0, 10**6)
    hs = moe.MoeHostStore(store.data_ptr() + 2, store.numel() - 2, TINY.E * TINY.expert_bytes,
                          TINY.expert_bytes)
    h = ctypes.c_void_p()
    assert moe.lib().moe_cache_init(ctypes.byref(cfg), ctypes.byref(hs), None, ctypes.byref(h)) \
        == moe.MOE_ERR_HOST_STORE
    hs = moe.MoeHostStore(store.data_ptr(), 1000, TINY.E * TINY.expert_bytes, TINY.expert_bytes)
    assert moe.lib().moe_cache_init(ctypes.byref(cfg), ctypes.byref(hs), None, ctypes.byref(h)) \
        == moe.MOE_ERR_HOST_STORE


def test_unpinned_store_is_registered():
    # an ordinary (pageable) numpy buffer is registered at init and released at destroy
    import torch
    buf = synth.store(1, TINY.E, TINY.H, TINY.F, seed=0)
    c = moe.MoECache(n_layers=1, n_experts=TINY.E, top_k=TINY.k, hidden=TINY.H, ffn=TINY.F,
                     slots_per_layer=TINY.S, max_tokens=4, store=(buf.ctypes.data, buf.nbytes))
    lg, x = _inputs(4)
    out = c.forward(0, lg, x)
    torch.cuda.synchronize()
    assert torch.isfinite(out).all()
    c.close()


def test_timing_and_launch_count(store):
    import torch
    c = _cache(store)
    lg, x = _inputs(4)
    c.set_timing(True)
    for _ in range(3):
        c.forward(0, lg, x)
    t = c.timing()
    c.set_timing(False)
    assert t["plan"]["launches"] == 3 and t["plan"]["ms"] > 0
    assert c.launch_count() >= 3 * 3      # plan, gate/up, down(+combine) at least
    assert c.probe_h2d(5) > 0.1
    c.close()
