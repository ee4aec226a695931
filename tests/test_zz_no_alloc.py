"""The allocation-free expert entry point (moe_expert_ffn_static), through the C ABI.

It serves callers that cannot allocate device memory: code running while a CUDA
graph is being captured (allocation calls cannot be captured), real-time paths
that must not block on an allocator, and plugins that do not own the process's
memory pool.  Its output is checked against the CPU oracle's expert FFN (exact,
in double) and against the library's regular entry point for the same expert (a
one-expert cache: E = k = 1, so the router weight is exactly 1 and the layer
output is the expert's y), on two calls in a row.
Collected last on purpose: the fixed scratch array it uses is shared by every
call in the process."""
import os

import numpy as np
import pytest

import oracle
import router_softmax_top_gb300 as moe
from tests.gpu_util import DECODE_TOL, pinned_store, row_rel_err

pytestmark = pytest.mark.gpu


def _oracle_y(block: np.ndarray, H: int, F: int, x: np.ndarray) -> np.ndarray:
    return np.stack([oracle.expert_ffn(block, H, F, x[t].astype(np.float64)) for t in range(x.shape[0])])


@pytest.mark.parametrize("H,F,T", [(2816, 704, 1), (256, 512, 8), (4096, 1536, 8)])
def test_static_entry_matches_oracle_and_layer_forward(H, F, T):
    import torch
    store = pinned_store(1, 1, H, F, seed=11)           # one expert
    block_d = store.cuda()                               # canonical block in device memory
    cache = moe.MoECache(n_layers=1, n_experts=1, top_k=1, hidden=H, ffn=F, slots_per_layer=1,
                         max_tokens=T, store=store)
    rng = np.random.default_rng(H + T)
    for call in range(2):                                # two calls in a row, fresh inputs each
        xh = rng.standard_normal((T, H)).astype(np.float32)
        x = torch.from_numpy(xh).cuda()
        y = torch.full((T, H), float("nan"), dtype=torch.float32, device="cuda")
        rc = moe.moe_expert_ffn_static(block_d.data_ptr(), H, F, x.data_ptr(), T, y.data_ptr())
        assert rc == moe.MOE_OK
        torch.cuda.synchronize()
        got = y.cpu().numpy()
        assert np.all(np.isfinite(got)), call
        err = row_rel_err(got, _oracle_y(store.numpy(), H, F, xh))
        assert err.max() <= DECODE_TOL, (call, err.max())
        logits = torch.zeros((T, 1), dtype=torch.float32, device="cuda")
        ref = cache.forward(0, logits, x)
        err2 = row_rel_err(got, ref.cpu().numpy())
        assert err2.max() <= DECODE_TOL, (call, err2.max())
    cache.close()


def test_static_entry_reads_mapped_host_block():
    # the block stays in page-locked host memory: with unified addressing its
    # host address is also its device address, read over the host link
    import torch
    H, F, T = 2816, 704, 2
    store = pinned_store(1, 1, H, F, seed=12)
    rng = np.random.default_rng(7)
    for call in range(2):
        xh = rng.standard_normal((T, H)).astype(np.float32)
        x = torch.from_numpy(xh).cuda()
        y = torch.full((T, H), float("nan"), dtype=torch.float32, device="cuda")
        assert moe.moe_expert_ffn_static(store.data_ptr(), H, F, x.data_ptr(), T, y.data_ptr()) == moe.MOE_OK
        torch.cuda.synchronize()
        err = row_rel_err(y.cpu().numpy(), _oracle_y(store.numpy(), H, F, xh))
        assert err.max() <= DECODE_TOL, (call, err.max())


def test_static_entry_reports_a_wait_that_gave_up():
    # MOE_STATIC_INJECT_WAIT=1 makes the down tiles wait for a count that is
    # never reached (a test hook; no GPU fault): their bounded wait gives up,
    # they write NaN, and the next call reports MOE_ERR_TIMEOUT once
    import torch
    H, F, T = 256, 512, 3
    store = pinned_store(1, 1, H, F, seed=13)
    block_d = store.cuda()
    xh = np.random.default_rng(3).standard_normal((T, H)).astype(np.float32)
    x = torch.from_numpy(xh).cuda()
    y = torch.zeros((T, H), dtype=torch.float32, device="cuda")
    os.environ["MOE_STATIC_INJECT_WAIT"] = "1"
    try:
        assert moe.moe_expert_ffn_static(block_d.data_ptr(), H, F, x.data_ptr(), T, y.data_ptr()) == moe.MOE_OK
        torch.cuda.synchronize()
    finally:
        del os.environ["MOE_STATIC_INJECT_WAIT"]
    assert np.all(np.isnan(y.cpu().numpy()))             # no stale values that look valid
    assert moe.moe_expert_ffn_static(block_d.data_ptr(), H, F, x.data_ptr(), T, y.data_ptr()) \
        == moe.MOE_ERR_TIMEOUT                           # the record, reported once
    assert moe.moe_expert_ffn_static(block_d.data_ptr(), H, F, x.data_ptr(), T, y.data_ptr()) == moe.MOE_OK
    torch.cuda.synchronize()
    err = row_rel_err(y.cpu().numpy(), _oracle_y(store.numpy(), H, F, xh))
    assert err.max() <= DECODE_TOL


def test_static_entry_limits():
    import torch
    x = torch.zeros((9, 256), dtype=torch.float32, device="cuda")
    y = torch.zeros_like(x)
    blk = torch.zeros(moe.moe_expert_bytes(256, 512), dtype=torch.uint8, device="cuda")
    assert moe.moe_expert_ffn_static(blk.data_ptr(), 256, 512, x.data_ptr(), 9, y.data_ptr()) \
        == moe.MOE_ERR_UNSUPPORTED                        # more than 8 tokens
    assert moe.moe_expert_ffn_static(blk.data_ptr(), 8192, 512, x.data_ptr(), 1, y.data_ptr()) \
        == moe.MOE_ERR_UNSUPPORTED                        # hidden above 4096
    assert moe.moe_expert_ffn_static(0, 256, 512, x.data_ptr(), 1, y.data_ptr()) \
        == moe.MOE_ERR_INVALID_ARG
    assert moe.moe_expert_ffn_static(blk.data_ptr(), 256, 512, x.data_ptr(), 0, y.data_ptr()) \
        == moe.MOE_OK                                     # no-op
