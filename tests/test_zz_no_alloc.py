"""The allocation-free expert entry point (moe_expert_ffn_static), through the C ABI.

It serves callers that cannot allocate (graph capture, real-time paths, plugins
without their own pool).  Its output must match what the library's regular
entry point computes for the same expert: a one-expert cache (E = k = 1, so
the router weight is exactly 1 and the layer output is the expert's y).
Collected last on purpose: the fixed scratch array it uses is shared by every
call in the process."""
import numpy as np
import pytest

import router_softmax_top_gb300 as moe
import synth
from tests.gpu_util import DECODE_TOL, pinned_store, row_rel_err

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("H,F,T", [(2816, 704, 1), (256, 512, 8), (4096, 1536, 8)])
def test_static_entry_matches_layer_forward(H, F, T):
    import torch
    store = pinned_store(1, 1, H, F, seed=11)           # one expert
    block_d = store.cuda()                               # canonical block in device memory
    cache = moe.MoECache(n_layers=1, n_experts=1, top_k=1, hidden=H, ffn=F, slots_per_layer=1,
                         max_tokens=T, store=store)
    rng = np.random.default_rng(H + T)
    for call in range(2):                                # two calls in a row, fresh inputs each
        x = torch.from_numpy(rng.standard_normal((T, H)).astype(np.float32)).cuda()
        logits = torch.zeros((T, 1), dtype=torch.float32, device="cuda")
        ref = cache.forward(0, logits, x)
        y = torch.full((T, H), float("nan"), dtype=torch.float32, device="cuda")
        rc = moe.moe_expert_ffn_static(block_d.data_ptr(), H, F, x.data_ptr(), T, y.data_ptr())
        assert rc == moe.MOE_OK
        torch.cuda.synchronize()
        err = row_rel_err(y.cpu().numpy(), ref.cpu().numpy())
        assert np.all(np.isfinite(y.cpu().numpy())), call
        assert err.max() <= DECODE_TOL, (call, err.max())
    cache.close()


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
