"""The product path has no CPU fallback (CPU only): without the built library
the binding raises, and without a GPU the cache's init fails with a CUDA error
instead of computing anything on the host."""
import pytest
import torch

import router_softmax_top_gb300 as moe
import synth


def test_missing_library_raises(monkeypatch, tmp_path):
    monkeypatch.setattr(moe, "LIB_PATH", str(tmp_path / "libmoe_cache.so"))
    monkeypatch.setattr(moe, "_lib", None)
    with pytest.raises(RuntimeError, match="is missing"):
        moe.lib()


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the behaviour without a GPU")
def test_no_gpu_means_an_error_not_a_host_computation():
    sh = synth.TINY
    store = torch.zeros(sh.L * sh.E * synth.expert_bytes(sh.H, sh.F), dtype=torch.uint8)
    with pytest.raises(moe.MoeError) as e:
        moe.MoECache(n_layers=1, n_experts=sh.E, top_k=sh.k, hidden=sh.H, ffn=sh.F,
                     slots_per_layer=sh.S, max_tokens=4, store=store, stream=0)
    assert e.value.code == moe.MOE_ERR_CUDA
