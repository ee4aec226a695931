"""Helpers for the GPU parity tests: one CUDA cache and one oracle cache fed the
same seeded inputs, compared call by call."""
import numpy as np

import oracle
import synth

DECODE_TOL = 1e-3   # max relative error per token row, fp32-accumulate paths
PREFILL_TOL = 2e-2  # bf16 tensor-core path


def torch():
    import torch as _t
    return _t


def pinned_store(L, E, H, F, seed=0, threads=0):
    t = torch()
    eb = synth.expert_bytes(H, F)
    buf = t.empty(L * E * eb, dtype=t.uint8, pin_memory=True)
    synth.fill_store(buf.data_ptr(), L, E, H, F, seed, threads)
    return buf


def row_rel_err(gpu, ref):
    """Per token row: max_i |gpu - ref| / max_i |ref|."""
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.maximum(np.abs(ref).max(axis=-1), 1e-30)
    return np.abs(gpu - ref).max(axis=-1) / den


class Pair:
    """A CUDA cache and an oracle cache over the same pinned host store."""

    def __init__(self, L, E, k, H, F, S, store, max_tokens, fill_mode=0, act="f32",
                 weight_mode=0, gemm_min_tokens=0, timeout_us=20_000_000, policy=0, admit_budget=0,
                 sticky=0):
        import router_softmax_top_gb300 as moe
        self.moe = moe
        self.L, self.E, self.k, self.H, self.F, self.S = L, E, k, H, F, S
        self.act = act
        self.store = store
        self.gpu = moe.MoECache(n_layers=L, n_experts=E, top_k=k, hidden=H, ffn=F,
                                slots_per_layer=S, max_tokens=max_tokens, store=store,
                                weight_mode=weight_mode, act_dtype=act, fill_mode=fill_mode,
                                gemm_min_tokens=gemm_min_tokens, timeout_us=timeout_us,
                                policy=policy, admit_budget=admit_budget, sticky_permille=sticky)
        self.orc = oracle.Cache(L, E, k, H, F, S, store.numpy(), weight_mode=weight_mode, policy=policy,
                                admit_budget=admit_budget, sticky=sticky)

    def close(self):
        self.gpu.close()

    def step(self, layer, logits, x, compute_oracle=True):
        """Run one layer call on both sides; returns (gpu_out, gpu_plan, oracle_result)."""
        t = torch()
        T = logits.shape[0]
        lg = t.from_numpy(np.ascontiguousarray(logits, np.float32)).cuda()
        if self.act == "bf16":
            xd = t.from_numpy(np.ascontiguousarray(x).view(np.int16)).cuda().view(t.bfloat16)
        else:
            xd = t.from_numpy(np.ascontiguousarray(x, np.float32)).cuda()
        out = self.gpu.forward(layer, lg, xd)
        plan = self.gpu.last_plan(layer, T)
        gout = out.cpu().numpy()
        res = self.orc.forward(layer, logits, x if compute_oracle else None, compute=compute_oracle)
        return gout, plan, res


def assert_plan_equal(plan, res, where=""):
    assert np.array_equal(plan["ids"], res["ids"]), f"ids {where}"
    assert np.array_equal(plan["gpu_slot"], res["gpu_slot"]), f"gpu_slot {where}"
    assert np.array_equal(plan["stage"], res["stage"]), f"stage {where}"
    for key in ("miss_expert", "miss_slot", "miss_evicted", "miss_stage"):
        assert np.array_equal(plan[key], res[key]), f"{key} {where}"
    assert plan["n_stages"] == res["info"]["n_stages"], f"n_stages {where}"
    # router weights: fp32 softmax on the device vs double in the oracle
    np.testing.assert_allclose(plan["w"], res["w"], rtol=2e-6, atol=1e-9, err_msg=f"w {where}")


def assert_stats_equal(gpu_stats, orc_stats):
    for key in ("calls", "pick_hits", "pick_misses", "unique_hits", "unique_misses", "evictions",
                "bytes_uploaded", "stages", "staged_calls", "bypassed"):
        assert gpu_stats[key] == orc_stats[key], key


def anonymous_store(nbytes: int):
    """A host store in ordinary anonymous memory (transparent huge pages
    requested), as a torch uint8 tensor; the library pins and maps it at init.
    For stores too large for cudaHostAlloc to be quick (the large model's
    130 GB)."""
    import mmap
    t = torch()
    mm = mmap.mmap(-1, nbytes, flags=mmap.MAP_PRIVATE | mmap.MAP_ANONYMOUS)
    if hasattr(mmap, "MADV_HUGEPAGE"):
        mm.madvise(mmap.MADV_HUGEPAGE)
    arr = np.frombuffer(mm, dtype=np.uint8, count=nbytes)
    ten = t.from_numpy(arr)
    ten._moe_mmap = mm          # keep the mapping alive with the tensor
    return ten


def mem_available_bytes():
    """MemAvailable of the host (bytes), or None when unknown."""
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) * 1024
    except OSError:
        pass
    return None
