"""Routed-MoE layer over a GPU-resident expert-slot cache (GB300, sm_103a).

Thin ctypes binding of ``libmoe_cache.so``: argument marshalling only, every
step of the layer runs in the library's CUDA kernels.  The functions keep the C
names (``moe_cache_init``, ``moe_layer_forward``, ``moe_cache_stats``, ...);
``MoECache`` wraps them for PyTorch tensors (device memory and streams).

There is no fallback: if the compiled library is missing, loading fails with an
error telling how to build it.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe_cache.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_CUDA = 2
MOE_ERR_OOM = 3
MOE_ERR_TIMEOUT = 4
MOE_ERR_HOST_STORE = 5
MOE_ERR_POISONED = 6
MOE_ERR_UNSUPPORTED = 7
MOE_ERR_CHECK = 8

MOE_FILL_MEMCPY = 0
MOE_FILL_PULL = 1

MOE_INJECT_DECODE_WAIT = 1
MOE_INJECT_MEMCPY_FAIL = 2

MOE_POLICY_LRU = 0
MOE_POLICY_SCORE = 1
MOE_POLICY_ADOPT = 2

# every symbol include/moe_cache.h declares
EXPORTS = ("moe_cache_init", "moe_layer_forward", "moe_cache_sync", "moe_cache_stats",
           "moe_layer_last_plan", "moe_cache_preload", "moe_cache_inject", "moe_cache_set_timing",
           "moe_cache_timing",
           "moe_cache_probe_h2d", "moe_expert_bytes", "moe_cache_launch_count",
           "moe_cache_destroy", "moe_strerror", "moe_expert_ffn_static", "moe_cache_usage",
           "moe_cache_state_size", "moe_cache_save_state", "moe_cache_load_state")

MOE_STATE_MAGIC = 0x53454F4D
MOE_STATE_VERSION = 1


class MoeCacheConfig(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int32), ("n_experts", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("hidden", ctypes.c_int32), ("ffn", ctypes.c_int32),
                ("slots_per_layer", ctypes.c_int32), ("max_tokens", ctypes.c_int32),
                ("weight_mode", ctypes.c_int32), ("act_dtype", ctypes.c_int32),
                ("fill_mode", ctypes.c_int32), ("gemm_min_tokens", ctypes.c_int32),
                ("policy", ctypes.c_int32), ("admit_budget", ctypes.c_int32),
                ("sticky_permille", ctypes.c_int32), ("timeout_us", ctypes.c_int64)]


class MoeHostStore(ctypes.Structure):
    _fields_ = [("base", ctypes.c_void_p), ("bytes", ctypes.c_uint64),
                ("layer_stride", ctypes.c_uint64), ("expert_stride", ctypes.c_uint64)]


class MoeCacheStats(ctypes.Structure):
    _fields_ = [("calls", ctypes.c_uint64), ("pick_hits", ctypes.c_uint64),
                ("pick_misses", ctypes.c_uint64), ("unique_hits", ctypes.c_uint64),
                ("unique_misses", ctypes.c_uint64), ("evictions", ctypes.c_uint64),
                ("bytes_uploaded", ctypes.c_uint64), ("stages", ctypes.c_uint64),
                ("staged_calls", ctypes.c_uint64), ("bypassed", ctypes.c_uint64),
                ("poisoned", ctypes.c_int32),
                ("last_error", ctypes.c_int32), ("cuda_error", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]

    def as_dict(self):
        return {f: int(getattr(self, f)) for f, _ in self._fields_}


class MoeStateHeader(ctypes.Structure):
    """moe_cache_state_header: the first 48 bytes of a saved state."""
    _fields_ = [("magic", ctypes.c_uint32), ("version", ctypes.c_uint32), ("n_layers", ctypes.c_int32),
                ("n_experts", ctypes.c_int32), ("slots_per_layer", ctypes.c_int32), ("policy", ctypes.c_int32),
                ("expert_bytes", ctypes.c_uint64), ("total_bytes", ctypes.c_uint64),
                ("reserved", ctypes.c_uint64)]


class MoeError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {strerror(code)} ({code})")


_lib = None


def lib() -> ctypes.CDLL:
    """Load the compiled library (no fallback)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               f"`python -m router_softmax_top_gb300.build` (nvcc, sm_103a)")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, u64, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_uint64, ctypes.c_int64
        L.moe_cache_init.restype = ctypes.c_int
        L.moe_cache_init.argtypes = [ctypes.POINTER(MoeCacheConfig), ctypes.POINTER(MoeHostStore),
                                     vp, ctypes.POINTER(vp)]
        L.moe_layer_forward.restype = ctypes.c_int
        L.moe_layer_forward.argtypes = [vp, i32, vp, vp, i32, vp, vp]
        L.moe_cache_sync.restype = ctypes.c_int
        L.moe_cache_sync.argtypes = [vp, vp]
        L.moe_cache_stats.restype = ctypes.c_int
        L.moe_cache_stats.argtypes = [vp, i32, ctypes.POINTER(MoeCacheStats)]
        L.moe_layer_last_plan.restype = ctypes.c_int
        L.moe_layer_last_plan.argtypes = [vp, i32] + [vp] * 10
        L.moe_cache_set_timing.restype = ctypes.c_int
        L.moe_cache_set_timing.argtypes = [vp, i32]
        L.moe_cache_timing.restype = ctypes.c_int
        L.moe_cache_timing.argtypes = [vp, ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(u64),
                                       ctypes.POINTER(ctypes.c_double), i32, ctypes.POINTER(i32)]
        L.moe_cache_preload.restype = ctypes.c_int
        L.moe_cache_preload.argtypes = [vp, vp, vp]
        L.moe_cache_inject.restype = ctypes.c_int
        L.moe_cache_inject.argtypes = [vp, i32]
        L.moe_cache_usage.argtypes = [vp, vp]
        L.moe_cache_state_size.argtypes = [vp, ctypes.POINTER(u64)]
        L.moe_cache_save_state.argtypes = [vp, vp, u64]
        L.moe_cache_load_state.argtypes = [vp, vp, u64, vp]
        L.moe_cache_probe_h2d.restype = ctypes.c_int
        L.moe_cache_probe_h2d.argtypes = [vp, i32, ctypes.POINTER(ctypes.c_double)]
        L.moe_expert_bytes.restype = u64
        L.moe_expert_bytes.argtypes = [i32, i32]
        L.moe_cache_launch_count.restype = u64
        L.moe_cache_launch_count.argtypes = [vp]
        L.moe_cache_destroy.restype = None
        L.moe_cache_destroy.argtypes = [vp]
        L.moe_strerror.restype = ctypes.c_char_p
        L.moe_strerror.argtypes = [ctypes.c_int]
        L.moe_expert_ffn_static.restype = ctypes.c_int
        L.moe_expert_ffn_static.argtypes = [vp, i32, i32, vp, i32, vp, vp]
        _lib = L
    return _lib


def strerror(code: int) -> str:
    return lib().moe_strerror(code).decode()


def _check(rc: int, where: str):
    if rc != MOE_OK:
        raise MoeError(rc, where)


def _stream_handle(stream):
    if stream is None:
        import torch
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


# ------------------------------------------------- C names, marshalling only
def moe_expert_bytes(hidden: int, ffn: int) -> int:
    return int(lib().moe_expert_bytes(hidden, ffn))


def moe_cache_init(cfg: MoeCacheConfig, store: MoeHostStore, stream=None) -> ctypes.c_void_p:
    h = ctypes.c_void_p()
    _check(lib().moe_cache_init(ctypes.byref(cfg), ctypes.byref(store), _stream_handle(stream),
                                ctypes.byref(h)), "moe_cache_init")
    return h


def moe_layer_forward(handle, layer: int, d_logits: int, d_x: int, n_tokens: int, d_out: int,
                      stream=None) -> int:
    return int(lib().moe_layer_forward(handle, layer, ctypes.c_void_p(d_logits), ctypes.c_void_p(d_x),
                                       n_tokens, ctypes.c_void_p(d_out), _stream_handle(stream)))


def moe_cache_sync(handle, stream=None) -> int:
    return int(lib().moe_cache_sync(handle, _stream_handle(stream)))


def moe_cache_stats(handle, layer: int = -1) -> dict:
    s = MoeCacheStats()
    _check(lib().moe_cache_stats(handle, layer, ctypes.byref(s)), "moe_cache_stats")
    return s.as_dict()


def moe_cache_destroy(handle) -> None:
    lib().moe_cache_destroy(handle)


def moe_expert_ffn_static(d_expert_block: int, hidden: int, ffn: int, d_x: int, n_tokens: int,
                          d_y: int, stream=None) -> int:
    """One expert's FFN on up to 8 tokens with no allocation (for callers that cannot
    allocate, e.g. during graph capture); returns the status code."""
    return int(lib().moe_expert_ffn_static(ctypes.c_void_p(d_expert_block), hidden, ffn,
                                           ctypes.c_void_p(d_x), n_tokens, ctypes.c_void_p(d_y),
                                           _stream_handle(stream)))


# ------------------------------------------------------- tensor-level API
class MoECache:
    """One cache over a host store, for PyTorch tensors.

    store: a CPU uint8 tensor or a (host address, nbytes) pair, holding
    canonical Q4_0 expert blocks [layer][expert] (block = gate | up | down).
    Ordinary memory is pinned and mapped by the library (cudaHostRegister) for
    the lifetime of the cache; already pinned memory is used as it is.  On a
    Grace host, ordinary (e.g. mmap'd) memory registered this way reads over
    the host link faster and more steadily than a cudaHostAlloc buffer."""

    def __init__(self, *, n_layers, n_experts, top_k, hidden, ffn, slots_per_layer, max_tokens,
                 store, weight_mode=0, act_dtype="f32", fill_mode=MOE_FILL_MEMCPY,
                 gemm_min_tokens=0, timeout_us=10_000_000, layer_stride=None,
                 expert_stride=None, stream=None, policy=MOE_POLICY_LRU, admit_budget=0,
                 sticky_permille=0):
        self.cfg = MoeCacheConfig(n_layers=n_layers, n_experts=n_experts, top_k=top_k, hidden=hidden,
                                  ffn=ffn, slots_per_layer=slots_per_layer, max_tokens=max_tokens,
                                  weight_mode=weight_mode, act_dtype=1 if act_dtype == "bf16" else 0,
                                  fill_mode=fill_mode, gemm_min_tokens=gemm_min_tokens, policy=policy,
                                  admit_budget=admit_budget, sticky_permille=sticky_permille, timeout_us=timeout_us)
        eb = moe_expert_bytes(hidden, ffn)
        self.expert_bytes = eb
        if isinstance(store, tuple):
            addr, nbytes = store
            self._store_ref = None
        else:
            addr, nbytes = store.data_ptr(), store.numel() * store.element_size()
            self._store_ref = store
        es = eb if expert_stride is None else expert_stride
        ls = n_experts * es if layer_stride is None else layer_stride
        self.store = MoeHostStore(addr, nbytes, ls, es)
        self.handle = moe_cache_init(self.cfg, self.store, stream)
        self.L, self.k, self.E, self.H, self.F = n_layers, top_k, n_experts, hidden, ffn

    def close(self):
        if getattr(self, "handle", None):
            moe_cache_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def forward(self, layer: int, logits, x, out=None, stream=None):
        """logits: cuda fp32 [T, E]; x: cuda [T, H] (fp32 or bf16); returns out fp32 [T, H]."""
        import torch
        T = logits.shape[0]
        assert logits.is_cuda and logits.dtype == torch.float32 and logits.is_contiguous()
        assert x.is_cuda and x.is_contiguous() and x.shape[0] == T
        if out is None:
            out = torch.empty((T, self.H), dtype=torch.float32, device=logits.device)
        rc = moe_layer_forward(self.handle, layer, logits.data_ptr(), x.data_ptr(), T,
                               out.data_ptr(), stream)
        _check(rc, "moe_layer_forward")
        return out

    def forward_rc(self, layer: int, logits, x, out, stream=None) -> int:
        """Same as forward but returns the status code instead of raising."""
        return moe_layer_forward(self.handle, layer, logits.data_ptr(), x.data_ptr(),
                                 logits.shape[0], out.data_ptr(), stream)

    def sync(self, stream=None) -> int:
        return moe_cache_sync(self.handle, stream)

    def stats(self, layer: int = -1) -> dict:
        return moe_cache_stats(self.handle, layer)

    def last_plan(self, layer: int, n_tokens: int) -> dict:
        import numpy as np
        P = n_tokens * self.k
        m = max(1, min(self.E, P))
        ids = np.empty(P, np.int32); w = np.empty(P, np.float32)
        gs = np.empty(P, np.int32); stg = np.empty(P, np.int32)
        me = np.empty(m, np.int32); ms = np.empty(m, np.int32)
        mv = np.empty(m, np.int32); mst = np.empty(m, np.int32)
        nm = ctypes.c_int32(); ns = ctypes.c_int32()
        p = lambda a: ctypes.c_void_p(a.ctypes.data)
        _check(lib().moe_layer_last_plan(self.handle, layer, p(ids), p(w), p(gs), p(stg), p(me),
                                         p(ms), p(mv), p(mst), ctypes.byref(nm), ctypes.byref(ns)),
               "moe_layer_last_plan")
        n = nm.value
        return {"ids": ids.reshape(n_tokens, self.k), "w": w.reshape(n_tokens, self.k),
                "gpu_slot": gs.reshape(n_tokens, self.k), "stage": stg.reshape(n_tokens, self.k),
                "miss_expert": me[:n].copy(), "miss_slot": ms[:n].copy(),
                "miss_evicted": mv[:n].copy(), "miss_stage": mst[:n].copy(), "n_stages": ns.value}

    def preload(self, counts, stream=None):
        """Warm start: per layer the most-used experts of counts [L, E] (moe_cache_preload)."""
        import numpy as np
        c = np.ascontiguousarray(counts, dtype=np.uint32)
        if c.shape != (self.L, self.E):
            raise ValueError(f"counts must be [{self.L}, {self.E}]")
        if stream is None:
            import torch
            stream = torch.cuda.current_stream().cuda_stream
        _check(lib().moe_cache_preload(self.handle, ctypes.c_void_p(c.ctypes.data), ctypes.c_void_p(stream)),
               "moe_cache_preload")

    def usage(self):
        """Lifetime activation counts [L, E] u32 (moe_cache_usage)."""
        import numpy as np
        out = np.empty((self.L, self.E), np.uint32)
        _check(lib().moe_cache_usage(self.handle, ctypes.c_void_p(out.ctypes.data)), "moe_cache_usage")
        return out

    def save_state(self) -> bytes:
        """The handle's slot tables, stamps, clocks, scores and usage (moe_cache_save_state)."""
        n = ctypes.c_uint64(0)
        _check(lib().moe_cache_state_size(self.handle, ctypes.byref(n)), "moe_cache_state_size")
        buf = ctypes.create_string_buffer(n.value)
        _check(lib().moe_cache_save_state(self.handle, buf, n.value), "moe_cache_save_state")
        return buf.raw

    def load_state_rc(self, state: bytes, stream=None) -> int:
        """moe_cache_load_state; returns its code."""
        if stream is None:
            import torch
            stream = torch.cuda.current_stream().cuda_stream
        buf = ctypes.create_string_buffer(bytes(state), len(state))
        return lib().moe_cache_load_state(self.handle, buf, len(state), ctypes.c_void_p(stream))

    def load_state(self, state: bytes, stream=None):
        """Resume a saved state (moe_cache_load_state)."""
        _check(self.load_state_rc(state, stream), "moe_cache_load_state")

    def inject(self, what: int):
        """Test hook: fault injection without a GPU fault (moe_cache_inject)."""
        _check(lib().moe_cache_inject(self.handle, what), "moe_cache_inject")

    def set_timing(self, enable: bool):
        _check(lib().moe_cache_set_timing(self.handle, 1 if enable else 0), "moe_cache_set_timing")

    def timing(self) -> dict:
        cap = 16
        names = (ctypes.c_char_p * cap)()
        launches = (ctypes.c_uint64 * cap)()
        ms = (ctypes.c_double * cap)()
        n = ctypes.c_int32()
        _check(lib().moe_cache_timing(self.handle, names, launches, ms, cap, ctypes.byref(n)),
               "moe_cache_timing")
        return {names[i].decode(): {"launches": int(launches[i]), "ms": float(ms[i])}
                for i in range(min(cap, n.value))}

    def probe_h2d(self, iters: int = 20) -> float:
        g = ctypes.c_double()
        _check(lib().moe_cache_probe_h2d(self.handle, iters, ctypes.byref(g)), "moe_cache_probe_h2d")
        return float(g.value)

    def launch_count(self) -> int:
        return int(lib().moe_cache_launch_count(self.handle))
