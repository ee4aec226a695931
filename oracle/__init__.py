"""CPU oracle for the routed-MoE expert-slot-cache layer (ctypes wrapper of oracle.c).

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the bench's CPU-baseline
and reference legs use it; the product path (``router_softmax_top_gb300``) never
imports it, and the two share no code.  All arithmetic is in oracle.c, in double.
Every function below is a thin marshalling layer.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_SO = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

NSTAT = 10
STAT_NAMES = ("calls", "pick_hits", "pick_misses", "unique_hits", "unique_misses",
              "evictions", "bytes_uploaded", "stages", "staged_calls", "bypassed")

POLICY_LRU = 0
POLICY_SCORE = 1
POLICY_ADOPT = 2   # LRU; a call of more than one stage ends holding its most-used experts


class PlanInfo(ctypes.Structure):
    _fields_ = [("n_unique", ctypes.c_int32), ("n_hits", ctypes.c_int32),
                ("n_miss", ctypes.c_int32), ("n_stages", ctypes.c_int32),
                ("n_evict", ctypes.c_int32), ("pick_hits", ctypes.c_int32),
                ("pick_misses", ctypes.c_int32), ("n_bypass", ctypes.c_int32)]

    def as_dict(self):
        return {f: int(getattr(self, f)) for f, _ in self._fields_}


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (gcc, OpenMP over independent pairs only)."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-shared", "-fPIC",
                        "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _SO)
    return _SO


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_SO)
            vp, i32, u64, dbl = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64, ctypes.c_double
            L.orc_fp16_to_double.restype = dbl
            L.orc_fp16_to_double.argtypes = [ctypes.c_uint16]
            L.orc_bf16_to_double.restype = dbl
            L.orc_bf16_to_double.argtypes = [ctypes.c_uint16]
            L.orc_q4_0_decode.argtypes = [vp, vp]
            L.orc_router.restype = i32
            L.orc_router.argtypes = [vp, i32, i32, i32, i32, vp, vp]
            L.orc_lru_new.restype = vp
            L.orc_lru_new.argtypes = [i32, i32]
            L.orc_lru_free.argtypes = [vp]
            L.orc_lru_get.argtypes = [vp, vp, vp, vp, vp]
            L.orc_lru_set_policy.argtypes = [vp, i32, i32]
            L.orc_lru_set_sticky.argtypes = [vp, i32]
            L.orc_cache_set_sticky.argtypes = [vp, i32]
            L.orc_lru_scores.argtypes = [vp, vp]
            L.orc_slot_map.restype = i32
            L.orc_slot_map.argtypes = [vp, vp, i32, i32, vp, vp, vp, vp, vp, vp, ctypes.POINTER(PlanInfo)]
            L.orc_expert_ffn_parts.argtypes = [vp, i32, i32, vp, vp, vp, vp, vp]
            L.orc_expert_ffn.argtypes = [vp, i32, i32, vp, vp]
            L.orc_cache_new.restype = vp
            L.orc_cache_new.argtypes = [i32, i32, i32, i32, i32, i32, i32, vp, u64, u64, i32, i32, i32]
            L.orc_cache_free.argtypes = [vp]
            L.orc_cache_lru.restype = vp
            L.orc_cache_lru.argtypes = [vp, i32]
            L.orc_cache_stats.argtypes = [vp, i32, vp]
            L.orc_cache_preload.argtypes = [vp, vp]
            L.orc_cache_usage.argtypes = [vp, vp]
            L.orc_cache_set_state.restype = i32
            L.orc_cache_set_state.argtypes = [vp, i32, vp, vp, u64, vp, vp]
            L.orc_layer_forward.restype = i32
            L.orc_layer_forward.argtypes = [vp, i32, vp, vp, i32, i32, i32, vp,
                                            vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                            ctypes.POINTER(PlanInfo)]
            L.orc_max_threads.restype = i32
            _lib = L
    return _lib


def _p(a):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "arrays passed to the oracle must be C-contiguous"
    return ctypes.c_void_p(a.ctypes.data)


# ------------------------------------------------------------------ formats
def fp16_to_double(h: int) -> float:
    return float(lib().orc_fp16_to_double(h))


def bf16_to_double(b: int) -> float:
    return float(lib().orc_bf16_to_double(b))


def q4_0_decode(block: bytes | np.ndarray) -> np.ndarray:
    blk = np.frombuffer(bytes(block), dtype=np.uint8).copy()
    assert blk.size == 18
    out = np.empty(32, dtype=np.float64)
    lib().orc_q4_0_decode(_p(blk), _p(out))
    return out


# ------------------------------------------------------------------- router
def router(logits: np.ndarray, k: int, weight_mode: int = 0):
    """Returns (ids int32 [T,k], w float64 [T,k]); raises ValueError on a non-finite logit."""
    lg = np.ascontiguousarray(logits, dtype=np.float32)
    T, E = lg.shape
    ids = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float64)
    if lib().orc_router(_p(lg), T, E, k, weight_mode, _p(ids), _p(w)) != 0:
        raise ValueError("non-finite router logit")
    return ids, w


# ---------------------------------------------------------------------- LRU
class LRU:
    """One layer's slot-map state (S slots, E experts)."""

    def __init__(self, S: int, E: int, policy: int = POLICY_LRU, budget: int = 0, sticky: int = 0):
        self.S, self.E = S, E
        self._h = lib().orc_lru_new(S, E)
        self._own = True
        if policy != POLICY_LRU:
            lib().orc_lru_set_policy(self._h, policy, budget)
        if sticky:
            lib().orc_lru_set_sticky(self._h, sticky)

    @classmethod
    def _borrow(cls, handle, S, E):
        o = cls.__new__(cls)
        o.S, o.E, o._h, o._own = S, E, handle, False
        return o

    def __del__(self):
        if getattr(self, "_own", False) and self._h:
            lib().orc_lru_free(self._h)
            self._h = None

    def plan(self, ids: np.ndarray) -> dict:
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        T, k = ids.shape
        P = T * k
        m = min(self.E, P)
        gs = np.empty(P, np.int32); stg = np.empty(P, np.int32)
        me = np.empty(m, np.int32); ms = np.empty(m, np.int32)
        mv = np.empty(m, np.int32); mst = np.empty(m, np.int32)
        info = PlanInfo()
        if lib().orc_slot_map(self._h, _p(ids), T, k, _p(gs), _p(stg), _p(me), _p(ms), _p(mv),
                              _p(mst), ctypes.byref(info)) != 0:
            raise ValueError("the score policy plans single-stage calls only")
        n = info.n_miss
        return {"gpu_slot": gs.reshape(T, k), "stage": stg.reshape(T, k),
                "miss_expert": me[:n].copy(), "miss_slot": ms[:n].copy(),
                "miss_evicted": mv[:n].copy(), "miss_stage": mst[:n].copy(),
                "info": info.as_dict()}

    def state(self) -> dict:
        se = np.empty(self.S, np.int32); es = np.empty(self.E, np.int32)
        ss = np.empty(self.S, np.uint64); clk = ctypes.c_uint64(0)
        lib().orc_lru_get(self._h, _p(se), _p(es), _p(ss), ctypes.byref(clk))
        return {"slot_expert": se, "expert_slot": es, "slot_stamp": ss, "clock": int(clk.value)}

    def scores(self) -> np.ndarray:
        """The decayed usage scores [E] (policy 1, fp32)."""
        out = np.empty(self.E, np.float32)
        lib().orc_lru_scores(self._h, _p(out))
        return out


# ---------------------------------------------------------------------- FFN
def expert_ffn(block: np.ndarray, H: int, F: int, x: np.ndarray, parts: bool = False):
    blk = np.ascontiguousarray(block, dtype=np.uint8)
    assert blk.size == 3 * F * H // 32 * 18
    xd = np.ascontiguousarray(x, dtype=np.float64)
    y = np.empty(H, np.float64)
    if not parts:
        lib().orc_expert_ffn(_p(blk), H, F, _p(xd), _p(y))
        return y
    g = np.empty(F, np.float64); u = np.empty(F, np.float64); h = np.empty(F, np.float64)
    lib().orc_expert_ffn_parts(_p(blk), H, F, _p(xd), _p(g), _p(u), _p(h), _p(y))
    return {"g": g, "u": u, "h": h, "y": y}


# -------------------------------------------------------------------- layer
class Cache:
    """Whole-model oracle: per-layer LRU state, simulated slots, stats.

    ``store`` is a uint8 array (or an integer host address plus ``nbytes``) of
    canonical Q4_0 expert blocks, [layer][expert] with the given strides."""

    def __init__(self, L, E, k, H, F, S, store, weight_mode=0, layer_stride=None,
                 expert_stride=None, threads=0, policy=POLICY_LRU, admit_budget=0, sticky=0):
        self.L, self.E, self.k, self.H, self.F, self.S = L, E, k, H, F, S
        eb = 3 * F * H // 32 * 18
        self.expert_stride = eb if expert_stride is None else expert_stride
        self.layer_stride = E * self.expert_stride if layer_stride is None else layer_stride
        if isinstance(store, np.ndarray):
            self._store_ref = store
            addr = store.ctypes.data
        else:
            self._store_ref = None
            addr = int(store)
        self._h = lib().orc_cache_new(L, E, k, H, F, S, weight_mode, ctypes.c_void_p(addr),
                                      self.layer_stride, self.expert_stride, threads, policy,
                                      admit_budget)
        if sticky:
            lib().orc_cache_set_sticky(self._h, sticky)

    def __del__(self):
        if getattr(self, "_h", None):
            lib().orc_cache_free(self._h)
            self._h = None

    def lru(self, layer: int) -> LRU:
        return LRU._borrow(lib().orc_cache_lru(self._h, layer), self.S, self.E)

    def preload(self, counts: np.ndarray):
        """Warm start: per layer the S most-used experts (counts [L, E]) in slots 0, 1, ..."""
        c = np.ascontiguousarray(counts, dtype=np.uint32)
        assert c.shape == (self.L, self.E)
        lib().orc_cache_preload(self._h, _p(c))

    def usage(self) -> np.ndarray:
        """Lifetime activation counts [L, E] (u32): one per routed (token, pick) of every accepted call."""
        out = np.empty((self.L, self.E), np.uint32)
        lib().orc_cache_usage(self._h, _p(out))
        return out

    def state(self, layer: int) -> dict:
        """One layer's resumable state: slot_expert, slot_stamp, clock, score (fp32), usage (u32)."""
        st = self.lru(layer).state()
        return {"slot_expert": st["slot_expert"], "slot_stamp": st["slot_stamp"], "clock": st["clock"],
                "score": self.lru(layer).scores(), "usage": self.usage()[layer].copy()}

    def set_state(self, layer: int, slot_expert, slot_stamp, clock: int, score, usage) -> bool:
        """Resume one layer from a saved state; False (state untouched) when the tables are invalid."""
        se = np.ascontiguousarray(slot_expert, dtype=np.int32)
        ss = np.ascontiguousarray(slot_stamp, dtype=np.uint64)
        sc = np.ascontiguousarray(score, dtype=np.float32)
        us = np.ascontiguousarray(usage, dtype=np.uint32)
        assert se.shape == (self.S,) and ss.shape == (self.S,) and sc.shape == (self.E,) and us.shape == (self.E,)
        return lib().orc_cache_set_state(self._h, layer, _p(se), _p(ss), int(clock), _p(sc), _p(us)) == 0

    def forward(self, layer: int, logits: np.ndarray, x: np.ndarray | None, compute: bool = True):
        lg = np.ascontiguousarray(logits, dtype=np.float32)
        T = lg.shape[0]
        k, H = self.k, self.H
        P = T * k
        m = max(1, min(self.E, P))
        out = np.zeros((T, H), np.float32)
        ids = np.empty(P, np.int32); w = np.empty(P, np.float64)
        gs = np.empty(P, np.int32); stg = np.empty(P, np.int32)
        me = np.empty(m, np.int32); ms = np.empty(m, np.int32)
        mv = np.empty(m, np.int32); mst = np.empty(m, np.int32)
        visits = np.empty(P, np.int32)
        info = PlanInfo()
        if x is None:
            xa, is_bf16 = np.zeros((T, H), np.float32), 0
        else:
            xa = np.ascontiguousarray(x)
            is_bf16 = 1 if xa.dtype == np.uint16 else 0
            if not is_bf16:
                xa = np.ascontiguousarray(xa, dtype=np.float32)
        rc = lib().orc_layer_forward(self._h, layer, _p(lg), _p(xa), is_bf16, T, int(bool(compute)),
                                     _p(out), _p(ids), _p(w), _p(gs), _p(stg), _p(me), _p(ms),
                                     _p(mv), _p(mst), _p(visits), ctypes.byref(info))
        if rc == -2:
            raise ValueError("the score policy plans single-stage calls only")
        if rc != 0:
            raise ValueError("non-finite router logit")
        n = info.n_miss
        return {"out": out if compute else None, "ids": ids.reshape(T, k), "w": w.reshape(T, k),
                "gpu_slot": gs.reshape(T, k), "stage": stg.reshape(T, k),
                "miss_expert": me[:n].copy(), "miss_slot": ms[:n].copy(),
                "miss_evicted": mv[:n].copy(), "miss_stage": mst[:n].copy(),
                "visits": visits.reshape(T, k), "info": info.as_dict()}

    def stats(self, layer: int) -> dict:
        """Counters of one layer (0 <= layer < L)."""
        if not 0 <= layer < self.L:
            raise IndexError(f"layer {layer} out of range [0, {self.L})")
        out = np.empty(NSTAT, np.uint64)
        lib().orc_cache_stats(self._h, layer, _p(out))
        return dict(zip(STAT_NAMES, (int(v) for v in out)))


def max_threads() -> int:
    return int(lib().orc_max_threads())
