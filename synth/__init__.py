"""Seeded synthetic inputs shared by the CPU oracle tests and the CUDA path.

This package only generates inputs (random Q4_0 expert stores, routing traces,
router logits, activations) and describes the workloads' shapes.  It contains
none of the routed-MoE method's arithmetic and imports neither the oracle nor
the CUDA library.  The generator itself is ``synth.c`` (SplitMix64-seeded PCG32
streams, Box-Muller normals, inverse-CDF Zipf), compiled on first use.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_SO = os.path.join(_HERE, "libsynth.so")
_lock = threading.Lock()
_lib = None

PURPOSE_X = 5
PURPOSE_IID_LOGITS = 6


def build(force: bool = False) -> str:
    """Compile synth.c into libsynth.so next to it (gcc, OpenMP)."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.run(
            ["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-shared", "-fPIC",
             "-o", tmp, _SRC, "-lm"],
            check=True,
        )
        os.replace(tmp, _SO)
    return _SO


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_SO)
            u64, i32, vp, dbl = ctypes.c_uint64, ctypes.c_int, ctypes.c_void_p, ctypes.c_double
            L.synth_expert_bytes.restype = u64
            L.synth_expert_bytes.argtypes = [i32, i32]
            L.synth_fill_expert.argtypes = [vp, i32, i32, i32, i32, u64]
            L.synth_fill_store.argtypes = [vp, i32, i32, i32, i32, u64, i32]
            L.synth_permutation.argtypes = [vp, i32, u64, i32]
            L.synth_trace.argtypes = [vp, i32, i32, i32, dbl, dbl, u64, i32, i32]
            L.synth_logits_from_picks.argtypes = [vp, vp, i32, i32, i32, u64, i32, i32, u64]
            L.synth_normal_f32.argtypes = [vp, u64, u64, u64, u64, u64]
            L.synth_normal_bf16.argtypes = [vp, u64, u64, u64, u64, u64]
            L.synth_pcg32_raw.argtypes = [vp, i32, u64, u64]
            L.synth_splitmix64_raw.argtypes = [vp, i32, u64]
            L.synth_fp16_rne.restype = ctypes.c_uint16
            L.synth_fp16_rne.argtypes = [dbl]
            L.synth_bf16_rne.restype = ctypes.c_uint16
            L.synth_bf16_rne.argtypes = [ctypes.c_float]
            _lib = L
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


# ---------------------------------------------------------------- primitives
def expert_bytes(H: int, F: int) -> int:
    """Bytes of one expert block: gate, up (F x H) and down (H x F) at 18 B per 32 values."""
    return int(lib().synth_expert_bytes(H, F))


def fill_store(dst_addr: int, L: int, E: int, H: int, F: int, seed: int = 0, threads: int = 0) -> None:
    """Write the whole [layer][expert] store at host address ``dst_addr``."""
    lib().synth_fill_store(ctypes.c_void_p(dst_addr), L, E, H, F, seed, threads)


def store(L: int, E: int, H: int, F: int, seed: int = 0, threads: int = 0) -> np.ndarray:
    buf = np.empty(L * E * expert_bytes(H, F), dtype=np.uint8)
    fill_store(_ptr(buf), L, E, H, F, seed, threads)
    return buf


def expert_block(layer: int, expert: int, H: int, F: int, seed: int = 0) -> np.ndarray:
    buf = np.empty(expert_bytes(H, F), dtype=np.uint8)
    lib().synth_fill_expert(_ptr(buf), layer, expert, H, F, seed)
    return buf


def permutation(E: int, seed: int, layer: int) -> np.ndarray:
    out = np.empty(E, dtype=np.int32)
    lib().synth_permutation(_ptr(out), E, seed, layer)
    return out


def trace(n_tok: int, E: int, k: int, zipf_s: float, p_sticky: float,
          seed: int = 0, layer: int = 0, stream: int = 0) -> np.ndarray:
    picks = np.empty((n_tok, k), dtype=np.int32)
    lib().synth_trace(_ptr(picks), n_tok, E, k, float(zipf_s), float(p_sticky), seed, layer, stream)
    return picks


def logits_from_picks(picks: np.ndarray, E: int, seed: int = 0, layer: int = 0,
                      stream: int = 0, key: int = 0) -> np.ndarray:
    picks = np.ascontiguousarray(picks, dtype=np.int32)
    n_tok, k = picks.shape
    out = np.empty((n_tok, E), dtype=np.float32)
    lib().synth_logits_from_picks(_ptr(out), _ptr(picks), n_tok, E, k, seed, layer, stream, key)
    return out


def normal_f32(n: int, seed: int, purpose: int, a: int = 0, b: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.float32)
    lib().synth_normal_f32(_ptr(out), n, seed, purpose, a, b)
    return out


def normal_bf16_bits(n: int, seed: int, purpose: int, a: int = 0, b: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.uint16)
    lib().synth_normal_bf16(_ptr(out), n, seed, purpose, a, b)
    return out


def pcg32_raw(n: int, initstate: int, initseq: int) -> np.ndarray:
    out = np.empty(n, dtype=np.uint32)
    lib().synth_pcg32_raw(_ptr(out), n, initstate, initseq)
    return out


def splitmix64_raw(n: int, seed: int) -> np.ndarray:
    out = np.empty(n, dtype=np.uint64)
    lib().synth_splitmix64_raw(_ptr(out), n, seed)
    return out


# ---------------------------------------------------------------- workloads
@dataclass(frozen=True)
class Shape:
    """Model shape of one workload: L layers, E experts, top-k, hidden H, FFN F, S slots."""
    name: str
    L: int
    E: int
    k: int
    H: int
    F: int
    S: int
    act: str = "f32"        # activation dtype: "f32" or "bf16"
    zipf: float = 0.0       # 0 = i.i.d. N(0,1) logits (no trace)
    sticky: float = 0.0
    extra: dict = field(default_factory=dict)

    @property
    def expert_bytes(self) -> int:
        return 3 * self.F * self.H // 32 * 18

    @property
    def store_bytes(self) -> int:
        return self.L * self.E * self.expert_bytes


TINY = Shape("tiny", L=1, E=8, k=2, H=256, F=512, S=4, act="f32")
DECODE = Shape("decode", L=30, E=128, k=8, H=2816, F=704, S=32, act="f32", zipf=1.1, sticky=0.39,
               extra={"steps": 512, "T": 1})
PREFILL = Shape("prefill", L=30, E=128, k=8, H=2816, F=704, S=32, act="bf16", zipf=1.1, sticky=0.39,
                extra={"batches": 4, "T": 512})
LARGE = Shape("large", L=48, E=256, k=8, H=4096, F=1536, S=64, act="f32", zipf=1.0, sticky=0.30,
              extra={"steps": 256, "T": (1, 8)})
SWEEP = Shape("sweep", L=1, E=128, k=8, H=2816, F=704, S=32, act="f32", zipf=1.2, sticky=0.0,
              extra={"batches": 16, "T": 64, "budgets": (8, 16, 32, 64, 128)})

SHAPES = {s.name: s for s in (TINY, DECODE, PREFILL, LARGE, SWEEP)}


def tiny_inputs(seed: int = 0):
    """Tiny workload: 4 tokens, logits i.i.d. N(0,1) [4, 8], x N(0,1) [4, 256] fp32."""
    T = 4
    logits = normal_f32(T * TINY.E, seed, PURPOSE_IID_LOGITS, 0, 0).reshape(T, TINY.E)
    x = normal_f32(T * TINY.H, seed, PURPOSE_X, 0, 0).reshape(T, TINY.H)
    return logits, x


def decode_inputs(shape: Shape, steps: int, batch: int = 1, seed: int = 0, layers=None,
                  p_override=None, zipf_override=None):
    """Decode workload: ``batch`` independent token streams, each sticky to its own
    previous step.  Returns (picks [steps, L, B, k], logits [steps, L, B, E], x [steps, L, B, H])."""
    layers = range(shape.L) if layers is None else layers
    nl = len(layers)
    zs = shape.zipf if zipf_override is None else zipf_override
    ps = shape.sticky if p_override is None else p_override
    picks = np.empty((steps, nl, batch, shape.k), dtype=np.int32)
    logits = np.empty((steps, nl, batch, shape.E), dtype=np.float32)
    x = np.empty((steps, nl, batch, shape.H), dtype=np.float32)
    for li, l in enumerate(layers):
        for b in range(batch):
            p = trace(steps, shape.E, shape.k, zs, ps, seed, l, b)
            picks[:, li, b] = p
            logits[:, li, b] = logits_from_picks(p, shape.E, seed, l, b, 0)
        x[:, li] = normal_f32(steps * batch * shape.H, seed, PURPOSE_X, l, 1000 + batch).reshape(
            steps, batch, shape.H)
    return picks, logits, x


def batch_inputs(shape: Shape, n_batches: int, T: int, seed: int = 0, layers=None,
                 zipf=None, sticky=None, act=None):
    """Batched (prefill-like) workload: per layer and batch, a T-token sticky trace
    (stickiness within the batch).  x is fp32, or bf16 raw bits when act == 'bf16'.
    Returns (picks [n_batches, L, T, k], logits [n_batches, L, T, E], x [n_batches, L, T, H])."""
    layers = range(shape.L) if layers is None else layers
    nl = len(layers)
    zs = shape.zipf if zipf is None else zipf
    ps = shape.sticky if sticky is None else sticky
    act = shape.act if act is None else act
    picks = np.empty((n_batches, nl, T, shape.k), dtype=np.int32)
    logits = np.empty((n_batches, nl, T, shape.E), dtype=np.float32)
    xdt = np.uint16 if act == "bf16" else np.float32
    x = np.empty((n_batches, nl, T, shape.H), dtype=xdt)
    for li, l in enumerate(layers):
        for b in range(n_batches):
            stream = 10000 + b
            p = trace(T, shape.E, shape.k, zs, ps, seed, l, stream)
            picks[b, li] = p
            logits[b, li] = logits_from_picks(p, shape.E, seed, l, stream, 1)
            n = T * shape.H
            if act == "bf16":
                x[b, li] = normal_bf16_bits(n, seed, PURPOSE_X, l, stream).reshape(T, shape.H)
            else:
                x[b, li] = normal_f32(n, seed, PURPOSE_X, l, stream).reshape(T, shape.H)
    return picks, logits, x


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen raw bf16 bits to fp32 (exact)."""
    return (bits.astype(np.uint32) << 16).view(np.float32)
