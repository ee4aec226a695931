"""Pins for the oracle's expert FFN (CPU only).

SwiGLU with merged gate/up ("llama.cpp + MoE expert cache", "Limitations": merged
gate/up tensors, SiLU activation): g = W_gate x, u = W_up x, h = silu(g) u,
y = W_down h, weights in Q4_0 rows of the expert block [gate | up | down].
"""
import math

import numpy as np
import pytest

import oracle


def _blk_bytes(rows, cols, d_bits, nibble_fn):
    """A Q4_0 matrix whose element (r, c) has nibble nibble_fn(r, c) and scale d_bits."""
    nb = cols // 32
    out = bytearray()
    for r in range(rows):
        for b in range(nb):
            out += bytes([d_bits & 0xFF, d_bits >> 8])
            for j in range(16):
                lo = nibble_fn(r, 32 * b + j)
                hi = nibble_fn(r, 32 * b + 16 + j)
                out.append(lo | (hi << 4))
    return bytes(out)


def _expert(H, F, d, g_fn, u_fn, dn_fn):
    return np.frombuffer(_blk_bytes(F, H, d, g_fn) + _blk_bytes(F, H, d, u_fn)
                         + _blk_bytes(H, F, d, dn_fn), dtype=np.uint8).copy()


def test_integer_exact_gate_up():
    # d = 1 and integer x in {-2..2}: g and u are exact integers; computed here
    # with Python integers straight from the nibble rule.
    H, F = 64, 32
    rng = np.random.default_rng(1)
    G = rng.integers(0, 16, size=(F, H))
    U = rng.integers(0, 16, size=(F, H))
    D = rng.integers(0, 16, size=(H, F))
    blk = _expert(H, F, 0x3C00, lambda r, c: int(G[r, c]), lambda r, c: int(U[r, c]),
                  lambda r, c: int(D[r, c]))
    x = rng.integers(-2, 3, size=H).astype(np.float64)
    parts = oracle.expert_ffn(blk, H, F, x, parts=True)
    g_int = [sum((int(G[r, c]) - 8) * int(x[c]) for c in range(H)) for r in range(F)]
    u_int = [sum((int(U[r, c]) - 8) * int(x[c]) for c in range(H)) for r in range(F)]
    assert parts["g"].tolist() == [float(v) for v in g_int]
    assert parts["u"].tolist() == [float(v) for v in u_int]


def test_power_of_two_scale_exact():
    H, F = 32, 32
    rng = np.random.default_rng(2)
    G = rng.integers(0, 16, size=(F, H))
    blk = _expert(H, F, 0x3000, lambda r, c: int(G[r, c]), lambda r, c: 9, lambda r, c: 8)  # d = 0.125
    x = rng.integers(-2, 3, size=H).astype(np.float64)
    parts = oracle.expert_ffn(blk, H, F, x, parts=True)
    want = [sum((int(G[r, c]) - 8) * int(x[c]) for c in range(H)) * 0.125 for r in range(F)]
    assert parts["g"].tolist() == want
    assert parts["u"].tolist() == [0.125 * float(x.sum())] * F   # up nibbles 9 -> weight +d
    assert np.all(parts["y"] == 0)                         # down nibbles 8 -> zero weights


def test_all_eights_give_zero():
    H, F = 64, 64
    blk = _expert(H, F, 0x3C00, lambda r, c: 8, lambda r, c: 8, lambda r, c: 8)
    x = np.random.default_rng(3).standard_normal(H)
    y = oracle.expert_ffn(blk, H, F, x)
    assert np.all(y == 0.0)


def test_silu_and_gate_up_roles():
    # x = e_0; gate row r has weight 2 at column 0 (g = 2), up weight 1 (u = 1):
    # h = silu(2) * 1 = 2 / (1 + e^-2) = 1.7615941559557649; with the roles
    # swapped it would be silu(1) * 2 = 1.4621171572600098.
    H, F = 32, 32
    blk = _expert(H, F, 0x3C00,
                  lambda r, c: 10 if c == 0 else 8,
                  lambda r, c: 9 if c == 0 else 8,
                  lambda r, c: 9 if c == r else 8)      # down = identity on the first 32 rows
    x = np.zeros(H); x[0] = 1.0
    parts = oracle.expert_ffn(blk, H, F, x, parts=True)
    assert parts["g"].tolist() == [2.0] * F
    assert parts["u"].tolist() == [1.0] * F
    np.testing.assert_allclose(parts["h"], 1.7615941559557649, rtol=1e-15)
    np.testing.assert_allclose(parts["y"], 1.7615941559557649, rtol=1e-15)


def test_silu_special_values():
    H, F = 32, 32
    # g = 0 -> h = 0; g = 1 -> silu(1) = sigmoid(1) = 0.7310585786300049 (u = 1)
    for gq, want in ((8, 0.0), (9, 0.7310585786300049)):
        blk = _expert(H, F, 0x3C00, lambda r, c, gq=gq: gq if c == 0 else 8,
                      lambda r, c: 9 if c == 0 else 8, lambda r, c: 8)
        x = np.zeros(H); x[0] = 1.0
        parts = oracle.expert_ffn(blk, H, F, x, parts=True)
        np.testing.assert_allclose(parts["h"], want, rtol=1e-15, atol=0)
    # very negative g: silu -> 0 without overflow trouble (d = 8, q = 0 -> -64 per x)
    blk = _expert(H, F, 0x4800, lambda r, c: 0, lambda r, c: 9, lambda r, c: 8)
    x = np.full(H, 20.0)
    parts = oracle.expert_ffn(blk, H, F, x, parts=True)
    assert np.all(parts["g"] == -64.0 * 20 * H)
    assert np.all(np.abs(parts["h"]) < 1e-300)


def test_layout_row_and_column_positions():
    # one non-neutral weight in gate at (row 5, column 37) and in down at
    # (row 11, column 5): pins row-major rows of blocks along the input dimension
    H, F = 64, 32
    blk = _expert(H, F, 0x3C00,
                  lambda r, c: 11 if (r, c) == (5, 37) else 8,
                  lambda r, c: 9,
                  lambda r, c: 12 if (r, c) == (11, 5) else 8)
    x = np.zeros(H); x[37] = 1.0
    parts = oracle.expert_ffn(blk, H, F, x, parts=True)
    g = np.zeros(F); g[5] = 3.0
    assert parts["g"].tolist() == g.tolist()
    assert parts["u"].tolist() == [1.0] * F
    y = np.zeros(H); y[11] = 4.0 * (3.0 / (1.0 + math.exp(-3.0)))
    np.testing.assert_allclose(parts["y"], y, rtol=1e-15, atol=0)


def _dequant_numpy(mat_bytes, rows, cols):
    a = np.frombuffer(mat_bytes, dtype=np.uint8).reshape(rows, cols // 32, 18)
    d = a[:, :, 0:2].copy().view(np.float16)[:, :, 0].astype(np.float64)
    qs = a[:, :, 2:]
    q = np.concatenate([qs & 0xF, qs >> 4], axis=2).astype(np.float64) - 8.0
    return (q * d[:, :, None]).reshape(rows, cols)


def test_dense_random_block_against_numpy():
    # random canonical block: oracle vs a vectorised numpy decode + float64 matmul
    import synth
    H, F = 256, 512
    blk = synth.expert_block(0, 3, H, F, seed=0)
    x = np.random.default_rng(4).standard_normal(H)
    mat = F * H // 32 * 18
    Wg = _dequant_numpy(blk[:mat].tobytes(), F, H)
    Wu = _dequant_numpy(blk[mat:2 * mat].tobytes(), F, H)
    Wd = _dequant_numpy(blk[2 * mat:].tobytes(), H, F)
    g, u = Wg @ x, Wu @ x
    y = Wd @ (g / (1 + np.exp(-g)) * u)
    np.testing.assert_allclose(oracle.expert_ffn(blk, H, F, x), y, rtol=1e-12, atol=1e-12)
