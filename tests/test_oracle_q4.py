"""Pins for the oracle's number formats and Q4_0 decode (CPU only).

Q4_0: 18 bytes per 32 values ("Multi-GPU LLM Calculator: VRAM Split and RAM
Offload", "Memory placement"), fp16 scale plus 16 nibble bytes, w = (q - 8) d.
"""
import os

import numpy as np
import pytest

import oracle


def _load_blocks(golden_dir):
    blocks, cur = [], {}
    with open(os.path.join(golden_dir, "q4_0_blocks.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, rest = line.partition(" ")
            if key == "name":
                cur = {"name": rest}
            elif key == "d":
                cur["d"] = int(rest, 16)
            elif key == "qs":
                cur["qs"] = bytes(int(t, 16) for t in rest.split())
            elif key == "values":
                cur["values"] = [float(t) for t in rest.split()]
                blocks.append(cur)
    return blocks


def test_golden_blocks(golden_dir):
    blocks = _load_blocks(golden_dir)
    assert len(blocks) >= 7
    for b in blocks:
        raw = bytes([b["d"] & 0xFF, b["d"] >> 8]) + b["qs"]
        assert len(raw) == 18 and len(b["values"]) == 32
        got = oracle.q4_0_decode(raw)
        assert np.array_equal(got, np.array(b["values"])), b["name"]


def test_fp16_all_patterns_match_numpy():
    # every binary16 bit pattern against numpy's float16 -> float64 widening
    bits = np.arange(65536, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.fp16_to_double(int(h)) for h in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # signed zeros keep their sign
    assert np.signbit(oracle.fp16_to_double(0x8000))


def test_bf16_exact():
    for v in (1.0, -2.5, 3.140625, 1e-30, -7.0e30, 0.0):
        b = np.float32(v).view(np.uint32) >> 16
        f = float((np.uint32(b) << 16).view(np.float32))
        assert oracle.bf16_to_double(int(b)) == f


def test_nibble_order_single_position():
    # one non-8 nibble at each position in turn: exactly one output moves
    for pos in range(32):
        qs = bytearray([0x88] * 16)
        j = pos % 16
        if pos < 16:
            qs[j] = (qs[j] & 0xF0) | 0x3     # low nibble 3 -> value -5
        else:
            qs[j] = (qs[j] & 0x0F) | 0xC0    # high nibble 12 -> value +4
        got = oracle.q4_0_decode(bytes([0x00, 0x3C]) + bytes(qs))
        want = np.zeros(32)
        want[pos] = -5.0 if pos < 16 else 4.0
        assert np.array_equal(got, want), pos


def test_block_size_matches_pages():
    # 18 bytes per 32 values; the decode-model expert block of 3 matrices
    # 704 x 2816 is 3,345,408 bytes, the pages' "~3.35 MB per expert at 4-bit"
    # ("llama.cpp + MoE expert cache", "The problem").
    H, F = 2816, 704
    assert 3 * F * H // 32 * 18 == 3_345_408
    assert abs(3_345_408 / 1e6 - 3.35) < 0.01
