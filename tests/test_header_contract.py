"""The int8 quantiser as include/pa.h states it, held against the oracle
(CPU only).

The header is the contract a caller reproduces bytes from, so its formula must
be the one the pinned oracle computes ("A Rust inference server for Qwen2 on
Apple Silicon", Day 4 "int8 KV"): q = RN(x * (127 / m)) with one fp32 division
per group, not RN(x / s) with the stored scale s = m / 127. The two round
differently for some inputs, and this test builds rows where they do.
"""

import re
from pathlib import Path

import numpy as np

import oracle

HEADER = Path(__file__).resolve().parents[1] / "include" / "pa.h"


def _header_text():
    return " ".join(HEADER.read_text().replace("*", " ").split())


def test_header_states_the_multiply_form():
    text = _header_text()
    assert re.search(r"s = m / 127", text), "the stored scale"
    assert re.search(r"q = RN\(x \s*\(127 / m\)\)", text), "codes from one division per group, then a multiply"
    assert "x / s" not in text, "the per-element division form is not what the library computes"


def _header_codes(x32: np.ndarray) -> np.ndarray:
    """The header's formula, element by element in float32."""
    m = np.float32(np.abs(x32).max())
    if m == 0:
        return np.full(x32.shape, 128, np.uint8)
    inv = np.float32(127.0) / m
    r = np.rint((x32 * inv).astype(np.float32))
    return (np.clip(r, -127, 127).astype(np.int32) + 128).astype(np.uint8)


def _division_codes(x32: np.ndarray) -> np.ndarray:
    m = np.float32(np.abs(x32).max())
    s = m / np.float32(127.0)
    r = np.rint((x32 / s).astype(np.float32))
    return (np.clip(r, -127, 127).astype(np.int32) + 128).astype(np.uint8)


def test_oracle_v_codes_follow_the_header_formula():
    rng = np.random.default_rng(2024)
    rows = 64
    x = rng.standard_normal((rows, 128)).astype(np.float32)
    bits = (x.view(np.uint32) + 0x8000) >> 16  # bf16 bit patterns (round half up is fine for inputs)
    bits = bits.astype(np.uint16)
    x32 = (bits.astype(np.uint32) << 16).view(np.float32)
    # One V row per slot: each row is a group of its own.
    nb = rows // 16
    kq = np.full((1, nb, 16, 128), 128, np.uint8)
    vq = np.full((1, nb, 16, 128), 128, np.uint8)
    ks = np.zeros((1, nb, 128), np.float32)
    vs = np.zeros((1, nb, 16), np.float32)
    rows_in = bits.reshape(rows, 1, 128)
    assert oracle.cache_write_q8(kq, vq, ks, vs, rows_in, rows_in, np.arange(rows, dtype=np.int32)) == 0
    got = vq.reshape(rows, 128)
    differ = 0
    for r in range(rows):
        want = _header_codes(x32[r])
        assert np.array_equal(got[r], want), f"row {r}"
        assert vs.reshape(rows)[r] == np.float32(np.abs(x32[r]).max()) / np.float32(127.0)
        differ += int((_division_codes(x32[r]) != want).sum())
    # The rows exercise inputs on which the two forms disagree, so a header
    # that stated the division form would describe different bytes.
    assert differ > 0
