"""Byte accounting against the numbers the Qwen2 page prints (CPU only)."""

import json
import os

import numpy as np

from paged_kv_decode_pa_gb300 import accounting

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "kv_bytes.json")


def test_kv_bytes_per_token_matches_page():
    g = json.load(open(GOLDEN))["qwen2_1p5b"]
    assert accounting.kv_bytes_per_token(g["layers"], g["kv_heads"], g["head_dim"], 2) == \
        g["kv_bytes_per_token_bf16"]
    assert accounting.kv_bytes_per_token(g["layers"], g["kv_heads"], g["head_dim"], 4) == \
        g["kv_bytes_per_token_f32"]
    assert accounting.kv_bytes_per_token(g["layers"], g["kv_heads"], g["head_dim"], 1) == \
        g["int8_codes_per_token"]
    # 32k tokens of context is the page's 0.94 GB (decimal gigabytes).
    gb = 32768 * g["kv_bytes_per_token_bf16"] / 1e9
    assert round(gb, 2) == g["context_32k_gb"]


def test_one_layer_call_is_the_per_token_formula_over_valid_tokens():
    lens = np.array([1, 17, 33, 64])
    per_token_one_layer = accounting.kv_bytes_per_token(1, 2, 128, 2)
    assert accounting.kv_read_bytes(lens, 2, 128, 2) == lens.sum() * per_token_one_layer
    b = accounting.decode_bytes(lens, q_heads=12, kv_heads=2, head_dim=128, elem=2)
    assert b["kv"] == lens.sum() * per_token_one_layer
    assert b["q_out"] == 2 * 4 * 12 * 128 * 2
    assert b["tables"] == (1 + 2 + 3 + 4) * 4 + 4 * 4


def test_flops_count_visible_pairs_only():
    lens = np.array([3, 5])
    assert accounting.attention_flops(lens, q_heads=2, head_dim=4) == 4 * 4 * 2 * 8
    # verify with two queries: rows see L-1 and L tokens
    assert accounting.attention_flops(lens, q_heads=1, head_dim=1, num_queries=2) == 4 * (2 + 4 + 3 + 5)


def test_q8_bytes_per_block():
    """One full 16-token block of one KV head in the int8 pool: 2 x 2048 code
    bytes, 16 V scales and 128 K scales of 4 bytes = 4,672 bytes (against 8,192
    in bf16)."""
    from paged_kv_decode_pa_gb300 import accounting

    assert accounting.q8_kv_read_bytes([16], 1, 128) == 4672
    assert accounting.kv_read_bytes([16], 1, 128, 2) == 8192
    # a partial block still carries the block's K scales
    assert accounting.q8_kv_read_bytes([1], 1, 128) == 2 * 128 + 4 + 512
    b = accounting.decode_bytes_q8([17, 0], q_heads=2, kv_heads=1, head_dim=128, num_queries=2)
    # new tokens at positions 15, 16: two touched blocks for the first sequence, none for L = 0
    assert b["new_writes"] == 2 * (16 * 128 + 128 * 4) + 4 * (2 * 128 * 2 + 128 + 4) + 4 * 4
