"""Algorithmic byte and flop counts for the paged-attention calls.

These are the bytes a call must move at minimum, used as the numerator of the
roofline fraction. Only tokens inside each sequence's context count; the
unused rows of a partial last block do not, and neither do the split-K
partials (an artefact of the kernel, not of the method).

The per-token KV formula is the one the Qwen2 page prints for its model: K and
V, times layers, KV heads, head_dim and element size ("A Rust inference server
for Qwen2 on Apple Silicon", "Target architecture"). For one layer call it is
2 * kv_heads * head_dim * elem_bytes per token.
"""

from __future__ import annotations

import numpy as np


def elem_bytes(dtype: str) -> int:
    return {"bf16": 2, "f32": 4}[dtype]


def kv_bytes_per_token(layers: int, kv_heads: int, head_dim: int, elem: int) -> int:
    """KV-cache bytes one token occupies across a whole model (K and V)."""
    return 2 * layers * kv_heads * head_dim * elem


def kv_read_bytes(context_lens, kv_heads: int, head_dim: int, elem: int) -> int:
    """K and V bytes read for one layer call: every valid token of every sequence."""
    total_tokens = int(np.asarray(context_lens, dtype=np.int64).sum())
    return total_tokens * kv_heads * 2 * head_dim * elem


def decode_bytes(context_lens, q_heads: int, kv_heads: int, head_dim: int, elem: int,
                 num_queries: int = 1, block_size: int = 16, fused_write: bool | None = None) -> dict:
    """Algorithmic bytes of one decode or fused verify call.

    With the fused write (pa_verify, the default whenever num_queries > 1) the
    new tokens' K/V are read from the inputs instead of the cache (same count)
    and written once to the cache.
    """
    if fused_write is None:
        fused_write = num_queries > 1
    lens = np.asarray(context_lens, dtype=np.int64)
    batch = lens.size
    kv = kv_read_bytes(lens, kv_heads, head_dim, elem)
    qo = 2 * batch * num_queries * q_heads * head_dim * elem          # q read + out written
    tables = int(((lens + block_size - 1) // block_size).sum()) * 4 + batch * 4
    new_writes = 0
    if fused_write:
        new_writes = batch * num_queries * kv_heads * 2 * head_dim * elem + batch * num_queries * 4
    total = kv + qo + tables + new_writes
    return {"kv": kv, "q_out": qo, "tables": tables, "new_writes": new_writes, "total": total}


def cache_write_bytes(num_tokens: int, kv_heads: int, head_dim: int, elem: int) -> int:
    """New K and V rows read from the inputs and written into the pool, plus the slots."""
    return num_tokens * (2 * 2 * kv_heads * head_dim * elem + 4)


def attention_flops(context_lens, q_heads: int, head_dim: int, num_queries: int = 1) -> int:
    """Multiply-adds of q.K and p.V (2 flops each), every visible (row, token) pair."""
    lens = np.asarray(context_lens, dtype=np.int64)
    pairs = 0
    for i in range(num_queries):
        pairs += int(np.clip(lens - num_queries + i + 1, 0, None).sum())
    return 4 * head_dim * q_heads * pairs


def q8_kv_read_bytes(context_lens, kv_heads: int, head_dim: int, block_size: int = 16) -> int:
    """int8 pool bytes read for one layer call: one byte per value of K and V for
    every valid token, its V scale (4 B), and the K scales (4 B per channel) of
    every block a sequence touches."""
    lens = np.asarray(context_lens, dtype=np.int64)
    tokens = int(lens.sum())
    blocks = int(((lens + block_size - 1) // block_size).sum())
    return tokens * kv_heads * (2 * head_dim + 4) + blocks * kv_heads * head_dim * 4


def decode_bytes_q8(context_lens, q_heads: int, kv_heads: int, head_dim: int, num_queries: int = 1,
                    block_size: int = 16, fused_write: bool | None = None) -> dict:
    """Algorithmic bytes of one decode or fused verify call over an int8 pool
    (queries, new rows and outputs are bf16). The fused write reads the new
    rows and rewrites, per touched block and KV head, the block's K bytes and
    scales (its requantisation) and the new V rows with their scales."""
    if fused_write is None:
        fused_write = num_queries > 1
    lens = np.asarray(context_lens, dtype=np.int64)
    batch = lens.size
    kv = q8_kv_read_bytes(lens, kv_heads, head_dim, block_size)
    qo = 2 * batch * num_queries * q_heads * head_dim * 2
    tables = int(((lens + block_size - 1) // block_size).sum()) * 4 + batch * 4
    new_writes = 0
    if fused_write:
        first = np.maximum(lens - num_queries, 0) // block_size
        last = np.maximum(lens - 1, 0) // block_size
        touched = int((last - first + 1)[lens > 0].sum())
        new_tokens = batch * num_queries
        new_writes = (touched * kv_heads * (block_size * head_dim + head_dim * 4)
                      + new_tokens * kv_heads * (2 * head_dim * 2 + head_dim + 4) + new_tokens * 4)
    total = kv + qo + tables + new_writes
    return {"kv": kv, "q_out": qo, "tables": tables, "new_writes": new_writes, "total": total}
