"""pa_verify_ragged (decode and verify sequences in one launch, no padding)
against the oracle: bf16 tensor-core, fp32 CUDA-core and int8 pools."""

from __future__ import annotations

import numpy as np
import pytest

import oracle
from gpu_util import assert_close, to_f64
from paged_kv_decode_pa_gb300 import inputs

pytestmark = pytest.mark.gpu


def _run(rw, kernel="auto", split=0, kv="native"):
    import torch

    import paged_kv_decode_pa_gb300 as pa

    w = rw.base
    dev = torch.device("cuda")
    scales = {}
    if kv == "int8":
        pool = inputs.q8_pool(w)
        host = [pool.k_codes, pool.v_codes, pool.k_scale, pool.v_scale]
        dev_pool = [pa.to_torch(a, dev) for a in host]
        kc, vc = dev_pool[0], dev_pool[1]
        scales = {"k_scale": dev_pool[2], "v_scale": dev_pool[3]}
    else:
        host = [w.k_cache, w.v_cache]
        dev_pool = [pa.to_torch(a, dev) for a in host]
        kc, vc = dev_pool
    ws = pa.new_workspace(w.spec.batch, rw.max_queries, w.spec.q_heads, w.spec.kv_heads, w.max_context_len, dev,
                          split)
    out = pa.pa_verify_ragged(kc, vc, pa.to_torch(rw.q, dev), pa.to_torch(rw.k_new, dev),
                              pa.to_torch(rw.v_new, dev), pa.to_torch(rw.slot_mapping, dev),
                              pa.to_torch(rw.query_start, dev), pa.to_torch(w.block_tables, dev),
                              pa.to_torch(w.context_lens, dev), w.max_context_len, w.scale, ws, rw.max_queries,
                              split_tokens=split, kernel=kernel, **scales)
    torch.cuda.synchronize()
    assert pa.pa_workspace_status(ws) == 0
    ref_pool = [a.copy() for a in host]
    if kv == "int8":
        ref = oracle.verify_ragged(ref_pool[0], ref_pool[1], rw.q, rw.k_new, rw.v_new, rw.slot_mapping,
                                   rw.query_start, w.block_tables, w.context_lens, w.scale,
                                   q8_scales=(ref_pool[2], ref_pool[3]))
    else:
        ref = oracle.verify_ragged(ref_pool[0], ref_pool[1], rw.q, rw.k_new, rw.v_new, rw.slot_mapping,
                                   rw.query_start, w.block_tables, w.context_lens, w.scale)
    for got_t, want in zip(dev_pool, ref_pool):
        assert pa.to_numpy(got_t).tobytes() == want.tobytes(), "pool after the write differs from the oracle's"
    return to_f64(pa.to_numpy(out)), ref


MIX = (1, 5, 0, 2, 1, 3, 5, 1, 4, 1, 2)


@pytest.mark.parametrize("hq,hkv", [(16, 8), (12, 2), (32, 4)])
@pytest.mark.parametrize("split", [0, 16, 48])
def test_ragged_bf16(hq, hkv, split):
    lens = (5, 16, 17, 18, 47, 48, 49, 300, 513, 1, 64)
    w = inputs.custom(batch=len(lens), q_heads=hq, kv_heads=hkv, context_lens=lens, num_blocks=120,
                      seed=hq * 10 + hkv, num_queries=5)
    rw = inputs.ragged(w, [min(n, L) for n, L in zip(MIX, lens)])
    got, ref = _run(rw, split=split)
    assert_close(got, ref, "bf16", f"ragged bf16 {hq}/{hkv} split {split}")


def test_ragged_fp32():
    lens = (3, 20, 64, 130, 1, 33)
    w = inputs.custom(batch=len(lens), q_heads=12, kv_heads=2, context_lens=lens, num_blocks=30, dtype="f32",
                      seed=77, num_queries=3)
    rw = inputs.ragged(w, [1, 3, 2, 0, 1, 3])
    got, ref = _run(rw)
    assert_close(got, ref, "f32", "ragged fp32")


@pytest.mark.parametrize("hq,hkv", [(16, 8), (12, 2)])
def test_ragged_int8(hq, hkv):
    """16/8 keeps one row group (the block requantised in the kernel); 12/2 with
    five tokens has two (the append runs first)."""
    lens = (5, 16, 17, 18, 47, 48, 49, 300, 513, 1, 64)
    w = inputs.custom(batch=len(lens), q_heads=hq, kv_heads=hkv, context_lens=lens, num_blocks=120,
                      seed=hq * 10 + hkv + 1, num_queries=5)
    rw = inputs.ragged(w, [min(n, L) for n, L in zip(MIX, lens)])
    got, ref = _run(rw, kv="int8")
    assert_close(got, ref, "bf16", f"ragged int8 {hq}/{hkv}")


def test_ragged_all_decode_equals_decode():
    """Every sequence with one token: the same as a decode step of those tokens."""
    w = inputs.make("c5", batch=12, num_blocks=1024)
    rw = inputs.ragged(w, [1] * 12)
    got, ref = _run(rw)
    assert_close(got, ref, "bf16", "ragged, all decode")


@pytest.mark.parametrize("kv,hq,hkv", [("native", 16, 8), ("native", 32, 4), ("int8", 16, 8), ("int8", 12, 2)])
def test_ragged_negative_slots(kv, hq, hkv):
    """Some new tokens of a ragged call have negative slots: not written, and
    attention sees the pool's rows at their positions (the fused write equals
    the append followed by attention)."""
    lens = (5, 16, 17, 18, 47, 48, 49, 300, 513, 1, 64)
    w = inputs.custom(batch=len(lens), q_heads=hq, kv_heads=hkv, context_lens=lens, num_blocks=120,
                      seed=hq * 10 + hkv + 7, num_queries=5)
    rw = inputs.ragged(w, [min(n, L) for n, L in zip(MIX, lens)])
    slots = rw.slot_mapping.copy()
    slots[[0, 3, 9, 17]] = -1  # tokens of sequences 0, 1, 5 and 7
    rw.slot_mapping = slots
    got, ref = _run(rw, kv=kv)
    assert_close(got, ref, "bf16", f"ragged negative slots {kv} {hq}/{hkv}")
