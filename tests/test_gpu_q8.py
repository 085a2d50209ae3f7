"""The int8 KV pool on the GPU against the oracle: the quantised append bit for
bit (bytes and scales), and decode / verify attention over the pool within
the bf16 output tolerance."""

from __future__ import annotations

import numpy as np
import pytest

import oracle
from gpu_util import assert_close, to_f64, workload
from paged_kv_decode_pa_gb300 import inputs

pytestmark = pytest.mark.gpu


def _dev_pool(pool):
    import paged_kv_decode_pa_gb300 as pa

    return [pa.to_torch(a) for a in (pool.k_codes, pool.v_codes, pool.k_scale, pool.v_scale)]


def _host(t):
    import paged_kv_decode_pa_gb300 as pa

    return pa.to_numpy(t)


def _same_pool(dev, ref, what):
    names = ("K bytes", "V bytes", "K scales", "V scales")
    for name, got, want in zip(names, map(_host, dev), ref):
        assert got.tobytes() == want.tobytes(), f"{what}: {name} differ from the oracle"


def _oracle_pool(pool):
    return [a.copy() for a in (pool.k_codes, pool.v_codes, pool.k_scale, pool.v_scale)]


def _gpu_q8(w, pool, verify: bool, split=0):
    import torch

    import paged_kv_decode_pa_gb300 as pa

    dev = _dev_pool(pool)
    kq, vq, ks, vs = dev
    q = w.q if (verify or w.q.ndim == 3) else w.q[:, 0]
    nq = w.spec.num_queries if verify else 1
    q4 = q if q.ndim == 4 else q[:, None]
    batch, hq = q4.shape[0], q4.shape[2]
    ws = pa.new_workspace(batch, nq, hq, w.spec.kv_heads, w.max_context_len, "cuda", split)
    tables, lens = pa.to_torch(w.block_tables), pa.to_torch(w.context_lens)
    if verify:
        out = pa.pa_verify(kq, vq, pa.to_torch(q4), pa.to_torch(w.k_new), pa.to_torch(w.v_new),
                           pa.to_torch(w.slot_mapping), tables, lens, w.max_context_len, w.scale, ws,
                           split_tokens=split, k_scale=ks, v_scale=vs)
    else:
        out = pa.pa_decode(kq, vq, pa.to_torch(q), tables, lens, w.max_context_len, w.scale, ws,
                           split_tokens=split, k_scale=ks, v_scale=vs)
    torch.cuda.synchronize()
    assert pa.pa_workspace_status(ws) == 0
    return pa.to_numpy(out), dev


@pytest.mark.parametrize("name", ["c2", "c3", "c5"])
def test_q8_append_bit_exact(name):
    """pa_cache_write into an int8 pool: every byte and scale equals the oracle's."""
    import torch

    import paged_kv_decode_pa_gb300 as pa

    w = workload(name)
    pool = inputs.q8_pool(w)
    ref = _oracle_pool(pool)
    assert oracle.cache_write_q8(*ref, w.k_new, w.v_new, w.slot_mapping) == 0
    dev = _dev_pool(pool)
    pa.pa_cache_write(dev[0], dev[1], pa.to_torch(w.k_new), pa.to_torch(w.v_new),
                      pa.to_torch(w.slot_mapping), k_scale=dev[2], v_scale=dev[3])
    torch.cuda.synchronize()
    _same_pool(dev, ref, name)


def test_q8_append_edge_slots():
    """Several rows into one block in one call, a repeated slot (the later token
    wins), negative and out-of-range slots (skipped), tokens out of order."""
    import torch

    import paged_kv_decode_pa_gb300 as pa

    w = inputs.custom(batch=4, q_heads=12, kv_heads=2, context_lens=(40, 3, 17, 64), num_blocks=40, seed=21)
    pool = inputs.q8_pool(w)
    rng = np.random.default_rng(5)
    n = 24
    slots = rng.choice(np.arange(40 * 16), size=n, replace=False).astype(np.int32)
    slots[3:9] = 16 * 7 + np.array([4, 0, 15, 9, 4, 2])  # six rows into block 7, slot 116 twice
    slots[10], slots[11] = -1, 40 * 16 + 3
    kn = inputs.f32_to_bf16_bits(rng.standard_normal((n, 2, 128)).astype(np.float32) * 3)
    vn = inputs.f32_to_bf16_bits(rng.standard_normal((n, 2, 128)).astype(np.float32) * 3)
    ref = _oracle_pool(pool)
    assert oracle.cache_write_q8(*ref, kn, vn, slots) == 1
    dev = _dev_pool(pool)
    pa.pa_cache_write(dev[0], dev[1], pa.to_torch(kn), pa.to_torch(vn), pa.to_torch(slots),
                      k_scale=dev[2], v_scale=dev[3])
    torch.cuda.synchronize()
    _same_pool(dev, ref, "edge slots")


@pytest.mark.parametrize("name,split", [("c1", 0), ("c2", 0), ("c2", 64), ("c3", 0), ("c4", 0), ("c4", 2048)])
def test_q8_decode_matches_oracle(name, split):
    w = workload(name) if name != "c1" else inputs.make("c1", dtype="bf16")
    pool = inputs.q8_pool(w)
    ref = oracle.decode_q8(pool.k_codes, pool.v_codes, pool.k_scale, pool.v_scale, w.q, w.block_tables,
                           w.context_lens, w.scale)
    out, dev = _gpu_q8(w, pool, verify=False, split=split)
    assert_close(to_f64(out), ref, "bf16", f"int8 decode {name} split {split}")
    _same_pool(dev, _oracle_pool(pool), "decode leaves the pool alone")


@pytest.mark.parametrize("name,split", [("c5", 0), ("c5", 256), ("c3", 0), ("c2", 32)])
def test_q8_verify_matches_oracle(name, split):
    """pa_verify on an int8 pool: the quantised append, then attention over the
    requantised blocks (decode workloads run as one-query verify)."""
    w = workload(name)
    pool = inputs.q8_pool(w)
    ref_pool = _oracle_pool(pool)
    q4 = w.q if w.q.ndim == 4 else w.q[:, None]
    ref = oracle.verify_q8(*ref_pool, q4, w.k_new, w.v_new, w.slot_mapping, w.block_tables,
                           w.context_lens, w.scale)
    out, dev = _gpu_q8(w, pool, verify=True, split=split)
    _same_pool(dev, ref_pool, f"verify {name}")
    assert_close(to_f64(out), ref, "bf16", f"int8 verify {name} split {split}")


@pytest.mark.parametrize("nq,hq,hkv", [(3, 16, 8), (5, 12, 2), (4, 32, 4)])
def test_q8_verify_shapes(nq, hq, hkv):
    """Row groups beyond 16 rows, new tokens straddling block and split edges,
    zero-length and one-token sequences."""
    lens = (0, 1, nq, 16, 17, 18, 47, 48, 49, 300, 513)
    lens = tuple(0 if x == 0 else max(nq, x) for x in lens)
    w = inputs.custom(batch=len(lens), q_heads=hq, kv_heads=hkv, context_lens=lens, num_blocks=90,
                      seed=nq * 1000 + hq, num_queries=nq)
    pool = inputs.q8_pool(w)
    for split in (0, 48):
        ref_pool = _oracle_pool(pool)
        ref = oracle.verify_q8(*ref_pool, w.q, w.k_new, w.v_new, w.slot_mapping, w.block_tables,
                               w.context_lens, w.scale)
        out, dev = _gpu_q8(w, pool, verify=True, split=split)
        _same_pool(dev, ref_pool, f"verify nq={nq} {hq}/{hkv} split {split}")
        assert_close(to_f64(out), ref, "bf16", f"int8 verify nq={nq} {hq}/{hkv} split {split}")


@pytest.mark.parametrize("hq,hkv", [(16, 8), (32, 4)])
def test_q8_verify_negative_slots(hq, hkv):
    """int8 pool: a new token with a negative slot is not written and its
    position keeps the pool's row, in the fused requantisation (one row group)
    and behind the separate append (two row groups)."""
    nq = 4
    w = inputs.custom(batch=4, q_heads=hq, kv_heads=hkv, context_lens=(4, 17, 33, 300), num_blocks=64,
                      seed=8765 + hq, num_queries=nq)
    slots = w.slot_mapping.copy()
    slots[[1, 4, 5, 15]] = -1
    w.slot_mapping = slots
    pool = inputs.q8_pool(w)
    ref_pool = _oracle_pool(pool)
    ref = oracle.verify_q8(*ref_pool, w.q, w.k_new, w.v_new, w.slot_mapping, w.block_tables,
                           w.context_lens, w.scale)
    out, dev = _gpu_q8(w, pool, verify=True)
    _same_pool(dev, ref_pool, f"negative slots {hq}/{hkv}")
    assert_close(to_f64(out), ref, "bf16", f"int8 negative slots {hq}/{hkv}")


def test_q8_verify_many_new_tokens():
    """int8 pool, 100 new tokens per sequence (several row groups: the append
    runs first), some with negative slots."""
    nq = 100
    w = inputs.custom(batch=3, q_heads=4, kv_heads=4, context_lens=(100, 150, 700), num_blocks=80,
                      seed=1357, num_queries=nq)
    slots = w.slot_mapping.copy()
    slots[[7, 99, 150, 298]] = -1
    w.slot_mapping = slots
    pool = inputs.q8_pool(w)
    ref_pool = _oracle_pool(pool)
    ref = oracle.verify_q8(*ref_pool, w.q, w.k_new, w.v_new, w.slot_mapping, w.block_tables,
                           w.context_lens, w.scale)
    out, dev = _gpu_q8(w, pool, verify=True)
    _same_pool(dev, ref_pool, "100 new tokens")
    assert_close(to_f64(out), ref, "bf16", "int8 100 new tokens")
