"""Seeded random sweep of small configurations against the oracle (GPU).

The fixed-shape tests cover the configurations the pages describe and their
edges one at a time. This sweep draws combinations none of them pins: query
head groups of 1 to 16 over 1 to 8 KV heads, 1 to 12 sequences of 1 to 1400
tokens (some at block and split edges), 1 to 8 new tokens per sequence,
explicit splits from 16 tokens up, and softmax scales from the standard
1/sqrt(128) to 1. Every case runs the fused path a caller would use (append
+ decode, or verify) and compares the output with the fp64 oracle at the
bf16 bound, and the pool with the oracle's write bit for bit. The draws are
seeded, so a failure names its case.
"""

from __future__ import annotations

import numpy as np
import pytest

import oracle
from gpu_util import assert_close, gpu_decode, gpu_verify, oracle_verify_of, to_f64
from paged_kv_decode_pa_gb300 import inputs

pytestmark = pytest.mark.gpu

CASES = range(12)


def _draw(case: int, max_len: int = 1400):
    rng = np.random.Generator(np.random.PCG64(7000 + case))
    hkv = int(rng.choice([1, 2, 4, 8]))
    g = int(rng.choice([1, 2, 3, 4, 6, 8, 12, 16]))
    batch = int(rng.integers(1, 13))
    nq = int(rng.choice([1, 1, 2, 3, 5, 8]))
    lens = rng.integers(nq, max_len + 1, size=batch)
    edges = np.array([nq, 16, 17, 32, 64, 65, 1024, 1025])
    pick = rng.random(batch) < 0.3
    lens[pick] = np.maximum(nq, edges[rng.integers(0, len(edges), size=int(pick.sum()))])
    split = int(rng.choice([0, 0, 16, 48, 64, 256, 1024]))
    scale = float(rng.choice([0.08838834764831845, 0.3, 1.0]))
    return hkv, g, batch, nq, [int(x) for x in lens], split, scale


def _workload(case, hkv, g, batch, nq, lens, scale):
    nb = sum(-(-x // 16) for x in lens) + 4
    w = inputs.custom(batch=batch, q_heads=g * hkv, kv_heads=hkv, context_lens=tuple(lens), num_blocks=nb,
                      seed=9000 + case, num_queries=nq)
    w.scale = scale
    return w


@pytest.mark.parametrize("case", CASES)
@pytest.mark.parametrize("kernel", ["auto", "simt"])
def test_random_bf16(case, kernel):
    hkv, g, batch, nq, lens, split, scale = _draw(case)
    w = _workload(case, hkv, g, batch, nq, lens, scale)
    what = f"case {case}: {batch} seqs {g * hkv}/{hkv} heads nq {nq} split {split} scale {scale:.3g} {kernel}"
    if nq == 1:
        kc, vc = w.k_cache.copy(), w.v_cache.copy()
        oracle.cache_write(kc, vc, w.k_new, w.v_new, w.slot_mapping)
        ref = oracle.decode(kc, vc, w.q, w.block_tables, w.context_lens, w.scale)
        out, gk, gv = gpu_decode(w, kernel=kernel, split_tokens=split)
    else:
        ref, kc, vc = oracle_verify_of(w)
        out, gk, gv = gpu_verify(w, kernel=kernel, split_tokens=split)
    assert gk.tobytes() == kc.tobytes() and gv.tobytes() == vc.tobytes(), f"{what}: pool differs"
    assert_close(to_f64(out), ref, "bf16", what)


@pytest.mark.parametrize("case", CASES)
def test_random_int8(case):
    import torch

    import paged_kv_decode_pa_gb300 as pa

    hkv, g, batch, nq, lens, split, scale = _draw(case)
    w = _workload(case, hkv, g, batch, nq, lens, scale)
    what = f"case {case}: int8 {batch} seqs {g * hkv}/{hkv} heads nq {nq} split {split} scale {scale:.3g}"
    pool = inputs.q8_pool(w)
    ref_pool = [a.copy() for a in (pool.k_codes, pool.v_codes, pool.k_scale, pool.v_scale)]
    dev = torch.device("cuda")
    kq, vq, ks, vs = (pa.to_torch(a, dev) for a in (pool.k_codes, pool.v_codes, pool.k_scale, pool.v_scale))
    q4 = w.q if w.q.ndim == 4 else w.q[:, None]
    ws = pa.new_workspace(batch, nq, g * hkv, hkv, w.max_context_len, dev, split)
    ref = oracle.verify_q8(*ref_pool, q4, w.k_new, w.v_new, w.slot_mapping, w.block_tables, w.context_lens,
                           w.scale)
    out = pa.pa_verify(kq, vq, pa.to_torch(q4, dev), pa.to_torch(w.k_new, dev), pa.to_torch(w.v_new, dev),
                       pa.to_torch(w.slot_mapping, dev), pa.to_torch(w.block_tables, dev),
                       pa.to_torch(w.context_lens, dev), w.max_context_len, w.scale, ws, split_tokens=split,
                       k_scale=ks, v_scale=vs)
    torch.cuda.synchronize()
    assert pa.pa_workspace_status(ws) == 0, what
    for got, want in zip((kq, vq, ks, vs), ref_pool):
        assert pa.to_numpy(got).tobytes() == want.tobytes(), f"{what}: pool differs"
    assert_close(to_f64(pa.to_numpy(out)), ref, "bf16", what)


@pytest.mark.parametrize("case", CASES)
@pytest.mark.parametrize("kernel", ["tc", "mma"])
def test_random_prefill(case, kernel):
    """Chunks of 1 .. the whole context after the remaining prefix, some empty."""
    import torch

    import paged_kv_decode_pa_gb300 as pa

    hkv, g, batch, _, lens, _, scale = _draw(case, max_len=900)
    rng = np.random.Generator(np.random.PCG64(8000 + case))
    chunks = [int(rng.integers(0, L + 1)) if rng.random() < 0.8 else L for L in lens]
    nq_max = max(1, max(chunks))
    w = inputs.custom(batch=batch, q_heads=g * hkv, kv_heads=hkv, context_lens=tuple(lens),
                      num_blocks=sum(-(-x // 16) for x in lens) + 4, seed=9500 + case, num_queries=nq_max)
    w.scale = scale
    rw = inputs.ragged(w, chunks)
    dev = torch.device("cuda")
    kc, vc = pa.to_torch(w.k_cache, dev), pa.to_torch(w.v_cache, dev)
    ws = torch.zeros(256, dtype=torch.uint8, device=dev)
    out = pa.pa_prefill(kc, vc, pa.to_torch(rw.q, dev), pa.to_torch(rw.query_start, dev),
                        pa.to_torch(w.block_tables, dev), pa.to_torch(w.context_lens, dev), w.max_context_len,
                        w.scale, rw.max_queries, workspace=ws, kernel=kernel)
    torch.cuda.synchronize()
    what = f"case {case}: prefill {batch} seqs {g * hkv}/{hkv} heads chunks {chunks} scale {scale:.3g} {kernel}"
    assert pa.pa_workspace_status(ws) == 0, what
    ref = oracle.attend_ragged(w.k_cache, w.v_cache, rw.q, rw.query_start, w.block_tables, w.context_lens,
                               w.scale)
    assert_close(to_f64(pa.to_numpy(out)), ref, "bf16", what)
