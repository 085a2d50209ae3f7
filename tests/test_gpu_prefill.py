"""pa_prefill (causal attention of prompt chunks over the paged cache) against
the oracle, bf16."""

from __future__ import annotations

import functools

import numpy as np
import pytest

import oracle
from gpu_util import assert_close, to_f64
from paged_kv_decode_pa_gb300 import inputs

pytestmark = pytest.mark.gpu


KERNELS = ["tc", "mma"]


def _prefill(w, chunks, kernel="auto"):
    """Run pa_prefill for chunks = per-sequence chunk lengths; returns (gpu, ref)."""
    import torch

    import paged_kv_decode_pa_gb300 as pa

    rw = inputs.ragged(w, chunks)
    dev = torch.device("cuda")
    kc, vc = pa.to_torch(w.k_cache, dev), pa.to_torch(w.v_cache, dev)
    ws = torch.zeros(256, dtype=torch.uint8, device=dev)
    out = pa.pa_prefill(kc, vc, pa.to_torch(rw.q, dev), pa.to_torch(rw.query_start, dev),
                        pa.to_torch(w.block_tables, dev), pa.to_torch(w.context_lens, dev), w.max_context_len,
                        w.scale, rw.max_queries, workspace=ws, kernel=kernel)
    torch.cuda.synchronize()
    assert pa.pa_workspace_status(ws) == 0
    ref = oracle.attend_ragged(w.k_cache, w.v_cache, rw.q, rw.query_start, w.block_tables, w.context_lens,
                               w.scale)
    return to_f64(pa.to_numpy(out)), ref


@pytest.mark.parametrize("kernel", KERNELS)
def test_prefill_64_prompts_of_256(kernel):
    """The 64-request workload's prompts: 256 tokens each, no prefix, 16/8 heads."""
    w = inputs.custom(batch=64, q_heads=16, kv_heads=8, context_lens=(256,) * 64, num_blocks=1100, seed=51,
                      num_queries=256)
    got, ref = _prefill(w, [256] * 64, kernel)
    assert_close(got, ref, "bf16", f"prefill 64 x 256 ({kernel})")


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("hq,hkv", [(16, 8), (12, 2), (32, 4), (8, 8), (10, 2), (20, 1)])
def test_prefill_chunks_with_prefixes(hq, hkv, kernel):
    """Chunks after prefixes of several lengths: tiles of whole tokens (groups
    of 1, 2, 5, 6, 8, 20: 125- and 120-row tiles included), ragged tails, chunk
    sizes 1 .. 300, context ends inside and at block edges."""
    prefixes = (0, 5, 100, 700, 16, 0, 31)
    chunks = (64, 1, 300, 129, 16, 17, 33)
    lens = tuple(p + c for p, c in zip(prefixes, chunks))
    w = inputs.custom(batch=len(lens), q_heads=hq, kv_heads=hkv, context_lens=lens, num_blocks=160,
                      seed=hq * 7 + hkv, num_queries=max(chunks))
    got, ref = _prefill(w, list(chunks), kernel)
    assert_close(got, ref, "bf16", f"prefill {hq}/{hkv} ({kernel})")


@pytest.mark.parametrize("kernel", KERNELS)
def test_prefill_zero_chunks_and_long_context(kernel):
    """A sequence with an empty chunk (no rows, nothing written) next to a
    256-token chunk after a 4096-token prefix."""
    lens = (10, 4096 + 256, 3)
    w = inputs.custom(batch=3, q_heads=12, kv_heads=2, context_lens=lens, num_blocks=300, seed=52,
                      num_queries=256)
    got, ref = _prefill(w, [0, 256, 3], kernel)
    assert_close(got, ref, "bf16", f"prefill long ({kernel})")


def _prefill_raw(w, rw, tables, lens, kernel):
    import torch

    import paged_kv_decode_pa_gb300 as pa

    dev = torch.device("cuda")
    kc, vc = pa.to_torch(w.k_cache, dev), pa.to_torch(w.v_cache, dev)
    ws = torch.zeros(256, dtype=torch.uint8, device=dev)
    out = pa.pa_prefill(kc, vc, pa.to_torch(rw.q, dev), pa.to_torch(rw.query_start, dev), pa.to_torch(tables, dev),
                        pa.to_torch(lens, dev), w.max_context_len, w.scale, rw.max_queries, workspace=ws,
                        kernel=kernel)
    torch.cuda.synchronize()
    return pa.to_numpy(out), pa.pa_workspace_status(ws)


@pytest.mark.parametrize("kernel", KERNELS)
def test_prefill_flags_bad_ids_and_lengths(kernel):
    """A block id outside the pool raises PA_FLAG_BAD_BLOCK and reads zeros; a
    length past max_context_len raises PA_FLAG_BAD_LENGTH and is clamped.
    Neither faults, and the other sequences' rows are unchanged."""
    from paged_kv_decode_pa_gb300 import _lib

    w = inputs.custom(batch=3, q_heads=12, kv_heads=2, context_lens=(40, 40, 40), num_blocks=16, seed=44,
                      num_queries=8)
    rw = inputs.ragged(w, [8, 8, 8])
    good, st = _prefill_raw(w, rw, w.block_tables, w.context_lens, kernel)
    assert st == 0
    tables = w.block_tables.copy()
    tables[1, 1] = 1 << 30
    bad, st = _prefill_raw(w, rw, tables, w.context_lens, kernel)
    assert st & _lib.PA_FLAG_BAD_BLOCK
    assert np.array_equal(bad[np.r_[0:8, 16:24]], good[np.r_[0:8, 16:24]])
    lens = w.context_lens.copy()
    lens[2] = w.max_context_len + 100
    bad, st = _prefill_raw(w, rw, w.block_tables, lens, kernel)
    assert st & _lib.PA_FLAG_BAD_LENGTH
    assert np.array_equal(bad[0:16], good[0:16])


def test_prefill_graph_replay():
    """pa_prefill captured in a CUDA graph: rewrite q and the lengths in place,
    replay, and match the oracle for the new inputs."""
    import torch

    import paged_kv_decode_pa_gb300 as pa

    dev = torch.device("cuda")
    w = inputs.custom(batch=4, q_heads=16, kv_heads=8, context_lens=(300, 200, 64, 129), num_blocks=80, seed=45,
                      num_queries=64)
    chunks = [64, 33, 1, 40]
    rw = inputs.ragged(w, chunks)
    kc, vc = pa.to_torch(w.k_cache, dev), pa.to_torch(w.v_cache, dev)
    q, qs = pa.to_torch(rw.q, dev), pa.to_torch(rw.query_start, dev)
    tb, ln = pa.to_torch(w.block_tables, dev), pa.to_torch(w.context_lens, dev)
    out = torch.empty_like(q)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        pa.pa_prefill(kc, vc, q, qs, tb, ln, w.max_context_len, w.scale, rw.max_queries, out=out)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        pa.pa_prefill(kc, vc, q, qs, tb, ln, w.max_context_len, w.scale, rw.max_queries, out=out)
    rng = np.random.default_rng(46)
    q2 = rng.standard_normal(rw.q.shape).astype(np.float32)
    q2 = pa.to_numpy(torch.from_numpy(q2).to(torch.bfloat16))
    lens2 = w.context_lens.copy()
    lens2[0] -= 5  # the chunk now ends 5 positions earlier
    q.copy_(pa.to_torch(q2, dev))
    ln.copy_(pa.to_torch(lens2, dev))
    g.replay()
    torch.cuda.synchronize()
    ref = oracle.attend_ragged(w.k_cache, w.v_cache, q2, rw.query_start, w.block_tables, lens2, w.scale)
    assert_close(to_f64(pa.to_numpy(out)), ref, "bf16", "prefill graph replay")


@pytest.mark.parametrize("hq,kernel", [(64, "tc"), (64, "mma"), (130, "auto")])
def test_prefill_large_groups(hq, kernel):
    """One KV head shared by 64 query heads (two tokens per tcgen05 tile), and
    by 130 (above the tcgen05 kernel's 128: AUTO takes the warp-level kernel)."""
    prefixes = (0, 37)
    chunks = (7, 19)
    lens = tuple(p + c for p, c in zip(prefixes, chunks))
    w = inputs.custom(batch=2, q_heads=hq, kv_heads=1, context_lens=lens, num_blocks=16, seed=hq,
                      num_queries=max(chunks))
    got, ref = _prefill(w, list(chunks), kernel)
    assert_close(got, ref, "bf16", f"prefill group {hq} ({kernel})")


_LONG = dict(batch=8, q_heads=12, kv_heads=2, context_lens=(4096,) * 8, num_blocks=2100, seed=61, num_queries=2048)
# Sampled rows of the long workload: (sequence, first row of its chunk, rows).
# The chunk's first rows see the shortest contexts, its last rows the longest;
# the middle samples cross several row tiles (21 tokens each for a group of 6)
# and so the persistent grid's item boundaries.
_LONG_SAMPLES = ((0, 0, 256), (3, 1000, 100), (5, 1337, 64), (7, 1536, 512))


@functools.lru_cache(maxsize=1)
def _long_reference():
    """The oracle's rows for _LONG_SAMPLES. A chunk's rows are its sequence's
    last positions, so rows [r0, r0 + n) of a 2048-token chunk ending at 4096
    are those of an n-token chunk ending at 2048 + r0 + n."""
    w = inputs.custom(**_LONG)
    rw = inputs.ragged(w, [2048] * 8)
    refs = []
    for b, r0, n in _LONG_SAMPLES:
        q0 = int(rw.query_start[b]) + r0
        refs.append(oracle.attend_ragged(w.k_cache, w.v_cache, rw.q[q0:q0 + n], np.array([0, n], dtype=np.int32),
                                         w.block_tables[b:b + 1], np.array([2048 + r0 + n], dtype=np.int32),
                                         w.scale))
    return refs


@pytest.mark.parametrize("kernel", KERNELS)
def test_prefill_long_chunks_full_size(kernel):
    """The benchmark's long workload at full size (8 sequences, 2048-token
    chunks after 2048-token prefixes, 12/2 heads), in the benchmark's launch
    configuration; the oracle checks sampled rows of four sequences, at the
    start, in the middle and at the end of their chunks."""
    import torch

    import paged_kv_decode_pa_gb300 as pa

    w = inputs.custom(**_LONG)
    rw = inputs.ragged(w, [2048] * 8)
    dev = torch.device("cuda")
    kc, vc = pa.to_torch(w.k_cache, dev), pa.to_torch(w.v_cache, dev)
    ws = torch.zeros(256, dtype=torch.uint8, device=dev)
    out = pa.pa_prefill(kc, vc, pa.to_torch(rw.q, dev), pa.to_torch(rw.query_start, dev),
                        pa.to_torch(w.block_tables, dev), pa.to_torch(w.context_lens, dev), w.max_context_len,
                        w.scale, rw.max_queries, workspace=ws, kernel=kernel)
    torch.cuda.synchronize()
    assert pa.pa_workspace_status(ws) == 0
    got = to_f64(pa.to_numpy(out))
    for (b, r0, n), ref in zip(_LONG_SAMPLES, _long_reference()):
        q0 = int(rw.query_start[b]) + r0
        assert_close(got[q0:q0 + n], ref, "bf16", f"prefill 8 x 2048 after 2048, sequence {b} rows {r0}+{n} ({kernel})")
