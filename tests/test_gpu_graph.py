"""The calls are CUDA-graph capturable: the grid depends on host arguments only,
and a replay after the inputs change in place gives the oracle's answer for the
new inputs (the engine pattern of one graph per batch bucket with fixed buffers)."""

from __future__ import annotations

import numpy as np
import pytest

import oracle
from gpu_util import assert_close, to_f64
from paged_kv_decode_pa_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,split", [("c5", 0), ("c2", 64)])
def test_graph_replay_tracks_inputs(name, split):
    import torch

    import paged_kv_decode_pa_gb300 as pa

    over = {"batch": 8, "num_blocks": 1024} if name == "c5" else {"batch": 8, "num_blocks": 512}
    w = inputs.make(name, **over)
    dev = torch.device("cuda")
    q_np = w.q if w.q.ndim == 4 else w.q[:, None]
    kc, vc = pa.to_torch(w.k_cache, dev), pa.to_torch(w.v_cache, dev)
    q = pa.to_torch(q_np, dev)
    kn, vn = pa.to_torch(w.k_new, dev), pa.to_torch(w.v_new, dev)
    slots, tables, lens = (pa.to_torch(w.slot_mapping, dev), pa.to_torch(w.block_tables, dev),
                           pa.to_torch(w.context_lens, dev))
    batch, nq, hq, _ = q.shape
    ws = pa.new_workspace(batch, nq, hq, w.spec.kv_heads, w.max_context_len, dev, split)
    out = torch.empty_like(q)

    def call():
        pa.pa_verify(kc, vc, q, kn, vn, slots, tables, lens, w.max_context_len, w.scale, ws, out=out,
                     split_tokens=split)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        call()
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()

    rng = np.random.default_rng(77)
    for trial in range(2):
        # New queries, new K/V rows and shorter lengths, written into the captured buffers.
        q2 = inputs.f32_to_bf16_bits(rng.standard_normal(q_np.shape).astype(np.float32))
        kn2 = inputs.f32_to_bf16_bits(rng.standard_normal(w.k_new.shape).astype(np.float32))
        vn2 = inputs.f32_to_bf16_bits(rng.standard_normal(w.v_new.shape).astype(np.float32))
        lens2 = w.context_lens.copy()
        if trial == 1:
            lens2 = np.maximum(lens2 - 3 * nq, nq).astype(np.int32)
        # Slots follow the lengths (position L - nq + i of each sequence).
        slots2 = inputs.slots_for(w.block_tables, lens2, nq)
        q.copy_(pa.to_torch(q2, dev))
        kn.copy_(pa.to_torch(kn2, dev))
        vn.copy_(pa.to_torch(vn2, dev))
        lens.copy_(pa.to_torch(lens2, dev))
        slots.copy_(pa.to_torch(slots2, dev))
        kc.copy_(pa.to_torch(w.k_cache, dev))
        vc.copy_(pa.to_torch(w.v_cache, dev))
        g.replay()
        torch.cuda.synchronize()
        assert pa.pa_workspace_status(ws) == 0
        kc0, vc0 = w.k_cache.copy(), w.v_cache.copy()
        ref = oracle.verify(kc0, vc0, q2, kn2, vn2, slots2, w.block_tables, lens2, w.scale)
        got = pa.to_numpy(out)
        assert_close(to_f64(got), ref, "bf16", f"{name} graph replay {trial}")
        assert np.array_equal(pa.to_numpy(kc), kc0) and np.array_equal(pa.to_numpy(vc), vc0)


@pytest.mark.parametrize("batch", [1, 8, 64])
def test_bucket_graph_write_then_decode(batch):
    """One graph per batch bucket: pa_cache_write + pa_decode captured over fixed
    buffers and replayed; the replay matches the oracle's write-then-decode."""
    import torch

    import paged_kv_decode_pa_gb300 as pa

    w = inputs.make("c2", batch=batch, num_blocks=max(4096, batch * 40))
    dev = torch.device("cuda")
    kc, vc = pa.to_torch(w.k_cache, dev), pa.to_torch(w.v_cache, dev)
    q, kn, vn = pa.to_torch(w.q, dev), pa.to_torch(w.k_new, dev), pa.to_torch(w.v_new, dev)
    slots, tables, lens = (pa.to_torch(w.slot_mapping, dev), pa.to_torch(w.block_tables, dev),
                           pa.to_torch(w.context_lens, dev))
    ws = pa.new_workspace(batch, 1, w.spec.q_heads, w.spec.kv_heads, w.max_context_len, dev)
    out = torch.empty_like(q)

    def step():
        pa.pa_cache_write(kc, vc, kn, vn, slots)
        pa.pa_decode(kc, vc, q, tables, lens, w.max_context_len, w.scale, ws, out=out)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    kc.copy_(pa.to_torch(w.k_cache, dev))
    vc.copy_(pa.to_torch(w.v_cache, dev))
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert pa.pa_workspace_status(ws) == 0
    rk, rv = w.k_cache.copy(), w.v_cache.copy()
    assert oracle.cache_write(rk, rv, w.k_new, w.v_new, w.slot_mapping) == 0
    ref = oracle.decode(rk, rv, w.q, w.block_tables, w.context_lens, w.scale)
    assert_close(to_f64(pa.to_numpy(out)), ref, "bf16", f"bucket {batch}")
    assert np.array_equal(pa.to_numpy(kc), rk) and np.array_equal(pa.to_numpy(vc), rv)
