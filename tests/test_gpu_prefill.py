"""pa_prefill (causal attention of prompt chunks over the paged cache) against
the oracle, bf16."""

from __future__ import annotations

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
@pytest.mark.parametrize("hq,hkv", [(16, 8), (12, 2), (32, 4), (8, 8)])
def test_prefill_chunks_with_prefixes(hq, hkv, kernel):
    """Chunks after prefixes of several lengths: tiles of 128 rows, ragged tails,
    chunk sizes 1 .. 300, context ends inside and at block edges."""
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
