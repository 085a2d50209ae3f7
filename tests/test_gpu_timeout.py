"""The bounded-wait path of the TMA kernels (GPU).

Every wait of a kernel's pipeline is bounded (pa_options.wait_limit_ns): one
that runs past its bound raises PA_FLAG_TIMEOUT, the CTA lets its own copies in
flight land and returns without writing its rows. Here the bound is set to 1 ns,
so the first wait that does not find its stage ready gives up: the call must
still return, raise the flag, and leave the device usable; the next call with
the default bound (on a re-initialised workspace) must match the oracle with
no flag raised. Nothing here faults or hangs the GPU: the waits give up on
their own and the copies they leave behind are drained under the default
bound.
"""

from __future__ import annotations

import pytest

import oracle
from gpu_util import assert_close, to_f64, workload
from paged_kv_decode_pa_gb300 import _lib, inputs

pytestmark = pytest.mark.gpu

TINY = 1  # ns


def _timed_out(ws):
    import paged_kv_decode_pa_gb300 as pa

    flags = pa.pa_workspace_status(ws)
    return flags & _lib.PA_FLAG_TIMEOUT


@pytest.mark.parametrize("name", ["c3", "c5"])
def test_bf16_pipeline_wait_gives_up_then_next_call_is_clean(name):
    """Fused append + decode (c3) and the k+1-token verify (c5) at full size."""
    import torch

    import paged_kv_decode_pa_gb300 as pa

    w = workload(name)
    q4 = w.q if w.q.ndim == 4 else w.q[:, None]
    batch, nq, hq, _ = q4.shape
    args = (pa.to_torch(q4), pa.to_torch(w.k_new), pa.to_torch(w.v_new), pa.to_torch(w.slot_mapping),
            pa.to_torch(w.block_tables), pa.to_torch(w.context_lens), w.max_context_len, w.scale)
    ws = pa.new_workspace(batch, nq, hq, w.spec.kv_heads, w.max_context_len)

    kc, vc = pa.to_torch(w.k_cache), pa.to_torch(w.v_cache)
    pa.pa_verify(kc, vc, *args, ws, wait_limit_ns=TINY)
    torch.cuda.synchronize()
    assert _timed_out(ws), "a 1 ns bound must make some wait give up"

    pa.pa_workspace_init(ws)
    kc, vc = pa.to_torch(w.k_cache), pa.to_torch(w.v_cache)
    out = pa.pa_verify(kc, vc, *args, ws)
    torch.cuda.synchronize()
    assert pa.pa_workspace_status(ws) == 0
    okc, ovc = w.k_cache.copy(), w.v_cache.copy()
    ref = oracle.verify(okc, ovc, q4, w.k_new, w.v_new, w.slot_mapping, w.block_tables, w.context_lens, w.scale)
    assert_close(to_f64(pa.to_numpy(out)), ref, "bf16", f"{name} after a timed-out call")
    assert pa.to_numpy(kc).tobytes() == okc.tobytes() and pa.to_numpy(vc).tobytes() == ovc.tobytes()


def test_bf16_long_context_split_merge_gives_up_then_next_call_is_clean():
    """The 32k-context decode: many splits per sequence and the merge kernel
    behind the attention grid."""
    import torch

    import paged_kv_decode_pa_gb300 as pa

    w = workload("c4")
    kc, vc = pa.to_torch(w.k_cache), pa.to_torch(w.v_cache)
    q, tb, ln = pa.to_torch(w.q), pa.to_torch(w.block_tables), pa.to_torch(w.context_lens)
    ws = pa.new_workspace(w.spec.batch, 1, w.spec.q_heads, w.spec.kv_heads, w.max_context_len)
    pa.pa_decode(kc, vc, q, tb, ln, w.max_context_len, w.scale, ws, wait_limit_ns=TINY)
    torch.cuda.synchronize()
    assert _timed_out(ws)
    pa.pa_workspace_init(ws)
    out = pa.pa_decode(kc, vc, q, tb, ln, w.max_context_len, w.scale, ws)
    torch.cuda.synchronize()
    assert pa.pa_workspace_status(ws) == 0
    ref = oracle.decode(w.k_cache, w.v_cache, w.q, w.block_tables, w.context_lens, w.scale)
    assert_close(to_f64(pa.to_numpy(out)), ref, "bf16", "c4 after a timed-out call")


def test_int8_pipeline_wait_gives_up_then_next_call_is_clean():
    """The int8 pool's kernel (c3 shape, decode)."""
    import torch

    import paged_kv_decode_pa_gb300 as pa

    w = workload("c3")
    pool = inputs.q8_pool(w)
    kq, vq, ks, vs = (pa.to_torch(a) for a in (pool.k_codes, pool.v_codes, pool.k_scale, pool.v_scale))
    q, tb, ln = pa.to_torch(w.q), pa.to_torch(w.block_tables), pa.to_torch(w.context_lens)
    ws = pa.new_workspace(w.spec.batch, 1, w.spec.q_heads, w.spec.kv_heads, w.max_context_len)
    pa.pa_decode(kq, vq, q, tb, ln, w.max_context_len, w.scale, ws, k_scale=ks, v_scale=vs, wait_limit_ns=TINY)
    torch.cuda.synchronize()
    assert _timed_out(ws)
    pa.pa_workspace_init(ws)
    out = pa.pa_decode(kq, vq, q, tb, ln, w.max_context_len, w.scale, ws, k_scale=ks, v_scale=vs)
    torch.cuda.synchronize()
    assert pa.pa_workspace_status(ws) == 0
    ref = oracle.decode_q8(pool.k_codes, pool.v_codes, pool.k_scale, pool.v_scale, w.q, w.block_tables,
                           w.context_lens, w.scale)
    assert_close(to_f64(pa.to_numpy(out)), ref, "bf16", "int8 c3 after a timed-out call")


def test_prefill_tensor_memory_kernel_gives_up_then_next_call_is_clean():
    """The tcgen05 prefill: on giving up it drains its loads and its products
    and frees its tensor memory, so the next call (whose CTAs allocate tensor
    memory on the same SMs) runs normally."""
    import torch

    import paged_kv_decode_pa_gb300 as pa

    w = inputs.custom(batch=64, q_heads=16, kv_heads=8, context_lens=(256,) * 64, num_blocks=1100, seed=51,
                      num_queries=256)
    rw = inputs.ragged(w, [256] * 64)
    kc, vc = pa.to_torch(w.k_cache), pa.to_torch(w.v_cache)
    q, qs = pa.to_torch(rw.q), pa.to_torch(rw.query_start)
    tb, ln = pa.to_torch(w.block_tables), pa.to_torch(w.context_lens)
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    pa.pa_prefill(kc, vc, q, qs, tb, ln, w.max_context_len, w.scale, rw.max_queries, workspace=ws, kernel="tc",
                  wait_limit_ns=TINY)
    torch.cuda.synchronize()
    assert _timed_out(ws)
    out = pa.pa_prefill(kc, vc, q, qs, tb, ln, w.max_context_len, w.scale, rw.max_queries, workspace=ws,
                        kernel="tc")
    torch.cuda.synchronize()
    assert pa.pa_workspace_status(ws) == 0
    ref = oracle.attend_ragged(w.k_cache, w.v_cache, rw.q, rw.query_start, w.block_tables, w.context_lens, w.scale)
    assert_close(to_f64(pa.to_numpy(out)), ref, "bf16", "prefill after a timed-out call")
