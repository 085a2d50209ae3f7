"""pa_decode_noalloc, the decode entry point for callers that cannot allocate
device memory when they call: a plugin inside a host program that owns every
device allocation, or code that must keep the device footprint fixed once it
runs. Its scratch is a fixed array inside the library, so the check here is
that it gives exactly what pa_decode gives with the same kernel and split
plan, call after call, with nothing left over from the previous call's
scratch (GPU).

This file is named to be collected last: if it fails, a run that stops at the
first failure has already run every other test.
"""

import ctypes

import numpy as np
import pytest

pytestmark = pytest.mark.gpu


def _call_c(lib, pa, kc, vc, w, out, split=0, kernel=0):
    """pa_decode_noalloc through the C ABI on the current stream."""
    import torch

    from paged_kv_decode_pa_gb300 import _lib

    cache = pa.make_cache(kc, vc)
    q, tables, ctx = pa.to_torch(w.q), pa.to_torch(w.block_tables), pa.to_torch(w.context_lens)
    opts = _lib.PaOptions(split, kernel, 0)
    status = lib.pa_decode_noalloc(
        ctypes.byref(cache), ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(out.data_ptr()),
        ctypes.c_void_p(tables.data_ptr()), w.max_blocks_per_seq, ctypes.c_void_p(ctx.data_ptr()),
        w.spec.batch, w.spec.q_heads, w.max_context_len, ctypes.c_float(w.scale), ctypes.byref(opts),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    return status


def _reference(pa, kc, vc, w, split=0, kernel="auto"):
    """pa_decode with its own workspace, same kernel and split plan."""
    s = w.spec
    ws = pa.new_workspace(s.batch, 1, s.q_heads, s.kv_heads, w.max_context_len, split_tokens=split)
    out = pa.pa_decode(kc, vc, pa.to_torch(w.q), pa.to_torch(w.block_tables), pa.to_torch(w.context_lens),
                       w.max_context_len, w.scale, ws, split_tokens=split, kernel=kernel)
    assert pa.pa_workspace_status(ws) == 0
    return pa.to_numpy(out)


def test_noalloc_equals_pa_decode_on_two_calls_in_a_row():
    """First a bf16 call whose first sequence has three splits, so its
    log-sum-exp partials land just past a small counter region; then an fp32
    call with more (sequence, KV head) units and an explicit 64-token split,
    whose in-kernel merge counts split arrivals in counters that now cover
    those partials. Without the clear of the counter region between calls the
    second merge would miscount and leave rows unwritten. Both results must
    equal pa_decode's bit for bit."""
    import torch

    import paged_kv_decode_pa_gb300 as pa
    from paged_kv_decode_pa_gb300 import _lib, inputs

    lib = _lib.load()
    calls = (
        (inputs.custom(batch=4, q_heads=12, kv_heads=2, context_lens=(4000, 2049, 1300, 17), num_blocks=512,
                       dtype="bf16", seed=101), 0, _lib.PA_KERNEL_AUTO, "auto"),
        (inputs.custom(batch=64, q_heads=12, kv_heads=2, context_lens=tuple(1 + (37 * i) % 300 for i in range(64)),
                       num_blocks=1400, dtype="f32", seed=202), 64, _lib.PA_KERNEL_SIMT, "simt"),
    )
    for w, split, kernel, kname in calls:
        kc, vc = pa.to_torch(w.k_cache), pa.to_torch(w.v_cache)
        want = _reference(pa, kc, vc, w, split, kname)
        out = torch.full_like(pa.to_torch(w.q), float("nan"))
        status = _call_c(lib, pa, kc, vc, w, out, split, kernel)
        assert status == _lib.PA_OK, pa.pa_status_string(status)
        got = pa.to_numpy(out)
        assert got.tobytes() == want.tobytes(), f"{w.spec.dtype} split {split}: differs from pa_decode"


def test_noalloc_python_binding_with_explicit_split():
    """The Python wrapper passes split_tokens and the kernel through: the
    bf16 tensor-core kernel with several splits per sequence (merge kernel),
    twice in a row, equals pa_decode with the same options bit for bit."""
    import paged_kv_decode_pa_gb300 as pa
    from paged_kv_decode_pa_gb300 import inputs

    for seed in (303, 304):
        w = inputs.custom(batch=6, q_heads=16, kv_heads=8, context_lens=(1, 16, 33, 200, 511, 700), num_blocks=300,
                          dtype="bf16", seed=seed)
        kc, vc = pa.to_torch(w.k_cache), pa.to_torch(w.v_cache)
        want = _reference(pa, kc, vc, w, 128, "mma")
        got = pa.pa_decode_noalloc(kc, vc, pa.to_torch(w.q), pa.to_torch(w.block_tables),
                                   pa.to_torch(w.context_lens), w.max_context_len, w.scale, split_tokens=128,
                                   kernel="mma")
        assert pa.to_numpy(got).tobytes() == want.tobytes()


def test_noalloc_int8_pool_equals_pa_decode():
    """The int8 pool through the wrapper (its K and V scales passed on), with
    a 64-token split so that the merge kernel runs: bit-identical to
    pa_decode with its own workspace."""
    import torch

    import paged_kv_decode_pa_gb300 as pa
    from paged_kv_decode_pa_gb300 import inputs

    w = inputs.custom(batch=5, q_heads=16, kv_heads=8, context_lens=(1, 17, 200, 640, 1025), num_blocks=200,
                      dtype="bf16", seed=404)
    pool = inputs.q8_pool(w)
    kq, vq, ks, vs = (pa.to_torch(a) for a in (pool.k_codes, pool.v_codes, pool.k_scale, pool.v_scale))
    q, tb, ln = pa.to_torch(w.q), pa.to_torch(w.block_tables), pa.to_torch(w.context_lens)
    s = w.spec
    ws = pa.new_workspace(s.batch, 1, s.q_heads, s.kv_heads, w.max_context_len, split_tokens=64)
    want = pa.pa_decode(kq, vq, q, tb, ln, w.max_context_len, w.scale, ws, split_tokens=64, k_scale=ks, v_scale=vs)
    got = pa.pa_decode_noalloc(kq, vq, q, tb, ln, w.max_context_len, w.scale, split_tokens=64, k_scale=ks,
                               v_scale=vs)
    torch.cuda.synchronize()
    assert pa.pa_workspace_status(ws) == 0
    assert pa.to_numpy(got).tobytes() == pa.to_numpy(want).tobytes()


def test_noalloc_rejects_sizes_beyond_its_scratch():
    import torch

    import paged_kv_decode_pa_gb300 as pa
    from paged_kv_decode_pa_gb300 import _lib

    lib = _lib.load()
    kc = torch.zeros((2, 64, 16, 128), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    cache = pa.make_cache(kc, vc)
    batch, max_ctx = 4096, 1 << 16  # needs far more than PA_NOALLOC_SCRATCH_BYTES
    assert pa.pa_workspace_size(batch, 1, 12, 2, max_ctx) > _lib.PA_NOALLOC_SCRATCH_BYTES
    status = lib.pa_decode_noalloc(ctypes.byref(cache), ctypes.c_void_p(16), ctypes.c_void_p(16),
                                   ctypes.c_void_p(16), max_ctx // 16, ctypes.c_void_p(16), batch, 12,
                                   max_ctx, ctypes.c_float(0.1), None, None)
    assert status == _lib.PA_ERR_WORKSPACE
