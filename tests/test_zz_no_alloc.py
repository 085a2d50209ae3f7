"""pa_decode_noalloc, the decode entry point for callers that cannot allocate
device memory when they call (a plugin inside a host program that owns every
device allocation, or code that must keep the device footprint fixed once it
runs). Its scratch is a fixed array inside the library, so the check here is
that it gives what pa_decode gives, call after call, with nothing left over
from the previous call's scratch (GPU).

This file is named to be collected last: if it fails, a run that stops at the
first failure has already run every other test.
"""

import ctypes

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

TOL = (3e-3, 1e-2)  # the bf16 tolerance of the parity tests: |a - b| <= 3e-3 + 1e-2 |b|


def _inputs(lens, seed):
    from paged_kv_decode_pa_gb300 import inputs

    return inputs.custom(batch=len(lens), q_heads=12, kv_heads=2, context_lens=lens, num_blocks=512,
                         dtype="bf16", seed=seed)


def _f64(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def test_noalloc_matches_pa_decode_on_two_calls_in_a_row():
    import torch

    import paged_kv_decode_pa_gb300 as pa
    from paged_kv_decode_pa_gb300 import _lib

    lib = _lib.load()
    # Two different calls: lengths spanning several splits (partials, counters
    # and the merge all live in the scratch), then a different batch shape.
    for lens, seed in (((1, 17, 500, 513, 1300, 2049), 101), ((2048, 16, 900, 3), 202)):
        w = _inputs(lens, seed)
        kc, vc = pa.to_torch(w.k_cache), pa.to_torch(w.v_cache)
        q, tables, ctx = pa.to_torch(w.q), pa.to_torch(w.block_tables), pa.to_torch(w.context_lens)
        ws = pa.new_workspace(len(lens), 1, 12, 2, w.max_context_len)
        ref = pa.pa_decode(kc, vc, q, tables, ctx, w.max_context_len, w.scale, ws)

        cache = pa.make_cache(kc, vc)
        out = torch.full_like(q, float("nan"))
        status = lib.pa_decode_noalloc(
            ctypes.byref(cache), ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(out.data_ptr()),
            ctypes.c_void_p(tables.data_ptr()), w.max_blocks_per_seq, ctypes.c_void_p(ctx.data_ptr()),
            len(lens), 12, w.max_context_len, ctypes.c_float(w.scale), None,
            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert status == _lib.PA_OK, pa.pa_status_string(status)
        torch.cuda.synchronize()
        got, want = _f64(pa.to_numpy(out)), _f64(pa.to_numpy(ref))
        assert np.all(np.isfinite(got))
        assert np.all(np.abs(got - want) <= TOL[0] + TOL[1] * np.abs(want))


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
