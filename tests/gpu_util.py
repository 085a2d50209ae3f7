"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI,
run the oracle on the same seeded inputs, compare."""

from __future__ import annotations

import functools

import numpy as np

import oracle
from paged_kv_decode_pa_gb300 import inputs

# Element-wise tolerance |gpu - ref| <= atol + rtol * |ref|: bf16 (max abs 3e-3,
# rel 1e-2, read in allclose form) and fp32 (1e-5).
TOL = {"bf16": (3e-3, 1e-2), "f32": (1e-5, 1e-5)}


@functools.lru_cache(maxsize=8)
def workload(name: str, **kw):
    return inputs.make(name, **kw) if kw else inputs.make(name)


def to_f64(arr):
    return oracle.to_f64(arr)


def assert_close(got: np.ndarray, ref: np.ndarray, dtype: str, what: str = ""):
    atol, rtol = TOL[dtype]
    assert got.shape == ref.shape
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    excess = np.abs(got - ref) - (atol + rtol * np.abs(ref))
    worst = np.unravel_index(np.argmax(excess), excess.shape)
    assert excess.max() <= 0, (f"{what}: outside tolerance at {worst}: got {got[worst]}, "
                               f"ref {ref[worst]}, max abs err {np.abs(got - ref).max():.3e}")


def gpu_decode(w, kernel="auto", split_tokens=0, write=True, rows=None):
    """Cache write (optional) + pa_decode on the device; returns (out f64, k, v) on the host."""
    import torch

    import paged_kv_decode_pa_gb300 as pa

    dev = torch.device("cuda")
    sel = slice(None) if rows is None else rows
    kc, vc = pa.to_torch(w.k_cache, dev), pa.to_torch(w.v_cache, dev)
    if write:
        pa.pa_cache_write(kc, vc, pa.to_torch(w.k_new, dev), pa.to_torch(w.v_new, dev),
                          pa.to_torch(w.slot_mapping, dev))
    q = np.ascontiguousarray(w.q[sel])
    tables = np.ascontiguousarray(w.block_tables[sel])
    lens = np.ascontiguousarray(w.context_lens[sel])
    batch, hq = q.shape[0], q.shape[1]
    ws = pa.new_workspace(batch, 1, hq, w.spec.kv_heads, w.max_context_len, dev, split_tokens)
    out = pa.pa_decode(kc, vc, pa.to_torch(q, dev), pa.to_torch(tables, dev), pa.to_torch(lens, dev),
                       w.max_context_len, w.scale, ws, split_tokens=split_tokens, kernel=kernel)
    torch.cuda.synchronize()
    status = pa.pa_workspace_status(ws)
    assert status == 0, f"device status flags {status:#x}"
    return pa.to_numpy(out), pa.to_numpy(kc), pa.to_numpy(vc)


def gpu_verify(w, kernel="auto", split_tokens=0):
    import torch

    import paged_kv_decode_pa_gb300 as pa

    dev = torch.device("cuda")
    kc, vc = pa.to_torch(w.k_cache, dev), pa.to_torch(w.v_cache, dev)
    batch, nq, hq, _ = w.q.shape
    ws = pa.new_workspace(batch, nq, hq, w.spec.kv_heads, w.max_context_len, dev, split_tokens)
    out = pa.pa_verify(kc, vc, pa.to_torch(w.q, dev), pa.to_torch(w.k_new, dev),
                       pa.to_torch(w.v_new, dev), pa.to_torch(w.slot_mapping, dev),
                       pa.to_torch(w.block_tables, dev), pa.to_torch(w.context_lens, dev),
                       w.max_context_len, w.scale, ws, split_tokens=split_tokens, kernel=kernel)
    torch.cuda.synchronize()
    status = pa.pa_workspace_status(ws)
    assert status == 0, f"device status flags {status:#x}"
    return pa.to_numpy(out), pa.to_numpy(kc), pa.to_numpy(vc)


@functools.lru_cache(maxsize=8)
def oracle_decode(name: str, **kw):
    """(reference output, caches after the write) for a standard workload."""
    w = workload(name, **kw)
    kc, vc = w.k_cache.copy(), w.v_cache.copy()
    assert oracle.cache_write(kc, vc, w.k_new, w.v_new, w.slot_mapping) == 0
    return oracle.decode(kc, vc, w.q, w.block_tables, w.context_lens, w.scale), kc, vc


def oracle_verify_of(w):
    kc, vc = w.k_cache.copy(), w.v_cache.copy()
    ref = oracle.verify(kc, vc, w.q, w.k_new, w.v_new, w.slot_mapping, w.block_tables,
                        w.context_lens, w.scale)
    return ref, kc, vc
