"""Python binding of libpa: the C entry points under the same names, taking torch tensors.

Argument marshalling only. Every operation runs in libpa's CUDA kernels on the
caller's current CUDA stream (or the one passed). PyTorch provides device
memory and streams; nothing here computes attention.
"""

from __future__ import annotations

import ctypes
import functools
from typing import Optional

import numpy as np
import torch

from . import _lib as L

_DTYPES = {torch.bfloat16: L.PA_DTYPE_BF16, torch.float32: L.PA_DTYPE_F32, torch.uint8: L.PA_DTYPE_INT8}
_KERNELS = {"auto": L.PA_KERNEL_AUTO, "mma": L.PA_KERNEL_MMA, "simt": L.PA_KERNEL_SIMT, "tc": L.PA_KERNEL_TC}


def _vp(t: Optional[torch.Tensor]):
    """Device address as a plain int (ctypes converts it for void* parameters)."""
    return t.data_ptr() if t is not None else None


# The current stream's raw handle without building a torch Stream object, which
# costs a few microseconds per call; the public accessor is the fallback.
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream: Optional[torch.cuda.Stream]):
    if stream is not None:
        return stream.cuda_stream
    if _raw_stream is not None:
        return _raw_stream(torch.cuda.current_device())
    return torch.cuda.current_stream().cuda_stream


def _need(cond: bool, msg: str):
    if not cond:
        raise ValueError(msg)


def make_cache(k_cache: torch.Tensor, v_cache: torch.Tensor, k_scale: Optional[torch.Tensor] = None,
               v_scale: Optional[torch.Tensor] = None) -> L.PaCache:
    """Describe two head-major pools [kv_heads, num_blocks, block_size, head_dim].

    bf16 or fp32 pools hold values. uint8 pools are the int8 format (bytes
    value + 128) and need fp32 scales: k_scale [kv_heads, num_blocks, head_dim]
    and v_scale [kv_heads, num_blocks, block_size].
    """
    _need(k_cache.shape == v_cache.shape and k_cache.dim() == 4, "caches must be equal 4-D tensors")
    _need(k_cache.dtype == v_cache.dtype and k_cache.dtype in _DTYPES, "cache dtype must be bf16, fp32 or uint8")
    _need(k_cache.is_cuda and v_cache.is_cuda, "caches must be CUDA tensors")
    _need(k_cache.is_contiguous() and v_cache.is_contiguous(), "caches must be contiguous")
    hkv, nb, bs, d = k_cache.shape
    dt = _DTYPES[k_cache.dtype]
    if dt != L.PA_DTYPE_INT8:
        return L.PaCache(k_cache.data_ptr(), v_cache.data_ptr(), hkv, nb, bs, d, dt, None, None)
    _need(k_scale is not None and v_scale is not None, "an int8 pool needs k_scale and v_scale")
    _need(k_scale.dtype == torch.float32 and v_scale.dtype == torch.float32, "scales must be fp32")
    _need(tuple(k_scale.shape) == (hkv, nb, d) and tuple(v_scale.shape) == (hkv, nb, bs),
          "k_scale must be [kv_heads, num_blocks, head_dim], v_scale [kv_heads, num_blocks, block_size]")
    _need(k_scale.is_cuda and v_scale.is_cuda and k_scale.is_contiguous() and v_scale.is_contiguous(),
          "scales must be contiguous CUDA tensors")
    return L.PaCache(k_cache.data_ptr(), v_cache.data_ptr(), hkv, nb, bs, d, dt, k_scale.data_ptr(),
                     v_scale.data_ptr())


def _row_dtype(k_cache: torch.Tensor):
    """dtype of queries, new rows and outputs for this pool (bf16 for int8)."""
    return torch.bfloat16 if k_cache.dtype == torch.uint8 else k_cache.dtype


@functools.lru_cache(maxsize=64)
def _options(split_tokens: int, kernel: str, wait_limit_ns: int = 0) -> L.PaOptions:
    """Options struct for these values (cached: libpa only reads it)."""
    return L.PaOptions(int(split_tokens), _KERNELS[kernel], int(wait_limit_ns))


def pa_workspace_size(batch: int, num_queries: int, q_heads: int, kv_heads: int,
                      max_context_len: int, split_tokens: int = 0, head_dim: int = 128) -> int:
    opts = _options(split_tokens, "auto")
    n = L.load().pa_workspace_size(batch, num_queries, q_heads, kv_heads, head_dim,
                                   max_context_len, ctypes.byref(opts))
    if n == 0:
        raise ValueError("pa_workspace_size: invalid sizes")
    return int(n)


def pa_workspace_init(workspace: torch.Tensor, stream=None) -> None:
    L.check("pa_workspace_init", L.load().pa_workspace_init(
        _vp(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))


def new_workspace(batch: int, num_queries: int, q_heads: int, kv_heads: int, max_context_len: int,
                  device="cuda", split_tokens: int = 0, stream=None) -> torch.Tensor:
    """Allocate (torch) and zero (libpa) a workspace for these sizes."""
    n = pa_workspace_size(batch, num_queries, q_heads, kv_heads, max_context_len, split_tokens)
    ws = torch.empty(n, dtype=torch.uint8, device=device)
    pa_workspace_init(ws, stream)
    return ws


def pa_workspace_status(workspace: torch.Tensor, stream=None) -> int:
    """Read and clear the PA_FLAG_* status word (synchronises the stream)."""
    flags = ctypes.c_uint32(0)
    L.check("pa_workspace_status", L.load().pa_workspace_status(
        _vp(workspace), ctypes.byref(flags), _stream(stream)))
    return int(flags.value)


def pa_cache_write(k_cache, v_cache, k_new, v_new, slot_mapping, stream=None, k_scale=None,
                   v_scale=None) -> None:
    cache = make_cache(k_cache, v_cache, k_scale, v_scale)
    n = int(slot_mapping.shape[0])
    _need(slot_mapping.dtype == torch.int32, "slot_mapping must be int32")
    rd = _row_dtype(k_cache)
    _need(k_new.dtype == rd and v_new.dtype == rd, "new rows must match the cache dtype (bf16 for int8)")
    _need(tuple(k_new.shape) == (n, cache.kv_heads, cache.head_dim) and k_new.shape == v_new.shape,
          "new rows must be [num_tokens, kv_heads, head_dim]")
    _need(k_new.is_contiguous() and v_new.is_contiguous() and slot_mapping.is_contiguous(),
          "inputs must be contiguous")
    L.check("pa_cache_write", L.load().pa_cache_write(
        ctypes.byref(cache), _vp(k_new), _vp(v_new), _vp(slot_mapping), n, _stream(stream)))


def _tables(block_tables, context_lens, batch):
    _need(block_tables.dtype == torch.int32 and context_lens.dtype == torch.int32,
          "block_tables and context_lens must be int32")
    _need(block_tables.dim() == 2 and block_tables.shape[0] == batch, "block_tables must be [batch, mbps]")
    _need(tuple(context_lens.shape) == (batch,), "context_lens must be [batch]")
    _need(block_tables.is_contiguous() and context_lens.is_contiguous(), "tables must be contiguous")
    return int(block_tables.shape[1])


def pa_decode(k_cache, v_cache, q, block_tables, context_lens, max_context_len: int, scale: float,
              workspace, out=None, split_tokens: int = 0, kernel: str = "auto", stream=None,
              k_scale=None, v_scale=None, wait_limit_ns: int = 0):
    """out[b, hq] = softmax(scale * q[b, hq] . K_b^T) V_b over sequence b's paged context.

    wait_limit_ns: bound on each device-side pipeline wait (0: one second);
    a wait past it raises PA_FLAG_TIMEOUT in the workspace status word."""
    cache = make_cache(k_cache, v_cache, k_scale, v_scale)
    _need(q.dim() == 3 and q.dtype == _row_dtype(k_cache) and q.is_contiguous(),
          "q must be [batch, q_heads, head_dim] of the row dtype")
    batch, q_heads, _ = q.shape
    mbps = _tables(block_tables, context_lens, batch)
    if out is None:
        out = torch.empty_like(q)
    opts = _options(split_tokens, kernel, wait_limit_ns)
    L.check("pa_decode", L.load().pa_decode(
        ctypes.byref(cache), _vp(q), _vp(out), _vp(block_tables), mbps, _vp(context_lens), batch,
        q_heads, int(max_context_len), float(scale), _vp(workspace),
        workspace.numel() * workspace.element_size(), ctypes.byref(opts), _stream(stream)))
    return out


def pa_decode_noalloc(k_cache, v_cache, q, block_tables, context_lens, max_context_len: int,
                      scale: float, out=None, split_tokens: int = 0, kernel: str = "auto", stream=None,
                      k_scale=None, v_scale=None):
    """pa_decode without a caller workspace, for callers that cannot allocate device memory.

    The scratch is a fixed library-owned device array (PA_NOALLOC_SCRATCH_BYTES);
    overlapping calls on the GPU race on it. Only ``out`` may be allocated here,
    and only when it is not passed.
    """
    cache = make_cache(k_cache, v_cache, k_scale, v_scale)
    _need(q.dim() == 3 and q.dtype == _row_dtype(k_cache) and q.is_contiguous(),
          "q must be [batch, q_heads, head_dim] of the row dtype")
    batch, q_heads, _ = q.shape
    mbps = _tables(block_tables, context_lens, batch)
    if out is None:
        out = torch.empty_like(q)
    opts = _options(split_tokens, kernel)
    L.check("pa_decode_noalloc", L.load().pa_decode_noalloc(
        ctypes.byref(cache), _vp(q), _vp(out), _vp(block_tables), mbps, _vp(context_lens), batch,
        q_heads, int(max_context_len), float(scale), ctypes.byref(opts), _stream(stream)))
    return out


def pa_verify(k_cache, v_cache, q, k_new, v_new, slot_mapping, block_tables, context_lens,
              max_context_len: int, scale: float, workspace, out=None, split_tokens: int = 0,
              kernel: str = "auto", stream=None, k_scale=None, v_scale=None, wait_limit_ns: int = 0):
    """Fused speculative verify: write the new K/V, attend causally. q: [batch, nq, q_heads, head_dim]."""
    cache = make_cache(k_cache, v_cache, k_scale, v_scale)
    _need(q.dim() == 4 and q.dtype == _row_dtype(k_cache) and q.is_contiguous(),
          "q must be [batch, num_queries, q_heads, head_dim]")
    batch, nq, q_heads, _ = q.shape
    mbps = _tables(block_tables, context_lens, batch)
    _need(slot_mapping.dtype == torch.int32 and tuple(slot_mapping.shape) == (batch * nq,),
          "slot_mapping must be int32 [batch * num_queries]")
    _need(tuple(k_new.shape) == (batch * nq, cache.kv_heads, cache.head_dim) and k_new.shape == v_new.shape
          and k_new.dtype == q.dtype and v_new.dtype == q.dtype,
          "new rows must be [batch * num_queries, kv_heads, head_dim] of the cache dtype")
    if out is None:
        out = torch.empty_like(q)
    opts = _options(split_tokens, kernel, wait_limit_ns)
    L.check("pa_verify", L.load().pa_verify(
        ctypes.byref(cache), _vp(q), _vp(out), _vp(k_new), _vp(v_new), _vp(slot_mapping), nq,
        _vp(block_tables), mbps, _vp(context_lens), batch, q_heads, int(max_context_len),
        float(scale), _vp(workspace), workspace.numel() * workspace.element_size(),
        ctypes.byref(opts), _stream(stream)))
    return out


def pa_verify_ragged(k_cache, v_cache, q, k_new, v_new, slot_mapping, query_start, block_tables,
                     context_lens, max_context_len: int, scale: float, workspace, max_queries: int,
                     out=None, split_tokens: int = 0, kernel: str = "auto", stream=None, k_scale=None,
                     v_scale=None, wait_limit_ns: int = 0):
    """Verify with a different number of new tokens per sequence, in one launch.

    q: [total, q_heads, head_dim]; sequence b owns rows query_start[b] ..
    query_start[b+1] - 1 (int32 [batch + 1] on the device); max_queries bounds
    every sequence's count (the workspace is sized with it as num_queries).
    """
    cache = make_cache(k_cache, v_cache, k_scale, v_scale)
    _need(q.dim() == 3 and q.dtype == _row_dtype(k_cache) and q.is_contiguous(),
          "q must be [total_queries, q_heads, head_dim] of the row dtype")
    total, q_heads, _ = q.shape
    batch = int(context_lens.shape[0])
    mbps = _tables(block_tables, context_lens, batch)
    _need(query_start.dtype == torch.int32 and query_start.shape == (batch + 1,) and query_start.is_contiguous(),
          "query_start must be int32 [batch + 1]")
    _need(slot_mapping.dtype == torch.int32 and slot_mapping.shape == (total,), "slot_mapping must be int32 [total]")
    _need(k_new.shape == (total, cache.kv_heads, cache.head_dim) and k_new.shape == v_new.shape
          and k_new.dtype == q.dtype and v_new.dtype == q.dtype,
          "new rows must be [total_queries, kv_heads, head_dim] of the row dtype")
    if out is None:
        out = torch.empty_like(q)
    opts = _options(split_tokens, kernel, wait_limit_ns)
    L.check("pa_verify_ragged", L.load().pa_verify_ragged(
        ctypes.byref(cache), _vp(q), _vp(out), _vp(k_new), _vp(v_new), _vp(slot_mapping), _vp(query_start),
        total, int(max_queries), _vp(block_tables), mbps, _vp(context_lens), batch, q_heads,
        int(max_context_len), float(scale), _vp(workspace), workspace.numel() * workspace.element_size(),
        ctypes.byref(opts), _stream(stream)))
    return out


def pa_prefill(k_cache, v_cache, q, query_start, block_tables, context_lens, max_context_len: int,
               scale: float, max_queries: int, out=None, workspace=None, stream=None, kernel: str = "auto",
               wait_limit_ns: int = 0):
    """Causal attention of each sequence's prompt chunk (its last n_b positions,
    already in the cache) over its paged context. q: [total, q_heads, head_dim]
    bf16; query_start: int32 [batch + 1]. workspace (optional) receives the
    status word. kernel: "auto" / "tc" (tcgen05) or "mma" (warp-level)."""
    cache = make_cache(k_cache, v_cache)
    _need(q.dim() == 3 and q.dtype == k_cache.dtype and q.is_contiguous(),
          "q must be [total_queries, q_heads, head_dim] of the cache dtype")
    total, q_heads, _ = q.shape
    batch = int(context_lens.shape[0])
    mbps = _tables(block_tables, context_lens, batch)
    _need(query_start.dtype == torch.int32 and query_start.shape == (batch + 1,) and query_start.is_contiguous(),
          "query_start must be int32 [batch + 1]")
    if out is None:
        out = torch.empty_like(q)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    L.check("pa_prefill", L.load().pa_prefill(
        ctypes.byref(cache), _vp(q), _vp(out), _vp(query_start), total, int(max_queries), _vp(block_tables),
        mbps, _vp(context_lens), batch, q_heads, int(max_context_len), float(scale), _vp(workspace), ws_bytes,
        ctypes.byref(_options(0, kernel, wait_limit_ns)), _stream(stream)))
    return out


def pa_validate(k_cache, v_cache, block_tables, context_lens, max_context_len: int,
                slot_mapping=None, num_queries: int = 1, report=None, stream=None, k_scale=None,
                v_scale=None):
    """Device check of tables, lengths and slots; returns the 4-word report tensor (int32 view)."""
    cache = make_cache(k_cache, v_cache, k_scale, v_scale)
    batch = int(context_lens.shape[0])
    mbps = _tables(block_tables, context_lens, batch)
    if report is None:
        report = torch.zeros(L.PA_VALIDATE_WORDS, dtype=torch.int32, device=k_cache.device)
    L.check("pa_validate", L.load().pa_validate(
        ctypes.byref(cache), _vp(block_tables), mbps, _vp(context_lens), batch, int(max_context_len),
        _vp(slot_mapping), int(num_queries), _vp(report), _stream(stream)))
    return report


def pa_status_string(status: int) -> str:
    return L.load().pa_status_string(int(status)).decode()


def pa_version() -> int:
    return int(L.load().pa_version())


def to_torch(arr: np.ndarray, device="cuda") -> torch.Tensor:
    """Copy a host array to the device; uint16 arrays are bf16 bit patterns."""
    if arr.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(arr).view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(np.ascontiguousarray(arr)).to(device)


def to_numpy(t: torch.Tensor) -> np.ndarray:
    """Copy a device tensor to the host; bf16 comes back as uint16 bit patterns."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()
