"""fp64 CPU oracle for paged-KV decode attention (TEST INFRASTRUCTURE).

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU
baseline leg may import this package. The product library never does, and this
package imports nothing from the product package: the two share no code. Inputs
come from the seeded generators, which hold none of the method's arithmetic.

The arithmetic lives in ``pa_oracle.c`` (plain C, double precision, one
contiguous gather per sequence followed by dense masked attention). Each
function there cites the passage of the pages it follows:

* the head-major cache layout and the per-step slot / block-table / length
  inputs: "From 183 ms to 19 ms per decode step", sections "2. Head-major KV
  cache" and "4. CUDA graphs per batch bucket";
* write-then-attend order and the plain softmax row: "Anatomy of a
  Decode-Step Stall", the engine's ``Model._layer``;
* grouped-query mapping: "From 183 ms to 19 ms per decode step", section
  "1. Grouped attention"; repeat_kv in "A Rust inference server for Qwen2 on
  Apple Silicon", Day 3;
* the causal verify rows: "From 183 ms to 19 ms per decode step", section
  "Then speculative decoding got slower".

Pins (tests/test_oracle.py) tie it to things other than itself: a pure-Python
brute force, torch's float64 scaled_dot_product_attention, one-hot and
constant value matrices (closed forms), single-token contexts, block-id
permutation invariance and a numpy fancy-index scatter for the cache write.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import sys
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent
_SRC = _HERE / "pa_oracle.c"
_LIB_DIR = _HERE / "_build"
_LIB = _LIB_DIR / "liboracle.so"

F32 = 0
BF16 = 1


def compile_oracle(src: Path, out: Path) -> Path:
    """Compile one oracle C source into a shared library with gcc (plain -O2, no fast-math,
    no fused multiply-add contraction: the int8 quantiser's fp32 steps stay IEEE-exact)."""
    out = Path(out)
    out.parent.mkdir(parents=True, exist_ok=True)
    tmp = out.with_name(out.name + f".tmp{os.getpid()}")
    cmd = ["gcc", "-O2", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared", "-std=c11",
           "-o", str(tmp), str(src), "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> Path:
    """Compile the C oracle into ``oracle/_build/liboracle.so`` (skipped when up to date)."""
    if _LIB.exists() and not force and _LIB.stat().st_mtime >= _SRC.stat().st_mtime:
        return _LIB
    return compile_oracle(_SRC, _LIB)


class Oracle:
    """ctypes binding of one compiled copy of ``pa_oracle.c``."""

    def __init__(self, lib_path: Path):
        lib = ctypes.CDLL(str(lib_path))
        i32, vp = ctypes.c_int, ctypes.c_void_p
        lib.oracle_cache_write.restype = i32
        lib.oracle_cache_write.argtypes = [vp, vp, i32, i32, i32, i32, i32, vp, vp, vp, i32]
        lib.oracle_attend.restype = i32
        lib.oracle_attend.argtypes = [vp, vp, i32, i32, i32, i32, i32, vp, vp, vp, i32, vp,
                                      i32, i32, i32, ctypes.c_double, i32, i32]
        lib.oracle_cache_write_q8.restype = i32
        lib.oracle_cache_write_q8.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, vp, vp, vp, i32]
        lib.oracle_dequant_q8.restype = None
        lib.oracle_dequant_q8.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, vp, vp]
        lib.oracle_max_threads.restype = i32
        lib.oracle_set_threads.argtypes = [i32]
        self.lib = lib
        self.path = Path(lib_path)

    def set_threads(self, n: int) -> None:
        self.lib.oracle_set_threads(int(n))

    def max_threads(self) -> int:
        return int(self.lib.oracle_max_threads())

    def cache_write(self, k_cache: np.ndarray, v_cache: np.ndarray, k_new: np.ndarray,
                    v_new: np.ndarray, slot_mapping: np.ndarray) -> int:
        """In place: cache[h, s // bs, s % bs, :] = new[i, h, :] for s = slot_mapping[i] >= 0.

        Caches are [kv_heads, num_blocks, block_size, head_dim]; new rows are
        [num_tokens, kv_heads, head_dim]. Returns the count of out-of-range slots.
        """
        code = _dtype_code(k_cache)
        hkv, nb, bs, d = k_cache.shape
        assert v_cache.shape == k_cache.shape and v_cache.dtype == k_cache.dtype
        assert k_new.dtype == k_cache.dtype and v_new.dtype == k_cache.dtype
        n = int(slot_mapping.shape[0])
        assert k_new.shape == (n, hkv, d) and v_new.shape == (n, hkv, d)
        slots = np.ascontiguousarray(slot_mapping, dtype=np.int32)
        return int(self.lib.oracle_cache_write(_ptr(k_cache), _ptr(v_cache), code, hkv, nb, bs, d,
                                               _ptr(np.ascontiguousarray(k_new)),
                                               _ptr(np.ascontiguousarray(v_new)), _ptr(slots), n))

    def attend(self, k_cache: np.ndarray, v_cache: np.ndarray, q: np.ndarray,
               block_tables: np.ndarray, context_lens: np.ndarray, scale: float,
               b_range: tuple[int, int] | None = None) -> np.ndarray:
        """Dense masked GQA attention per sequence, in float64.

        q is [batch, num_queries, q_heads, head_dim] (a decode q of shape
        [batch, q_heads, head_dim] is accepted and treated as num_queries = 1).
        Query i of sequence b attends to positions t <= L_b - num_queries + i.
        Returns float64 of q's shape; rows outside ``b_range`` are zero.
        """
        code = _dtype_code(k_cache)
        decode_shape = q.ndim == 3
        q4 = q[:, None] if decode_shape else q
        batch, nq, hq, d = q4.shape
        hkv, nb, bs, dk = k_cache.shape
        assert dk == d and q4.dtype == k_cache.dtype
        tables = np.ascontiguousarray(block_tables, dtype=np.int32)
        lens = np.ascontiguousarray(context_lens, dtype=np.int32)
        assert tables.shape[0] == batch and lens.shape == (batch,)
        out = np.zeros((batch, nq, hq, d), dtype=np.float64)
        b0, b1 = b_range if b_range is not None else (0, batch)
        rc = self.lib.oracle_attend(_ptr(k_cache), _ptr(v_cache), code, hkv, nb, bs, d,
                                    _ptr(np.ascontiguousarray(q4)), _ptr(out), _ptr(tables),
                                    int(tables.shape[1]), _ptr(lens), batch, hq, nq, float(scale),
                                    int(b0), int(b1))
        if rc != 0:
            raise ValueError(f"oracle_attend: {rc} sequence(s) with out-of-range lengths or block ids")
        return out[:, 0] if decode_shape else out

    def decode(self, k_cache, v_cache, q, block_tables, context_lens, scale, b_range=None):
        """Decode attention: one query token per sequence (q: [batch, q_heads, head_dim])."""
        return self.attend(k_cache, v_cache, q, block_tables, context_lens, scale, b_range)

    def verify(self, k_cache, v_cache, q, k_new, v_new, slot_mapping, block_tables,
               context_lens, scale, b_range=None):
        """Speculative verify: write the new K/V at their slots, then attend causally.

        Mutates the caches in place (the write is part of the step).
        q: [batch, num_queries, q_heads, head_dim]; k_new / v_new:
        [batch * num_queries, kv_heads, head_dim]; slot_mapping: [batch * num_queries].
        """
        bad = self.cache_write(k_cache, v_cache, k_new, v_new, slot_mapping)
        if bad:
            raise ValueError(f"oracle verify: {bad} out-of-range slot(s)")
        return self.attend(k_cache, v_cache, q, block_tables, context_lens, scale, b_range)


    # ---- int8 cache ("A Rust inference server for Qwen2 on Apple Silicon", Day 4) ----

    def cache_write_q8(self, k_codes: np.ndarray, v_codes: np.ndarray, k_scale: np.ndarray,
                       v_scale: np.ndarray, k_new: np.ndarray, v_new: np.ndarray,
                       slot_mapping: np.ndarray) -> int:
        """In place: quantised write of bf16 rows (see pa_oracle.c, "int8 KV cache").

        Codes [kv_heads, num_blocks, block_size, head_dim] uint8; k_scale
        [kv_heads, num_blocks, head_dim] float32; v_scale [kv_heads, num_blocks,
        block_size] float32; new rows [num_tokens, kv_heads, head_dim] uint16 (bf16
        bits). Returns the count of out-of-range slots.
        """
        hkv, nb, bs, d = k_codes.shape
        assert k_codes.dtype == np.uint8 and v_codes.dtype == np.uint8 and v_codes.shape == k_codes.shape
        assert k_scale.dtype == np.float32 and k_scale.shape == (hkv, nb, d)
        assert v_scale.dtype == np.float32 and v_scale.shape == (hkv, nb, bs)
        n = int(slot_mapping.shape[0])
        assert k_new.dtype == np.uint16 and k_new.shape == (n, hkv, d) and v_new.shape == k_new.shape
        slots = np.ascontiguousarray(slot_mapping, dtype=np.int32)
        return int(self.lib.oracle_cache_write_q8(
            _ptr(k_codes), _ptr(v_codes), _ptr(k_scale), _ptr(v_scale), hkv, nb, bs, d,
            _ptr(np.ascontiguousarray(k_new)), _ptr(np.ascontiguousarray(v_new)), _ptr(slots), n))

    def dequant_q8(self, k_codes, v_codes, k_scale, v_scale):
        """(K, V) as float32 caches of the plain layout: (byte - 128) * scale."""
        hkv, nb, bs, d = k_codes.shape
        ko = np.empty((hkv, nb, bs, d), dtype=np.float32)
        vo = np.empty((hkv, nb, bs, d), dtype=np.float32)
        self.lib.oracle_dequant_q8(_ptr(np.ascontiguousarray(k_codes)), _ptr(np.ascontiguousarray(v_codes)),
                                   _ptr(np.ascontiguousarray(k_scale)), _ptr(np.ascontiguousarray(v_scale)),
                                   hkv, nb, bs, d, _ptr(ko), _ptr(vo))
        return ko, vo

    def decode_q8(self, k_codes, v_codes, k_scale, v_scale, q, block_tables, context_lens, scale,
                  b_range=None):
        """Attention over the dequantised pool (q as bf16 bits, widened exactly)."""
        ko, vo = self.dequant_q8(k_codes, v_codes, k_scale, v_scale)
        qf = bf16_bits_to_f64(q).astype(np.float32) if q.dtype == np.uint16 else q.astype(np.float32)
        return self.attend(ko, vo, qf, block_tables, context_lens, scale, b_range)

    def verify_q8(self, k_codes, v_codes, k_scale, v_scale, q, k_new, v_new, slot_mapping,
                  block_tables, context_lens, scale, b_range=None):
        """Quantised write of the new rows (in place), then attention over the pool."""
        bad = self.cache_write_q8(k_codes, v_codes, k_scale, v_scale, k_new, v_new, slot_mapping)
        if bad:
            raise ValueError(f"oracle verify_q8: {bad} out-of-range slot(s)")
        return self.decode_q8(k_codes, v_codes, k_scale, v_scale, q, block_tables, context_lens,
                              scale, b_range)


    # ---- ragged verify: a different number of new tokens per sequence ----

    def verify_ragged(self, k_cache, v_cache, q, k_new, v_new, slot_mapping, query_start, block_tables,
                      context_lens, scale, q8_scales=None):
        """Write every new row (in place), then attend per sequence: sequence b's
        n_b = query_start[b+1] - query_start[b] query tokens (flat rows of q) sit
        at positions L_b - n_b + i, causal among themselves ("From 183 ms to
        19 ms per decode step", section "Then speculative decoding got slower").
        q8_scales = (k_scale, v_scale) for an int8 pool (k_cache / v_cache are
        then the code bytes). Returns float64 [total, q_heads, head_dim]."""
        if q8_scales is None:
            bad = self.cache_write(k_cache, v_cache, k_new, v_new, slot_mapping)
        else:
            bad = self.cache_write_q8(k_cache, v_cache, *q8_scales, k_new, v_new, slot_mapping)
        if bad:
            raise ValueError(f"oracle verify_ragged: {bad} out-of-range slot(s)")
        return self.attend_ragged(k_cache, v_cache, q, query_start, block_tables, context_lens, scale, q8_scales)

    def attend_ragged(self, k_cache, v_cache, q, query_start, block_tables, context_lens, scale,
                      q8_scales=None):
        """Attention only (nothing written): sequence b's query_start[b+1] -
        query_start[b] flat q rows are its last positions, causal among
        themselves. This is prefill / chunked prefill over a cache that already
        holds the chunk ("From 183 ms to 19 ms per decode step", section
        "What's next"). Returns float64 [total, q_heads, head_dim]."""
        qs = np.asarray(query_start, dtype=np.int64)
        out = np.zeros(q.shape, dtype=np.float64)
        for b in range(len(context_lens)):
            a, e = int(qs[b]), int(qs[b + 1])
            if e == a:
                continue
            qb = np.ascontiguousarray(q[a:e][None])
            tb = np.ascontiguousarray(block_tables[b:b + 1])
            lb = np.ascontiguousarray(context_lens[b:b + 1])
            if q8_scales is None:
                out[a:e] = self.attend(k_cache, v_cache, qb, tb, lb, scale)[0]
            else:
                out[a:e] = self.decode_q8(k_cache, v_cache, *q8_scales, qb, tb, lb, scale)[0]
        return out


def _dtype_code(arr: np.ndarray) -> int:
    if arr.dtype == np.float32:
        return F32
    if arr.dtype == np.uint16:  # bf16 bit patterns
        return BF16
    raise TypeError(f"cache dtype must be float32 or uint16 (bf16 bits), got {arr.dtype}")


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


_default: Oracle | None = None


def get() -> Oracle:
    """The oracle compiled from this directory's ``pa_oracle.c`` (built on first use)."""
    global _default
    if _default is None:
        _default = Oracle(build())
    return _default


def set_threads(n: int) -> None:
    get().set_threads(n)


def max_threads() -> int:
    return get().max_threads()


def cache_write(*args, **kwargs) -> int:
    return get().cache_write(*args, **kwargs)


def attend(*args, **kwargs) -> np.ndarray:
    return get().attend(*args, **kwargs)


def decode(*args, **kwargs) -> np.ndarray:
    return get().decode(*args, **kwargs)


def verify(*args, **kwargs) -> np.ndarray:
    return get().verify(*args, **kwargs)


def cache_write_q8(*args, **kwargs) -> int:
    return get().cache_write_q8(*args, **kwargs)


def dequant_q8(*args, **kwargs):
    return get().dequant_q8(*args, **kwargs)


def decode_q8(*args, **kwargs) -> np.ndarray:
    return get().decode_q8(*args, **kwargs)


def verify_q8(*args, **kwargs) -> np.ndarray:
    return get().verify_q8(*args, **kwargs)


def verify_ragged(*args, **kwargs) -> np.ndarray:
    return get().verify_ragged(*args, **kwargs)


def attend_ragged(*args, **kwargs) -> np.ndarray:
    return get().attend_ragged(*args, **kwargs)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to float64."""
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def to_f64(arr: np.ndarray) -> np.ndarray:
    if arr.dtype == np.uint16:
        return bf16_bits_to_f64(arr)
    return arr.astype(np.float64)


if __name__ == "__main__":  # pragma: no cover
    build(force="--force" in sys.argv)
    print(_LIB)
