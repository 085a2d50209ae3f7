"""The C-ABI library: it loads, exports every symbol include/pa.h declares, and
rejects bad host arguments before launching anything (CPU only: no call here
reaches the GPU)."""

import ctypes
import re
from pathlib import Path

import pytest

from paged_kv_decode_pa_gb300 import _lib

HEADER = Path(__file__).resolve().parents[1] / "include" / "pa.h"


@pytest.fixture(scope="module")
def lib():
    from paged_kv_decode_pa_gb300 import build

    build.build()
    return _lib.load()


def declared_functions():
    text = HEADER.read_text()
    return sorted(set(re.findall(r"^[a-z_ *]*?\b(pa_[a-z_]+)\s*\(", text, flags=re.M)))


def test_options_layout_matches_header():
    """pa_options as the header declares it: the binding's struct has the same
    fields in the same order and size."""
    text = HEADER.read_text()
    body = re.search(r"typedef struct pa_options \{(.*?)\} pa_options;", text, flags=re.S).group(1)
    body = re.sub(r"/\*.*?\*/", " ", body, flags=re.S)
    fields = re.findall(r"(int32_t|uint32_t)\s+(\w+);", body)
    ctypes_of = {"int32_t": ctypes.c_int32, "uint32_t": ctypes.c_uint32}
    assert [(n, ctypes_of[t]) for t, n in fields] == list(_lib.PaOptions._fields_)


def test_header_declares_the_binding_list():
    assert declared_functions() == sorted(_lib.EXPORTED)


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_header_constants_match_binding():
    text = HEADER.read_text()
    for name in ("PA_FLAG_BAD_BLOCK", "PA_FLAG_BAD_LENGTH", "PA_FLAG_BAD_SLOT", "PA_FLAG_TIMEOUT",
                 "PA_DEFAULT_SPLIT_TOKENS", "PA_VALIDATE_WORDS", "PA_DEFAULT_WAIT_LIMIT_NS",
                 "PA_LONG_CONTEXT_TOKENS", "PA_DEFAULT_SPLIT_LONG", "PA_DEFAULT_SPLIT_LONG_INT8",
                 "PA_DEFAULT_SPLIT_TOKENS_INT8"):
        m = re.search(rf"#define {name} (0x[0-9a-f]+|\d+)", text)
        assert m and int(m.group(1), 0) == getattr(_lib, name), name


def _cache(**kw):
    c = dict(k=0x10000, v=0x20000, kv_heads=2, num_blocks=64, block_size=16, head_dim=128,
             dtype=_lib.PA_DTYPE_BF16)
    c.update(kw)
    return _lib.PaCache(**c)


def _decode(lib, cache, q=0x30000, out=0x40000, tables=0x50000, lens=0x60000, mbps=4, batch=2,
            hq=12, max_ctx=64, ws=0x70000, ws_bytes=1 << 30, opts=None):
    return lib.pa_decode(ctypes.byref(cache), q, out, tables, mbps, lens, batch, hq, max_ctx,
                         ctypes.c_float(0.088), ws, ws_bytes,
                         ctypes.byref(opts) if opts is not None else None, None)


@pytest.mark.parametrize("kw,status", [
    (dict(head_dim=64), _lib.PA_ERR_UNSUPPORTED),
    (dict(block_size=32), _lib.PA_ERR_UNSUPPORTED),
    (dict(dtype=7), _lib.PA_ERR_UNSUPPORTED),
    (dict(k=0), _lib.PA_ERR_INVALID_ARG),
    (dict(v=0x20008), _lib.PA_ERR_INVALID_ARG),  # not 16-byte aligned
    (dict(kv_heads=0), _lib.PA_ERR_INVALID_ARG),
])
def test_bad_cache_rejected(lib, kw, status):
    assert _decode(lib, _cache(**kw)) == status


def test_bad_call_arguments_rejected(lib):
    c = _cache()
    assert _decode(lib, c, hq=13) == _lib.PA_ERR_INVALID_ARG          # q_heads % kv_heads
    assert _decode(lib, c, q=0) == _lib.PA_ERR_INVALID_ARG
    assert _decode(lib, c, out=0x40004) == _lib.PA_ERR_INVALID_ARG    # misaligned
    assert _decode(lib, c, max_ctx=65) == _lib.PA_ERR_INVALID_ARG     # > mbps * 16
    assert _decode(lib, c, batch=-1) == _lib.PA_ERR_INVALID_ARG
    assert _decode(lib, c, ws=0) == _lib.PA_ERR_WORKSPACE
    assert _decode(lib, c, ws_bytes=16) == _lib.PA_ERR_WORKSPACE
    assert _decode(lib, c, ws=0x70010) == _lib.PA_ERR_WORKSPACE       # not 256-aligned
    assert _decode(lib, c, opts=_lib.PaOptions(24, 0)) == _lib.PA_ERR_UNSUPPORTED  # not a multiple of 16
    assert _decode(lib, c, opts=_lib.PaOptions(0, 9)) == _lib.PA_ERR_UNSUPPORTED
    f32 = _cache(dtype=_lib.PA_DTYPE_F32)
    assert _decode(lib, f32, opts=_lib.PaOptions(0, _lib.PA_KERNEL_MMA)) == _lib.PA_ERR_UNSUPPORTED
    assert _decode(lib, c, opts=_lib.PaOptions(0, 3)) == _lib.PA_ERR_UNSUPPORTED    # no kernel 3
    assert _decode(lib, c, opts=_lib.PaOptions(0, _lib.PA_KERNEL_TC)) == _lib.PA_ERR_UNSUPPORTED  # prefill only
    assert _decode(lib, c, batch=0) == _lib.PA_OK                      # nothing to do, nothing launched
    # The split index is the grid's z: more than 65535 splits per sequence is refused before
    # anything is launched (16-token splits over 65537 blocks).
    assert _decode(lib, _cache(num_blocks=70000), mbps=65537, max_ctx=16 * 65537, batch=1, hq=2,
                   ws_bytes=1 << 45, opts=_lib.PaOptions(16, 0)) == _lib.PA_ERR_UNSUPPORTED


def test_verify_and_write_arguments(lib):
    c = _cache()
    assert lib.pa_verify(ctypes.byref(c), 0x30000, 0x40000, 0, 0x80000, 0x90000, 5, 0x50000, 4,
                         0x60000, 2, 12, 64, ctypes.c_float(0.1), 0x70000, 1 << 30, None,
                         None) == _lib.PA_ERR_INVALID_ARG
    assert lib.pa_verify(ctypes.byref(c), 0x30000, 0x40000, 0x80000, 0x90000, 0xa0000, 0, 0x50000, 4,
                         0x60000, 2, 12, 64, ctypes.c_float(0.1), 0x70000, 1 << 30, None,
                         None) == _lib.PA_ERR_INVALID_ARG
    assert lib.pa_cache_write(ctypes.byref(c), 0x80008, 0x90000, 0xa0000, 4, None) == _lib.PA_ERR_INVALID_ARG
    assert lib.pa_cache_write(ctypes.byref(c), 0x80000, 0x90000, 0xa0000, -1, None) == _lib.PA_ERR_INVALID_ARG
    assert lib.pa_cache_write(ctypes.byref(c), 0x80000, 0x90000, 0xa0000, 0, None) == _lib.PA_OK


def test_workspace_size(lib):
    opts = _lib.PaOptions(0, 0)
    n1 = lib.pa_workspace_size(8, 1, 12, 2, 128, 32768, ctypes.byref(opts))
    n2 = lib.pa_workspace_size(8, 1, 12, 2, 128, 512, ctypes.byref(opts))
    assert n1 > n2 > 0
    assert lib.pa_workspace_size(8, 1, 13, 2, 128, 512, None) == 0
    assert lib.pa_workspace_size(8, 1, 12, 2, 64, 512, None) == 0


def test_status_strings(lib):
    assert lib.pa_status_string(_lib.PA_ERR_WORKSPACE) == b"PA_ERR_WORKSPACE"
    assert lib.pa_version() >= 100


def test_int8_pool_arguments(lib):
    """An int8 pool needs 16-byte aligned scale arrays and runs only on the
    tensor-core kernel; the dtype value matches the header."""
    text = HEADER.read_text()
    assert re.search(r"PA_DTYPE_INT8 = (\d+)", text).group(1) == str(_lib.PA_DTYPE_INT8)
    ok = dict(dtype=_lib.PA_DTYPE_INT8, k_scale=0x110000, v_scale=0x120000)
    assert _decode(lib, _cache(**ok), batch=0) == _lib.PA_OK
    assert _decode(lib, _cache(**{**ok, "k_scale": None})) == _lib.PA_ERR_INVALID_ARG
    assert _decode(lib, _cache(**{**ok, "v_scale": 0x120004})) == _lib.PA_ERR_INVALID_ARG
    for kernel in (_lib.PA_KERNEL_SIMT, 3):
        assert _decode(lib, _cache(**ok), opts=_lib.PaOptions(0, kernel)) == _lib.PA_ERR_UNSUPPORTED
    assert lib.pa_cache_write(ctypes.byref(_cache(**{**ok, "k_scale": None})), 0x80000, 0x90000, 0xa0000, 4,
                              None) == _lib.PA_ERR_INVALID_ARG


def _prefill(lib, cache, opts=None, batch=2, total=8, max_q=4, hq=12, q=0x30000):
    return lib.pa_prefill(ctypes.byref(cache), q, 0x40000, 0x80000, total, max_q, 0x50000, 4, 0x60000, batch, hq,
                          64, ctypes.c_float(0.1), None, 0, ctypes.byref(opts) if opts is not None else None, None)


def test_prefill_arguments(lib):
    """pa_prefill runs the tcgen05 kernel (the default) or the warp-level one,
    bf16 only; the enum value matches the header."""
    text = HEADER.read_text()
    assert re.search(r"PA_KERNEL_TC = (\d+)", text).group(1) == str(_lib.PA_KERNEL_TC)
    c = _cache()
    for kernel in (_lib.PA_KERNEL_SIMT, 3, 9):
        assert _prefill(lib, c, _lib.PaOptions(0, kernel)) == _lib.PA_ERR_UNSUPPORTED
    for kernel in (_lib.PA_KERNEL_AUTO, _lib.PA_KERNEL_TC, _lib.PA_KERNEL_MMA):
        assert _prefill(lib, c, _lib.PaOptions(0, kernel), batch=0) == _lib.PA_OK
    assert _prefill(lib, c, batch=0) == _lib.PA_OK
    assert _prefill(lib, c, hq=13) == _lib.PA_ERR_INVALID_ARG
    assert _prefill(lib, c, max_q=0) == _lib.PA_ERR_INVALID_ARG
    assert _prefill(lib, c, q=0x30008) == _lib.PA_ERR_INVALID_ARG
    assert _prefill(lib, _cache(dtype=_lib.PA_DTYPE_F32)) == _lib.PA_ERR_UNSUPPORTED


def test_prefill_tc_needs_group_of_at_most_128(lib):
    """The tcgen05 prefill kernel takes whole tokens per 128-row tile."""
    c = _cache()
    assert _prefill(lib, c, _lib.PaOptions(0, _lib.PA_KERNEL_TC), hq=2 * 129) == _lib.PA_ERR_UNSUPPORTED


def test_noalloc_checks_arguments_like_pa_decode_first(lib):
    """pa_decode_noalloc returns pa_decode's status for a bad argument even
    when the sizes would also exceed its scratch: the checks run before the
    scratch is sized or touched (nothing here reaches the GPU)."""
    def noalloc(cache, batch=4096, max_ctx=1 << 16, hq=12, opts=None):
        return lib.pa_decode_noalloc(ctypes.byref(cache), 0x30000, 0x40000, 0x50000, max_ctx // 16, 0x60000, batch,
                                     hq, max_ctx, ctypes.c_float(0.1), ctypes.byref(opts) if opts else None, None)
    big = dict(batch=4096, max_ctx=1 << 16)
    assert noalloc(_cache(head_dim=64), **big) == _lib.PA_ERR_UNSUPPORTED
    assert noalloc(_cache(), opts=_lib.PaOptions(24, 0), **big) == _lib.PA_ERR_UNSUPPORTED
    assert noalloc(_cache(), opts=_lib.PaOptions(0, 9), **big) == _lib.PA_ERR_UNSUPPORTED
    assert noalloc(_cache(), hq=13, **big) == _lib.PA_ERR_INVALID_ARG
    assert noalloc(_cache(), **big) == _lib.PA_ERR_WORKSPACE
    assert noalloc(_cache(), batch=0, max_ctx=64) == _lib.PA_OK
