"""ctypes declarations of libpa's C ABI (include/pa.h).

Loading fails loudly when the shared library has not been built: there is no
fallback implementation of any operation.
"""

from __future__ import annotations

import ctypes
from pathlib import Path

from . import build as _build

PA_OK = 0
PA_ERR_INVALID_ARG = 1
PA_ERR_UNSUPPORTED = 2
PA_ERR_WORKSPACE = 3
PA_ERR_CUDA = 4

PA_DTYPE_F32 = 0
PA_DTYPE_BF16 = 1
PA_DTYPE_INT8 = 2

PA_KERNEL_AUTO = 0
PA_KERNEL_MMA = 1
PA_KERNEL_SIMT = 2
PA_KERNEL_TC = 4
PA_DEFAULT_WAIT_LIMIT_NS = 1000000000

PA_FLAG_BAD_BLOCK = 0x1
PA_FLAG_BAD_LENGTH = 0x2
PA_FLAG_BAD_SLOT = 0x4
PA_FLAG_TIMEOUT = 0x8

PA_DEFAULT_SPLIT_TOKENS = 768
PA_DEFAULT_SPLIT_TOKENS_INT8 = 1536
PA_LONG_CONTEXT_TOKENS = 4096
PA_DEFAULT_SPLIT_LONG = 1152
PA_DEFAULT_SPLIT_LONG_INT8 = 704
PA_VALIDATE_WORDS = 4
PA_NOALLOC_SCRATCH_BYTES = 16 << 20

# Every symbol include/pa.h declares.
EXPORTED = ("pa_cache_write", "pa_workspace_size", "pa_workspace_init", "pa_workspace_status",
            "pa_decode", "pa_verify", "pa_verify_ragged", "pa_prefill", "pa_validate", "pa_decode_noalloc",
            "pa_status_string",
            "pa_last_cuda_error", "pa_version")


class PaCache(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("kv_heads", ctypes.c_int32),
                ("num_blocks", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("k_scale", ctypes.c_void_p), ("v_scale", ctypes.c_void_p)]


class PaOptions(ctypes.Structure):
    _fields_ = [("split_tokens", ctypes.c_int32), ("kernel", ctypes.c_int32),
                ("wait_limit_ns", ctypes.c_uint32)]


class PaError(RuntimeError):
    def __init__(self, fn: str, status: int, cuda_error: int = 0):
        self.status = status
        self.cuda_error = cuda_error
        name = _STATUS_NAMES.get(status, f"status {status}")
        extra = f" (CUDA error {cuda_error})" if status == PA_ERR_CUDA else ""
        super().__init__(f"{fn} failed: {name}{extra}")


_STATUS_NAMES = {0: "PA_OK", 1: "PA_ERR_INVALID_ARG", 2: "PA_ERR_UNSUPPORTED",
                 3: "PA_ERR_WORKSPACE", 4: "PA_ERR_CUDA"}

_lib = None


def library_path() -> Path:
    return _build.LIB


def load(path: Path | None = None):
    """Load libpa.so (once) and declare its functions."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = Path(path) if path is not None else _build.LIB
    if not p.exists():
        raise ImportError(
            f"libpa.so not found at {p}: build it first "
            "(python -c 'import __graft_entry__ as g; g.build()'); there is no fallback")
    lib = ctypes.CDLL(str(p))
    vp, i32, u32p = ctypes.c_void_p, ctypes.c_int32, ctypes.POINTER(ctypes.c_uint32)
    cache_p, opts_p = ctypes.POINTER(PaCache), ctypes.POINTER(PaOptions)
    sig = {
        "pa_cache_write": (ctypes.c_int, [cache_p, vp, vp, vp, i32, vp]),
        "pa_workspace_size": (ctypes.c_size_t, [i32, i32, i32, i32, i32, i32, opts_p]),
        "pa_workspace_init": (ctypes.c_int, [vp, ctypes.c_size_t, vp]),
        "pa_workspace_status": (ctypes.c_int, [vp, u32p, vp]),
        "pa_decode": (ctypes.c_int, [cache_p, vp, vp, vp, i32, vp, i32, i32, i32, ctypes.c_float,
                                     vp, ctypes.c_size_t, opts_p, vp]),
        "pa_verify": (ctypes.c_int, [cache_p, vp, vp, vp, vp, vp, i32, vp, i32, vp, i32, i32, i32,
                                     ctypes.c_float, vp, ctypes.c_size_t, opts_p, vp]),
        "pa_verify_ragged": (ctypes.c_int, [cache_p, vp, vp, vp, vp, vp, vp, i32, i32, vp, i32, vp, i32, i32,
                                            i32, ctypes.c_float, vp, ctypes.c_size_t, opts_p, vp]),
        "pa_prefill": (ctypes.c_int, [cache_p, vp, vp, vp, i32, i32, vp, i32, vp, i32, i32, i32,
                                      ctypes.c_float, vp, ctypes.c_size_t, opts_p, vp]),
        "pa_validate": (ctypes.c_int, [cache_p, vp, i32, vp, i32, i32, vp, i32, vp, vp]),
        "pa_decode_noalloc": (ctypes.c_int, [cache_p, vp, vp, vp, i32, vp, i32, i32, i32,
                                             ctypes.c_float, opts_p, vp]),
        "pa_status_string": (ctypes.c_char_p, [ctypes.c_int]),
        "pa_last_cuda_error": (ctypes.c_int, []),
        "pa_version": (ctypes.c_int, []),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path is None:
        _lib = lib
    return lib


def check(fn: str, status: int) -> None:
    if status != PA_OK:
        raise PaError(fn, status, load().pa_last_cuda_error() if status == PA_ERR_CUDA else 0)
