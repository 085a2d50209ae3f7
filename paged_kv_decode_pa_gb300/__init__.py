"""GB300-native decode-time attention over a paged KV cache.

The hot path lives in libpa.so (hand-written CUDA for sm_103a, C ABI declared
in include/pa.h). This package builds it (``build``), binds it with ctypes
(``_lib``) and exposes the same entry points over torch tensors (``api``).
``inputs`` holds the seeded synthetic workloads and ``accounting`` the
algorithmic byte counts used for the roofline.
"""

from .api import (make_cache, new_workspace, pa_cache_write, pa_decode, pa_decode_noalloc,  # noqa: F401
                  pa_prefill, pa_status_string, pa_verify_ragged,
                  pa_validate, pa_verify, pa_version, pa_workspace_init, pa_workspace_size,
                  pa_workspace_status, to_numpy, to_torch)

__all__ = ["make_cache", "new_workspace", "pa_cache_write", "pa_decode", "pa_decode_noalloc", "pa_verify",
           "pa_verify_ragged", "pa_prefill",
           "pa_validate",
           "pa_workspace_size", "pa_workspace_init", "pa_workspace_status", "pa_status_string",
           "pa_version", "to_torch", "to_numpy"]
