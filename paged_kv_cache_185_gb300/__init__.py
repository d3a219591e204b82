"""GB300-native paged KV-cache decode: the KV append and paged decode attention.

The operations run in hand-written sm_103a CUDA kernels inside ``libwllm.so``
(C ABI declared in ``include/wllm.h``).  This package is the thin Python
binding over that library: it passes device pointers, sizes and the current
CUDA stream, and nothing else.  There is no CPU fallback: an op called while
the library is missing or no GPU is present raises.

``workloads`` draws the seeded synthetic decode steps used by tests and bench;
importing it does not load the CUDA library.
"""
from __future__ import annotations

__all__ = ["reshape_and_cache", "paged_attention_decode", "paged_attention_decode_noalloc",
           "workspace_bytes", "set_workspace",
           "partition_tokens", "device_errors", "selftest_wait_timeout", "launch_count", "version",
           "load_library",
           "decode_step", "WllmError", "library_path", "BlockManager",
           "reshape_and_cache_fp8", "paged_attention_decode_fp8", "decode_step_fp8",
           "paged_attention_prefill", "paged_attention_prefill_fp8"]


def __getattr__(name):
    if name in __all__:
        from . import binding
        return getattr(binding, name)
    raise AttributeError(name)
