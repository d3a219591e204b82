"""ctypes binding over libwllm.so (C ABI in include/wllm.h).

Argument marshalling only: each call turns torch tensors into ``wllm_tensor``
descriptors (device pointer, dtype code, sizes, strides in elements), passes
the current CUDA stream, and raises ``WllmError`` on a non-zero status.  Every
step of the computation runs in the library's CUDA kernels; there is no CPU
path.  Loading fails loudly when the library has not been built.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libwllm.so")

WLLM_OK, WLLM_ERR_INVALID_ARG, WLLM_ERR_UNSUPPORTED, WLLM_ERR_OUT_OF_RANGE, WLLM_ERR_CUDA = range(5)
# E4M3 caches may be passed as torch.float8_e4m3fn or as raw uint8 codes
_DTYPE = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2, torch.int32: 3, torch.int64: 4,
          torch.float8_e4m3fn: 5, torch.uint8: 5}

# every symbol include/wllm.h declares
EXPORTED = ("wllm_reshape_and_cache", "wllm_paged_attention_decode", "wllm_decode_step",
            "wllm_reshape_and_cache_fp8", "wllm_paged_attention_decode_fp8", "wllm_decode_step_fp8",
            "wllm_paged_attention_prefill", "wllm_paged_attention_prefill_fp8",
            "wllm_paged_attention_decode_noalloc",
            "wllm_paged_attention_workspace_bytes", "wllm_set_workspace",
            "wllm_partition_tokens", "wllm_device_errors", "wllm_selftest_wait_timeout", "wllm_launch_count",
            "wllm_last_error", "wllm_version",
            "wllm_bm_create", "wllm_bm_destroy", "wllm_bm_add_sequence", "wllm_bm_append_token",
            "wllm_bm_fork", "wllm_bm_free_sequence", "wllm_bm_block_table", "wllm_bm_num_free_blocks",
            "wllm_bm_num_cached_blocks", "wllm_bm_block_ref")


class WllmError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"wllm status {status}: {message}")
        self.status = status


class WllmTensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("ndim", ctypes.c_int32),
                ("shape", ctypes.c_int64 * 4), ("stride", ctypes.c_int64 * 4)]


_lib = None
_lock = threading.Lock()


def library_path() -> str:
    return _LIB_PATH


def load_library():
    """Load libwllm.so (raises if it is missing: build it with ``build()`` first)."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"{_LIB_PATH} is missing: run `python -m paged_kv_cache_185_gb300.build`")
        lib = ctypes.CDLL(_LIB_PATH)
        P = ctypes.POINTER(WllmTensor)
        lib.wllm_reshape_and_cache.argtypes = [P, P, P, P, P, ctypes.c_void_p]
        lib.wllm_reshape_and_cache.restype = ctypes.c_int
        lib.wllm_paged_attention_decode.argtypes = [P, P, P, P, P, P, ctypes.c_int, ctypes.c_float,
                                                    ctypes.c_int, ctypes.c_void_p]
        lib.wllm_paged_attention_decode.restype = ctypes.c_int
        lib.wllm_decode_step.argtypes = [P, P, P, P, P, P, P, P, P, ctypes.c_int, ctypes.c_float, ctypes.c_int,
                                         ctypes.c_void_p]
        lib.wllm_decode_step.restype = ctypes.c_int
        f32 = ctypes.c_float
        lib.wllm_reshape_and_cache_fp8.argtypes = [P, P, P, P, P, f32, f32, ctypes.c_void_p]
        lib.wllm_reshape_and_cache_fp8.restype = ctypes.c_int
        lib.wllm_paged_attention_decode_fp8.argtypes = [P, P, P, P, P, P, ctypes.c_int, f32, f32, f32,
                                                        ctypes.c_int, ctypes.c_void_p]
        lib.wllm_paged_attention_decode_fp8.restype = ctypes.c_int
        lib.wllm_decode_step_fp8.argtypes = [P, P, P, P, P, P, P, P, P, ctypes.c_int, f32, f32, f32, ctypes.c_int,
                                             ctypes.c_void_p]
        lib.wllm_decode_step_fp8.restype = ctypes.c_int
        lib.wllm_paged_attention_prefill.argtypes = [P, P, P, P, P, P, P, ctypes.c_int, ctypes.c_float,
                                                     ctypes.c_int, ctypes.c_void_p]
        lib.wllm_paged_attention_prefill.restype = ctypes.c_int
        lib.wllm_paged_attention_prefill_fp8.argtypes = [P, P, P, P, P, P, P, ctypes.c_int, f32, f32, f32,
                                                         ctypes.c_int, ctypes.c_void_p]
        lib.wllm_paged_attention_prefill_fp8.restype = ctypes.c_int
        lib.wllm_paged_attention_decode_noalloc.argtypes = [P, P, P, P, P, P, ctypes.c_int, ctypes.c_float,
                                                            ctypes.c_int, ctypes.c_void_p]
        lib.wllm_paged_attention_decode_noalloc.restype = ctypes.c_int
        lib.wllm_paged_attention_workspace_bytes.argtypes = [ctypes.c_int] * 6
        lib.wllm_paged_attention_workspace_bytes.restype = ctypes.c_size_t
        lib.wllm_set_workspace.argtypes = [ctypes.c_void_p, ctypes.c_size_t]
        lib.wllm_set_workspace.restype = ctypes.c_int
        lib.wllm_partition_tokens.argtypes = [ctypes.c_int] * 7
        lib.wllm_partition_tokens.restype = ctypes.c_int
        lib.wllm_device_errors.argtypes = []
        lib.wllm_device_errors.restype = ctypes.c_int
        lib.wllm_selftest_wait_timeout.argtypes = [ctypes.c_ulonglong, ctypes.c_void_p]
        lib.wllm_selftest_wait_timeout.restype = ctypes.c_int
        lib.wllm_launch_count.argtypes = []
        lib.wllm_launch_count.restype = ctypes.c_ulonglong
        lib.wllm_last_error.argtypes = []
        lib.wllm_last_error.restype = ctypes.c_char_p
        lib.wllm_version.argtypes = []
        lib.wllm_version.restype = ctypes.c_char_p
        vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32
        p64, p32 = ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_int32)
        lib.wllm_bm_create.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.POINTER(vp)]
        lib.wllm_bm_create.restype = ctypes.c_int
        lib.wllm_bm_destroy.argtypes = [vp]
        lib.wllm_bm_destroy.restype = None
        lib.wllm_bm_add_sequence.argtypes = [vp, i64, p32, i64, p64, p64]
        lib.wllm_bm_add_sequence.restype = ctypes.c_int
        lib.wllm_bm_append_token.argtypes = [vp, i64, i32, p64, p32, p32]
        lib.wllm_bm_append_token.restype = ctypes.c_int
        lib.wllm_bm_fork.argtypes = [vp, i64, i64]
        lib.wllm_bm_fork.restype = ctypes.c_int
        lib.wllm_bm_free_sequence.argtypes = [vp, i64]
        lib.wllm_bm_free_sequence.restype = ctypes.c_int
        lib.wllm_bm_block_table.argtypes = [vp, i64, p32, ctypes.c_int, p64]
        lib.wllm_bm_block_table.restype = ctypes.c_int
        lib.wllm_bm_num_free_blocks.argtypes = [vp]
        lib.wllm_bm_num_free_blocks.restype = i64
        lib.wllm_bm_num_cached_blocks.argtypes = [vp]
        lib.wllm_bm_num_cached_blocks.restype = i64
        lib.wllm_bm_block_ref.argtypes = [vp, i32]
        lib.wllm_bm_block_ref.restype = ctypes.c_int
        _lib = lib
    return _lib


def describe(t: torch.Tensor) -> WllmTensor:
    if t.dim() > 4:
        raise ValueError("at most 4 dims")
    d = WllmTensor()
    d.data = t.data_ptr() if t.numel() > 0 else None
    d.dtype = _DTYPE[t.dtype]
    d.ndim = t.dim()
    for i in range(t.dim()):
        d.shape[i] = t.shape[i]
        d.stride[i] = t.stride(i)
    return d


def _stream_handle(device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _check(rc: int) -> None:
    if rc != WLLM_OK:
        raise WllmError(rc, load_library().wllm_last_error().decode())


def _require_cuda(*ts):
    for t in ts:
        if not t.is_cuda:
            raise ValueError("all tensors must be CUDA tensors (the library has no CPU path)")
    dev = ts[0].device
    for t in ts:
        if t.device != dev:
            raise ValueError("all tensors must be on one device")
    return dev


def reshape_and_cache(key, value, k_cache, v_cache, slot_mapping) -> None:
    """KV append: scatter key/value [T,Hkv,D] into caches [N_b,Hkv,bs,D] at ``slot_mapping``."""
    dev = _require_cuda(key, value, k_cache, v_cache, slot_mapping)
    lib = load_library()
    with torch.cuda.device(dev):
        args = [describe(x) for x in (key, value, k_cache, v_cache, slot_mapping)]
        _check(lib.wllm_reshape_and_cache(*[ctypes.byref(a) for a in args], _stream_handle(dev)))


def paged_attention_decode(out, q, k_cache, v_cache, block_tables, context_lens,
                           num_kv_heads: int, scale: float, block_size: int) -> torch.Tensor:
    """Paged decode attention into ``out`` [B,Hq,D]; returns ``out``."""
    dev = _require_cuda(out, q, k_cache, v_cache, block_tables, context_lens)
    lib = load_library()
    with torch.cuda.device(dev):
        args = [describe(x) for x in (out, q, k_cache, v_cache, block_tables, context_lens)]
        _check(lib.wllm_paged_attention_decode(*[ctypes.byref(a) for a in args], int(num_kv_heads),
                                               float(scale), int(block_size), _stream_handle(dev)))
    return out


def paged_attention_decode_noalloc(out, q, k_cache, v_cache, block_tables, context_lens,
                                   num_kv_heads: int, scale: float, block_size: int) -> torch.Tensor:
    """Paged decode attention that allocates no device memory (fixed scratch
    inside the library; see wllm_paged_attention_decode_noalloc in wllm.h)."""
    dev = _require_cuda(out, q, k_cache, v_cache, block_tables, context_lens)
    lib = load_library()
    with torch.cuda.device(dev):
        args = [describe(x) for x in (out, q, k_cache, v_cache, block_tables, context_lens)]
        _check(lib.wllm_paged_attention_decode_noalloc(*[ctypes.byref(a) for a in args], int(num_kv_heads),
                                                       float(scale), int(block_size), _stream_handle(dev)))
    return out


def decode_step(out, q, key, value, k_cache, v_cache, slot_mapping, block_tables, context_lens,
                num_kv_heads: int, scale: float, block_size: int) -> torch.Tensor:
    """One decode step of one layer: append this step's K/V, then attend (one
    fused launch where the kernel allows; see wllm_decode_step)."""
    dev = _require_cuda(out, q, key, value, k_cache, v_cache, slot_mapping, block_tables, context_lens)
    lib = load_library()
    with torch.cuda.device(dev):
        args = [describe(x) for x in (out, q, key, value, k_cache, v_cache, slot_mapping, block_tables,
                                      context_lens)]
        _check(lib.wllm_decode_step(*[ctypes.byref(a) for a in args], int(num_kv_heads), float(scale),
                                    int(block_size), _stream_handle(dev)))
    return out


def reshape_and_cache_fp8(key, value, k_cache, v_cache, slot_mapping, k_scale: float, v_scale: float) -> None:
    """KV append into E4M3 caches (uint8 or float8_e4m3fn): stores E4M3(x * (1/scale))."""
    dev = _require_cuda(key, value, k_cache, v_cache, slot_mapping)
    lib = load_library()
    with torch.cuda.device(dev):
        args = [describe(x) for x in (key, value, k_cache, v_cache, slot_mapping)]
        _check(lib.wllm_reshape_and_cache_fp8(*[ctypes.byref(a) for a in args], float(k_scale), float(v_scale),
                                              _stream_handle(dev)))


def paged_attention_decode_fp8(out, q, k_cache, v_cache, block_tables, context_lens, num_kv_heads: int,
                               scale: float, k_scale: float, v_scale: float, block_size: int) -> torch.Tensor:
    """Paged decode attention over E4M3 caches (K = code * k_scale, V = code * v_scale); returns ``out``."""
    dev = _require_cuda(out, q, k_cache, v_cache, block_tables, context_lens)
    lib = load_library()
    with torch.cuda.device(dev):
        args = [describe(x) for x in (out, q, k_cache, v_cache, block_tables, context_lens)]
        _check(lib.wllm_paged_attention_decode_fp8(*[ctypes.byref(a) for a in args], int(num_kv_heads),
                                                   float(scale), float(k_scale), float(v_scale), int(block_size),
                                                   _stream_handle(dev)))
    return out


def decode_step_fp8(out, q, key, value, k_cache, v_cache, slot_mapping, block_tables, context_lens,
                    num_kv_heads: int, scale: float, k_scale: float, v_scale: float, block_size: int) -> torch.Tensor:
    """decode_step over E4M3 caches: the append quantises with the same scales the attention reads back."""
    dev = _require_cuda(out, q, key, value, k_cache, v_cache, slot_mapping, block_tables, context_lens)
    lib = load_library()
    with torch.cuda.device(dev):
        args = [describe(x) for x in (out, q, key, value, k_cache, v_cache, slot_mapping, block_tables,
                                      context_lens)]
        _check(lib.wllm_decode_step_fp8(*[ctypes.byref(a) for a in args], int(num_kv_heads), float(scale),
                                        float(k_scale), float(v_scale), int(block_size), _stream_handle(dev)))
    return out


def paged_attention_prefill(out, q, k_cache, v_cache, block_tables, context_lens, query_start_loc,
                            num_kv_heads: int, scale: float, block_size: int) -> torch.Tensor:
    """Chunked-prefill paged attention into ``out`` [T,Hq,D] (packed chunks, causal); returns ``out``."""
    dev = _require_cuda(out, q, k_cache, v_cache, block_tables, context_lens, query_start_loc)
    lib = load_library()
    with torch.cuda.device(dev):
        args = [describe(x) for x in (out, q, k_cache, v_cache, block_tables, context_lens, query_start_loc)]
        _check(lib.wllm_paged_attention_prefill(*[ctypes.byref(a) for a in args], int(num_kv_heads),
                                                float(scale), int(block_size), _stream_handle(dev)))
    return out


def paged_attention_prefill_fp8(out, q, k_cache, v_cache, block_tables, context_lens, query_start_loc,
                                num_kv_heads: int, scale: float, k_scale: float, v_scale: float,
                                block_size: int) -> torch.Tensor:
    """Chunked-prefill paged attention over E4M3 caches (K = code * k_scale, V = code * v_scale)."""
    dev = _require_cuda(out, q, k_cache, v_cache, block_tables, context_lens, query_start_loc)
    lib = load_library()
    with torch.cuda.device(dev):
        args = [describe(x) for x in (out, q, k_cache, v_cache, block_tables, context_lens, query_start_loc)]
        _check(lib.wllm_paged_attention_prefill_fp8(*[ctypes.byref(a) for a in args], int(num_kv_heads),
                                                    float(scale), float(k_scale), float(v_scale),
                                                    int(block_size), _stream_handle(dev)))
    return out


def workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq, block_size) -> int:
    return int(load_library().wllm_paged_attention_workspace_bytes(
        num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq, block_size))


def set_workspace(buf: torch.Tensor | None) -> None:
    """Use a caller-owned device buffer (uint8, 256-byte aligned) as workspace; None reverts."""
    lib = load_library()
    if buf is None:
        _check(lib.wllm_set_workspace(None, 0))
    else:
        with torch.cuda.device(buf.device):
            _check(lib.wllm_set_workspace(buf.data_ptr(), buf.numel() * buf.element_size()))


def partition_tokens(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq, block_size,
                     dtype: torch.dtype) -> int:
    return int(load_library().wllm_partition_tokens(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                                    max_blocks_per_seq, block_size, _DTYPE[dtype]))


def device_errors() -> int:
    return int(load_library().wllm_device_errors())


def selftest_wait_timeout(limit_ns: int, device=None) -> None:
    """Run the bounded-wait self-test kernel on the current stream (see
    wllm_selftest_wait_timeout); call device_errors() afterwards."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    lib = load_library()
    with torch.cuda.device(dev):
        _check(lib.wllm_selftest_wait_timeout(int(limit_ns), _stream_handle(dev)))


def launch_count() -> int:
    """Kernel launches the library has issued in this process."""
    return int(load_library().wllm_launch_count())


def version() -> str:
    return load_library().wllm_version().decode()


class BlockManager:
    """Prefix-caching manager of the physical KV blocks (host side; see the
    wllm_bm_* calls in wllm.h).  Argument marshalling only."""

    def __init__(self, num_blocks: int, block_size: int):
        self._lib = load_library()
        h = ctypes.c_void_p()
        rc = self._lib.wllm_bm_create(int(num_blocks), int(block_size), ctypes.byref(h))
        if rc != WLLM_OK:
            raise WllmError(rc, "wllm_bm_create")
        self._h = h
        self.num_blocks, self.block_size = int(num_blocks), int(block_size)

    def close(self):
        if self._h:
            self._lib.wllm_bm_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @staticmethod
    def _ok(rc: int, what: str):
        if rc != WLLM_OK:
            raise WllmError(rc, what)

    def add_sequence(self, seq_id: int, tokens):
        """Returns (slots [n] int64 tensor, number of leading tokens already cached)."""
        t = torch.as_tensor(tokens, dtype=torch.int32).contiguous()
        n = t.numel()
        slots = torch.empty(n, dtype=torch.int64)
        cached = ctypes.c_int64()
        self._ok(self._lib.wllm_bm_add_sequence(
            self._h, int(seq_id), ctypes.cast(t.data_ptr(), ctypes.POINTER(ctypes.c_int32)) if n else None, n,
            ctypes.cast(slots.data_ptr(), ctypes.POINTER(ctypes.c_int64)) if n else None, ctypes.byref(cached)),
            "wllm_bm_add_sequence")
        return slots, int(cached.value)

    def append_token(self, seq_id: int, token: int):
        """Returns (slot, copy) with copy = (src_block, dst_block) or None."""
        slot, src, dst = ctypes.c_int64(), ctypes.c_int32(), ctypes.c_int32()
        self._ok(self._lib.wllm_bm_append_token(self._h, int(seq_id), int(token), ctypes.byref(slot),
                                                ctypes.byref(src), ctypes.byref(dst)), "wllm_bm_append_token")
        return int(slot.value), (None if src.value < 0 else (int(src.value), int(dst.value)))

    def fork(self, parent: int, child: int):
        self._ok(self._lib.wllm_bm_fork(self._h, int(parent), int(child)), "wllm_bm_fork")

    def free_sequence(self, seq_id: int):
        self._ok(self._lib.wllm_bm_free_sequence(self._h, int(seq_id)), "wllm_bm_free_sequence")

    def block_table(self, seq_id: int, max_blocks: int):
        """Returns (row [max_blocks] int32 tensor, -1 past the last block; context length)."""
        row = torch.empty(int(max_blocks), dtype=torch.int32)
        n = ctypes.c_int64()
        self._ok(self._lib.wllm_bm_block_table(
            self._h, int(seq_id), ctypes.cast(row.data_ptr(), ctypes.POINTER(ctypes.c_int32)) if max_blocks else None,
            int(max_blocks), ctypes.byref(n)), "wllm_bm_block_table")
        return row, int(n.value)

    def num_free_blocks(self) -> int:
        return int(self._lib.wllm_bm_num_free_blocks(self._h))

    def num_cached_blocks(self) -> int:
        return int(self._lib.wllm_bm_num_cached_blocks(self._h))

    def block_ref(self, block: int) -> int:
        return int(self._lib.wllm_bm_block_ref(self._h, int(block)))
