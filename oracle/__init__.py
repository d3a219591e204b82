"""Plain fp64 CPU oracle for the paged KV-cache append and paged decode attention.

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this package.  The product path
(``paged_kv_cache_185_gb300``) never imports, links or runs it, and this package
imports nothing from there: the two share no code.

The arithmetic lives in ``oracle.c`` (plain C, binary64, optional OpenMP over
output rows); this module compiles it with gcc and marshals torch CPU tensors
(used here only as typed host buffers) through ctypes.

What it computes, with sources (page title, then section):

* ``reshape_and_cache`` -- "mini-vLLM" README, results paragraph on what changed:
  the K/V write is one indexed assignment; every token's key/value rows are copied
  unchanged into slot ``slot_mapping[t]`` = (block ``s // block_size``, offset
  ``s % block_size``).  A negative slot writes nothing.
* ``paged_decode`` -- "mini-vLLM" README, "How it works / Paged KV-cache" and the
  "Results / Correctness" table: single-query attention over the tokens found
  through each sequence's block table, equal to dense attention over the same
  tokens; query head ``h`` reads KV head ``h // (Hq // Hkv)``.
* ``paged_prefill`` -- "wLLM" project page, "Features / Core engine" (chunked
  prefill through the paged cache): every sequence's chunk of query tokens, the
  last ``n_b`` of its ``L`` cached tokens, attends causally (token at position
  ``P`` sees tokens ``0 .. P``).

Parity pins (tests/test_oracle.py) tie it to things other than itself: torch's
float64 scaled-dot-product attention on the dense tokens, numpy/torch decoding of
every 16-bit pattern, closed forms, invariants, and a pure-Python brute force.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "_oracle.so")
_lock = threading.Lock()
_lib = None

F32, F16, BF16, E4M3 = 0, 1, 2, 3
_DTYPE_CODE = {torch.float32: F32, torch.float16: F16, torch.bfloat16: BF16}

_ERRORS = {
    -1: "bad shape",
    -2: "bad dtype",
    -3: "slot out of range",
    -4: "context length out of range",
    -5: "block table entry out of range",
    -6: "out of memory",
}


class OracleError(RuntimeError):
    pass


def build(force: bool = False) -> str:
    """Compile oracle.c into an in-tree shared library (gcc, -O2, OpenMP, no fast-math)."""
    global _lib
    with _lock:
        stale = (not os.path.exists(_LIB)) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)
        if force or stale:
            tmp = _LIB + f".{os.getpid()}.tmp"
            cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fopenmp",
                   "-fno-fast-math", "-o", tmp, _SRC, "-lm"]
            subprocess.run(cmd, check=True)
            os.replace(tmp, _LIB)
            _lib = None
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        i64, i32, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
        lib.oracle_widen.argtypes = [vp, vp, i64, i32]
        lib.oracle_widen.restype = i32
        lib.oracle_reshape_and_cache.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i32]
        lib.oracle_reshape_and_cache.restype = i32
        lib.oracle_paged_decode_rows.argtypes = [
            vp, vp, i64, vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, i64,
            ctypes.c_float, i32, i32]
        lib.oracle_paged_decode_rows.restype = i32
        lib.oracle_paged_decode_rows_kv.argtypes = [
            vp, vp, i64, vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, i64,
            ctypes.c_float, i32, i32, ctypes.c_float, ctypes.c_float, i32]
        lib.oracle_paged_decode_rows_kv.restype = i32
        lib.oracle_e4m3_encode.argtypes = [vp, vp, i64]
        lib.oracle_e4m3_encode.restype = i32
        lib.oracle_reshape_and_cache_e4m3.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i32,
                                                      ctypes.c_float, ctypes.c_float]
        lib.oracle_reshape_and_cache_e4m3.restype = i32
        lib.oracle_paged_prefill_rows.argtypes = [
            vp, vp, i64, vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, i64, i64,
            ctypes.c_float, i32, i32]
        lib.oracle_paged_prefill_rows.restype = i32
        lib.oracle_paged_prefill_rows_kv.argtypes = [
            vp, vp, i64, vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, i64, i64,
            ctypes.c_float, i32, i32, ctypes.c_float, ctypes.c_float, i32]
        lib.oracle_paged_prefill_rows_kv.restype = i32
        lib.oracle_max_threads.argtypes = []
        lib.oracle_max_threads.restype = i32
        _lib = lib
    return _lib


def _check(rc: int) -> None:
    if rc != 0:
        raise OracleError(_ERRORS.get(rc, f"oracle status {rc}"))


def _host(t: torch.Tensor, dtype=None) -> torch.Tensor:
    if t.device.type != "cpu":
        raise ValueError("the oracle takes host tensors")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"expected {dtype}, got {t.dtype}")
    return t.contiguous()


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def widen(x: torch.Tensor) -> torch.Tensor:
    """Decode stored f32/f16/bf16 elements to float64 with the oracle's own decoder."""
    x = _host(x)
    out = torch.empty(x.shape, dtype=torch.float64)
    _check(_load().oracle_widen(x.data_ptr(), out.data_ptr(), x.numel(), _DTYPE_CODE[x.dtype]))
    return out


def widen_e4m3(codes: torch.Tensor) -> torch.Tensor:
    """Decode E4M3 codes (uint8) to float64 with the oracle's own decoder."""
    codes = _host(codes, torch.uint8)
    out = torch.empty(codes.shape, dtype=torch.float64)
    _check(_load().oracle_widen(codes.data_ptr(), out.data_ptr(), codes.numel(), E4M3))
    return out


def e4m3_encode(x: torch.Tensor) -> torch.Tensor:
    """Round float32 values to E4M3 codes (nearest, ties to even, saturating at +-448)."""
    x = _host(x, torch.float32)
    out = torch.empty(x.shape, dtype=torch.uint8)
    _check(_load().oracle_e4m3_encode(x.data_ptr(), out.data_ptr(), x.numel()))
    return out


def inv_scale(scale: float) -> float:
    """The binary32 reciprocal 1/scale that the FP8 append multiplies by."""
    import numpy as np
    return float(np.float32(1.0) / np.float32(scale))


def reshape_and_cache_e4m3(key: torch.Tensor, value: torch.Tensor, k_cache: torch.Tensor,
                           v_cache: torch.Tensor, slot_mapping: torch.Tensor, k_scale: float,
                           v_scale: float) -> None:
    """In-place KV append into E4M3 caches (uint8 [N_b,Hkv,bs,D]): every element x is
    stored as E4M3(fp32(x) * fp32(1/scale))."""
    if not (k_cache.is_contiguous() and v_cache.is_contiguous()):
        raise ValueError("caches must be contiguous")
    key, value = _host(key), _host(value)
    kc, vc = _host(k_cache, torch.uint8), _host(v_cache, torch.uint8)
    slots = _host(slot_mapping, torch.int64)
    T, Hkv, D = key.shape
    N_b, Hkv2, bs, D2 = kc.shape
    if value.shape != key.shape or vc.shape != kc.shape or (Hkv2, D2) != (Hkv, D) or value.dtype != key.dtype:
        raise ValueError("shape mismatch")
    _check(_load().oracle_reshape_and_cache_e4m3(
        key.data_ptr(), value.data_ptr(), kc.data_ptr(), vc.data_ptr(), slots.data_ptr(), T, Hkv, D, N_b, bs,
        _DTYPE_CODE[key.dtype], inv_scale(k_scale), inv_scale(v_scale)))


def reshape_and_cache(key: torch.Tensor, value: torch.Tensor, k_cache: torch.Tensor,
                      v_cache: torch.Tensor, slot_mapping: torch.Tensor) -> None:
    """In-place KV append on host tensors: key/value [T,Hkv,D], caches [N_b,Hkv,bs,D]."""
    if not (k_cache.is_contiguous() and v_cache.is_contiguous()):
        raise ValueError("caches must be contiguous")
    key, value = _host(key), _host(value)
    slots = _host(slot_mapping, torch.int64)
    T, Hkv, D = key.shape
    N_b, Hkv2, bs, D2 = k_cache.shape
    if value.shape != key.shape or v_cache.shape != k_cache.shape or (Hkv2, D2) != (Hkv, D):
        raise ValueError("shape mismatch")
    if not (key.dtype == value.dtype == k_cache.dtype == v_cache.dtype):
        raise ValueError("dtype mismatch")
    _check(_load().oracle_reshape_and_cache(
        key.data_ptr(), value.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
        slots.data_ptr(), T, Hkv, D, N_b, bs, _DTYPE_CODE[key.dtype]))


def paged_decode(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                 block_tables: torch.Tensor, context_lens: torch.Tensor, num_kv_heads: int,
                 scale: float, rows=None, num_threads: int = 0, k_scale: float = 1.0,
                 v_scale: float = 1.0) -> torch.Tensor:
    """Paged decode attention in float64.

    q [B,Hq,D]; caches [N_b,Hkv,bs,D] of q's dtype, or uint8 E4M3 codes whose
    values are code * k_scale (resp. v_scale); block_tables int32 [B,M_b];
    context_lens int32 [B].  Returns float64 [B,Hq,D], or [len(rows),D] for the
    flat row indices ``rows`` (r = b*Hq + h).  ``scale`` and the K/V scales are
    used as their binary32 values.
    """
    q = _host(q)
    kc, vc = _host(k_cache), _host(v_cache)
    bt = _host(block_tables, torch.int32)
    cl = _host(context_lens, torch.int32)
    B, Hq, D = q.shape
    N_b, Hkv, bs, D2 = kc.shape
    if Hkv != num_kv_heads or D2 != D or vc.shape != kc.shape:
        raise ValueError("shape mismatch")
    fp8 = kc.dtype == torch.uint8
    if vc.dtype != kc.dtype or not (fp8 or q.dtype == kc.dtype):
        raise ValueError("dtype mismatch")
    if bt.dim() != 2 or bt.shape[0] != B or cl.shape != (B,):
        raise ValueError("block_tables/context_lens shape mismatch")
    M_b = bt.shape[1]
    if rows is None:
        rows_t = None
        n_rows = B * Hq
        out = torch.empty((B, Hq, D), dtype=torch.float64)
    else:
        rows_t = torch.as_tensor(rows, dtype=torch.int64).contiguous()
        n_rows = rows_t.numel()
        out = torch.empty((n_rows, D), dtype=torch.float64)
    _check(_load().oracle_paged_decode_rows_kv(
        out.data_ptr(), None if rows_t is None else rows_t.data_ptr(), n_rows,
        q.data_ptr(), kc.data_ptr(), vc.data_ptr(), bt.data_ptr(), cl.data_ptr(),
        B, Hq, Hkv, D, N_b, bs, M_b, float(scale), _DTYPE_CODE[q.dtype], E4M3 if fp8 else _DTYPE_CODE[q.dtype],
        float(k_scale) if fp8 else 1.0, float(v_scale) if fp8 else 1.0, int(num_threads)))
    return out


def paged_prefill(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                  block_tables: torch.Tensor, context_lens: torch.Tensor, query_start_loc: torch.Tensor,
                  num_kv_heads: int, scale: float, rows=None, num_threads: int = 0, k_scale: float = 1.0,
                  v_scale: float = 1.0) -> torch.Tensor:
    """Chunked-prefill paged attention in float64.

    q [T,Hq,D] packed chunks (sequence b owns rows query_start_loc[b] ..
    query_start_loc[b+1]-1, the last n_b of its context_lens[b] tokens); caches
    [N_b,Hkv,bs,D] of q's dtype; block_tables int32 [B,M_b]; context_lens int32
    [B]; query_start_loc int32 [B+1].  Caches may instead be uint8 E4M3 codes
    whose values are code * k_scale (resp. v_scale).  Returns float64 [T,Hq,D],
    or [len(rows),D] for flat rows r = t*Hq + h.
    """
    q = _host(q)
    kc, vc = _host(k_cache), _host(v_cache)
    bt = _host(block_tables, torch.int32)
    cl = _host(context_lens, torch.int32)
    qsl = _host(query_start_loc, torch.int32)
    T, Hq, D = q.shape
    N_b, Hkv, bs, D2 = kc.shape
    B = cl.shape[0]
    if Hkv != num_kv_heads or D2 != D or vc.shape != kc.shape or qsl.shape != (B + 1,):
        raise ValueError("shape mismatch")
    fp8 = kc.dtype == torch.uint8
    if vc.dtype != kc.dtype or not (fp8 or kc.dtype == q.dtype):
        raise ValueError("dtype mismatch")
    if bt.dim() != 2 or bt.shape[0] != B:
        raise ValueError("block_tables shape mismatch")
    if rows is None:
        rows_t, n_rows = None, T * Hq
        out = torch.empty((T, Hq, D), dtype=torch.float64)
    else:
        rows_t = torch.as_tensor(rows, dtype=torch.int64).contiguous()
        n_rows = rows_t.numel()
        out = torch.empty((n_rows, D), dtype=torch.float64)
    _check(_load().oracle_paged_prefill_rows_kv(
        out.data_ptr(), None if rows_t is None else rows_t.data_ptr(), n_rows,
        q.data_ptr(), kc.data_ptr(), vc.data_ptr(), bt.data_ptr(), cl.data_ptr(), qsl.data_ptr(),
        B, T, Hq, Hkv, D, N_b, bs, bt.shape[1], float(scale), _DTYPE_CODE[q.dtype],
        E4M3 if fp8 else _DTYPE_CODE[q.dtype], float(k_scale) if fp8 else 1.0, float(v_scale) if fp8 else 1.0,
        int(num_threads)))
    return out
