"""The C ABI without a GPU: the library builds, loads, exports every symbol the
header declares, and rejects bad arguments on the host before any CUDA call."""
import ctypes
import os
import re

import pytest
import torch

from paged_kv_cache_185_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "wllm.h")
FAKE = 0x10000  # never dereferenced: every call below fails validation first


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(wllm_\w+)\s*\(", text)))


def test_header_declares_the_api():
    names = declared_functions()
    assert "wllm_reshape_and_cache" in names and "wllm_paged_attention_decode" in names
    assert set(names) == set(binding.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert "sm_103a" in binding.version()


def test_library_exports_nothing_else_with_c_linkage(lib):
    """Unmangled dynamic symbols of the library are exactly the header's calls."""
    import shutil
    import subprocess
    nm = shutil.which("nm")
    if nm is None:
        pytest.skip("nm not available")
    out = subprocess.run([nm, "-D", "--defined-only", build.LIB], capture_output=True, text=True, check=True)
    names = {ln.split()[-1] for ln in out.stdout.splitlines() if ln.strip()}
    plain = {n for n in names if not n.startswith("_Z") and not n.startswith("_")}
    assert plain == set(declared_functions()), plain ^ set(declared_functions())


def test_selftest_rejects_bad_limits_on_the_host(lib):
    for limit in (0, 2_000_000_000):
        assert lib.wllm_selftest_wait_timeout(limit, None) == binding.WLLM_ERR_INVALID_ARG
        assert b"limit_ns" in lib.wllm_last_error()


def test_launch_count_unchanged_by_rejected_calls(lib):
    n0 = lib.wllm_launch_count()
    q = desc([2, 4, 64], torch.float16)
    kc = desc([8, 2, 16, 64], torch.float16)
    bt = desc([2, 4], torch.int32)
    cl = desc([2], torch.int32)
    out = desc([2, 4, 64], torch.float32)  # wrong dtype: rejected on the host
    assert decode(lib, out, q, kc, kc, bt, cl) == binding.WLLM_ERR_INVALID_ARG
    assert lib.wllm_launch_count() == n0


def desc(shape, dtype, data=FAKE, stride=None):
    d = binding.WllmTensor()
    d.data = data
    d.dtype = binding._DTYPE[dtype]
    d.ndim = len(shape)
    if stride is None:
        stride, acc = [], 1
        for s in reversed(shape):
            stride.insert(0, acc)
            acc *= s
    for i, (s, st) in enumerate(zip(shape, stride)):
        d.shape[i] = s
        d.stride[i] = st
    return d


def decode(lib, out, q, kc, vc, bt, cl, hkv=2, scale=0.125, bs=16):
    r = lambda x: None if x is None else ctypes.byref(x)  # noqa: E731
    return lib.wllm_paged_attention_decode(r(out), r(q), r(kc), r(vc), r(bt), r(cl), hkv, scale, bs, None)


def good(B=2, Hq=4, Hkv=2, D=64, bs=16, nb=8, mb=4, dt=torch.bfloat16):
    return dict(out=desc((B, Hq, D), dt), q=desc((B, Hq, D), dt), kc=desc((nb, Hkv, bs, D), dt),
                vc=desc((nb, Hkv, bs, D), dt), bt=desc((B, mb), torch.int32),
                cl=desc((B,), torch.int32))


@pytest.mark.parametrize("mutate,status", [
    (lambda a: a.update(q=desc((2, 4), torch.bfloat16)), 1),                  # rank
    (lambda a: a.update(out=desc((2, 4, 64), torch.float16)), 1),            # dtype mismatch
    (lambda a: a.update(cl=desc((2,), torch.int64)), 1),                      # lens dtype
    (lambda a: a.update(bt=desc((3, 4), torch.int32)), 1),                    # table rows
    (lambda a: a.update(kc=desc((8, 2, 16, 64), torch.bfloat16, stride=(2048, 1024, 128, 1))), 1),
    (lambda a: a.update(q=desc((2, 4, 64), torch.bfloat16, stride=(256, 64, 2)), out=desc((2, 4, 64), torch.bfloat16, stride=(256, 64, 2))), 1),
    (lambda a: a.update(kc=None), 1),                                         # null descriptor
    (lambda a: a.update(q=desc((2, 4, 64), torch.bfloat16, data=None)), 1),   # null data
])
def test_decode_rejects_bad_arguments(lib, mutate, status):
    a = good()
    mutate(a)
    assert decode(lib, **a) == status
    assert lib.wllm_last_error().decode()


def test_decode_rejects_bad_sizes(lib):
    assert decode(lib, **good(), hkv=3) == 1                       # kv heads mismatch
    assert decode(lib, **good(), bs=8) == 1                        # block size mismatch
    assert decode(lib, **good(Hq=5, Hkv=2)) != 0                   # Hq % Hkv
    assert decode(lib, **good(D=96)) == 2                          # unsupported head_dim
    assert decode(lib, **good(bs=4), bs=4) == 2                    # unsupported block size
    assert decode(lib, **good(), scale=float("nan")) == 1
    assert decode(lib, **good(B=0)) == 0                           # empty batch: nothing to do


def test_append_rejects_bad_arguments(lib):
    r = ctypes.byref
    key = desc((3, 2, 64), torch.float16)
    kc = desc((4, 2, 16, 64), torch.float16)
    slots = desc((3,), torch.int64)
    call = lambda k, v, c1, c2, s: lib.wllm_reshape_and_cache(r(k), r(v), r(c1), r(c2), r(s), None)  # noqa
    assert call(desc((3, 2), torch.float16), key, kc, kc, slots) == 1
    assert call(key, desc((3, 2, 64), torch.bfloat16), kc, kc, slots) == 1
    assert call(key, key, kc, kc, desc((3,), torch.float32)) == 1
    assert call(key, key, kc, kc, desc((4,), torch.int64)) == 1
    assert call(key, key, desc((4, 3, 16, 64), torch.float16), kc, slots) == 1
    assert call(key, key, desc((4, 2, 16, 64), torch.float16, stride=(4096, 2048, 64, 2)), kc, slots) == 1
    assert call(key, key, desc((4, 2, 12, 64), torch.float16), desc((4, 2, 12, 64), torch.float16), slots) == 2
    empty = desc((0, 2, 64), torch.float16)
    assert call(empty, empty, kc, kc, desc((0,), torch.int64)) == 0


def test_binding_refuses_host_tensors():
    q = torch.zeros(1, 2, 64, dtype=torch.bfloat16)
    kc = torch.zeros(2, 1, 16, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        binding.paged_attention_decode(torch.empty_like(q), q, kc, kc,
                                       torch.zeros(1, 1, dtype=torch.int32),
                                       torch.ones(1, dtype=torch.int32), 1, 0.1, 16)


def decode_fp8(lib, out, q, kc, vc, bt, cl, hkv=2, scale=0.125, ks=0.5, vs=0.5, bs=16):
    r = lambda x: None if x is None else ctypes.byref(x)  # noqa: E731
    return lib.wllm_paged_attention_decode_fp8(r(out), r(q), r(kc), r(vc), r(bt), r(cl), hkv, scale, ks, vs, bs,
                                               None)


def good_fp8(B=2, Hq=4, Hkv=2, D=128, bs=16, nb=8, mb=4, dt=torch.bfloat16, q_stride=None):
    a = good(B, Hq, Hkv, D, bs, nb, mb, dt)
    a.update(kc=desc((nb, Hkv, bs, D), torch.uint8), vc=desc((nb, Hkv, bs, D), torch.uint8))
    if q_stride is not None:
        a.update(q=desc((B, Hq, D), dt, stride=q_stride))
    return a


def test_fp8_decode_rejects_bad_arguments(lib):
    assert decode_fp8(lib, **good_fp8(D=64, bs=8), bs=8) == 2                  # head_dim 64 with 8-token blocks
    assert decode_fp8(lib, **good_fp8(dt=torch.float32)) == 1                  # fp32 queries
    a = good_fp8()
    a.update(kc=desc((8, 2, 16, 128), torch.bfloat16))
    assert decode_fp8(lib, **a) == 1                                           # 16-bit K cache
    assert decode_fp8(lib, **good_fp8(), ks=0.0) == 1
    assert decode_fp8(lib, **good_fp8(), vs=float("nan")) == 1
    assert decode_fp8(lib, **good_fp8(), ks=float("inf")) == 1
    assert decode_fp8(lib, **good_fp8(q_stride=(4 * 132, 132, 1))) == 2       # rows not 16-byte aligned
    assert decode_fp8(lib, **good_fp8(B=0)) == 0
    # the 16-bit entry point refuses E4M3 caches
    assert decode(lib, **good_fp8()) == 1


def test_fp8_append_rejects_bad_arguments(lib):
    r = ctypes.byref
    key = desc((3, 2, 128), torch.float16)
    kc = desc((4, 2, 16, 128), torch.uint8)
    slots = desc((3,), torch.int64)

    def call(k, v, c1, c2, s, ks=1.0, vs=1.0):
        return lib.wllm_reshape_and_cache_fp8(r(k), r(v), r(c1), r(c2), r(s), ks, vs, None)

    assert call(key, key, desc((4, 2, 16, 128), torch.float16), kc, slots) == 1    # 16-bit cache
    assert call(key, desc((3, 2, 128), torch.bfloat16), kc, kc, slots) == 1       # key/value types
    assert call(key, key, kc, kc, slots, ks=-1.0) == 1
    assert call(key, key, kc, kc, slots, vs=float("inf")) == 1
    k6 = desc((3, 2, 6), torch.float16)
    c6 = desc((4, 2, 16, 6), torch.uint8)
    assert call(k6, k6, c6, c6, slots) == 2                                         # head_dim % 4
    empty = desc((0, 2, 128), torch.float16)
    assert call(empty, empty, kc, kc, desc((0,), torch.int64)) == 0
    # the bit-copy append refuses E4M3 caches
    assert lib.wllm_reshape_and_cache(r(key), r(key), r(kc), r(kc), r(slots), None) == 1


def prefill(lib, out, q, kc, vc, bt, cl, qsl, hkv=2, scale=0.125, bs=16):
    r = lambda x: None if x is None else ctypes.byref(x)  # noqa: E731
    return lib.wllm_paged_attention_prefill(r(out), r(q), r(kc), r(vc), r(bt), r(cl), r(qsl), hkv, scale, bs, None)


def good_prefill(T=10, B=2, Hq=4, Hkv=2, D=64, bs=16, nb=8, mb=4, dt=torch.bfloat16):
    a = good(B, Hq, Hkv, D, bs, nb, mb, dt)
    a.update(out=desc((T, Hq, D), dt), q=desc((T, Hq, D), dt), qsl=desc((B + 1,), torch.int32))
    return a


def test_prefill_rejects_bad_arguments(lib):
    assert prefill(lib, **good_prefill(D=256)) == 2                     # head_dim 256
    assert prefill(lib, **good_prefill(dt=torch.float32)) == 2          # fp32
    a = good_prefill()
    a.update(qsl=desc((2,), torch.int32))                               # B entries, not B + 1
    assert prefill(lib, **a) == 1
    a = good_prefill()
    a.update(qsl=desc((3,), torch.int64))                               # dtype
    assert prefill(lib, **a) == 1
    a = good_prefill()
    a.update(kc=desc((8, 2, 16, 64), torch.float16))                    # cache dtype
    assert prefill(lib, **a) == 1
    assert prefill(lib, **good_prefill(), hkv=3) == 1                   # kv heads mismatch
    assert prefill(lib, **good_prefill(), bs=8) == 1                    # block size mismatch
    assert prefill(lib, **good_prefill(bs=4), bs=4) == 2                # unsupported block size
    assert prefill(lib, **good_prefill(), scale=float("inf")) == 1
    a = good_prefill()
    a.update(q=desc((10, 4, 64), torch.bfloat16, stride=(257, 64, 1)))  # rows not 4-byte aligned
    assert prefill(lib, **a) == 1
    assert prefill(lib, **good_prefill(T=0)) == 0                       # nothing to do


def test_prefill_fp8_rejects_bad_arguments(lib):
    r = lambda x: None if x is None else ctypes.byref(x)  # noqa: E731

    def call(a, ks=0.5, vs=0.5, bs=16, hkv=2):
        return lib.wllm_paged_attention_prefill_fp8(r(a["out"]), r(a["q"]), r(a["kc"]), r(a["vc"]), r(a["bt"]),
                                                    r(a["cl"]), r(a["qsl"]), hkv, 0.125, ks, vs, bs, None)

    def good8(**kw):
        a = good_prefill(**kw)
        D, bs = kw.get("D", 64), kw.get("bs", 16)
        a.update(kc=desc((8, 2, bs, D), torch.uint8), vc=desc((8, 2, bs, D), torch.uint8))
        return a

    assert call(good8(D=64, bs=8), bs=8) == 2                      # head_dim 64 with 8-token blocks
    assert call(good8(D=256)) == 2                                 # head_dim 256
    assert call(good_prefill()) == 1                               # 16-bit caches
    assert call(good8(), ks=0.0) == 1
    assert call(good8(), vs=float("nan")) == 1
    a = good8()
    a.update(q=desc((10, 4, 64), torch.bfloat16, stride=(258, 64, 1)))  # rows 4- but not 8-byte aligned
    assert call(a) == 1
    assert call(good8(T=0)) == 0
